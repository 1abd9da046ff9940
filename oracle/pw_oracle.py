"""fp64 CPU oracle for the routed any-precision (bit-plane + LUT) MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of bench.py
may call it.  It shares no code with the CUDA library (different language,
independent implementation of every step); both sides only share the seeded
input generators in ``synth/``.

What is computed, and where it comes from
-----------------------------------------
PagedWeight (zhichai.net/topic/178446964, section "核心洞察") stores every
expert weight as an any-precision code split into bit-planes plus a lookup
table, switchable among 3/4/5/6 bits or a 16-bit fallback; lowering an
expert's precision detaches its low planes ("章节可以独立拆装").  Read plainly:

* plane p (p = 0..5) holds bit (5 - p) of the 6-bit parent code, so plane 0 is
  the most significant bit; a b-bit code is the top b planes, i.e.
  code_b = code6 >> (6 - b)   (nested planes);
* the dequantised weight is LUT_b[row][code_b] (one fp16 table of 2^b entries
  per output row and bitwidth); at b = 16 the fp16 page W16 is used instead.

The layer around it is the standard routed MoE block (the write-up names the
router and its imbalance in "三层感知" and "为什么这很重要"):
routing softmax + top-K, a stable permutation of (token, k) slots by expert,
a SwiGLU FFN per expert, and a weighted combine.  Readings taken where the
pages are silent are listed with each function.

Parity pins: every function here is checked in tests/test_oracle_*.py against
brute force, closed forms, invariants or special cases that do not reuse this
code.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------


def router_logits(x16: np.ndarray, wr16: np.ndarray, bias=None) -> np.ndarray:
    """l = x . W_r^T + bias in fp64 (inputs are the fp16 values, exactly widened)."""
    l = x16.astype(np.float64) @ wr16.astype(np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l


def softmax(l: np.ndarray) -> np.ndarray:
    """Row softmax, stabilised by subtracting the row max."""
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    return p / p.sum(axis=1, keepdims=True)


def route_topk(x16, wr16, bias, K: int, renormalize: int):
    """Router softmax over all E experts, then the K most probable experts.

    Readings: softmax over all E, then top-K by descending probability with
    exact ties going to the lower expert index; the kept weights are the
    softmax probabilities, rescaled to sum 1 when ``renormalize``.
    Returns (idx int32 [T,K], w fp64 [T,K], logits fp64 [T,E]).
    """
    l = router_logits(x16, wr16, bias)
    p = softmax(l)
    # a stable sort of -l keeps lower indices first among equal logits
    idx = np.argsort(-l, axis=1, kind="stable")[:, :K]
    w = np.take_along_axis(p, idx, axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), w, l


def near_tie_tokens(logits: np.ndarray, K: int, rel: float = 1e-4) -> np.ndarray:
    """Tokens whose K-th and (K+1)-th logits are within rel*(1+|l_K|).

    For these tokens an fp32 router may legitimately pick either expert; the
    parity tests accept both choices there and recompute the rest of the layer
    with the GPU's choice.
    """
    T, E = logits.shape
    if K >= E:
        return np.zeros(T, dtype=bool)
    s = -np.sort(-logits, axis=1)
    gap = s[:, K - 1] - s[:, K]
    return gap < rel * (1.0 + np.abs(s[:, K - 1]))


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------


def permute(idx: np.ndarray, E: int):
    """Stable counting sort of the S = T*K slots (flat index t*K + k) by expert.

    Reading: inside an expert's bucket, slots keep ascending flat order.
    Returns offsets [E+1], perm_src [S] (token of each sorted slot) and
    inv_slot [S] (sorted position of flat slot t*K + k).
    """
    T, K = idx.shape
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    perm_src = (order // K).astype(np.int32)
    inv_slot = np.empty(T * K, dtype=np.int32)
    inv_slot[order] = np.arange(T * K, dtype=np.int32)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, perm_src, inv_slot


# ---------------------------------------------------------------------------
# any-precision dequantisation
# ---------------------------------------------------------------------------


def code_at_bits(code6: np.ndarray, b: int) -> np.ndarray:
    """The b-bit code of a weight is the top b of its 6 parent bits."""
    if not 1 <= b <= 6:
        raise ValueError(b)
    return (code6.astype(np.int64) >> (6 - b))


def dequant(code6: np.ndarray, luts, b: int, w16=None) -> np.ndarray:
    """Weight matrix in fp64 at bitwidth b.

    b in {3,4,5,6}: W[r,c] = LUT_b[r][code6[r,c] >> (6-b)]  (fp16 table value,
    widened exactly).  b == 16: the fp16 fallback page.
    ``luts`` is the list [LUT_3, LUT_4, LUT_5, LUT_6] of fp16 [rows, 2^b].
    """
    if b == 16:
        if w16 is None:
            raise ValueError("b=16 needs the fp16 page")
        return w16.astype(np.float64)
    lut = np.asarray(luts[b - 3])
    code = code_at_bits(code6, b)
    rows = np.arange(code6.shape[0])[:, None]
    return lut[rows, code].astype(np.float64)


# ---------------------------------------------------------------------------
# expert FFN, combine, full layer
# ---------------------------------------------------------------------------


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def swiglu_ffn(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, X: np.ndarray) -> np.ndarray:
    """y = Wd (silu(Wg x) * (Wu x)) for each row x of X, all fp64, no rounding.

    Matrices are "out x in": Wg, Wu [f, d]; Wd [d, f]; X [n, d] -> [n, d].
    """
    g = X @ Wg.T
    u = X @ Wu.T
    return (silu(g) * u) @ Wd.T


def expert_weights(expert: dict, b: int):
    """Dequantised (Wg, Wu, Wd) of one expert at bitwidth b."""
    w16 = expert.get("w16")
    return [dequant(expert["code6"][m], expert["lut"][m], b,
                    None if w16 is None else w16[m]) for m in range(3)]


def combine(y_perm: np.ndarray, inv_slot: np.ndarray, w: np.ndarray, shared=None) -> np.ndarray:
    """y[t] = sum_k w[t,k] * y_perm[inv_slot[t*K+k]]  (+ shared[t], added unweighted)."""
    T, K = w.shape
    y = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    slots = inv_slot.reshape(T, K)
    for k in range(K):
        y += w[:, k:k + 1] * y_perm[slots[:, k]]
    if shared is not None:
        y += shared
    return y


def moe_layer(x16, wr16, bias, experts, bits, K: int, renormalize: int,
              shared=None, idx_override=None):
    """The whole hot path, step by step.

    experts: list (length E) of dicts from ``synth.make_expert`` (code6, lut,
    w16); bits: per-expert bitwidths; shared: fp16 [gate, up, down] or None.
    idx_override: routing indices to use instead of the oracle's own top-K
    (used only for near-tie tokens, where the fp32 choice is accepted).
    Returns a dict of every intermediate.
    """
    E = len(experts)
    idx, w, logits = route_topk(x16, wr16, bias, K, renormalize)
    if idx_override is not None:
        idx = np.asarray(idx_override, dtype=np.int32)
        p = softmax(logits)
        w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        if renormalize:
            w = w / w.sum(axis=1, keepdims=True)
    offsets, perm_src, inv_slot = permute(idx, E)
    x = x16.astype(np.float64)
    S = idx.size
    y_perm = np.zeros((S, x.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        Wg, Wu, Wd = expert_weights(experts[e], int(bits[e]))
        y_perm[lo:hi] = swiglu_ffn(Wg, Wu, Wd, x[perm_src[lo:hi]])
    y_shared = None
    if shared is not None:
        y_shared = swiglu_ffn(*[m.astype(np.float64) for m in shared], x)
    y = combine(y_perm, inv_slot, w, y_shared)
    return {"idx": idx, "w": w, "logits": logits, "offsets": offsets,
            "perm_src": perm_src, "inv_slot": inv_slot, "y_perm": y_perm,
            "y_shared": y_shared, "y": y}


def moe_tokens(x16, wr16, bias, get_expert, bits, K: int, renormalize: int,
               tokens, shared=None, idx_override=None):
    """Layer output for a few selected tokens only (for sampled checks at full size).

    get_expert(e) returns the expert dict; only the experts the sampled tokens
    route to are materialised.  Per token the result equals ``moe_layer``'s row,
    because a token's output depends only on its own routing.
    """
    tokens = np.asarray(tokens)
    xs = x16[tokens]
    idx, w, logits = route_topk(xs, wr16, bias, K, renormalize)
    if idx_override is not None:
        idx = np.asarray(idx_override, dtype=np.int32)
        p = softmax(logits)
        w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        if renormalize:
            w = w / w.sum(axis=1, keepdims=True)
    x = xs.astype(np.float64)
    y = np.zeros_like(x)
    for e in sorted(set(idx.reshape(-1).tolist())):
        Wg, Wu, Wd = expert_weights(get_expert(e), int(bits[e]))
        rows, ks = np.nonzero(idx == e)
        ye = swiglu_ffn(Wg, Wu, Wd, x[rows])
        y[rows] += w[rows, ks][:, None] * ye
    if shared is not None:
        y += swiglu_ffn(*[m.astype(np.float64) for m in shared], x)
    return {"idx": idx, "w": w, "logits": logits, "y": y}


# ---------------------------------------------------------------------------
# stored layout of the bit-planes and of the fp16 pages
# ---------------------------------------------------------------------------
# The pages fix only that weights are bit-planes plus LUTs; the order of bits
# inside the stored words is this library's own convention, chosen so that a
# GPU thread finds its tensor-core fragment in one 32-bit word per plane:
#
#   matrix [R, C] (R % 16 == 0, C % 64 == 0), tile tau = r // 16 (16 rows),
#   chunk kappa = c // 64.  Inside the tile: g = (r % 16) % 8,
#   rowsel = (r % 16) // 8; inside the chunk: s = (c % 64) // 16,
#   cs = c % 16, colhalf = cs // 8, t = (cs % 8) // 2, h = cs % 2.
#   lane L = 4 g + t, k = 2 rowsel + colhalf, q = 8 k + 4 h + s.
#   plane p keeps the weight's bit (5 - p) at bit (q + 5 - p) mod 32 of the
#   word of (tile, chunk, lane).  Words of a tile are grouped by 4 chunks:
#   a full group gamma holds 32 lanes x 4 words (word = gamma*128 + 4 L + i for
#   chunk 4 gamma + i); a final partial group of r < 4 chunks holds
#   32 lanes x r words (word = base + r L + i).  Tile tau starts at word
#   tau * (C / 64) * 32.
#
#   fp16 page: per (tile, chunk, step s) a block of 32 lanes x 8 halves; the
#   lane's halves are registers a = rowsel + 2 colhalf (0..3), each holding
#   (even column, odd column) = h.  half index =
#   (((tau * C/64 + kappa) * 4 + s) * 32 + L) * 8 + 2 a + h.


def _plane_index(R: int, C: int):
    if R % 16 or C % 64:
        raise ValueError("rows must be a multiple of 16 and cols of 64")
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    tau, rr = r // 16, r % 16
    g, rowsel = rr % 8, rr // 8
    kappa, cc = c // 64, c % 64
    s, cs = cc // 16, cc % 16
    colhalf, t, h = cs // 8, (cs % 8) // 2, cs % 2
    L = 4 * g + t
    k = 2 * rowsel + colhalf
    q = 8 * k + 4 * h + s
    nk = C // 64
    full, rem = nk // 4, nk % 4
    gamma, i = kappa // 4, kappa % 4
    in_full = gamma < full
    rem_div = max(rem, 1)
    word_in_tile = np.where(in_full, gamma * 128 + L * 4 + i, full * 128 + L * rem_div + i)
    word = tau * (nk * 32) + word_in_tile
    return np.broadcast_to(word, (R, C)), np.broadcast_to(q, (R, C))


def pack_planes(code6: np.ndarray):
    """6 uint32 plane arrays (length R*C/32 each) in the stored word order."""
    R, C = code6.shape
    word, q = _plane_index(R, C)
    word = word.reshape(-1)
    q = q.reshape(-1)
    nwords = R * C // 32
    c = code6.reshape(-1).astype(np.int64)
    planes = []
    for p in range(6):
        bit = (c >> (5 - p)) & 1
        pos = (q + 5 - p) % 32
        vals = (bit << pos).astype(np.float64)  # disjoint bits: exact integer sums
        planes.append(np.bincount(word, weights=vals, minlength=nwords).astype(np.uint32))
    return planes


def codes_from_planes(planes, R: int, C: int) -> np.ndarray:
    """Read the top len(planes) planes back into b-bit codes (b = len(planes))."""
    b = len(planes)
    word, q = _plane_index(R, C)
    code = np.zeros((R, C), dtype=np.int64)
    for p in range(b):
        pos = (q + 5 - p) % 32
        bit = (planes[p].astype(np.int64)[word] >> pos) & 1
        code |= bit << (b - 1 - p)
    return code


def unpack_planes(planes, R: int, C: int) -> np.ndarray:
    return codes_from_planes(planes[:6], R, C).astype(np.uint8)


def _f16_index(R: int, C: int):
    if R % 16 or C % 64:
        raise ValueError("rows must be a multiple of 16 and cols of 64")
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    tau, rr = r // 16, r % 16
    g, rowsel = rr % 8, rr // 8
    kappa, cc = c // 64, c % 64
    s, cs = cc // 16, cc % 16
    colhalf, t, h = cs // 8, (cs % 8) // 2, cs % 2
    L = 4 * g + t
    a = rowsel + 2 * colhalf
    nk = C // 64
    return (((tau * nk + kappa) * 4 + s) * 32 + L) * 8 + 2 * a + h


def pack_f16(w16: np.ndarray) -> np.ndarray:
    """fp16 page in stored order (as uint16 bit patterns)."""
    R, C = w16.shape
    out = np.empty(R * C, dtype=np.uint16)
    out[_f16_index(R, C).reshape(-1)] = w16.view(np.uint16).reshape(-1)
    return out


def unpack_f16(packed: np.ndarray, R: int, C: int) -> np.ndarray:
    return packed[_f16_index(R, C)].view(np.float16).reshape(R, C)
