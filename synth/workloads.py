"""Workload shapes and seeded generators (no layer arithmetic lives here).

Shapes follow the MoE models named in the PagedWeight write-up
(zhichai.net/topic/178446964, section "数据说话": Qwen1.5-MoE-A2.7B with 60
experts, Mixtral-8x7B with 8 experts, a 128-expert 25B-class model) plus a
tiny layer for exhaustive checks.  Value recipe (the pages give none, so these
are synthetic stand-ins for trained weights):

* hidden states x ~ N(0, 1) rounded to fp16, shape [T, d];
* router weight W_r ~ N(0, 0.02) fp16 [E, d]; optional Zipf(s) router bias
  bias_e = -s * ln(rank_e + 1) with rank a seeded permutation of 0..E-1;
* 6-bit parent codes code6 ~ U{0..63} (uint8) per expert matrix, matrices
  stored "out x in": gate [f, d], up [f, d], down [d, f];
* per-row lookup tables: LUT_b[r] = sort(N(0, 0.02) draws of size 2^b) in fp16,
  drawn independently per (matrix, row, b) for b = 3, 4, 5, 6;
* fp16 fallback pages W16 ~ N(0, 0.02) fp16, drawn independently of the codes;
* shared FFN (Qwen-shaped only) ~ N(0, 0.02) fp16.

Every tensor comes from its own generator ``default_rng([seed, purpose,
layer, expert, matrix, extra])`` so any single expert can be regenerated
without drawing the others (needed for sampled checks at full size).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

# generator purpose keys
_ROUTER, _BIASPERM, _CODE, _LUT, _W16, _SHARED, _TOKENS, _BITS, _SWEEP, _SENS = range(1, 11)

BITS_ALLOWED = (3, 4, 5, 6, 16)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    d: int                 # hidden size
    f: int                 # expert FFN size
    E: int                 # routed experts
    K: int                 # experts per token
    renormalize: int       # 1: top-K weights rescaled to sum 1
    shared_ffn: int = 0    # fp16 shared FFN size (0 = none)
    zipf_s: float = 0.0    # router-bias skew (0 = no bias)
    bits_rule: str = "uniform"
    decode_T: tuple = ()
    prefill_T: tuple = ()
    n_layers: int = 1


CONFIGS = {
    "tiny": LayerConfig("tiny", d=512, f=1024, E=8, K=2, renormalize=1,
                        bits_rule="uniform", decode_T=(16,)),
    "qwen": LayerConfig("qwen", d=2048, f=1408, E=60, K=4, renormalize=0,
                        shared_ffn=5632, zipf_s=1.1, bits_rule="greedy",
                        decode_T=(1, 8, 64, 256)),
    "mixtral": LayerConfig("mixtral", d=4096, f=14336, E=8, K=2, renormalize=1,
                           bits_rule="cycle6543", decode_T=(1, 8, 64, 256),
                           prefill_T=(4096,)),
    "e128": LayerConfig("e128", d=2816, f=704, E=128, K=8, renormalize=1,
                        zipf_s=1.2, bits_rule="e128", decode_T=(128,),
                        prefill_T=(8192,)),
    "sweep": LayerConfig("sweep", d=4096, f=14336, E=8, K=2, renormalize=1,
                         bits_rule="sweep", decode_T=(1, 8, 64, 256), n_layers=32),
}


def get_config(name: str, **overrides) -> LayerConfig:
    """Named config, optionally with fields replaced (e.g. smaller d for tests)."""
    return dataclasses.replace(CONFIGS[name], **overrides)


def _rng(seed, *key):
    return np.random.default_rng([int(seed)] + [int(k) for k in key])


def matrix_shapes(cfg: LayerConfig):
    """(rows, cols) of gate, up, down: rows are output channels."""
    return [(cfg.f, cfg.d), (cfg.f, cfg.d), (cfg.d, cfg.f)]


def zipf_bias(cfg: LayerConfig, seed: int = 0, layer: int = 0) -> Optional[np.ndarray]:
    if cfg.zipf_s == 0.0:
        return None
    rank = _rng(seed, _BIASPERM, layer).permutation(cfg.E)
    return (-cfg.zipf_s * np.log(rank + 1.0)).astype(np.float32)


def make_router(cfg: LayerConfig, seed: int = 0, layer: int = 0):
    """Router weight [E, d] fp16 and bias [E] fp32 (or None)."""
    wr = (_rng(seed, _ROUTER, layer).standard_normal((cfg.E, cfg.d)) * 0.02).astype(np.float16)
    return wr, zipf_bias(cfg, seed, layer)


def make_expert(cfg: LayerConfig, e: int, seed: int = 0, layer: int = 0,
                with_w16: Optional[bool] = None):
    """One expert's stored form.

    Returns dict with
      code6: [gate, up, down] uint8 arrays of 6-bit parent codes,
      lut:   [[LUT_3, LUT_4, LUT_5, LUT_6] per matrix], each fp16 [rows, 2^b],
      w16:   [gate, up, down] fp16 arrays or None.
    with_w16=None draws the fp16 page only if the expert's planned bitwidth is 16.
    """
    if with_w16 is None:
        with_w16 = 16 in {int(b) for b in np.atleast_1d(initial_bits_for(cfg, e, seed, layer))}
    code6, lut, w16 = [], [], []
    for m, (R, C) in enumerate(matrix_shapes(cfg)):
        code6.append(_rng(seed, _CODE, layer, e, m).integers(0, 64, size=(R, C), dtype=np.uint8))
        luts = []
        for b in (3, 4, 5, 6):
            t = _rng(seed, _LUT, layer, e, m, b).standard_normal((R, 1 << b)) * 0.02
            luts.append(np.sort(t, axis=1).astype(np.float16))
        lut.append(luts)
        if with_w16:
            w16.append((_rng(seed, _W16, layer, e, m).standard_normal((R, C)) * 0.02).astype(np.float16))
    return {"code6": code6, "lut": lut, "w16": w16 if with_w16 else None}


def make_shared(cfg: LayerConfig, seed: int = 0, layer: int = 0):
    """Shared fp16 FFN [gate (fs,d), up (fs,d), down (d,fs)] or None."""
    if cfg.shared_ffn == 0:
        return None
    fs = cfg.shared_ffn
    out = []
    for m, shp in enumerate([(fs, cfg.d), (fs, cfg.d), (cfg.d, fs)]):
        out.append((_rng(seed, _SHARED, layer, m).standard_normal(shp) * 0.02).astype(np.float16))
    return out


def make_tokens(cfg: LayerConfig, T: int, seed: int = 0, layer: int = 0, stream: int = 0):
    """Hidden states x [T, d] ~ N(0, 1) in fp16."""
    return _rng(seed, _TOKENS, layer, T, stream).standard_normal((T, cfg.d)).astype(np.float16)


def _greedy_plan(importance: np.ndarray, budget: float, floor: int = 3) -> np.ndarray:
    """Greedy floor-respecting bitwidth plan used to generate the Qwen-shaped bits.

    Experts are visited by descending importance (ties: lower index first);
    each gets the largest b in {16, 6, 5, 4, 3} whose cost (b plane units, 16
    units for the fp16 page) still leaves `floor` units for every expert not
    yet visited.
    """
    E = importance.shape[0]
    order = np.argsort(-importance, kind="stable")
    bits = np.full(E, floor, dtype=np.int32)
    left = float(budget)
    for i, e in enumerate(order):
        rest = E - i - 1
        for b in (16, 6, 5, 4, 3):
            if left - b >= floor * rest - 1e-9:
                bits[e] = b
                left -= b
                break
    return bits


def bits_plan(cfg: LayerConfig, seed: int = 0, layer: int = 0) -> np.ndarray:
    """Initial per-expert bitwidths (int32 [E]) for one layer of the config."""
    E = cfg.E
    rule = cfg.bits_rule
    if rule == "uniform":
        return _rng(seed, _BITS, layer).choice(np.array(BITS_ALLOWED), size=E).astype(np.int32)
    if rule == "greedy":
        bias = zipf_bias(cfg, seed, layer)
        imp = np.exp(bias.astype(np.float64)) if bias is not None else np.ones(E)
        return _greedy_plan(imp, budget=4.0 * E)
    if rule == "cycle6543":
        return np.array([(6, 5, 4, 3)[e % 4] for e in range(E)], dtype=np.int32)
    if rule == "e128":
        base = [3] * 45 + [4] * 45 + [6] * 30 + [16] * 8
        base = (base + [3] * E)[:E]
        return _rng(seed, _BITS, layer).permutation(np.array(base, dtype=np.int32))
    if rule == "sweep":
        return np.array([(6, 5, 4, 3, 16)[(e + layer) % 5] for e in range(E)], dtype=np.int32)
    raise ValueError(rule)


def make_sensitivity(cfg: LayerConfig, seed: int = 0, layer: int = 0) -> np.ndarray:
    """Synthetic offline sensitivity table, float64 [E, 4] for b = 3, 4, 5, 6.

    Stand-in for the Hessian-weighted sensitivity table that the write-up
    builds offline from calibration data (section "三层感知"; no trained
    weights or data exist here): expert e's damage at b bits is
    s_e * 4^(6 - b) (quantisation noise power drops 4x per bit), with
    s_e ~ lognormal(0, 1) drawn per (layer, expert).
    """
    s = _rng(seed, _SENS, layer).lognormal(0.0, 1.0, size=cfg.E)
    return np.stack([s * 4.0 ** (6 - b) for b in (3, 4, 5, 6)], axis=1)


def initial_bits_for(cfg: LayerConfig, e: int, seed: int = 0, layer: int = 0) -> int:
    return int(bits_plan(cfg, seed, layer)[e])


def sweep_changes(cfg: LayerConfig, step: int, initial: List[np.ndarray], seed: int = 0):
    """Bitwidth requests for one step of the multi-layer sweep.

    A seeded 25% of the (layer, expert) pairs each get a new bitwidth drawn from
    the allowed values that do not exceed the pair's initial bitwidth.
    Returns a list of (layer, expert, bits).
    """
    rng = _rng(seed, _SWEEP, step)
    L = len(initial)
    pairs = [(l, e) for l in range(L) for e in range(cfg.E)]
    n = max(1, len(pairs) // 4)
    pick = rng.choice(len(pairs), size=n, replace=False)
    out = []
    for i in sorted(pick.tolist()):
        l, e = pairs[i]
        allowed = [b for b in BITS_ALLOWED if b <= int(initial[l][e])]
        out.append((l, e, int(rng.choice(allowed))))
    return out
