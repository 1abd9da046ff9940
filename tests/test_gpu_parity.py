"""GPU parity: every hot-path call of libpw.so against the fp64 oracle.

Bar (from the layer's spec): routing indices, the permutation and the
dequantised weights bit-exact; router weights within 1e-5; FFN and layer
outputs within max|err| <= 2e-3 * (1 + |ref|) (fp32 accumulation, h rounded
to fp16, output rounded to fp16).
"""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from oracle import pw_oracle as O
from synth import get_config, make_router, make_tokens

from gpu_layers import GpuLayer, assert_close

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# dequantisation through the page table (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [dict(d=512, f=1024, E=2), dict(d=2816, f=704, E=2),
                                   dict(d=2048, f=1408, E=2), dict(d=320, f=192, E=2)])
def test_dequant_bit_exact_every_bitwidth(shape):
    cfg = get_config("tiny", **shape)
    gl = GpuLayer(cfg, seed=3, bits=[16, 16], with_w16=True)
    try:
        for b in (16, 6, 5, 4, 3, 6, 16):  # lower plane by plane, then raise from reclaimable pages
            gl.set_bits(0, b)
            for m in range(3):
                R, C = (cfg.f, cfg.d) if m < 2 else (cfg.d, cfg.f)
                out = torch.empty((R, C), dtype=torch.float16, device="cuda")
                gl.layer.debug_dequant(0, m, out)
                torch.cuda.synchronize()
                ex = gl.experts[0]
                ref = O.dequant(ex["code6"][m], ex["lut"][m], b, ex["w16"][m]).astype(np.float16)
                assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.view(np.uint16)), (b, m)
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,T,kw", [("tiny", 16, {}), ("qwen", 256, {}), ("e128", 300, {}),
                                       ("mixtral", 64, {}), ("tiny", 1, {}), ("e128", 8192, {})])
def test_route_topk(name, T, kw):
    cfg = get_config(name, **kw)
    wr, bias = make_router(cfg, seed=1)
    x = make_tokens(cfg, T, seed=1)
    pool = pw.Pool(cfg.E * (2 * cfg.f + cfg.d) * 240 + (64 << 20))  # resident LUTs of every expert
    layer = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize)
    try:
        xd = torch.from_numpy(x).cuda()
        idx = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
        cnt = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
        layer.route_topk(xd, torch.from_numpy(wr).cuda(),
                         torch.from_numpy(bias).cuda() if bias is not None else None, T, idx, w, cnt)
        torch.cuda.synchronize()
        ridx, rw, logits = O.route_topk(x, wr, bias, cfg.K, cfg.renormalize)
        gidx = idx.cpu().numpy()
        diff = (gidx != ridx).any(1)
        near = O.near_tie_tokens(logits, cfg.K)
        assert near[diff].all(), np.nonzero(diff & ~near)[0]
        ok = ~diff
        assert_close(w.cpu().numpy()[ok], rw[ok], tol=1e-5, what="weights")
        assert np.array_equal(cnt.cpu().numpy(), np.bincount(gidx.reshape(-1), minlength=cfg.E))
        for row in gidx:
            assert len(set(row.tolist())) == cfg.K
    finally:
        layer.destroy()
        pool.close()


def test_route_exact_ties_lower_index():
    cfg = get_config("tiny", d=64, E=8, K=3)
    wr = np.tile(np.linspace(-1, 1, cfg.d, dtype=np.float16), (cfg.E, 1))
    bias = np.array([5, 4, 1, -3, -3, 1, -9, -9], dtype=np.float32)
    x = np.ones((5, cfg.d), dtype=np.float16)
    pool = pw.Pool(16 << 20)
    layer = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, 0)
    try:
        idx = torch.empty((5, 3), dtype=torch.int32, device="cuda")
        w = torch.empty((5, 3), dtype=torch.float32, device="cuda")
        layer.route_topk(torch.from_numpy(x).cuda(), torch.from_numpy(wr).cuda(), torch.from_numpy(bias).cuda(),
                         5, idx, w)
        torch.cuda.synchronize()
        assert (idx.cpu().numpy() == [0, 1, 2]).all()
    finally:
        layer.destroy()
        pool.close()


# ---------------------------------------------------------------------------
# permutation (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,K", [(0, 8, 2), (1, 8, 2), (16, 8, 2), (1000, 60, 4), (8192, 128, 8), (300, 8, 8)])
def test_permute_bit_exact(T, E, K):
    d = 128
    rng = np.random.default_rng(T + E)
    if T:
        # skewed routing so some buckets are large and some empty
        p = np.exp(-0.15 * np.arange(E))
        idx = np.stack([rng.choice(E, size=K, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    else:
        idx = np.zeros((0, K), dtype=np.int32)
    x = rng.standard_normal((max(T, 1), d)).astype(np.float16)[:T]
    pool = pw.Pool(16 << 20)
    layer = pw.Layer(pool, d, 128, E, K, 1)
    try:
        S = T * K
        ws = torch.empty(max(layer.workspace_size(T), 256), dtype=torch.uint8, device="cuda")
        off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        ps = torch.empty(max(S, 1), dtype=torch.int32, device="cuda")
        inv = torch.empty(max(S, 1), dtype=torch.int32, device="cuda")
        xp = torch.empty((max(S, 1), d), dtype=torch.float16, device="cuda")
        xd = torch.from_numpy(x).cuda() if T else torch.empty((1, d), dtype=torch.float16, device="cuda")
        layer.permute(torch.from_numpy(idx).cuda() if T else ps, T, xd, off, ps, inv, xp, ws)
        torch.cuda.synchronize()
        ro, rp, ri = O.permute(idx, E)
        assert np.array_equal(off.cpu().numpy(), ro)
        if T:
            assert np.array_equal(ps.cpu().numpy()[:S], rp)
            assert np.array_equal(inv.cpu().numpy()[:S], ri)
            assert np.array_equal(xp.cpu().numpy()[:S].view(np.uint16), x[rp].view(np.uint16))
    finally:
        layer.destroy()
        pool.close()


# ---------------------------------------------------------------------------
# expert FFN and the whole layer
# ---------------------------------------------------------------------------

def test_expert_ffn_per_slot():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=0)
    try:
        for T in (16, 100):
            x = gl.tokens(T)
            r = gl.check_forward(x)
            ref = r["ref"]
            yp = r["buf"].y_perm[:T * cfg.K].cpu().numpy()
            assert_close(yp, ref["y_perm"], what="y_perm")
    finally:
        gl.close()


@pytest.mark.parametrize("T", [1, 16, 64])
def test_layer_tiny_all_bitwidths(T):
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=0)
    try:
        assert set(gl.bits.tolist()) >= {3, 16}
        gl.check_forward(gl.tokens(T))
    finally:
        gl.close()


def test_layer_qwen_shaped_with_shared_ffn():
    cfg = get_config("qwen", E=12, shared_ffn=5632)
    gl = GpuLayer(cfg, seed=2, with_w16=False)
    try:
        for T in (1, 8, 64):
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()


def test_layer_e128_shaped_tail_chunks():
    # f = 704 is 11 chunks of 64 columns: the down projection ends in a ragged group
    cfg = get_config("e128", E=24, K=8)
    gl = GpuLayer(cfg, seed=4, bits=[3, 4, 6, 16, 5] * 4 + [3, 4, 6, 16], with_w16=False)
    try:
        gl.check_forward(gl.tokens(40))
    finally:
        gl.close()


def test_bitwidth_changes_follow_stream_order():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=5, bits=[16] * 8, with_w16=True)
    try:
        x = gl.tokens(24)
        y16, buf = gl.forward(x)
        gl.check_forward(x, buf)
        for e, b in enumerate([3, 4, 5, 6, 3, 16, 4, 5]):
            gl.set_bits(e, b)
        gl.check_forward(x, buf)
        for e in range(8):
            gl.set_bits(e, 16)
        y16b, _ = gl.forward(x, buf)
        assert np.array_equal(y16, y16b)  # raising back re-maps the same pages
    finally:
        gl.close()


def test_one_expert_gets_every_token():
    cfg = get_config("tiny", K=1)
    gl = GpuLayer(cfg, seed=6, bits=[4] * 8, with_w16=False)
    try:
        gl.bias = np.array([50, 0, 0, 0, 0, 0, 0, 0], dtype=np.float32)
        gl.bias_d = torch.from_numpy(gl.bias).cuda()
        r = gl.check_forward(gl.tokens(100))   # 100 tokens: four 32-token chunks
        assert (r["buf"].idx[:100].cpu().numpy() == 0).all()
    finally:
        gl.close()


def test_top_k_equals_expert_count():
    cfg = get_config("tiny", K=8)
    gl = GpuLayer(cfg, seed=7, with_w16=False)
    try:
        gl.check_forward(gl.tokens(9))
    finally:
        gl.close()


def test_empty_batch():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=0, with_w16=False)
    try:
        buf = pw.Buffers(gl.layer, 4)
        x = torch.empty((0, cfg.d), dtype=torch.float16, device="cuda")
        y = pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, buf)
        torch.cuda.synchronize()
        assert y.shape == (0, cfg.d)
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


# ---------------------------------------------------------------------------
# prefill path: experts with many tokens go through the tcgen05 GEMM
# ---------------------------------------------------------------------------

@pytest.fixture
def decode_max_tok(monkeypatch):
    def set_(v):  # routed experts and the shared FFN switch at the same batch size
        monkeypatch.setenv("PW_DECODE_MAX_TOK", str(v))
        monkeypatch.setenv("PW_DECODE_MAX_TOK_SHARED", str(v))
    return set_


def test_prefill_tiny_all_bitwidths(decode_max_tok):
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=8)
    try:
        decode_max_tok(16)
        r = gl.check_forward(gl.tokens(400))   # ~100 tokens per expert: ragged 256-token tiles
        assert r["buf"].idx is not None
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


def test_prefill_tiles_past_512_tokens(decode_max_tok):
    # top-4 of 4 experts: every expert takes every token.  Down tiles hold
    # 512 tokens (600: one full, one of 88 -- a half of padding; 1100: two
    # full, one of 76), gate/up tiles 256.
    cfg = get_config("tiny", E=4, K=4)
    gl = GpuLayer(cfg, seed=12, bits=[3, 4, 6, 16], with_w16=False)
    try:
        decode_max_tok(32)
        for T in (600, 1100):
            gl.check_forward(gl.tokens(T))
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


def test_prefill_matches_decode_path(decode_max_tok):
    cfg = get_config("tiny", d=1024, f=2048, E=4, K=2)
    gl = GpuLayer(cfg, seed=9, bits=[3, 5, 16, 6], with_w16=False)
    try:
        x = gl.tokens(300)
        decode_max_tok(0)            # every expert through tcgen05
        a = gl.check_forward(x)
        decode_max_tok(100000)       # every expert through mma.sync
        b = gl.check_forward(x)
        assert np.abs(a["y"] - b["y"]).max() < 4e-3 * (1 + np.abs(b["y"]).max())
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


def test_prefill_ragged_rows_e128_shape(decode_max_tok):
    # ffn = 704 rows is 5.5 tiles of 128 rows for gate/up
    cfg = get_config("e128", E=8, K=2)
    gl = GpuLayer(cfg, seed=10, bits=[3, 4, 6, 16, 5, 3, 4, 6], with_w16=False)
    try:
        decode_max_tok(8)
        gl.check_forward(gl.tokens(260))
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


def test_prefill_shared_ffn(decode_max_tok):
    cfg = get_config("qwen", E=6, K=2, shared_ffn=512)
    gl = GpuLayer(cfg, seed=11, with_w16=False)
    try:
        decode_max_tok(32)
        gl.check_forward(gl.tokens(200))
        assert gl.layer.check_device() == 0
    finally:
        gl.close()
