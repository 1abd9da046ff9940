"""Library checks that need no GPU: exported symbols, host packers against the
oracle's packer, and page-pool / page-table bookkeeping in host-sim mode."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import any_precision_expert_gb300 as pw
from any_precision_expert_gb300 import _lib
from oracle import pw_oracle as O
from synth import get_config, make_expert

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pw_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported():
    names = _declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(_lib.lib, n), n
        assert n in _lib.EXPORTED, n


def test_status_strings():
    assert _lib.lib.pw_status_str(0) == b"PW_OK"
    assert _lib.lib.pw_status_str(4) == b"PW_ERR_NOT_RESIDENT"


@pytest.mark.parametrize("R,C", [(16, 64), (32, 256), (48, 320), (64, 704), (16, 1408), (32, 2816)])
def test_library_packers_match_oracle(R, C):
    rng = np.random.default_rng(R * 7 + C)
    code6 = rng.integers(0, 64, size=(R, C), dtype=np.uint8)
    for a, b in zip(pw.pack_planes(code6), O.pack_planes(code6)):
        assert np.array_equal(a, b)
    w = rng.standard_normal((R, C)).astype(np.float16)
    assert np.array_equal(pw.pack_f16(w), O.pack_f16(w))


def test_packer_rejects_bad_shapes():
    code6 = np.zeros((16, 96), dtype=np.uint8)
    with pytest.raises(pw.PwError):
        pw.pack_planes(code6)


# ---------------------------------------------------------------------------
# host-simulated device: pool and page table without a GPU
# ---------------------------------------------------------------------------

PAGE = 64 << 10


@pytest.fixture
def sim():
    _lib.lib.pw_testing_host_sim(1)
    yield
    _lib.lib.pw_testing_host_sim(0)


def _layer(pool, E=4, d=128, f=128, K=2):
    return pw.Layer(pool, d, f, E, K, 1)


def _expert(e, d=128, f=128, w16=True):
    cfg = get_config("tiny", d=d, f=f)
    return make_expert(cfg, e, seed=11, with_w16=w16)


def _load(layer, e, bits, ex):
    layer.load_expert(e, bits, ex["code6"], ex["lut"], ex["w16"] if bits == 16 else None, stream=0)


def _page_bytes(pool, addr, n):
    base = pool.buffer.data_ptr()
    off = addr - base
    return pool.buffer[off:off + n].numpy()


def test_load_places_packed_tiles_in_pages(sim):
    import torch  # noqa: F401
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    ex = _expert(0)
    _load(layer, 0, 4, ex)
    st = pool.stats()
    assert st["mapped_pages"] == 4  # four planes, one page each at this size
    # plane p of the gate matrix: 8 tiles of 2*d bytes from the start of page 0 of the block
    ref = O.pack_planes(ex["code6"][0])
    for p in range(4):
        addr = layer.page_address(0, p, 0)
        assert addr != 0
        got = _page_bytes(pool, addr, ref[p].nbytes).view(np.uint32)
        assert np.array_equal(got, ref[p])
        # down matrix follows gate and up in the same page
        refd = O.pack_planes(ex["code6"][2])[p]
        got = _page_bytes(pool, addr + 2 * ref[p].nbytes, refd.nbytes).view(np.uint32)
        assert np.array_equal(got, refd)
    assert layer.page_address(0, 4, 0) == 0  # planes >= b are never uploaded
    layer.destroy()
    assert pool.stats()["free_pages"] == pool.stats()["total_pages"]
    pool.close()


def test_lower_raise_moves_no_data(sim):
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    ex = _expert(1)
    _load(layer, 1, 16, ex)
    st = pool.stats()
    assert st["mapped_pages"] == 6 + 2  # six planes + two fp16 pages
    addrs = [layer.page_address(1, p, 0) for p in range(6)]
    layer.set_expert_bitwidth(1, 3, stream=0)
    assert layer.get_expert_bitwidth(1) == 3
    st = pool.stats()
    assert st["mapped_pages"] == 3 and st["reclaimable_pages"] == 5
    layer.set_expert_bitwidth(1, 5, stream=0)  # raise from still-intact pages
    assert [layer.page_address(1, p, 0) for p in range(6)] == addrs
    st = pool.stats()
    assert st["mapped_pages"] == 5 and st["reclaimable_pages"] == 3
    layer.set_expert_bitwidth(1, 16, stream=0)
    assert pool.stats()["reclaimable_pages"] == 0
    layer.destroy()
    pool.close()


def test_raise_without_planes_is_not_resident(sim):
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    _load(layer, 0, 3, _expert(0))
    assert layer.try_set_expert_bitwidth(0, 4) == 4  # PW_ERR_NOT_RESIDENT
    assert layer.try_set_expert_bitwidth(0, 16) == 4
    assert layer.get_expert_bitwidth(0) == 3
    layer.destroy()
    pool.close()


def test_freed_pages_wait_for_the_safe_boundary(sim):
    # 6 resident pages (LUTs and tables) + expert 0 at 6 planes + experts 1, 2 at
    # 3 planes leave one free page in a 19-page pool
    pool = pw.Pool(19 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    _load(layer, 0, 6, _expert(0))
    _load(layer, 1, 3, _expert(1))
    _load(layer, 2, 3, _expert(2))
    assert pool.stats()["free_pages"] == 1
    layer.set_expert_bitwidth(0, 3, stream=0)        # planes 3..5 -> reclaimable
    assert pool.stats()["reclaimable_pages"] == 3
    ex = _expert(3)
    with pytest.raises(pw.PwError) as ei:             # safe boundary not reached: no reuse
        _load(layer, 3, 3, ex)
    assert ei.value.status == 3
    assert layer.try_set_expert_bitwidth(0, 6) == 0   # still intact: raise works
    layer.set_expert_bitwidth(0, 3, stream=0)
    _lib.lib.pw_testing_complete_events()
    _load(layer, 3, 3, ex)                            # now the freed pages are reused
    assert layer.try_set_expert_bitwidth(0, 6) == 4   # those planes are gone
    assert layer.get_expert_bitwidth(0) == 3
    layer.destroy()
    pool.close()


def test_invalid_arguments_have_no_side_effects(sim):
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    with pytest.raises(pw.PwError):
        pw.Layer(pool, 96, 128, 4, 2, 1)       # d not a multiple of 64
    with pytest.raises(pw.PwError):
        pw.Layer(pool, 128, 128, 4, 5, 1)      # K > E
    with pytest.raises(pw.PwError):
        pw.Layer(pool, 128, 128, 300, 2, 1)    # E > 256
    layer = _layer(pool)
    before = pool.stats()
    ex = _expert(0)
    for bad_bits in (0, 2, 7, 8, 15, 17):
        with pytest.raises(pw.PwError):
            _load(layer, 0, bad_bits, ex)
    with pytest.raises(pw.PwError):
        _load(layer, 4, 3, ex)                 # expert out of range
    with pytest.raises(pw.PwError):
        layer.load_expert(0, 16, ex["code6"], ex["lut"], None, stream=0)  # 16 needs fp16 page
    assert pool.stats() == before
    _load(layer, 0, 4, ex)
    for bad in (2, 7, 0):
        assert layer.try_set_expert_bitwidth(0, bad) == 1
    assert layer.try_set_expert_bitwidth(1, 3) == 1  # never loaded
    assert layer.get_expert_bitwidth(0) == 4
    layer.destroy()
    pool.close()


def test_pool_exhaustion_is_oom(sim):
    pool = pw.Pool(12 * PAGE, page_bytes=PAGE, device="cpu")
    with pytest.raises(pw.PwError) as ei:
        _layer(pool, E=64)                     # LUT blocks do not fit
    assert ei.value.status == 3
    layer = _layer(pool, E=2)
    _load(layer, 0, 3, _expert(0))
    before = pool.stats()
    with pytest.raises(pw.PwError) as ei:
        _load(layer, 1, 16, _expert(1))
    assert ei.value.status == 3
    assert pool.stats()["mapped_pages"] == before["mapped_pages"]
    layer.destroy()
    pool.close()


def test_compute_calls_refuse_in_host_sim(sim):
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    rc = _lib.lib.pw_route_topk(layer.handle, 256, 256, None, 1, 256, 256, None, None)
    assert rc == 2
    rc = _lib.lib.pw_combine(layer.handle, 256, 256, 256, 1, None, 256, None)
    assert rc == 2
    layer.destroy()
    pool.close()


def test_forward_call_checks_arguments_on_the_host(sim):
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool, E=4, d=128, f=128, K=2)
    for e in range(4):
        _load(layer, e, 3, _expert(e, w16=False))
    n1, n8 = layer.forward_workspace_size(1), layer.forward_workspace_size(8)
    assert 0 < n1 < n8 and n8 >= layer.workspace_size(8)
    f = _lib.lib.pw_moe_forward
    assert f(layer.handle, 256, 256, None, -1, 256, 256, 256, 256, n8, None) == 1  # T < 0
    assert f(layer.handle, 256, 256, None, 8, None, 256, 256, 256, n8, None) == 1  # no idx
    assert f(layer.handle, 264, 256, None, 8, 256, 256, 256, 256, n8, None) == 1  # x not 16-byte aligned
    assert f(layer.handle, 256, 256, None, 8, 256, 256, 256, 256, n8 - 1, None) == 3  # scratch too small
    assert f(layer.handle, 256, 256, None, 8, 256, 256, 256, 256, n8, None) == 2  # no device in host-sim
    assert f(layer.handle, 256, 256, None, 0, None, None, None, None, 0, None) == 2  # empty batch: nothing to check
    big = (1 << 20) + 1  # past the token cap: refused before any size is computed
    assert f(layer.handle, 256, 256, None, big, 256, 256, 256, 256, 1 << 62, None) == 1
    size = C.c_size_t()
    assert _lib.lib.pw_moe_forward_workspace_size(layer.handle, big, C.byref(size)) == 1
    assert _lib.lib.pw_workspace_size(layer.handle, big, C.byref(size)) == 1
    assert _lib.lib.pw_route_topk(layer.handle, 256, 256, None, big, 256, 256, None, None) == 1
    assert _lib.lib.pw_moe_forward_workspace_size(layer.handle, 1 << 20, C.byref(size)) == 0
    layer.destroy()
    pool.close()


def test_debug_bounds_add_a_canary_after_every_scratch_region(sim):
    # pw_layer_set_debug_bounds: 256 canary bytes after each region of the
    # whole-layer scratch (7 regions of its own + the 3 of the hot-path
    # scratch) and of the hot-path scratch (3 regions)
    pool = pw.Pool(48 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool, E=4, d=128, f=128, K=2)
    for e in range(4):
        _load(layer, e, 3, _expert(e, w16=False))
    for T in (1, 8, 300):
        nf, nw = layer.forward_workspace_size(T), layer.workspace_size(T)
        layer.set_debug_bounds(True)
        assert layer.forward_workspace_size(T) == nf + 10 * 256
        assert layer.workspace_size(T) == nw + 3 * 256
        layer.set_debug_bounds(False)
        assert layer.forward_workspace_size(T) == nf
    L = _lib.lib
    assert L.pw_debug_check_workspace(layer.handle, 8, 256, 1 << 20, None) == 1  # debug bounds off
    layer.set_debug_bounds(True)
    n = layer.forward_workspace_size(8)
    assert L.pw_debug_check_workspace(layer.handle, 8, 256, n - 1, None) == 3  # too small
    assert L.pw_debug_check_workspace(layer.handle, 8, 256, n, None) == 2  # no device in host-sim
    layer.destroy()
    pool.close()


def test_scratch_must_be_16_byte_aligned(sim):
    # h and hs are carved out of ws and read back with 16-byte copies, so a
    # misaligned ws is refused on the host (status 1) instead of reaching a kernel
    pool = pw.Pool(64 * PAGE, page_bytes=PAGE, device="cpu")
    layer = pw.Layer(pool, 128, 128, 4, 2, 1, 128)
    for e in range(4):
        _load(layer, e, 3, _expert(e, w16=False))
    rng = np.random.default_rng(5)
    layer.load_shared([(rng.standard_normal(s) * 0.02).astype(np.float16)
                       for s in ((128, 128), (128, 128), (128, 128))], stream=0)
    n = layer.workspace_size(8)
    L = _lib.lib
    h = layer.handle
    for ws, want in ((258, 1), (264, 1), (256, 2)):  # aligned scratch reaches the "no device" refusal
        assert L.pw_expert_ffn_bitplane(h, 256, 256, 8, 256, ws, n, None) == want
        assert L.pw_moe_ffn(h, 256, 256, 256, 8, 256, 256, ws, n, None) == want
        assert L.pw_shared_ffn(h, 256, 8, 256, ws, n, None) == want
        assert L.pw_permute(h, 256, 8, 256, 256, 256, 256, 256, ws, n, None) == want
    layer.destroy()
    pool.close()


def test_copy_expert_between_layers(sim):
    pool = pw.Pool(96 * PAGE, page_bytes=PAGE, device="cpu")
    a = _layer(pool)
    b = _layer(pool)
    ex = _expert(2)
    _load(a, 2, 16, ex)
    for bits in (3, 5, 16):
        b.copy_expert(1, a, 2, bits, stream=0)
        assert b.get_expert_bitwidth(1) == bits
        np_ = 6 if bits == 16 else bits
        for p in range(6):
            src, dst = a.page_address(2, p, 0), b.page_address(1, p, 0)
            if p < np_:
                assert dst != 0 and dst != src
                assert np.array_equal(_page_bytes(pool, dst, PAGE), _page_bytes(pool, src, PAGE))
            else:
                assert dst == 0
    # the fp16 page came along at 16 bits
    assert np.array_equal(_page_bytes(pool, b.page_address(1, 6, 0), PAGE), _page_bytes(pool, a.page_address(2, 6, 0), PAGE))
    # a lowered source no longer offers its detached planes
    a.set_expert_bitwidth(2, 4, stream=0)
    with pytest.raises(pw.PwError) as ei:
        b.copy_expert(0, a, 2, 5, stream=0)
    assert ei.value.status == 4
    b.copy_expert(0, a, 2, 4, stream=0)
    # shapes must agree
    c = pw.Layer(pool, 128, 192, 4, 2, 1)
    with pytest.raises(pw.PwError):
        c.copy_expert(0, a, 2, 3, stream=0)
    for L in (a, b, c):
        L.destroy()
    assert pool.stats()["free_pages"] == pool.stats()["total_pages"]
    pool.close()


def test_raise_async_uploads_missing_planes_only(sim):
    pool = pw.Pool(64 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    ex = _expert(3)
    _load(layer, 1, 3, ex)
    packed = [pw.pack_planes(ex["code6"][m]) for m in range(3)]
    with pytest.raises(pw.PwError):                      # planes 3, 4 are gone and none were given
        layer.raise_expert_async(1, 5, stream=0, copy_stream=0)
    layer.raise_expert_async(1, 5, planes=packed, stream=0, copy_stream=0)
    assert layer.get_expert_bitwidth(1) == 5
    for p in range(5):
        addr = layer.page_address(1, p, 0)
        got = _page_bytes(pool, addr, packed[0][p].nbytes).view(np.uint32)
        assert np.array_equal(got, packed[0][p])        # gate tiles at the start of the block
        got = _page_bytes(pool, addr + 2 * packed[0][p].nbytes, packed[2][p].nbytes).view(np.uint32)
        assert np.array_equal(got, packed[2][p])        # down follows gate and up
    addrs = [layer.page_address(1, p, 0) for p in range(5)]
    layer.set_expert_bitwidth(1, 3, stream=0)
    layer.raise_expert_async(1, 5, stream=0, copy_stream=0)  # still reclaimable: re-mapped, nothing copied
    assert [layer.page_address(1, p, 0) for p in range(5)] == addrs
    with pytest.raises(pw.PwError):
        layer.raise_expert_async(1, 4, stream=0, copy_stream=0)  # not a raise
    with pytest.raises(pw.PwError):
        layer.raise_expert_async(1, 16, planes=packed, stream=0, copy_stream=0)  # fp16 page missing
    w16 = [pw.pack_f16(m) for m in _expert(3, w16=True)["w16"]]
    layer.raise_expert_async(1, 16, planes=packed, w16=w16, stream=0, copy_stream=0)
    assert layer.get_expert_bitwidth(1) == 16
    got = _page_bytes(pool, layer.page_address(1, 6, 0), w16[0].nbytes).view(np.uint16)
    assert np.array_equal(got, w16[0])
    layer.destroy()
    assert pool.stats()["free_pages"] == pool.stats()["total_pages"]
    pool.close()


def test_prefetch_then_raise(sim):
    pool = pw.Pool(64 * PAGE, page_bytes=PAGE, device="cpu")
    layer = _layer(pool)
    ex = _expert(4)
    _load(layer, 0, 3, ex)
    packed = [pw.pack_planes(ex["code6"][m]) for m in range(3)]
    assert layer.try_set_expert_bitwidth(0, 6) == 4          # planes 3..5 are not resident
    layer.prefetch_expert(0, 6, planes=packed, copy_stream=0)
    assert layer.get_expert_bitwidth(0) == 3                 # nothing committed yet
    got = _page_bytes(pool, layer.page_address(0, 5, 0), packed[0][5].nbytes).view(np.uint32)
    assert np.array_equal(got, packed[0][5])
    layer.set_expert_bitwidth(0, 6, stream=0)                # the commit
    assert layer.get_expert_bitwidth(0) == 6
    layer.set_expert_bitwidth(0, 3, stream=0)                # lower: planes 3..5 reclaimable again
    assert pool.stats()["reclaimable_pages"] == 3
    layer.prefetch_expert(0, 5, copy_stream=0)               # held off the reclaim queue, no data needed
    assert pool.stats()["reclaimable_pages"] == 1
    layer.set_expert_bitwidth(0, 5, stream=0)
    assert layer.get_expert_bitwidth(0) == 5
    layer.destroy()
    pool.close()


# ---------------------------------------------------------------------------
# virtual-memory pool (pw_pool_create_vmm), host-simulated: physical pages are
# pages of one shared memory file, mapped into reserved ranges with mmap
# ---------------------------------------------------------------------------

VPAGE = 2 << 20


def _at(addr, n):
    return np.frombuffer(C.string_at(addr, n), dtype=np.uint8)


def test_vmm_pool_fixed_addresses_and_mappings_only_on_reuse(sim):
    # one resident page (the layer's tables and LUTs), 4 + 3 + 3 plane pages, 2 free
    pool = pw.Pool.from_vmm_handles(list(range(13)), page_bytes=VPAGE)
    layer = pw.Layer(pool, 128, 128, 4, 2, 1)
    assert pool.vmm_counts() == (1, 0)                 # the resident run is mapped
    ex = _expert(0)
    _load(layer, 0, 4, ex)
    assert pool.vmm_counts() == (5, 0)                 # one page per plane block
    va = [layer.page_address(0, p, 0) for p in range(4)]
    assert len(set(va)) == 4 and all(a != 0 for a in va)
    ref = O.pack_planes(ex["code6"][0])
    for p in range(4):
        assert np.array_equal(_at(va[p], ref[p].nbytes).view(np.uint32), ref[p])
    # lowering and raising move no data and change no mapping
    layer.set_expert_bitwidth(0, 3, stream=0)
    assert layer.try_set_expert_bitwidth(0, 4) == 0
    layer.set_expert_bitwidth(0, 3, stream=0)
    assert pool.vmm_counts() == (5, 0)
    assert [layer.page_address(0, p, 0) for p in range(4)] == va
    for e in (1, 2):
        _load(layer, e, 3, _expert(e))
    assert pool.stats()["free_pages"] == 2 and pool.stats()["reclaimable_pages"] == 1
    # the reclaimable page goes to another expert only after its safe boundary,
    # and is unmapped from expert 0's range then
    with pytest.raises(pw.PwError):
        _load(layer, 3, 3, _expert(3))
    assert pool.vmm_counts() == (11, 0)
    _lib.lib.pw_testing_complete_events()
    _load(layer, 3, 3, _expert(3))
    assert pool.vmm_counts() == (14, 1)
    assert layer.page_address(0, 3, 0) == 0            # plane 3 of expert 0 is gone
    assert layer.try_set_expert_bitwidth(0, 4) == 4    # PW_ERR_NOT_RESIDENT
    layer.destroy()
    assert pool.vmm_counts()[0] == pool.vmm_counts()[1]
    assert pool.stats()["free_pages"] == 13
    pool.close()


def test_vmm_pool_reupload_keeps_the_block_address(sim):
    pool = pw.Pool.from_vmm_handles(list(range(16)), page_bytes=VPAGE)
    layer = pw.Layer(pool, 128, 128, 4, 2, 1)
    ex = _expert(5)
    _load(layer, 1, 5, ex)
    va = [layer.page_address(1, p, 0) for p in range(5)]
    layer.set_expert_bitwidth(1, 3, stream=0)          # planes 3 and 4 reclaimable
    _lib.lib.pw_testing_complete_events()
    for e in (0, 2, 3):                                # 12 pages: 10 free + the 2 reclaimable
        _load(layer, e, 4, _expert(e))
    assert layer.page_address(1, 3, 0) == 0 and layer.page_address(1, 4, 0) == 0
    for e in (2, 3):
        layer.set_expert_bitwidth(e, 3, stream=0)      # two pages reclaimable again
    _lib.lib.pw_testing_complete_events()
    packed = [pw.pack_planes(ex["code6"][m]) for m in range(3)]
    layer.raise_expert_async(1, 5, planes=packed, stream=0, copy_stream=0)
    assert layer.get_expert_bitwidth(1) == 5
    assert [layer.page_address(1, p, 0) for p in range(5)] == va   # same virtual addresses
    for p in range(5):
        assert np.array_equal(_at(va[p], packed[0][p].nbytes).view(np.uint32), packed[0][p])
        down = _at(va[p] + 2 * packed[0][p].nbytes, packed[2][p].nbytes).view(np.uint32)
        assert np.array_equal(down, packed[2][p])
    layer.destroy()
    assert pool.vmm_counts()[0] == pool.vmm_counts()[1]
    pool.close()


def test_vmm_pool_checks_arguments(sim):
    h = (C.c_ulonglong * 4)(1, 2, 3, 4)
    out = C.c_void_p()
    assert _lib.lib.pw_pool_create_vmm(h, 4, 64 << 10, 0, C.byref(out)) == 1   # not whole 2 MiB granules
    assert _lib.lib.pw_pool_create_vmm(None, 4, VPAGE, 0, C.byref(out)) == 1
    assert _lib.lib.pw_pool_create_vmm(h, 0, VPAGE, 0, C.byref(out)) == 1
    assert _lib.lib.pw_pool_create_vmm(h, 4, VPAGE, -1, C.byref(out)) == 1


def test_decode_plan_thresholds(monkeypatch):
    # host-only query of the decode / tensor-core split the kernels take
    monkeypatch.delenv("PW_DECODE_MAX_TOK", raising=False)
    monkeypatch.delenv("PW_DECODE_MAX_TOK_SHARED", raising=False)

    def plan(name, T):
        c = get_config(name)
        return pw.decode_plan(c.d, c.f, c.E, c.K, T, c.shared_ffn)
    # wide experts (ffn 14336, 8 experts, top-2): up to 64 tokens while the
    # batch averages at most 32 slots per expert, else 32
    assert plan("mixtral", 16) == {"routed_max": 64, "shared_max": 256, "fused": True}
    assert plan("mixtral", 17)["fused"] is False
    assert plan("mixtral", 64)["routed_max"] == 64
    assert plan("mixtral", 128)["routed_max"] == 64
    assert plan("mixtral", 129)["routed_max"] == 32
    assert plan("mixtral", 4096)["routed_max"] == 32
    # narrow experts: 64 up to 64-token batches; 128 for batches spread over
    # 128+ experts at <= 32 slots per expert; else 32
    assert plan("qwen", 64)["routed_max"] == 64
    assert plan("qwen", 65)["routed_max"] == 32
    assert plan("e128", 128)["routed_max"] == 128
    assert plan("e128", 512)["routed_max"] == 128
    assert plan("e128", 513)["routed_max"] == 32
    assert plan("qwen", 0)["fused"] is False
    # the kernels' environment overrides apply
    monkeypatch.setenv("PW_DECODE_MAX_TOK", "8")
    monkeypatch.setenv("PW_DECODE_MAX_TOK_SHARED", "4")
    p = plan("qwen", 8)
    assert (p["routed_max"], p["shared_max"], p["fused"]) == (8, 4, False)
    with pytest.raises(pw.PwError):
        pw.decode_plan(512, 1024, 8, 2, -1)
    with pytest.raises(pw.PwError):
        pw.decode_plan(512, 0, 8, 2, 4)
