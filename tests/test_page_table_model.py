"""Random sequences of bitwidth changes against the page table, on the host
(host-simulated device, no GPU).

PagedWeight (write-up "内存的饥饿游戏", sections 核心洞察 and 安全边界与异步搬运):
lowering an expert detaches its low planes without moving data; raising
reuses planes that are still intact or uploads them again; pages freed by a
lowering are reused only after the safe boundary.  Each step applies one
random operation (lower, raise in place, prefetch, raise with an upload,
re-load, reaching the safe boundary) and then checks, for every expert:
  - the host mirror of the bitwidth is the one the sequence implies;
  - the pages the page table maps for the expert's mapped blocks (planes
    0..b-1 and the fp16 page at 16 bits, plus whatever a prefetch brought
    back ahead of a raise) hold exactly that expert's packed data -- so no
    page was reused while still mapped, and no raise re-mapped a block that
    had been reused;
  - the pool's books balance: free + mapped + reclaimable + resident = total,
    and mapped = the pages of the mapped blocks;
  - a refused call (not resident, out of pages) changed nothing.
"""
import numpy as np
import pytest

import any_precision_expert_gb300 as pw
from any_precision_expert_gb300 import _lib
from synth import get_config, make_expert

PAGE = 64 << 10
D = F = 128
E = 4
LEVELS = (3, 4, 5, 6, 16)


@pytest.fixture
def sim():
    _lib.lib.pw_testing_host_sim(1)
    yield
    _lib.lib.pw_testing_host_sim(0)


def _experts():
    cfg = get_config("tiny", d=D, f=F)
    out = []
    for e in range(E):
        ex = make_expert(cfg, e, seed=21, with_w16=True)
        planes = [pw.pack_planes(ex["code6"][m]) for m in range(3)]
        f16 = [pw.pack_f16(ex["w16"][m]) for m in range(3)]
        out.append({"ex": ex, "planes": planes, "f16": f16,
                    "block": [np.concatenate([planes[m][p] for m in range(3)]) for p in range(6)],
                    "f16_block": np.concatenate(f16)})
    return out


def _read(pool, addr, nbytes):
    off = addr - pool.buffer.data_ptr()
    assert 0 <= off and off + nbytes <= pool.buffer.numel()
    return pool.buffer[off:off + nbytes].numpy()


def _blocks(b):
    # (mapped plane blocks, fp16 block mapped) that bitwidth b reads; mapped
    # plane blocks are always a prefix 0..n-1
    return (6, True) if b == 16 else (b, False)


def _check_books(pool, mapped):
    st = pool.stats()
    resident = st["resident_bytes"] // PAGE
    assert st["free_pages"] + st["mapped_pages"] + st["reclaimable_pages"] + resident == st["total_pages"]
    # one page per plane block at this size, two for the fp16 block
    assert st["mapped_pages"] == sum(n + 2 * f for n, f in mapped)


def _check(pool, layer, data, bits, mapped, books=True):
    if books:
        _check_books(pool, mapped)
    for e, b in enumerate(bits):
        assert layer.get_expert_bitwidth(e) == b
        n, f16 = mapped[e]
        for p in range(n):
            blk = data[e]["block"][p]
            got = _read(pool, layer.page_address(e, p, 0), blk.nbytes).view(np.uint32)
            assert np.array_equal(got, blk), (e, b, p)
        if f16:
            ref = data[e]["f16_block"].view(np.uint8)
            got = np.concatenate([_read(pool, layer.page_address(e, 6, 0), PAGE),
                                  _read(pool, layer.page_address(e, 6, 1), ref.nbytes - PAGE)])
            assert np.array_equal(got, ref), (e, "fp16")


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_bitwidth_sequences_keep_the_page_table_consistent(sim, seed):
    rng = np.random.default_rng(seed)
    data = _experts()
    # six resident pages (LUTs, tables) + 8 + 6 + 3 + 3 pages of planes: a full pool
    pool = pw.Pool(26 * PAGE, page_bytes=PAGE, device="cpu")
    layer = pw.Layer(pool, D, F, E, 2, 1)
    bits = [16, 6, 3, 3]
    for e, b in enumerate(bits):
        ex = data[e]["ex"]
        layer.load_expert(e, b, ex["code6"], ex["lut"], ex["w16"] if b == 16 else None, stream=0)
    mapped = [_blocks(b) for b in bits]
    _check(pool, layer, data, bits, mapped)
    counts = dict(lower=0, raise_ok=0, raise_refused=0, prefetch_ok=0, prefetch_oom=0, upload_ok=0, upload_oom=0,
                  reload_ok=0, reload_oom=0, boundary=0)
    for _ in range(400):
        op = rng.choice(["lower", "raise", "prefetch", "upload", "reload", "boundary"],
                        p=[0.25, 0.25, 0.15, 0.1, 0.1, 0.15])
        e = int(rng.integers(E))
        b = bits[e]
        if op == "lower" and b > 3:
            nb = int(rng.choice([v for v in LEVELS if v < b and v <= 6]))
            keep = [layer.page_address(e, p, 0) for p in range(nb)]
            layer.set_expert_bitwidth(e, nb, stream=0)
            assert [layer.page_address(e, p, 0) for p in range(nb)] == keep  # no data moved
            bits[e], mapped[e] = nb, _blocks(nb)  # blocks above the new bitwidth go, prefetched ones too
            counts["lower"] += 1
        elif op == "raise" and b < 16:
            nb = int(rng.choice([v for v in LEVELS if v > b]))
            before = pool.stats()
            rc = layer.try_set_expert_bitwidth(e, nb)
            assert rc in (0, 4), rc
            if rc == 0:
                bits[e], mapped[e] = nb, _blocks(nb)
                counts["raise_ok"] += 1
            else:
                assert pool.stats() == before
                counts["raise_refused"] += 1
        elif op == "prefetch" and b < 16:
            nb = int(rng.choice([v for v in LEVELS if v > b]))
            before = pool.stats()
            try:
                layer.prefetch_expert(e, nb, planes=data[e]["planes"], w16=data[e]["f16"], copy_stream=0)
                n, f = _blocks(nb)
                mapped[e] = (max(mapped[e][0], n), mapped[e][1] or f)  # bitwidth unchanged
                counts["prefetch_ok"] += 1
            except pw.PwError as err:
                assert err.status == 3, err.status
                assert pool.stats() == before and layer.get_expert_bitwidth(e) == b
                counts["prefetch_oom"] += 1
        elif op == "upload" and b < 16:
            nb = int(rng.choice([v for v in LEVELS if v > b]))
            before = pool.stats()
            try:
                layer.raise_expert_async(e, nb, planes=data[e]["planes"], w16=data[e]["f16"], stream=0,
                                         copy_stream=0)
                bits[e], mapped[e] = nb, _blocks(nb)
                counts["upload_ok"] += 1
            except pw.PwError as err:
                assert err.status == 3, err.status  # out of pages: nothing changed
                assert pool.stats() == before and layer.get_expert_bitwidth(e) == b
                counts["upload_oom"] += 1
        elif op == "reload":
            nb = int(rng.choice(LEVELS))
            ex = data[e]["ex"]
            before = pool.stats()
            try:
                layer.load_expert(e, nb, ex["code6"], ex["lut"], ex["w16"] if nb == 16 else None, stream=0)
                bits[e], mapped[e] = nb, _blocks(nb)
                counts["reload_ok"] += 1
            except pw.PwError as err:
                assert err.status == 3, err.status  # the pool cannot hold it: expert and pool as they were
                assert pool.stats() == before and layer.get_expert_bitwidth(e) == b
                counts["reload_oom"] += 1
        elif op == "boundary":
            _lib.lib.pw_testing_complete_events()
            counts["boundary"] += 1
        _check(pool, layer, data, bits, mapped)
    # the sequence exercised every outcome
    assert all(v > 0 for v in counts.values()), counts
    layer.destroy()
    assert pool.stats()["free_pages"] == pool.stats()["total_pages"]
    pool.close()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_copies_between_layers_keep_both_page_tables_consistent(sim, seed):
    """Two layers on one pool: expert copies (layer to layer and inside a layer)
    mixed with lowering, raising and the safe boundary; every expert's mapped
    pages must hold the data of the expert it was last copied or loaded from."""
    rng = np.random.default_rng(100 + seed)
    data = _experts()
    # 2 x 6 resident pages + 20 + 13 pages of planes, one page to spare
    pool = pw.Pool(46 * PAGE, page_bytes=PAGE, device="cpu")
    layers = [pw.Layer(pool, D, F, E, 2, 1) for _ in range(2)]
    bits = [[16, 6, 3, 3], [3, 3, 4, 3]]
    origin = [[0, 1, 2, 3], [3, 2, 1, 0]]  # which expert's data each slot holds
    for L in range(2):
        for e in range(E):
            ex = data[origin[L][e]]["ex"]
            b = bits[L][e]
            layers[L].load_expert(e, b, ex["code6"], ex["lut"], ex["w16"] if b == 16 else None, stream=0)
    mapped = [[_blocks(b) for b in bits[L]] for L in range(2)]

    def check():
        _check_books(pool, mapped[0] + mapped[1])
        for L in range(2):
            _check(pool, layers[L], [data[o] for o in origin[L]], bits[L], mapped[L], books=False)

    check()
    counts = dict(lower=0, raise_ok=0, raise_refused=0, upload_ok=0, copy_ok=0, copy_not_resident=0, copy_oom=0,
                  boundary=0)
    for _ in range(300):
        op = rng.choice(["lower", "raise", "upload", "copy", "boundary"], p=[0.2, 0.15, 0.2, 0.3, 0.15])
        L, e = int(rng.integers(2)), int(rng.integers(E))
        layer, b = layers[L], bits[L][e]
        if op == "lower" and b > 3:
            nb = int(rng.choice([v for v in LEVELS if v < b and v <= 6]))
            layer.set_expert_bitwidth(e, nb, stream=0)
            bits[L][e], mapped[L][e] = nb, _blocks(nb)
            counts["lower"] += 1
        elif op == "raise" and b < 16:
            nb = int(rng.choice([v for v in LEVELS if v > b]))
            before = pool.stats()
            rc = layer.try_set_expert_bitwidth(e, nb)
            assert rc in (0, 4), rc
            if rc == 0:
                bits[L][e], mapped[L][e] = nb, _blocks(nb)
                counts["raise_ok"] += 1
            else:
                assert pool.stats() == before
                counts["raise_refused"] += 1
        elif op == "upload" and b < 16:
            nb = int(rng.choice([v for v in LEVELS if v > b]))
            src = data[origin[L][e]]
            before = pool.stats()
            try:
                layer.raise_expert_async(e, nb, planes=src["planes"], w16=src["f16"], stream=0, copy_stream=0)
                bits[L][e], mapped[L][e] = nb, _blocks(nb)
                counts["upload_ok"] += 1
            except pw.PwError as err:
                assert err.status == 3, err.status
                assert pool.stats() == before and layer.get_expert_bitwidth(e) == b
        elif op == "copy":
            Ls, es = int(rng.integers(2)), int(rng.integers(E))
            if (Ls, es) == (L, e):
                continue
            held = [v for v in LEVELS if _blocks(v)[0] <= mapped[Ls][es][0] and
                    (not _blocks(v)[1] or mapped[Ls][es][1])]
            nb = int(rng.choice(held if rng.random() < 0.7 else LEVELS))
            n, f = _blocks(nb)
            resident = n <= mapped[Ls][es][0] and (not f or mapped[Ls][es][1])
            before = pool.stats()
            try:
                layer.copy_expert(e, layers[Ls], es, nb, stream=0)
                assert resident, (nb, mapped[Ls][es])
                bits[L][e], mapped[L][e], origin[L][e] = nb, _blocks(nb), origin[Ls][es]
                counts["copy_ok"] += 1
            except pw.PwError as err:
                if not resident:
                    assert err.status == 4, err.status  # the source does not read those blocks
                    counts["copy_not_resident"] += 1
                else:
                    assert err.status == 3, err.status  # out of pages
                    counts["copy_oom"] += 1
                assert pool.stats() == before and layer.get_expert_bitwidth(e) == b
        elif op == "boundary":
            _lib.lib.pw_testing_complete_events()
            counts["boundary"] += 1
        check()
    assert all(v > 0 for v in counts.values()), counts
    for layer in layers:
        layer.destroy()
    assert pool.stats()["free_pages"] == pool.stats()["total_pages"]
    pool.close()
