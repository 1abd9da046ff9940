"""Bitwidth planner of the library (pw_plan_bitwidths, pw_expert_resident_bytes)
against the planner oracle, on the host: no GPU needed.

PagedWeight (zhichai.net/topic/178446964), sections "三层感知" and
"安全边界与异步搬运"; "动态量化优化MoE模型服务", section 方法与技术路线.
"""
import numpy as np
import pytest

import any_precision_expert_gb300 as pw
from any_precision_expert_gb300 import _lib
from oracle import pw_planner as P
from synth import get_config, make_expert, make_sensitivity


def _instance(rng, E):
    sens = rng.random((E, 4)) * 10 * (rng.random((E, 1)) > 0.1)
    sens = -np.sort(-sens, axis=1)
    mass = rng.random(E) * (rng.random(E) > 0.25)
    resid = mass * (0.3 + 2 * rng.random(E))
    floors = rng.choice([3, 3, 3, 4, 5, 6], E)
    ceils = np.maximum(floors, rng.choice([16, 16, 16, 6, 5], E))
    ceils = np.where(ceils == 6, np.maximum(floors, 6), ceils)
    plane, f16 = int(rng.integers(1, 5)), int(rng.integers(3, 20))
    sizes = np.array([P.expert_bytes(plane, f16, 4096) for _ in range(E)], dtype=np.uint64)
    return sens, mass, resid, floors, ceils, sizes


def _both(sens, sizes, budget, mass, resid, floors, ceils):
    got = pw.plan_bitwidths(sens, sizes, budget, mass=mass, resid=resid, floors=floors, ceils=ceils)
    use_mass = mass is not None
    use_resid = use_mass and resid is not None
    ref = P.plan_bitwidths(sens.tolist(), None if mass is None else mass.tolist(),
                           None if resid is None else resid.tolist(),
                           None if floors is None else floors.tolist(), None if ceils is None else ceils.tolist(),
                           sizes.tolist(), int(budget), use_mass=use_mass, use_resid=use_resid)
    return got, ref


def test_native_plan_equals_oracle_plan():
    rng = np.random.default_rng(7)
    n_infeasible = 0
    for trial in range(300):
        E = int(rng.integers(1, 70))
        sens, mass, resid, floors, ceils, sizes = _instance(rng, E)
        top = int(sum(s[P.LEVELS.index(c)] for s, c in zip(sizes.tolist(), ceils.tolist())))
        for budget in rng.integers(0, top + 4096, 6).tolist() + [top]:
            sig = trial % 3
            m = mass if sig < 2 else None
            r = resid if sig == 0 else None
            (bits, used, ok), (rbits, rused, rok) = _both(sens, sizes, budget, m, r, floors, ceils)
            assert bits.tolist() == rbits and used == rused and ok == rok, (trial, budget)
            n_infeasible += not ok
    assert n_infeasible > 0  # the infeasible branch ran too


def test_native_plan_hand_worked():
    sens = np.array([[64.0, 16.0, 4.0, 1.0]] * 3)
    sizes = np.array([[100, 36, 30, 24, 18]] * 3, dtype=np.uint64)
    mass = np.array([1.0, 2.0, 3.0])
    assert pw.plan_bitwidths(sens, sizes, 100, mass=mass, resid=mass)[0].tolist() == [5, 5, 6]
    bits, used, ok = pw.plan_bitwidths(sens, sizes, 60, mass=mass, resid=mass, floors=[3, 5, 3])
    assert (bits.tolist(), used, ok) == ([3, 5, 3], 66, False)


@pytest.mark.parametrize("kw", [dict(floors=[7, 3]), dict(floors=[6, 3], ceils=[5, 16]),
                                dict(sens=[[1.0, 1.0, 1.0, -1.0], [0.0] * 4]), dict(mass=[1.0, float("nan")])])
def test_native_plan_rejects_bad_arguments(kw):
    args = dict(sens=[[1.0] * 4] * 2, sizes=[[9, 6, 5, 4, 3]] * 2, budget=20)
    args.update(kw)
    with pytest.raises(pw.PwError):
        pw.plan_bitwidths(args.pop("sens"), args.pop("sizes"), args.pop("budget"), **args)


PAGE = 64 << 10


@pytest.fixture
def sim():
    _lib.lib.pw_testing_host_sim(1)
    yield
    _lib.lib.pw_testing_host_sim(0)


def test_resident_bytes_match_the_pool(sim):
    cfg = get_config("tiny", d=128, f=192)
    ex = make_expert(cfg, 0, seed=3, with_w16=True)
    pool = pw.Pool(64 * PAGE, page_bytes=PAGE, device="cpu")
    layer = pw.Layer(pool, cfg.d, cfg.f, 2, 1, 1)
    layer.load_expert(0, 16, ex["code6"], ex["lut"], ex["w16"], stream=0)
    sizes = layer.plan_sizes()
    assert sizes == [layer.expert_resident_bytes(b) for b in (16, 6, 5, 4, 3)]
    for b, n in zip((16, 6, 5, 4, 3), sizes):
        layer.set_expert_bitwidth(0, b, stream=0)
        assert pool.stats()["mapped_pages"] * PAGE == n, b
    assert sizes[1] == 2 * sizes[4] and sizes[0] > sizes[1]
    layer.destroy()
    pool.close()


def test_apply_plan_reports_experts_needing_upload(sim):
    cfg = get_config("tiny", d=128, f=128)
    pool = pw.Pool(64 * PAGE, page_bytes=PAGE, device="cpu")
    layer = pw.Layer(pool, cfg.d, cfg.f, 3, 1, 1)
    for e, b in enumerate((16, 6, 3)):
        ex = make_expert(cfg, e, seed=4, with_w16=b == 16)
        layer.load_expert(e, b, ex["code6"], ex["lut"], ex["w16"] if b == 16 else None, stream=0)
    missing = layer.apply_plan([6, 4, 5], stream=0)  # lower, lower, raise past what expert 2 holds
    assert missing == [2]
    assert [layer.get_expert_bitwidth(e) for e in range(3)] == [6, 4, 3]
    layer.destroy()
    pool.close()


def test_plans_under_changing_budgets_land_in_the_pool(sim):
    """KV pressure grows, then shrinks: each budget is planned, applied (lowering
    unmaps, raising re-maps what is still held) and the experts whose planes
    are gone are uploaded again after the safe boundary; the pool then holds
    exactly the plan's bytes and every mapped page the right data."""
    cfg = get_config("tiny", d=128, f=128)
    E = 6
    pool = pw.Pool(64 * PAGE, page_bytes=PAGE, device="cpu")
    layer = pw.Layer(pool, cfg.d, cfg.f, E, 2, 1)
    exs = [make_expert(cfg, e, seed=9, with_w16=True) for e in range(E)]
    planes = [[pw.pack_planes(ex["code6"][m]) for m in range(3)] for ex in exs]
    f16 = [[pw.pack_f16(ex["w16"][m]) for m in range(3)] for ex in exs]
    for e, ex in enumerate(exs):
        layer.load_expert(e, 16, ex["code6"], ex["lut"], ex["w16"], stream=0)
    sizes = np.array([layer.plan_sizes()] * E, dtype=np.uint64)
    rng = np.random.default_rng(5)
    mass = rng.random(E) + 0.1
    resid = mass * (0.5 + rng.random(E))
    sens = make_sensitivity(get_config("qwen", E=E), seed=5)
    top = int(sizes[:, 0].sum())
    uploads = 0
    for frac in (1.0, 0.8, 0.6, 0.45, "other", 0.7, 1.0):
        if frac == "other":
            # another owner takes the freed pages for a while, so that some
            # lowered planes are really gone when the budget grows again
            other = pw.Layer(pool, cfg.d, cfg.f, 4, 2, 1)
            for e in range(4):
                other.load_expert(e, 6, exs[e]["code6"], exs[e]["lut"], None, stream=0)
            other.destroy()
            continue
        budget = int(top * frac)
        bits, used, ok = pw.plan_bitwidths(sens, sizes, budget, mass=mass, resid=resid)
        assert ok and used <= budget
        missing = layer.apply_plan(bits, stream=0)
        _lib.lib.pw_testing_complete_events()  # the safe boundary: freed pages may be reused
        for e in missing:
            layer.raise_expert_async(e, int(bits[e]), planes=planes[e], w16=f16[e], stream=0, copy_stream=0)
        uploads += len(missing)
        assert [layer.get_expert_bitwidth(e) for e in range(E)] == bits.tolist()
        assert pool.stats()["mapped_pages"] * PAGE == used
        for e, b in enumerate(bits.tolist()):
            for p in range(min(b, 6)):
                off = layer.page_address(e, p, 0) - pool.buffer.data_ptr()
                got = pool.buffer[off:off + planes[e][0][p].nbytes].numpy().view(np.uint32)
                assert np.array_equal(got, planes[e][0][p]), (frac, e, p)  # gate tiles open the block
    assert uploads > 0  # shrinking KV pressure brought back planes that were gone
    layer.destroy()
    pool.close()
