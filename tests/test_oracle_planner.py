"""Pins of the planner oracle (oracle/pw_planner.py) against hand-worked
plans, closed forms and invariants that do not reuse its code.

PagedWeight (zhichai.net/topic/178446964): sections "三层感知" (offline
sensitivity, routing statistics, prompt residual) and "安全边界与异步搬运"
(bitwidth floors, staged search); "动态量化优化MoE模型服务", section
方法与技术路线 (budget M_w = M_total - M_kv, greedy approximation).
"""
import numpy as np
import pytest

from oracle import pw_planner as P

# three experts of equal size: 16 -> 100 bytes, 6 -> 36, 5 -> 30, 4 -> 24, 3 -> 18
SIZES3 = [[100, 36, 30, 24, 18]] * 3
# damage grows 4x per bit removed (quantisation noise power)
SENS3 = [[64.0, 16.0, 4.0, 1.0]] * 3


def test_route_stats_hand_example():
    # token norms 5 (3-4-0-0) and 3 (1-2-2-0)
    x = np.array([[3, 4, 0, 0], [1, 2, 2, 0]], dtype=np.float16)
    idx = np.array([[0, 2], [2, 1]], dtype=np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5]])
    mass, resid = P.route_stats(x, idx, w, E=3)
    assert np.allclose(mass, [0.75, 0.5, 0.75])
    assert np.allclose(resid, [0.75 * 5, 0.5 * 3, 0.25 * 5 + 0.5 * 3])


def test_route_stats_invariants():
    rng = np.random.default_rng(0)
    T, K, E = 40, 3, 7
    x = rng.normal(size=(T, 16)).astype(np.float16)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, K))
    mass, resid = P.route_stats(x, idx, w, E)
    assert np.isclose(mass.sum(), w.sum())
    # every token at the same norm c: resid = c * mass
    xc = np.zeros((T, 16), dtype=np.float16)
    xc[:, 0] = 2.0
    _, r2 = P.route_stats(xc, idx, w, E)
    assert np.allclose(r2, 2.0 * mass)
    # token order does not matter
    perm = rng.permutation(T)
    m3, r3 = P.route_stats(x[perm], idx[perm], w[perm], E)
    assert np.allclose(m3, mass) and np.allclose(r3, resid)


def test_expert_weight_is_residual_share():
    mass = [1.0, 2.0, 5.0]
    resid = [4.0, 1.0, 3.0]
    wts = P.expert_weights(mass, resid, 3)
    # mass share x residual ratio = resid_e / sum(resid) when every expert has mass
    assert np.allclose(wts, [0.5, 0.125, 0.375])
    assert np.allclose(P.expert_weights(mass, resid, 3, use_resid=False), [1 / 8, 2 / 8, 5 / 8])
    assert np.allclose(P.expert_weights(mass, resid, 3, use_mass=False, use_resid=False), [1 / 3] * 3)
    # an idle expert keeps ratio 1 and a zero share
    assert P.expert_weights([0.0, 1.0], [0.0, 2.0], 2) == [0.0, 1.0]


@pytest.mark.parametrize("budget,bits,used", [
    (400, [16, 16, 16], 300),   # everything fits
    (200, [6, 6, 16], 172),     # stage 1 only: the two lightest experts lose their fp16 page
    (100, [5, 5, 6], 96),       # stage 1 for all, then 6 -> 5 lightest first
    (60, [3, 3, 4], 60),        # down to stage 4
])
def test_plan_hand_worked(budget, bits, used):
    # weights 1/6, 2/6, 3/6 (mass shares; residual ratio 1)
    mass = [1.0, 2.0, 3.0]
    got, u, ok = P.plan_bitwidths(SENS3, mass, mass, None, None, SIZES3, budget)
    assert ok and got == bits and u == used


def test_plan_floors_and_infeasible():
    mass = [1.0, 2.0, 3.0]
    got, u, ok = P.plan_bitwidths(SENS3, mass, mass, [3, 5, 3], None, SIZES3, 70)
    assert ok and got == [3, 5, 3] and u == 66
    got, u, ok = P.plan_bitwidths(SENS3, mass, mass, [3, 5, 3], None, SIZES3, 60)
    assert not ok and got == [3, 5, 3] and u == 66
    got, u, ok = P.plan_bitwidths(SENS3, mass, mass, None, None, SIZES3, 53)
    assert not ok and got == [3, 3, 3] and u == 54


def test_plan_residual_changes_the_order():
    mass = [1.0, 1.0, 1.0]
    resid = [3.0, 1.0, 1.0]  # expert 0 sees large-norm tokens: protected
    got, _, _ = P.plan_bitwidths(SENS3, mass, resid, None, None, SIZES3, 236)
    assert got == [16, 6, 16]  # experts 1 and 2 tie; the lower index goes first
    got, _, _ = P.plan_bitwidths(SENS3, mass, resid, None, None, SIZES3, 236, use_resid=False)
    assert got == [6, 16, 16]  # all equal without the residual: expert 0 goes first


def test_plan_ceilings():
    mass = [1.0, 2.0, 3.0]
    got, u, ok = P.plan_bitwidths(SENS3, mass, mass, None, [6, 16, 16], SIZES3, 400)
    assert ok and got == [6, 16, 16] and u == 236


def _random_instance(rng, E):
    sens = [sorted(rng.random(4) * 10, reverse=True) for _ in range(E)]
    mass = list(rng.random(E) * (rng.random(E) > 0.2))
    resid = [m * (0.5 + rng.random()) for m in mass]
    floors = list(rng.choice([3, 3, 3, 4, 5], E))
    plane = int(rng.integers(2, 6))
    f16 = int(rng.integers(8, 20))
    sizes = [P.expert_bytes(plane, f16, 1) for _ in range(E)]
    return sens, mass, resid, floors, sizes


def test_plan_invariants_random():
    rng = np.random.default_rng(1)
    for _ in range(200):
        E = int(rng.integers(1, 9))
        sens, mass, resid, floors, sizes = _random_instance(rng, E)
        top = sum(s[0] for s in sizes)
        prev = None
        for budget in sorted({int(v) for v in rng.integers(0, top + 5, 12)} | {top}, reverse=True):
            bits, used, ok = P.plan_bitwidths(sens, mass, resid, floors, None, sizes, budget)
            assert all(b >= f for b, f in zip(bits, floors))
            assert used == sum(sizes[e][P.LEVELS.index(bits[e])] for e in range(E))
            if ok:
                assert used <= budget
                # stage discipline: an expert below level L means every expert
                # is at L's predecessor level or below (or at its floor)
                for k in range(2, len(P.LEVELS)):
                    if any(b < P.LEVELS[k - 1] for b in bits):
                        assert all(b <= max(P.LEVELS[k - 1], f) for b, f in zip(bits, floors))
                # a smaller budget never raises an expert
                if prev is not None:
                    assert all(b <= a for a, b in zip(prev, bits))
                prev = bits
            else:
                assert bits == floors


def test_plan_stage_one_lowers_least_damage_per_byte():
    # brute force over which experts lose their fp16 page at a budget that
    # stage 1 alone can meet: the chosen set is the one the per-byte keys order
    rng = np.random.default_rng(2)
    for _ in range(50):
        E = 5
        sens = [sorted(rng.random(4) * 10, reverse=True) for _ in range(E)]
        mass = list(rng.random(E) + 0.1)
        sizes = [[100, 36, 30, 24, 18]] * E
        wts = P.expert_weights(mass, mass, E)
        order = sorted(range(E), key=lambda e: (wts[e] * sens[e][3] / 64.0, e))
        for n in range(E + 1):
            budget = 100 * E - 64 * n
            bits, _, ok = P.plan_bitwidths(sens, mass, mass, None, None, sizes, budget)
            lowered = {e for e in range(E) if bits[e] == 6}
            assert ok and lowered == set(order[:n]) and all(b in (6, 16) for b in bits)


def test_expert_bytes():
    assert P.expert_bytes(3, 10, 2) == [(18 + 10) * 2, 36, 30, 24, 18]
