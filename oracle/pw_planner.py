"""fp64 CPU oracle for the quality-aware bitwidth planner and its online signals.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only tests/ may call it.  It shares no code with the library (the native
planner in libpw.so and the CUDA statistics kernels are written separately);
both sides only share the seeded input generators in ``synth/``.

What is computed, and where it comes from
-----------------------------------------
PagedWeight (zhichai.net/topic/178446964, section "三层感知") chooses whose
precision to lower from three signals: an offline sensitivity table (how much
worse an expert gets at a lower bitwidth), online routing statistics (busy
experts are protected, idle ones lowered first) and a prompt residual taken
from the routing-weighted input norm, which corrects the offline table for
the current prompts.  Section "安全边界与异步搬运" adds a per-expert bitwidth
floor and a staged search: the least aggressive lowering first, more
aggressive stages only under memory pressure.  The second write-up
("动态量化优化MoE模型服务", section 方法与技术路线) states the budget
M_w = M_total - M_kv and a greedy approximation of the budgeted choice.

Readings taken (the pages give no formulas for these):

* routing mass of expert e: the sum of the routing weights of the (token, k)
  slots routed to e; prompt residual: the same sum weighted by the L2 norm of
  the slot's token;
* expert weight = (mass share) x (residual ratio), where the mass share is
  mass_e / sum(mass) and the residual ratio is the expert's routing-weighted
  mean input norm relative to the layer's, (resid_e / mass_e) / (sum(resid) /
  sum(mass)) (1 when the expert saw no tokens); either factor can be switched
  off (1/E and 1 respectively);
* damage of running expert e at bitwidth b = weight_e x sens[e][b], 0 at 16;
* stages: the levels are 16, 6, 5, 4, 3; stage k allows lowering down to
  level k (never below the expert's floor).  Inside a stage, while the plan
  is over budget, the expert whose next step down costs the least damage per
  byte saved moves one level down (ties to the lower expert index); the next
  stage starts only when no expert can move further in this one;
* the plan starts from every expert's ceiling (16 unless given) and is
  infeasible when even the floors do not fit; the plan is then the floors.

Sums run in index order with plain float additions (no pairwise or
compensated summation), so a native implementation that adds in the same
order reaches the same decisions.
"""
from __future__ import annotations

import numpy as np

LEVELS = (16, 6, 5, 4, 3)   # bitwidth levels, least aggressive first
SENS_BITS = (3, 4, 5, 6)    # columns of the sensitivity table


def route_stats(x16: np.ndarray, idx: np.ndarray, w: np.ndarray, E: int):
    """Routing mass and prompt residual per expert (fp64).

    mass[e]  = sum of w[t, k] over slots with idx[t, k] == e
    resid[e] = sum of w[t, k] * ||x[t]||_2 over the same slots
    """
    x = np.asarray(x16, dtype=np.float64)
    norms = np.sqrt((x * x).sum(axis=1))
    mass = np.zeros(E)
    resid = np.zeros(E)
    T, K = idx.shape
    for t in range(T):
        for k in range(K):
            e = int(idx[t, k])
            mass[e] += float(w[t, k])
            resid[e] += float(w[t, k]) * norms[t]
    return mass, resid


def _seq_sum(values) -> float:
    s = 0.0
    for v in values:
        s += float(v)
    return s


def expert_weights(mass, resid, E: int, use_mass: bool = True, use_resid: bool = True):
    """Online weight of each expert: mass share times residual ratio."""
    if mass is None:
        use_mass = use_resid = False
    if resid is None:
        use_resid = False
    M = _seq_sum(mass) if use_mass or use_resid else 0.0
    R = _seq_sum(resid) if use_resid else 0.0
    out = []
    for e in range(E):
        share = float(mass[e]) / M if (use_mass and M > 0.0) else 1.0 / E
        ratio = 1.0
        if use_resid and float(mass[e]) > 0.0 and R > 0.0 and M > 0.0:
            ratio = (float(resid[e]) / float(mass[e])) / (R / M)
        out.append(share * ratio)
    return out


def _damage(weight: float, sens_row, b: int) -> float:
    if b == 16:
        return 0.0
    return weight * float(sens_row[SENS_BITS.index(b)])


def plan_bitwidths(sens, mass, resid, floors, ceils, sizes, budget: int,
                   use_mass: bool = True, use_resid: bool = True):
    """Greedy staged plan.  sens [E][4] (b = 3..6), sizes [E][5] bytes at the
    levels 16, 6, 5, 4, 3; floors / ceils [E] (None: 3 / 16).  Returns
    (bits [E], bytes used, feasible)."""
    E = len(sens)
    floors = [3] * E if floors is None else [int(f) for f in floors]
    ceils = [16] * E if ceils is None else [int(c) for c in ceils]
    weight = expert_weights(mass, resid, E, use_mass, use_resid)

    def size(e, b):
        return int(sizes[e][LEVELS.index(b)])

    bits = list(ceils)
    used = sum(size(e, bits[e]) for e in range(E))
    for stage in range(1, len(LEVELS)):
        if used <= budget:
            break
        level = LEVELS[stage]
        while used > budget:
            best, best_key = -1, None
            for e in range(E):
                b = bits[e]
                if b <= max(level, floors[e]):
                    continue
                nb = LEVELS[LEVELS.index(b) + 1]
                saved = size(e, b) - size(e, nb)
                if saved <= 0:
                    continue
                key = (_damage(weight[e], sens[e], nb) - _damage(weight[e], sens[e], b)) / saved
                if best_key is None or key < best_key:
                    best, best_key = e, key
            if best < 0:
                break
            b = bits[best]
            nb = LEVELS[LEVELS.index(b) + 1]
            used -= size(best, b) - size(best, nb)
            bits[best] = nb
    if used > budget:
        bits = [max(f, 3) for f in floors]
        return bits, sum(size(e, bits[e]) for e in range(E)), False
    return bits, used, True


def expert_bytes(pages_per_plane: int, pages_f16: int, page_bytes: int):
    """Pool bytes one expert holds at the levels 16, 6, 5, 4, 3: b plane
    blocks at b <= 6; at 16 the fp16 block and all six plane blocks (a 16-bit
    expert lowered to any b reads planes it still holds)."""
    return [(6 * pages_per_plane + pages_f16) * page_bytes] + [b * pages_per_plane * page_bytes for b in (6, 5, 4, 3)]
