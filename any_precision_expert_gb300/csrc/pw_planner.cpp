// Quality-aware bitwidth planner (host only).
//
// PagedWeight (write-up "内存的饥饿游戏"): section 三层感知 ranks experts by
// an offline sensitivity table corrected online by routing statistics (busy
// experts are protected) and a prompt residual (the routing-weighted input
// norm); section 安全边界与异步搬运 gives every expert a bitwidth floor and
// searches bitwidth stages from the least aggressive one, moving to a more
// aggressive stage only under pressure.  "动态量化优化MoE模型服务" (section
// 方法与技术路线) states the budget M_w = M_total - M_kv and approximates the
// budgeted choice greedily.  This file implements the staged greedy plan
// declared in include/pw.h (pw_plan_bitwidths).
//
// The decisions compare doubles: sums run in index order and this file is
// compiled without floating-point contraction, so the plan does not depend
// on the host (x86 or Arm) or on the compiler's fused multiply-adds.
#include <cmath>
#include <cstdint>
#include <vector>

#include "pw.h"

namespace {

constexpr int kLevels[5] = {16, 6, 5, 4, 3};  // least aggressive first

int level_of(int b) {
  for (int i = 0; i < 5; ++i)
    if (kLevels[i] == b) return i;
  return -1;
}

bool finite_nonneg(double v) { return std::isfinite(v) && v >= 0.0; }

}  // namespace

extern "C" pw_status pw_plan_bitwidths(int E, const double* sens, const double* mass, const double* resid,
                                       const int* floors, const int* ceils, const uint64_t* sizes,
                                       uint64_t budget, int* bits, uint64_t* used) {
  if (E < 1 || !sens || !sizes || !bits || !used) return PW_ERR_INVALID_ARG;
  std::vector<int> lo(E), hi(E);  // level indices: floor (largest index allowed), ceiling (start)
  for (int e = 0; e < E; ++e) {
    lo[e] = level_of(floors ? floors[e] : 3);
    hi[e] = level_of(ceils ? ceils[e] : 16);
    if (lo[e] < 0 || hi[e] < 0 || hi[e] > lo[e]) return PW_ERR_INVALID_ARG;
    for (int j = 0; j < 4; ++j)
      if (!finite_nonneg(sens[(size_t)e * 4 + j])) return PW_ERR_INVALID_ARG;
    if (mass && !finite_nonneg(mass[e])) return PW_ERR_INVALID_ARG;
    if (resid && !finite_nonneg(resid[e])) return PW_ERR_INVALID_ARG;
  }
  const bool use_mass = mass != nullptr;
  const bool use_resid = use_mass && resid != nullptr;

  // expert weight: routing-mass share times the residual ratio
  double M = 0.0, R = 0.0;
  if (use_mass)
    for (int e = 0; e < E; ++e) M += mass[e];
  if (use_resid)
    for (int e = 0; e < E; ++e) R += resid[e];
  std::vector<double> wt(E);
  for (int e = 0; e < E; ++e) {
    const double share = (use_mass && M > 0.0) ? mass[e] / M : 1.0 / E;
    double ratio = 1.0;
    if (use_resid && mass[e] > 0.0 && R > 0.0 && M > 0.0) ratio = (resid[e] / mass[e]) / (R / M);
    wt[e] = share * ratio;
  }
  auto damage = [&](int e, int level) -> double {
    const int b = kLevels[level];
    return b == 16 ? 0.0 : wt[e] * sens[(size_t)e * 4 + (b - 3)];
  };
  auto size_at = [&](int e, int level) -> uint64_t { return sizes[(size_t)e * 5 + level]; };

  std::vector<int> lv(hi);  // current level of every expert
  uint64_t total = 0;
  for (int e = 0; e < E; ++e) total += size_at(e, lv[e]);
  for (int stage = 1; stage < 5 && total > budget; ++stage) {
    while (total > budget) {
      int pick = -1;
      double best = 0.0;
      for (int e = 0; e < E; ++e) {
        // may step down if still above both the stage level and its floor
        if (lv[e] >= stage || lv[e] >= lo[e]) continue;
        const uint64_t cur = size_at(e, lv[e]), nxt = size_at(e, lv[e] + 1);
        if (nxt >= cur) continue;
        const double key = (damage(e, lv[e] + 1) - damage(e, lv[e])) / (double)(cur - nxt);
        if (pick < 0 || key < best) {
          pick = e;
          best = key;
        }
      }
      if (pick < 0) break;
      total -= size_at(pick, lv[pick]) - size_at(pick, lv[pick] + 1);
      ++lv[pick];
    }
  }
  if (total > budget) {
    uint64_t fl = 0;
    for (int e = 0; e < E; ++e) {
      bits[e] = kLevels[lo[e]];
      fl += size_at(e, lo[e]);
    }
    *used = fl;
    return PW_ERR_OOM;
  }
  for (int e = 0; e < E; ++e) bits[e] = kLevels[lv[e]];
  *used = total;
  return PW_OK;
}
