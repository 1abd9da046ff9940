// Router arithmetic shared by the router kernel and the fused decode step, so
// that both give the same logits, indices and weights bit for bit.
//
// The router is the standard MoE gate around PagedWeight's experts (write-up
// "内存的饥饿游戏", section 三层感知 reads its routing statistics): for token
// t, l = W_r x_t + bias with fp32 accumulation, p = softmax(l) over the E
// experts, the K largest l (ties to the lower index), weights p[idx] divided
// by their sum when the layer renormalises.
//
// Order of the fp32 sums: d is cut into 1024-column slices (128 pieces of 8
// columns); a unit is (4 experts, one slice); lane i of the warp that takes a
// unit adds dot products of its pieces i, i + 32, i + 64, i + 96 in that
// order, a butterfly over the lanes gives the slice sum, and a logit is bias
// + the slice sums in slice order.  None of this depends on which warp or CTA
// takes a unit.
#pragma once

#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "pw_internal.h"

namespace pw {

constexpr int kRouteEB = 4;      // experts of one unit
constexpr int kRoutePieces = 4;  // 16-byte pieces of one lane per slice (route_slices: 1024 columns)

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  const __half2* ha = reinterpret_cast<const __half2*>(&a);
  const __half2* hb = reinterpret_cast<const __half2*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __half22float2(ha[i]);
    const float2 fb = __half22float2(hb[i]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

// The lane's four W_r pieces of unit (experts e0.., slice sl); zeros past E or d.
__device__ __forceinline__ void route_load_w(const __half* wr, int d8, int E, int e0, int sl, int lane,
                                             uint4 (&wv)[kRouteEB][kRoutePieces]) {
#pragma unroll
  for (int q = 0; q < kRouteEB; ++q)
#pragma unroll
    for (int i = 0; i < kRoutePieces; ++i) {
      const int c = (sl * kRoutePieces + i) * 32 + lane;
      wv[q][i] = (e0 + q < E && c < d8) ? __ldg(reinterpret_cast<const uint4*>(wr) + (size_t)(e0 + q) * d8 + c)
                                        : make_uint4(0, 0, 0, 0);
    }
}

// Butterfly sum of a lane value over the warp (the fixed order of both kernels).
__device__ __forceinline__ float route_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Softmax over the E logits lg[0..E) and the top-K selection for one token,
// by one warp; lane 0 writes idx[0..K), w[0..K) (and bumps counts).
__device__ __forceinline__ void route_select(const float* lg, int E, int K, int renorm, int* idx, float* wout,
                                             int* counts) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = kMaxExperts / 32;
  float v[kPer];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? lg[e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) z += (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
#pragma unroll
  for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);

  unsigned taken = 0;  // bit i: expert lane + 32 i already chosen
  float wsel[kMaxTopK];
  int esel[kMaxTopK];
  float wsum = 0.f;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    esel[k] = be;
    wsel[k] = expf(bv - m) / z;
    wsum += wsel[k];
  }
  if (lane == 0) {
    for (int k = 0; k < K; ++k) {
      idx[k] = esel[k];
      wout[k] = renorm ? wsel[k] / wsum : wsel[k];
      if (counts) atomicAdd(counts + esel[k], 1);
    }
  }
}

}  // namespace pw
