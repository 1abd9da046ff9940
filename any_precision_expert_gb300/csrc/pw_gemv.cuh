// Warp-level building blocks of the decode-side expert GEMV: cp.async weight
// rings, the 3-bit byte-permute decode, activation (B-fragment) loads and the
// K loops over bit-plane groups or fp16 chunks of one 16-row weight tile.
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): an expert at
// bitwidth b reads only its top b bit-planes; each code is looked up in the
// row's LUT and the weights feed the expert's SwiGLU FFN.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "pw_device.cuh"

namespace pw {

constexpr int kTok = 16;       // tokens per work item
constexpr int kNT = kTok / 8;  // mma n-tiles per item

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// 3-bit codes: byte-permute lookups from registers.
// lut[r] = {lo bytes of entries 0-3, lo 4-7, hi 0-3, hi 4-7} of row g (r = 0)
// or g + 8 (r = 1).  Plane p keeps code bit 2-p of weight (s, nibble n) at bit
// 4n + s + 5 - p; masking with rotl(0x11111111, s+5-p) and rotating right by
// s+3 puts the code of (s, n) in nibble n (bit 3 clear), so the low half
// selects row g's four codes and the high half row g+8's.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void decode_step_prmt3(const uint32_t (&w)[3], const int s, const uint32_t (&lut)[2][4],
                                                  uint32_t (&a)[4]) {
  uint32_t m = 0;
#pragma unroll
  for (int p = 0; p < 3; ++p) m |= w[p] & rotl_c(0x11111111u, s + 5 - p);
  const uint32_t sel0 = rotr(m, s + 3), sel1 = rotr(m, s + 19);
  uint32_t lo = prmt(lut[0][0], lut[0][1], sel0), hi = prmt(lut[0][2], lut[0][3], sel0);
  a[0] = prmt(lo, hi, 0x5140u);
  a[2] = prmt(lo, hi, 0x7362u);
  lo = prmt(lut[1][0], lut[1][1], sel1);
  hi = prmt(lut[1][2], lut[1][3], sel1);
  a[1] = prmt(lo, hi, 0x5140u);
  a[3] = prmt(lo, hi, 0x7362u);
}

__device__ __forceinline__ void load_lut3(const __half* row, uint32_t (&r)[4]) {
  const uint4 v = *reinterpret_cast<const uint4*>(row);
  r[0] = prmt(v.x, v.y, 0x6420u);
  r[1] = prmt(v.z, v.w, 0x6420u);
  r[2] = prmt(v.x, v.y, 0x7531u);
  r[3] = prmt(v.z, v.w, 0x7531u);
}

__device__ __forceinline__ uint32_t ldg_cg32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// B fragments (tokens) of one 16-column mma step.  CG: read through L2 only,
// for activations written earlier by the same launch.
template <bool CG = false>
__device__ __forceinline__ void load_bfrag(const __half* act, const int (&rowoff)[kNT], int NT, int col,
                                           uint32_t (&bf)[kNT][2]) {
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    if (nt < NT) {
      const __half* xp = act + rowoff[nt] + col;
      if constexpr (CG) {
        bf[nt][0] = ldg_cg32(xp);
        bf[nt][1] = ldg_cg32(xp + 8);
      } else {
        bf[nt][0] = *reinterpret_cast<const uint32_t*>(xp);
        bf[nt][1] = *reinterpret_cast<const uint32_t*>(xp + 8);
      }
    }
  }
}

// Issue the copies of plane group gamma (NM matrices, B planes) into ring slot `slot`:
// slot layout [matrix*B + plane][lane] x 16 bytes.
template <int B, int NM, int PB>
__device__ __forceinline__ void issue_group(const char* const (&base)[NM][PB], int gamma, int G, int rem, int lane,
                                            uint32_t slot) {
  if (gamma < G) {
    const size_t off = (size_t)(gamma * 128 + lane * 4) * 4;
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int p = 0; p < B; ++p) cp_async16(slot + ((mi * B + p) * 32 + lane) * 16, base[mi][p] + off);
  } else {
    const size_t off = (size_t)(G * 128 + lane * rem) * 4;
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int p = 0; p < B; ++p)
        for (int i = 0; i < rem; ++i) cp_async4(slot + ((mi * B + p) * 32 + lane) * 16 + 4 * i, base[mi][p] + off + 4 * i);
  }
}

// K loop of one warp over its plane groups (gamma = g0, g0 + gstep, ...).
// lut3: register LUTs (B == 3); tab: smem table of (tile, matrix 0) (B >= 4).
template <int B, int NM, int RING, int PB, bool CG = false>
__device__ __forceinline__ void warp_planes(const __half* act, const char* const (&base)[NM][PB], int K, int g0,
                                            int gstep, const int (&rowoff)[kNT], int NT,
                                            const uint32_t (&lut3)[NM][2][4], uint32_t tab, uint32_t tab_stride,
                                            uint32_t ring, float (&acc)[NM][kNT][4]) {
  const int lane = threadIdx.x & 31;
  const int nk = K / 64, G = nk / 4, rem = nk % 4, NG = G + (rem ? 1 : 0);
  const uint32_t lb0 = lane * 4, lb1 = 128 + lane * 4;
  constexpr uint32_t kSlot = NM * B * 32 * 16;
  const int nu = g0 < NG ? (NG - 1 - g0) / gstep + 1 : 0;
#pragma unroll
  for (int i = 0; i < RING - 1; ++i) {
    if (i < nu) issue_group<B, NM, PB>(base, g0 + i * gstep, G, rem, lane, ring + (i % RING) * kSlot);
    cp_commit();
  }
  // B fragments (tokens) of the next chunk are loaded while the current one is computed
  uint32_t bcur[4][kNT][2], bnxt[4][kNT][2];
  auto bload = [&](int kappa, uint32_t (&b)[4][kNT][2]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) load_bfrag<CG>(act, rowoff, NT, kappa * 64 + s * 16, b[s]);
  };
  if (nu > 0) bload(4 * g0, bcur);
  for (int i = 0; i < nu; ++i) {
    const int inext = i + RING - 1;
    if (inext < nu) issue_group<B, NM, PB>(base, g0 + inext * gstep, G, rem, lane, ring + (inext % RING) * kSlot);
    cp_commit();
    cp_wait<RING - 1>();
    const int gamma = g0 + i * gstep;
    const uint32_t slot = ring + (i % RING) * kSlot;
    uint32_t cur[NM][B][4];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int p = 0; p < B; ++p) {
        const uint4 v = lds128(slot + ((mi * B + p) * 32 + lane) * 16);
        cur[mi][p][0] = v.x;
        cur[mi][p][1] = v.y;
        cur[mi][p][2] = v.z;
        cur[mi][p][3] = v.w;
      }
    const int nch = gamma < G ? 4 : rem;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c >= nch) break;
      const int kappa = 4 * gamma + c;
      const int knext = c + 1 < nch ? kappa + 1 : (i + 1 < nu ? 4 * (gamma + gstep) : -1);
      if (knext >= 0) bload(knext, bnxt);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          uint32_t w[B];
#pragma unroll
          for (int p = 0; p < B; ++p) w[p] = cur[mi][p][c];
          uint32_t a[4];
          if constexpr (B == 3) {
            decode_step_prmt3(w, s, lut3[mi], a);
          } else {
            decode_step_lut<B>(w, s, tab + mi * tab_stride, lb0, lb1, a);
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
            if (nt < NT) mma16816(acc[mi][nt], a, bcur[s][nt][0], bcur[s][nt][1]);
        }
      }
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          bcur[s][nt][0] = bnxt[s][nt][0];
          bcur[s][nt][1] = bnxt[s][nt][1];
        }
    }
  }
  cp_wait<0>();
}

// K loop of one warp over its 64-column chunks of fp16 weights (fallback pages
// or the shared FFN): chunk kappa = k0, k0 + kstep, ...
template <int NM, int RING, bool CG = false>
__device__ __forceinline__ void warp_f16(const __half* act, const char* const (&base16)[NM], int K, int k0,
                                         int kstep, const int (&rowoff)[kNT], int NT, uint32_t ring,
                                         float (&acc)[NM][kNT][4]) {
  const int lane = threadIdx.x & 31;
  const int nk = K / 64;
  constexpr uint32_t kSlot = NM * 4 * 32 * 16;
  const int nu = k0 < nk ? (nk - 1 - k0) / kstep + 1 : 0;
  auto issue = [&](int kappa, uint32_t slot) {
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int s = 0; s < 4; ++s)
        cp_async16(slot + ((mi * 4 + s) * 32 + lane) * 16, base16[mi] + ((size_t)(kappa * 4 + s) * 32 + lane) * 16);
  };
#pragma unroll
  for (int i = 0; i < RING - 1; ++i) {
    if (i < nu) issue(k0 + i * kstep, ring + (i % RING) * kSlot);
    cp_commit();
  }
  uint32_t bcur[4][kNT][2], bnxt[4][kNT][2];
  auto bload = [&](int kappa, uint32_t (&b)[4][kNT][2]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) load_bfrag<CG>(act, rowoff, NT, kappa * 64 + s * 16, b[s]);
  };
  if (nu > 0) bload(k0, bcur);
  for (int i = 0; i < nu; ++i) {
    const int inext = i + RING - 1;
    if (inext < nu) issue(k0 + inext * kstep, ring + (inext % RING) * kSlot);
    cp_commit();
    cp_wait<RING - 1>();
    const int kappa = k0 + i * kstep;
    if (i + 1 < nu) bload(kappa + kstep, bnxt);
    const uint32_t slot = ring + (i % RING) * kSlot;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int mi = 0; mi < NM; ++mi) {
        const uint4 v = lds128(slot + ((mi * 4 + s) * 32 + lane) * 16);
        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          if (nt < NT) mma16816(acc[mi][nt], a, bcur[s][nt][0], bcur[s][nt][1]);
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        bcur[s][nt][0] = bnxt[s][nt][0];
        bcur[s][nt][1] = bnxt[s][nt][1];
      }
  }
  cp_wait<0>();
}

}  // namespace pw
