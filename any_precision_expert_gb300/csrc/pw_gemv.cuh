// Warp-level building blocks of the decode-side expert GEMV: cp.async
// helpers and the 3-bit byte-permute decode from register LUTs.
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): an expert at
// bitwidth b reads only its top b bit-planes; each code is looked up in the
// row's LUT and the weights feed the expert's SwiGLU FFN.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "pw_device.cuh"

namespace pw {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// 4-byte copy of which the first n bytes (0 or 4) come from src, the rest zeros.
__device__ __forceinline__ void cp_async4_n(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
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

// 16-bit shared load, zero-extended into a 32-bit register.
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Decode mma step s of one chunk of B-bit codes (B = 4..6) into the A
// fragment through a LUT table in shared memory: the entry of code v for this
// lane is at tabl + (v << TSHIFT) and holds LUT[row g][v] in its low and
// LUT[row g+8][v] in its high half, g and g + 8 being the lane's two fragment
// rows (the tables' layouts are the kernels').
// Plane p keeps code bit B-1-p of weight (h, s, byte
// k) at bit 8k + 4h + s + 5 - p (mod 32): masking one bit per byte and
// rotating right by 4h + s + 6 - B leaves the codes of R[h] in the low B
// bits of its bytes.  Each lookup reads the one 16-bit half it needs (row g:
// +0, row g+8: +2), zero-extended, so the two columns of a fragment register
// join with an integer multiply-add (the FMA pipe, beside the busy ALU).
template <int B, int TSHIFT>
__device__ __forceinline__ void decode_step_rt(const uint32_t (&w)[B], const int s, uint32_t tabl, uint32_t (&a)[4]) {
  uint32_t R[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t m = 0;
#pragma unroll
    for (int p = 0; p < B; ++p) m |= w[p] & rotl_c(0x01010101u, 4 * h + s + 5 - p);
    R[h] = rotr(m, 4 * h + s + 6 - B);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // k = 2 * rowsel + colhalf
    const uint32_t half = (k >> 1) * 2;
    const uint32_t e0 = lds16(tabl + half + (prmt(R[0], 0u, 0x4440u | (uint32_t)k) << TSHIFT));
    const uint32_t e1 = lds16(tabl + half + (prmt(R[1], 0u, 0x4440u | (uint32_t)k) << TSHIFT));
    const int reg = (k == 0) ? 0 : (k == 1) ? 2 : (k == 2) ? 1 : 3;
    a[reg] = e1 * 65536u + e0;
  }
}

// 16-bit shared load at addr + OFF (OFF folded into the instruction).
template <int OFF>
__device__ __forceinline__ uint32_t lds16_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}

// Rotation amount r reduced to [0, 32).
__host__ __device__ constexpr int rot_amt(int r) { return ((r % 32) + 32) % 32; }

// The decode of decode_step_rt against a table at a fixed shared-memory
// address, where one byte permute gives the whole lookup address: entry
// (code v) of this lane sits at tb + 512 v + 256 q with tb = 0x10000 + c
// (c < 256: the lane's byte offset, byte 1 zero) and q = 0 or 1 chosen by
// the warp (qbit = 0 or 0x01010101).  The code words are rotated so that
// byte k holds (code << 1) | q; prmt then replaces byte 1 of tb with it.
template <int B>
__device__ __forceinline__ void decode_step_px(const uint32_t (&w)[B], const int s, uint32_t qbit, uint32_t tb,
                                               uint32_t (&a)[4]) {
  uint32_t R[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    // q sits one bit below each byte's code field (a bit no mask selects);
    // the planes are gathered in two independent chains (half the depth)
    uint32_t m0 = rotl_c(qbit, rot_amt(4 * h + s + 5 - B)), m1 = 0;
#pragma unroll
    for (int p = 0; p < B; ++p) {
      const uint32_t v = w[p] & rotl_c(0x01010101u, 4 * h + s + 5 - p);
      if (p < (B + 1) / 2) m0 |= v;
      else m1 |= v;
    }
    R[h] = rotr(m0 | m1, rot_amt(4 * h + s + 5 - B));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // k = 2 * rowsel + colhalf
    const uint32_t sel = 0x7604u | ((uint32_t)k << 4);
    uint32_t e0, e1;
    if (k >> 1) {
      e0 = lds16_at<2>(prmt(R[0], tb, sel));
      e1 = lds16_at<2>(prmt(R[1], tb, sel));
    } else {
      e0 = lds16_at<0>(prmt(R[0], tb, sel));
      e1 = lds16_at<0>(prmt(R[1], tb, sel));
    }
    const int reg = (k == 0) ? 0 : (k == 1) ? 2 : (k == 2) ? 1 : 3;
    a[reg] = e1 * 65536u + e0;
  }
}

__device__ __forceinline__ void load_lut3(const __half* row, uint32_t (&r)[4]) {
  const uint4 v = *reinterpret_cast<const uint4*>(row);
  r[0] = prmt(v.x, v.y, 0x6420u);
  r[1] = prmt(v.z, v.w, 0x6420u);
  r[2] = prmt(v.x, v.y, 0x7531u);
  r[3] = prmt(v.z, v.w, 0x7531u);
}

}  // namespace pw
