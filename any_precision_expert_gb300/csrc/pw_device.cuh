// Device helpers shared by the kernels: PTX wrappers, the bit-plane decode and
// the tensor-core fragment conventions of the stored layout.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "pw_internal.h"

namespace pw {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__host__ __device__ constexpr uint32_t rotl_c(uint32_t x, int r) {
  return r % 32 == 0 ? x : ((x << (r % 32)) | (x >> (32 - r % 32)));
}

__device__ __forceinline__ uint32_t rotr(uint32_t x, int r) { return __funnelshift_r(x, x, r); }

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// D += A(16x16 fp16, row) * B(16x8 fp16, col), fp32 accumulate.
// A pure register operation: not volatile, so the compiler may schedule it
// among the shared-memory loads of the decode.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Bit-plane decode.
//
// One lane's word of plane p (for one 16-row x 64-column chunk) holds the bit
// (5 - p) of 32 weights: weight (s, k, h) sits at bit (8k + 4h + s + 5 - p) mod
// 32, where s is the 16-column mma step, k the A-fragment register (k = 2 rowsel
// + colhalf) and h the even/odd column of the register's half pair.  Masking
// plane p with rotl(0x01010101, 4h + s + 5 - p) keeps the four weights
// (s, k = 0..3, h); OR-ing the masked planes and rotating right by
// 4h + s + 6 - b leaves the b-bit code of weight (s, k, h) alone in byte k.
//
// LUT tables in shared memory: entry (v, rowset rho, lane) at byte offset
// v*256 + rho*128 + 4*lane holds LUT_b[row][v] in its low half, where row =
// tile row g + 8 rho of the lane (g = lane / 4).  Every lane reads its own
// copy, so a warp's 32 lookups never conflict on a bank.  With the lane offset
// in byte 0 of `lb[rho]`, one prmt builds the lookup offset: byte 1 = code.
// ---------------------------------------------------------------------------

// Decode mma step s (0..3) of one chunk into the four A-fragment registers.
// w[p]: the lane's word of plane p (p < B).  tab: smem table of this matrix.
template <int B>
__device__ __forceinline__ void decode_step_lut(const uint32_t (&w)[B], const int s, uint32_t tab, uint32_t lb0,
                                                uint32_t lb1, uint32_t (&a)[4]) {
  uint32_t R[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t m = 0;
#pragma unroll
    for (int p = 0; p < B; ++p) m |= w[p] & rotl_c(0x01010101u, 4 * h + s + 5 - p);
    R[h] = rotr(m, 4 * h + s + 6 - B);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lb = (k >> 1) ? lb1 : lb0;
    const uint32_t sel = 0x5504u | ((uint32_t)k << 4);
    const uint32_t e0 = lds32(tab + prmt(R[0], lb, sel));
    const uint32_t e1 = lds32(tab + prmt(R[1], lb, sel));
    // A-fragment register order: a0 (row g, cols 2t..), a1 (row g+8), a2 (row g, cols 2t+8..), a3
    const int reg = (k == 0) ? 0 : (k == 1) ? 2 : (k == 2) ? 1 : 3;
    a[reg] = prmt(e0, e1, 0x5410u);
  }
}

// Build the per-lane LUT copies of one 16-row tile of one matrix at bitwidth B.
// lut: the tile's LUT_b rows (16 rows x 2^B fp16, row-major).  tab: smem table.
// Called by nthreads threads with index tid.
template <int B>
__device__ __forceinline__ void build_lut_table(const __half* lut, uint32_t* tab, int tid, int nthreads) {
  constexpr int V = 1 << B;
  // one uint4 store per (v, rho, g): the four lanes t = 0..3 of row g+8rho
  for (int i = tid; i < V * 16; i += nthreads) {
    const int v = i >> 4, rg = i & 15;  // rg = rho*8 + g
    const uint32_t val = __half_as_ushort(lut[rg * V + v]);
    const uint32_t dup = val | (val << 16);
    reinterpret_cast<uint4*>(tab)[(v * 256 + rg * 16) / 16] = make_uint4(dup, dup, dup, dup);
  }
}

// Address of tile `tau` of matrix m, plane p (p < 6) or the fp16 page (p == 6)
// of expert e, through the page table.
__device__ __forceinline__ const char* tile_addr(const DevLayer& L, int e, int m, int p, int tau) {
  if (p < kPlanes) {
    const uint2 loc = L.tmap[m * L.tmax + tau];
    const unsigned long long base = L.plane_pt[((size_t)e * kPlanes + p) * L.pmax + loc.x];
    return reinterpret_cast<const char*>(base) + loc.y;
  }
  const uint2 loc = L.tmap16[m * L.tmax + tau];
  const unsigned long long base = L.f16_pt[(size_t)e * L.pmax16 + loc.x];
  return reinterpret_cast<const char*>(base) + loc.y;
}

__device__ __forceinline__ const __half* lut_rows(const DevLayer& L, int e, int m, int b, int row0) {
  const char* base = reinterpret_cast<const char*>(L.lut_base[e]) + L.lut_off[m][b - 3];
  return reinterpret_cast<const __half*>(base) + (size_t)row0 * (1 << b);
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + __expf(-v)); }

}  // namespace pw
