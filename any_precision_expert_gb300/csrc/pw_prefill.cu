// Prefill-side grouped expert GEMM on the 5th-generation tensor cores.
//
// For experts that receive many tokens the expert FFN is a dense contraction,
// so it runs as a grouped GEMM: each CTA owns a tile of 128 weight rows x 256
// tokens of one expert and walks the reduction in 64-column stages.  Warp
// roles (one CTA per SM, persistent over a device-built tile list):
//   * dequant warps (two per 64-row slab and matrix, alternating stages) take
//     the expert's top-b bit-planes through the page table, a plane group (4
//     stages) at a time copied by cp.async into the pair's shared buffer one
//     group ahead (whole 16-byte pieces: every sector is read once), decode them with
//     the same mask/rotate + per-lane LUT scheme as the decode kernel, and
//     write fp16 weights into shared memory in the 128-byte swizzled K-major
//     layout; afterwards they are the epilogue (TMEM -> registers -> global);
//   * one thread loads the tokens' activation tile of every stage with a TMA
//     tensor copy (128-byte swizzle; rows past the end of the tensor read as zeros);
//   * one thread issues tcgen05.mma (kind::f16, fp32 accumulators in tensor
//     memory) and releases stages with tcgen05.commit.
// Phase 0 accumulates gate and up side by side in TMEM (2 x 256 columns) and
// writes h = silu(gate) * up as fp16; phase 1 (down) writes y as fp32.
// Every wait is bounded: on a timeout the kernel flags the layer's error word
// (PW_ERR_TIMEOUT), drains its MMAs and frees its tensor memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdlib>
#include <type_traits>

#include "pw_device.cuh"
#include "pw_gemv.cuh"
#include "pw_tc.cuh"

namespace pw {

constexpr int PF_BM = 128, PF_BN = 256, PF_BK = 64;
constexpr uint32_t PF_A_BYTES = PF_BM * PF_BK * 2;  // 16 KB
constexpr uint32_t PF_B_BYTES = PF_BN * PF_BK * 2;  // 32 KB
constexpr int PF_BWARPS = 1;  // the TMA producer warp
constexpr uint32_t PF_TAB_BYTES = 64 * 128;          // LUT table of one (matrix, 64-row slab), b <= 6
constexpr uint32_t PF_PBUF_BYTES = 4 * 6 * 512;      // plane group of one warp pair's four 16-row tiles, b <= 6

template <int NM>
struct Pf {
  static constexpr int DQ = 4 * NM;                  // (matrix, slab, stage parity)
  // tokens of one tile: gate/up fills tensor memory with its two 256-column
  // accumulators; down takes 512 tokens in two, so each dequantised weight
  // tile feeds twice the MMA work
  static constexpr int NH = NM == 2 ? 1 : 2;  // 256-token halves of a tile
  static constexpr int BN = NH * PF_BN;
  static constexpr int NS = 2;
  static constexpr int WARPS = DQ + PF_BWARPS + 1;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr uint32_t STAGE = NM * PF_A_BYTES + NH * PF_B_BYTES;
  static constexpr uint32_t TABS = NM * 2 * PF_TAB_BYTES;
  // gate/up stages plane groups through a buffer per warp pair (one group in
  // flight); down loads each stage's plane words straight into registers
  static constexpr bool STAGED = NM == 2;
  // gate/up (FIXED) places its buffers at fixed addresses of the CTA's
  // shared-memory window, so that one byte permute forms a LUT lookup's whole
  // address (decode_step_px): the four LUT tables at 64 KB (entry (v, mi,
  // slab, lane) at 64 KB + 512 v + 256 mi + 128 slab + 4 lane), the stage
  // buffers from 96 KB to the window's end, plane-group buffers and barriers
  // from the dynamic base below 64 KB.  The kernel checks at entry that its
  // window holds this layout (kErrLayout otherwise).
  static constexpr bool FIXED = NM == 2;
  static constexpr int NB = 1;  // plane-group buffers per warp pair
  static constexpr uint32_t PBUFS = STAGED ? (DQ / 2) * NB * PF_PBUF_BYTES : 0;
  static constexpr uint32_t BARS = 256;
  static constexpr uint32_t SMEM = 1024 + NS * STAGE + TABS + PBUFS + BARS;  // !FIXED
  static constexpr uint32_t TAB_AT = 64 * 1024, STAGE_AT = 96 * 1024, END = STAGE_AT + NS * STAGE;  // FIXED
  static constexpr uint32_t TMEM_COLS = NM * NH * PF_BN;
  static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");
  static constexpr uint32_t FULL_COUNT = NM * 2 + 1;  // dequant warps + the TMA producer's expect_tx
  static constexpr int PAIRS = DQ / 2;                        // warps sharing one LUT table
};

struct PfParams {
  DevLayer L;
  int mode;             // 0 routed, 1 shared fp16 FFN
  const __half* act;    // [slots][K] fp16 (x_perm / x for phase 0, h for phase 1)
  const int* offsets;   // routed: [E+1]
  int n_slots;
  int min_tokens;       // experts with more tokens than this are handled here
  __half* h;            // phase 0 output [slots][fe]
  float* y;             // phase 1 output [slots][d]
};

struct PfTile {
  int e, mt, nt, slot0, nvalid;
};

template <int BN>
__device__ __forceinline__ PfTile pf_tile(int t, const int* s_pref, const int* s_off, int E, int mtiles) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= t) lo = mid; else hi = mid;
  }
  // the token tiles of one 128-row weight tile are consecutive, so they run
  // at the same time on neighbouring CTAs and read its planes from DRAM once
  const int ntiles = (s_off[lo + 1] - s_off[lo] + BN - 1) / BN;
  PfTile T;
  T.e = lo;
  const int local = t - s_pref[lo];
  T.nt = local % ntiles;
  T.mt = local / ntiles;
  T.slot0 = s_off[lo] + T.nt * BN;
  T.nvalid = min(BN, s_off[lo + 1] - T.slot0);
  return T;
}

__device__ __forceinline__ uint32_t sw128_offset(int row, int c16) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((c16 ^ (row & 7)) << 4));
}

// Decode mma steps S0 .. S0 + N - 1 (16 columns each) of one 64-column stage
// of this lane's two rows (g, g+8 of its 16-row tile) into out[s - S0][q]:
// q = 0 row g cols 16s..+7, 1 row g cols 16s+8..+15, 2 row g+8 cols 16s..+7,
// 3 row g+8 cols 16s+8..+15 (fp16 x 8 each).  tabl: this lane's entries in
// the slab's LUT table (pf_build_tab_half).
// PX: the table at fixed addresses (tabl = 0x10000 + the lane's byte offset,
// qbit its parity word; decode_step_px), else tabl = the lane's base address
// and entries 128 bytes apart (decode_step_rt).
template <int B, int S0, int N, bool PX>
__device__ __forceinline__ void pf_decode_planes(const uint32_t (&w)[4][B], uint32_t tabl, uint32_t qbit,
                                                 uint4 (&out)[N][4]) {
#pragma unroll
  for (int s = S0; s < S0 + N; ++s) {
    uint32_t a[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t wt[B];
#pragma unroll
      for (int p = 0; p < B; ++p) wt[p] = w[t][p];
      if constexpr (PX) decode_step_px<B>(wt, s, qbit, tabl, a[t]);
      else decode_step_rt<B, 7>(wt, s, tabl, a[t]);
    }
    out[s - S0][0] = make_uint4(a[0][0], a[1][0], a[2][0], a[3][0]);
    out[s - S0][1] = make_uint4(a[0][2], a[1][2], a[2][2], a[3][2]);
    out[s - S0][2] = make_uint4(a[0][1], a[1][1], a[2][1], a[3][1]);
    out[s - S0][3] = make_uint4(a[0][3], a[1][3], a[2][3], a[3][3]);
  }
}

// 3-bit codes: byte permutes from this lane's register LUTs (rows g, g+8).
template <int S0, int N>
__device__ __forceinline__ void pf_decode_planes3(const uint32_t (&w)[4][3], const uint32_t (&lut3)[2][4],
                                                  uint4 (&out)[N][4]) {
#pragma unroll
  for (int s = S0; s < S0 + N; ++s) {
    uint32_t a[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t wt[3] = {w[t][0], w[t][1], w[t][2]};
      decode_step_prmt3(wt, s, lut3, a[t]);
    }
    out[s - S0][0] = make_uint4(a[0][0], a[1][0], a[2][0], a[3][0]);
    out[s - S0][1] = make_uint4(a[0][2], a[1][2], a[2][2], a[3][2]);
    out[s - S0][2] = make_uint4(a[0][1], a[1][1], a[2][1], a[3][1]);
    out[s - S0][3] = make_uint4(a[0][3], a[1][3], a[2][3], a[3][3]);
  }
}

// Plane groups through shared memory.  A plane group (4 stages, 256 columns)
// of one 16-row tile and plane is 512 contiguous bytes: piece ln (16 bytes,
// the words of stages 0..3 of fragment lane ln).  A warp pair's buffer holds
// the group for its four tiles: block (tile tis, plane p) at 512 (6 tis + p),
// piece ln at slot ln ^ (ln >> 3), so that the eight lanes (tis, g = 0..7)
// of a quarter warp reading pieces 4g + t hit eight different 16-byte bank
// groups.  Lane (tis, g) copies pieces 4g .. 4g + 3 of its own tile: one
// 16-byte cp.async per piece for whole groups (each 32-byte sector is read
// once by the pair, instead of once per stage and lane), word by word (zeros
// past the end) for the ragged last group of rem < 4 words per lane.
__device__ __forceinline__ uint32_t pf_piece(int tis, int p, int ln) {
  return (uint32_t)((tis * 6 + p) * 512 + ((ln ^ (ln >> 3)) << 4));
}

template <int B>
__device__ __forceinline__ void pf_copy_group(const char* const (&pb)[6], int gamma, int nk, int tis, int g,
                                              uint32_t buf) {
  const int G = nk / 4, rem = nk % 4;
#pragma unroll
  for (int p = 0; p < B; ++p)
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int ln = 4 * g + t;
      const uint32_t dst = buf + pf_piece(tis, p, ln);
      if (gamma < G) {
        cp_async16(dst, pb[p] + (size_t)(gamma * 128 + ln * 4) * 4);
      } else {
        const char* q = pb[p] + (size_t)(G * 128 + ln * rem) * 4;
#pragma unroll 1
        for (int i = 0; i < 4; ++i) cp_async4_n(dst + 4 * i, q + 4 * min(i, rem - 1), i < rem ? 4u : 0u);
      }
    }
}

// This lane's words of its two stages par and par + 2 of the group (fragment
// lanes 4g + t of tile tis, every plane): w0 for stage par, w1 for par + 2.
template <int B>
__device__ __forceinline__ void pf_read_group(uint32_t buf, int par, int tis, int g, uint32_t (&w0)[4][B],
                                              uint32_t (&w1)[4][B]) {
#pragma unroll
  for (int p = 0; p < B; ++p) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 v = lds128(buf + pf_piece(tis, p, 4 * g + t));
      w0[t][p] = par ? v.y : v.x;
      w1[t][p] = par ? v.w : v.z;
    }
    // one plane's four pieces at a time in registers
#pragma unroll
    for (int t = 0; t < 4; ++t) asm volatile("" ::"r"(w0[t][p]), "r"(w1[t][p]));
  }
}

// Direct loads: the plane words of stage kb for this lane's fragment lanes
// 4g + t of its 16-row tile (null plane: zeros).
template <int B>
__device__ __forceinline__ void pf_load_planes(const char* const (&pb)[6], int kb, int nk, int g,
                                               uint32_t (&w)[4][B]) {
  const int G = nk / 4, rem = nk % 4, gamma = kb / 4, i = kb % 4;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int ln = 4 * g + t;
    const int word = gamma < G ? gamma * 128 + ln * 4 + i : G * 128 + ln * rem + i;
#pragma unroll
    for (int p = 0; p < B; ++p)
      w[t][p] = pb[p] ? *reinterpret_cast<const uint32_t*>(pb[p] + (size_t)word * 4) : 0u;
  }
}

// 3-bit register LUTs of this lane's rows g and g + 8 of the 16-row tile at
// row0 (rows past R repeat the last row).
__device__ __forceinline__ void pf_load_lut3(const DevLayer& L, int e, int mm, int row0, int g, int R,
                                             uint32_t (&lut3)[2][4]) {
  const int r0 = min(row0 + g, R - 1), r1 = min(row0 + g + 8, R - 1);
  load_lut3(lut_rows(L, e, mm, 3, r0), lut3[0]);
  load_lut3(lut_rows(L, e, mm, 3, r1), lut3[1]);
}

// Warp `par` of a pair writes its half (codes v with v / 2^(b-1) = par) of
// the per-lane LUT table of one 64-row slab starting at row slab0: entry (v,
// lane lx) at tbase + v * vstride + 4 lx holds LUT_b[row][v] | LUT_b[row +
// 8][v] << 16 for row = slab0 + 16 (lx / 8) + lx % 8, the lane's two rows, so
// a warp's 32 lookups fall on 32 different banks (rows past R repeat the last
// row).  b = 4..6.
__device__ __forceinline__ void pf_build_tab_half(const DevLayer& L, int e, int mm, int b, int slab0, int R,
                                                  int par, uint32_t tbase, uint32_t vstride) {
  const int lx = threadIdx.x & 31, half = 1 << (b - 1);
  const int row = slab0 + (lx >> 3) * 16 + (lx & 7);
  const uint4* q0 = reinterpret_cast<const uint4*>(lut_rows(L, e, mm, b, min(row, R - 1)) + par * half);
  const uint4* q1 = reinterpret_cast<const uint4*>(lut_rows(L, e, mm, b, min(row + 8, R - 1)) + par * half);
  uint4 lo[4], hi[4];  // the lane's half of both rows, loaded at once (8 entries per 16 bytes)
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < (half >> 3)) {
      lo[i] = __ldg(q0 + i);
      hi[i] = __ldg(q1 + i);
    }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < (half >> 3)) {
      const uint32_t l4[4] = {lo[i].x, lo[i].y, lo[i].z, lo[i].w}, h4[4] = {hi[i].x, hi[i].y, hi[i].z, hi[i].w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        sts32(tbase + (uint32_t)(par * half + 8 * i + j) * vstride + lx * 4,
              prmt(l4[j >> 1], h4[j >> 1], (j & 1) ? 0x7632u : 0x5410u));
    }
}

// fp16 page: stage kb of this lane's rows, gathered from the four fragment
// lanes (g, t = 0..3) of the stored tile at fb (null: zeros).
__device__ __forceinline__ void pf_gather_f16(const char* fb, int kb, int g, uint4 (&out)[4][4]) {
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    uint4 a[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      a[t] = fb ? *reinterpret_cast<const uint4*>(fb + ((size_t)(kb * 4 + st) * 32 + 4 * g + t) * 16)
                : make_uint4(0, 0, 0, 0);
    out[st][0] = make_uint4(a[0].x, a[1].x, a[2].x, a[3].x);
    out[st][1] = make_uint4(a[0].z, a[1].z, a[2].z, a[3].z);
    out[st][2] = make_uint4(a[0].y, a[1].y, a[2].y, a[3].y);
    out[st][3] = make_uint4(a[0].w, a[1].w, a[2].w, a[3].w);
  }
}

template <int NM>
__global__ void __launch_bounds__(Pf<NM>::THREADS, 1)
    ffn_prefill_kernel(PfParams Q, const __grid_constant__ CUtensorMap act_map) {
  using C = Pf<NM>;
  extern __shared__ unsigned char pf_raw[];
  __shared__ int s_pref[kMaxExperts + 1];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_bits[kMaxExperts];

  const DevLayer& L = Q.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool routed = Q.mode == 0;
  const int E = routed ? L.E : 1;
  const int fe = routed ? L.f : L.fs;
  const int K = NM == 2 ? L.d : fe;   // reduction length
  const int R = NM == 2 ? fe : L.d;   // output rows
  const int mtiles = (R + PF_BM - 1) / PF_BM;
  const int nkb = K / PF_BK;

  if (routed) {
    for (int i = tid; i <= E; i += C::THREADS) s_off[i] = Q.offsets[i];
    for (int i = tid; i < E; i += C::THREADS) s_bits[i] = L.bits[i];
  } else if (tid == 0) {
    s_off[0] = 0;
    s_off[1] = Q.n_slots;
    s_bits[0] = 16;
  }
  __syncthreads();
  if (routed && tid == 0) {
    // the caller's offsets, made monotone inside the slot rows [0, n_slots):
    // a bad table flags the layer's error word and no tile leaves those rows
    int prev = 0;
    bool bad = false;
    for (int i = 0; i <= E; ++i) {
      const int v = s_off[i], c = min(max(v, prev), Q.n_slots);
      bad |= v != c;
      s_off[i] = prev = c;
    }
    if (bad) atomicExch(L.err, kErrOffsets);
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int c = 0;
      if (e < E) {
        const int n = s_off[e + 1] - s_off[e];
        c = n > Q.min_tokens ? mtiles * ((n + C::BN - 1) / C::BN) : 0;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) s_pref[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_pref[E] = run;
  }
  __syncthreads();
  const int total = s_pref[E];
  if ((int)blockIdx.x >= total) return;  // uniform across the CTA

  // shared memory carve-up (stage buffers 1024-byte aligned for the swizzle)
  const uint32_t raw = smem_u32(pf_raw);
  uint32_t base, tabs, pbufs, bars;
  if constexpr (C::FIXED) {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t o = (raw + 127u) & ~127u;
    if (o + C::PBUFS + C::BARS > C::TAB_AT || raw + dyn < C::END) {  // uniform; nothing touched yet
      if (tid == 0) atomicExch(L.err, kErrLayout);
      return;
    }
    pbufs = o;
    bars = o + C::PBUFS;
    tabs = C::TAB_AT;
    base = C::STAGE_AT;
  } else {
    base = (raw + 1023u) & ~1023u;
    tabs = base + C::NS * C::STAGE;
    pbufs = tabs + C::TABS;
    bars = pbufs + C::PBUFS;
  }
  auto gptr = [&](uint32_t a) { return pf_raw + (a - raw); };  // generic pointer of a shared address
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::NS + s); };
  const uint32_t acc_full = bars + 16u * C::NS;
  const uint32_t acc_empty = acc_full + 8;
  const uint32_t fin_bar = acc_full + 16;
  const uint32_t tmem_slot = acc_full + 24;
  const uint32_t pair_bars = acc_full + 40;  // one per LUT-sharing warp pair
  // per (pair, buffer): the plane group in it has landed / the pair's first warp has read it
  const uint32_t landed_bars = pair_bars + 8u * C::PAIRS;
  const uint32_t read_bars = landed_bars + 8u * C::PAIRS * C::NB;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gptr(bars + 16u * C::NS + 32));
  uint32_t* tmem_slot_g = reinterpret_cast<uint32_t*>(gptr(bars + 16u * C::NS + 24));
  static_assert(16 * Pf<NM>::NS + 40 + 8 * Pf<NM>::PAIRS * (1 + 2 * Pf<NM>::NB) <= Pf<NM>::BARS, "barrier area");

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(full_bar(s), C::FULL_COUNT);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, C::DQ);
    mbar_init(fin_bar, 1);
    for (int i = 0; i < C::PAIRS; ++i) mbar_init(pair_bars + 8u * i, 2);
    for (int i = 0; i < C::PAIRS * C::NB; ++i) {
      mbar_init(landed_bars + 8u * i, 32);  // the copying warp's 32 lanes
      mbar_init(read_bars + 8u * i, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_g;

  if (warp < C::DQ) {
    // ---------------- dequant warps, then epilogue ----------------
    const int mi = NM == 2 ? (warp >> 2) : 0;
    const int mm = NM == 2 ? mi : 2;  // matrix index: 0 gate, 1 up, 2 down
    const int slab = (warp >> 1) & 1, par = warp & 1;
    const uint32_t pair_bar = pair_bars + 8u * (warp >> 1);
    uint32_t pair_use = 0;
    // both warps of the pair reach this point (bounded wait; false on abort)
    auto pair_sync = [&]() {
      if (lane == 0) mbar_arrive(pair_bar);
      const bool r = __all_sync(0xffffffffu, mbar_wait(pair_bar, pair_use & 1, abort_flag, L.err));
      ++pair_use;
      return r;
    };
    const int tis = lane >> 3, g = lane & 7;
    // this warp's LUT table: where its pair writes entry v of lane lx (tbase +
    // v vstride + 4 lx) and the lane's lookup base (tabl) and parity (qbit)
    const uint32_t tbase = C::FIXED ? C::TAB_AT + 256u * mi + 128u * slab : tabs + (uint32_t)(mi * 2 + slab) * PF_TAB_BYTES;
    const uint32_t vstride = C::FIXED ? 512u : 128u;
    const uint32_t tabl = C::FIXED ? 0x10000u + 128u * slab + 4u * lane : tbase + 4u * lane;
    const uint32_t qbit = C::FIXED && mi ? 0x01010101u : 0u;
    uint32_t it = 0, tc = 0, grp = 0;  // stages and tiles done, plane groups passed
    // plane group j of the pair (counted over all its tiles) sits in buffer j % NB
    const uint32_t pbuf0 = pbufs + (uint32_t)(warp >> 1) * C::NB * PF_PBUF_BYTES;
    const uint32_t landed0 = landed_bars + 8u * (warp >> 1) * C::NB, readb0 = read_bars + 8u * (warp >> 1) * C::NB;
    auto pbuf = [&](uint32_t j) { return pbuf0 + (j % C::NB) * PF_PBUF_BYTES; };
    auto landed = [&](uint32_t j) { return landed0 + 8u * (j % C::NB); };
    auto readb = [&](uint32_t j) { return readb0 + 8u * (j % C::NB); };
    auto jphase = [&](uint32_t j) { return (j / C::NB) & 1; };
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const PfTile T = pf_tile<C::BN>(t, s_pref, s_off, E, mtiles);
      const int b = s_bits[T.e];
      const int row0 = T.mt * PF_BM + slab * 64 + tis * 16;  // this lane's 16-row tile
      const bool tile_ok = row0 < R;
      const int tau = row0 / 16;
      uint32_t lut3[2][4] = {};
      if (b == 3) {  // register LUTs of this lane's row pair; no shared table
        pf_load_lut3(L, T.e, mm, row0, g, R, lut3);
      } else if (b <= 6) {
        ok = pair_sync();  // both warps of the pair finished the previous tile
        if (!ok) break;
        pf_build_tab_half(L, T.e, mm, b, T.mt * PF_BM + slab * 64, R, par, tbase, vstride);
        ok = pair_sync();
        if (!ok) break;
      }
      const char* pb[6];
#pragma unroll
      for (int p = 0; p < 6; ++p) pb[p] = (tile_ok && b <= 6 && p < b) ? tile_addr(L, T.e, mm, p, tau) : nullptr;
      const char* fb = nullptr;
      if (tile_ok && b == 16)
        fb = routed ? tile_addr(L, T.e, mm, kPlanes, tau)
                    : reinterpret_cast<const char*>(L.shared16[mm]) + (size_t)tau * 32 * K;

      // this warp's stages kb = par, par + 2, ... (two per plane group): the
      // pair's second warp copies each group into the pair's buffer after both
      // have read the previous one (a group ahead of its use by the first warp)
      // Steps S0 .. S0 + N - 1 of stage kb into its buffer: the first part
      // waits for the buffer (after being decoded), the last one hands the
      // stage to the MMA.
      auto store_part = [&](int kb, auto s0c, auto& out) {
        constexpr int S0 = decltype(s0c)::value;
        constexpr int N = std::extent<std::remove_reference_t<decltype(out)>>::value;
        const int s = (it + kb) % C::NS;
        if (!tile_ok) {
#pragma unroll
          for (int st = 0; st < N; ++st)
#pragma unroll
            for (int q = 0; q < 4; ++q) out[st][q] = make_uint4(0, 0, 0, 0);
        }
        if constexpr (S0 == 0) {
          const uint32_t ph = ((it + kb) / C::NS) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(s), ph ^ 1, abort_flag, L.err))) return false;
        }
        const uint32_t A = base + s * C::STAGE + mi * PF_A_BYTES;
#pragma unroll
        for (int st = 0; st < N; ++st)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = slab * 64 + tis * 16 + g + 8 * (q >> 1);
            sts128(A + sw128_offset(r, 2 * (S0 + st) + (q & 1)), out[st][q]);
          }
        if constexpr (S0 + N == 4) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
        }
        return true;
      };
      auto store_stage = [&](int kb, uint4 (&out)[4][4]) {
        return store_part(kb, std::integral_constant<int, 0>{}, out);
      };
      // gate/up: plane groups staged through the pair's buffer
      auto plane_loop_staged = [&](auto tag) {
        constexpr int BB = decltype(tag)::value;
        const int ngr = (nkb + 3) / 4;
        // The pair's second warp copies group j (into buffer j % NB) after
        // reading group j - 1, once the first warp has read group j - NB too
        // (the buffer's previous group): with two buffers that is the group
        // before, so the second warp never waits on the first one's progress.
        if (par == 1) {  // the tile's first group (its buffer's previous group was waited for)
          if (tile_ok) pf_copy_group<BB>(pb, 0, nkb, tis, g, pbuf(grp));
          cp_async_arrive(landed(grp));
        }
        for (int gm = 0; gm < ngr && ok; ++gm) {
          uint32_t w0[4][BB], w1[4][BB];
          ok = __all_sync(0xffffffffu, mbar_wait(landed(grp), jphase(grp), abort_flag, L.err));
          if (!ok) break;
          pf_read_group<BB>(pbuf(grp), par, tis, g, w0, w1);
          // the words are in registers before the buffer may be refilled
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int p = 0; p < BB; ++p) asm volatile("" ::"r"(w0[q][p]), "r"(w1[q][p]));
          __syncwarp();
          if (par == 0) {
            if (lane == 0) mbar_arrive(readb(grp));
          } else {
            const uint32_t prev = grp + 1 - C::NB;  // group whose buffer the next copy reuses
            if (grp + 1 >= (uint32_t)C::NB) {
              ok = __all_sync(0xffffffffu, mbar_wait(readb(prev), jphase(prev), abort_flag, L.err));
              if (!ok) break;
            }
            if (gm + 1 < ngr) {
              if (tile_ok) pf_copy_group<BB>(pb, gm + 1, nkb, tis, g, pbuf(grp + 1));
              cp_async_arrive(landed(grp + 1));
            }
          }
          ++grp;
          // a stage in two halves of two mma steps (fewer live registers)
          auto stage = [&](int kb, const uint32_t (&w)[4][BB]) {
            uint4 o[2][4];
            if constexpr (BB == 3) pf_decode_planes3<0, 2>(w, lut3, o);
            else pf_decode_planes<BB, 0, 2, C::FIXED>(w, tabl, qbit, o);
            if (!store_part(kb, std::integral_constant<int, 0>{}, o)) return false;
            if constexpr (BB == 3) pf_decode_planes3<2, 2>(w, lut3, o);
            else pf_decode_planes<BB, 2, 2, C::FIXED>(w, tabl, qbit, o);
            return store_part(kb, std::integral_constant<int, 2>{}, o);
          };
          const int kb = 4 * gm + par;
          if (kb < nkb) ok = stage(kb, w0);
          if (ok && kb + 2 < nkb) ok = stage(kb + 2, w1);
        }
      };
      // down: this warp's stages kb = par, par + 2, ...: decode one while the
      // plane words of the next are in flight
      auto plane_loop_direct = [&](auto tag) {
        constexpr int BB = decltype(tag)::value;
        uint32_t wn[4][BB];
        if (par < nkb) pf_load_planes<BB>(pb, par, nkb, g, wn);
        for (int kb = par; kb < nkb && ok; kb += 2) {
          uint32_t w[4][BB];
#pragma unroll
          for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int p = 0; p < BB; ++p) w[t][p] = wn[t][p];
          if (kb + 2 < nkb) pf_load_planes<BB>(pb, kb + 2, nkb, g, wn);
          uint4 out[4][4];
          if constexpr (BB == 3) pf_decode_planes3<0, 4>(w, lut3, out);
          else pf_decode_planes<BB, 0, 4, C::FIXED>(w, tabl, qbit, out);
          ok = store_stage(kb, out);
        }
      };
      auto plane_loop = [&](auto tag) {
        if constexpr (C::STAGED) plane_loop_staged(tag);
        else plane_loop_direct(tag);
      };
      switch (b) {
        case 3: plane_loop(std::integral_constant<int, 3>{}); break;
        case 4: plane_loop(std::integral_constant<int, 4>{}); break;
        case 5: plane_loop(std::integral_constant<int, 5>{}); break;
        case 6: plane_loop(std::integral_constant<int, 6>{}); break;
        default:  // fp16 page: the lane gathers the four fragment lanes (g, t)
          for (int kb = par; kb < nkb && ok; kb += 2) {
            uint4 out[4][4];
            pf_gather_f16(fb, kb, g, out);
            ok = store_stage(kb, out);
          }
      }
      it += nkb;
      if (!ok) break;
      // epilogue: this warp reads TMEM lanes 32*(warp%4).. of the tile's accumulators
      ok = __all_sync(0xffffffffu, mbar_wait(acc_full, tc & 1, abort_flag, L.err));
      if (!ok) break;
      tc_fence_after();
      const int lg = warp & 3;
      const int row = T.mt * PF_BM + 32 * lg + lane;
      const uint32_t tl = tmem + ((uint32_t)(32 * lg) << 16);
      if (NM == 2) {
        const int c0 = (warp >> 2) * 128;
        for (int c = 0; c < 4; ++c) {
          float gv[32], uv[32];
          tmem_ld32(tl + c0 + 32 * c, gv);
          tmem_ld32(tl + 256 + c0 + 32 * c, uv);
          if (row < R) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = c0 + 32 * c + j;
              if (n < T.nvalid)
                Q.h[(size_t)(T.slot0 + n) * fe + row] = __float2half_rn(silu_f(gv[j]) * uv[j]);
            }
          }
        }
      } else {
        const int nc = (min(T.nvalid, C::BN) + 31) / 32;  // column groups holding tokens
        for (int c = 0; c < nc; ++c) {
          float acc[32];
          tmem_ld32(tl + 32 * c, acc);
          if (row < R) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = 32 * c + j;
              if (n < T.nvalid) Q.y[(size_t)(T.slot0 + n) * L.d + row] = acc[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      ++tc;
    }
    cp_wait<0>();  // no copy into shared memory outlives the loop (also after an abort)
  } else if (warp < C::DQ + PF_BWARPS) {
    // ---------------- activation producer: one TMA copy per stage ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const PfTile T = pf_tile<C::BN>(t, s_pref, s_off, E, mtiles);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % C::NS;
          const uint32_t ph = (it / C::NS) & 1;
          ok = mbar_wait(empty_bar(s), ph ^ 1, abort_flag, L.err);
          if (!ok) break;
          const uint32_t Bs = base + s * C::STAGE + NM * PF_A_BYTES;
          const int nh = T.nvalid > PF_BN ? C::NH : 1;  // 256-row boxes holding tokens
          mbar_arrive_expect_tx(full_bar(s), nh * PF_B_BYTES);
          for (int hh = 0; hh < nh; ++hh)
            tma_load_2d(Bs + hh * PF_B_BYTES, &act_map, kb * PF_BK, T.slot0 + hh * PF_BN, full_bar(s));
        }
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_f16(PF_BM, PF_BN);
    uint32_t it = 0, tc = 0;
    bool issued = false, ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      // halves of the tile holding tokens (a tile of at most 256 takes one)
      const int nh = C::NH == 1 || pf_tile<C::BN>(t, s_pref, s_off, E, mtiles).nvalid > PF_BN ? C::NH : 1;
      ok = mbar_wait(acc_empty, (tc & 1) ^ 1, abort_flag, L.err);
      if (!ok) break;
      tc_fence_after();
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % C::NS;
        const uint32_t ph = (it / C::NS) & 1;
        ok = mbar_wait(full_bar(s), ph, abort_flag, L.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = base + s * C::STAGE;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const uint64_t adesc = sw128_desc(st + m * PF_A_BYTES);
#pragma unroll
          for (int hh = 0; hh < C::NH; ++hh) {  // accumulator columns (m * NH + hh) * 256 ..
            if (hh >= nh) break;
            const uint64_t bdesc = sw128_desc(st + NM * PF_A_BYTES + hh * PF_B_BYTES);
#pragma unroll
            for (int k = 0; k < PF_BK / 16; ++k)
              umma_f16(tmem + (m * C::NH + hh) * PF_BN, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
          }
        }
        issued = true;
        umma_commit(empty_bar(s));
      }
      if (!ok) break;
      umma_commit(acc_full);
      ++tc;
    }
    if (issued) {  // drain: every MMA must be done before tensor memory is freed
      umma_commit(fin_bar);
      volatile int never = 0;  // drain even after an abort
      mbar_wait(fin_bar, 0, &never, L.err);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// Debug: the decoded weights of expert e's matrix m exactly as the dequant
// warps of this kernel produce them (same LUT set-up, plane loads -- staged
// plane groups for gate and up, direct loads for down -- and decode
// routines), written to out[rows][cols] instead of the swizzled A tile.  One
// CTA per 128-row tile; warps (slab, parity) as in the kernel.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) prefill_dump_kernel(DevLayer L, int e, int m, __half* out) {
  extern __shared__ __align__(16) unsigned char pfd_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slab = (warp >> 1) & 1, par = warp & 1, tis = lane >> 3, g = lane & 7;
  const int R = m < 2 ? L.f : L.d, C = m < 2 ? L.d : L.f;
  const int nkb = C / PF_BK;
  const int row0 = blockIdx.x * PF_BM + slab * 64 + tis * 16;
  const bool tile_ok = row0 < R;
  const int tau = row0 / 16;
  const int b = L.bits[e];
  // shared memory: the down kernel's tables (2 x 8 KB) and the slabs' plane-group
  // buffers from the dynamic base, the gate/up kernel's fixed tables at 64 KB
  const uint32_t raw = smem_u32(pfd_smem);
  {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (raw + 2 * PF_TAB_BYTES + 2 * PF_PBUF_BYTES > Pf<2>::TAB_AT || raw + dyn < Pf<2>::TAB_AT + 32 * 1024) {
      if (threadIdx.x == 0) atomicExch(L.err, kErrLayout);
      return;
    }
  }
  const bool px = m < 2;  // gate / up: the fixed layout of ffn_prefill_kernel<2>
  const uint32_t tbase = px ? Pf<2>::TAB_AT + 256u * m + 128u * slab : raw + (uint32_t)slab * PF_TAB_BYTES;
  const uint32_t vstride = px ? 512u : 128u;
  const uint32_t tabl = px ? 0x10000u + 128u * slab + 4u * lane : tbase + 4u * lane;
  const uint32_t qbit = px && m ? 0x01010101u : 0u;
  uint32_t lut3[2][4] = {};
  if (b == 3) {
    pf_load_lut3(L, e, m, row0, g, R, lut3);
  } else if (b >= 4 && b <= 6) {
    pf_build_tab_half(L, e, m, b, blockIdx.x * PF_BM + slab * 64, R, par, tbase, vstride);
    __syncthreads();  // b is the same for the whole CTA
  }
  const char* pb[6];
#pragma unroll
  for (int p = 0; p < 6; ++p) pb[p] = (tile_ok && b <= 6 && p < b) ? tile_addr(L, e, m, p, tau) : nullptr;
  const char* fb = (tile_ok && b == 16) ? tile_addr(L, e, m, kPlanes, tau) : nullptr;
  auto put = [&](int kb, const uint4 (&o)[4][4]) {
    if (!tile_ok) return;
#pragma unroll
    for (int st = 0; st < 4; ++st)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = row0 + g + 8 * (q >> 1), c = kb * PF_BK + 16 * st + 8 * (q & 1);
        *reinterpret_cast<uint4*>(out + (size_t)r * C + c) = o[st][q];
      }
  };
  const uint32_t pbuf = raw + 2 * PF_TAB_BYTES + (uint32_t)slab * PF_PBUF_BYTES;
  auto planes = [&](auto tag) {
    constexpr int BB = decltype(tag)::value;
    if (m == 2) {  // down: direct loads
      for (int kb = par; kb < nkb; kb += 2) {
        uint32_t w[4][BB];
        pf_load_planes<BB>(pb, kb, nkb, g, w);
        uint4 o[4][4];
        if constexpr (BB == 3) pf_decode_planes3<0, 4>(w, lut3, o);
        else pf_decode_planes<BB, 0, 4, false>(w, tabl, qbit, o);
        put(kb, o);
      }
      return;
    }
    const int ngr = (nkb + 3) / 4;
    for (int gm = 0; gm < ngr; ++gm) {  // gate / up: plane groups through the slab's buffer
      if (par == 1 && tile_ok) pf_copy_group<BB>(pb, gm, nkb, tis, g, pbuf);
      cp_commit();
      cp_wait<0>();
      __syncthreads();  // the group is in the slab's buffer
      uint32_t w0[4][BB], w1[4][BB];
      pf_read_group<BB>(pbuf, par, tis, g, w0, w1);
      __syncthreads();  // both warps of the slab have read it
      uint4 o[4][4];
      const int kb = 4 * gm + par;
      if (kb < nkb) {
        if constexpr (BB == 3) pf_decode_planes3<0, 4>(w0, lut3, o);
        else pf_decode_planes<BB, 0, 4, true>(w0, tabl, qbit, o);
        put(kb, o);
      }
      if (kb + 2 < nkb) {
        if constexpr (BB == 3) pf_decode_planes3<0, 4>(w1, lut3, o);
        else pf_decode_planes<BB, 0, 4, true>(w1, tabl, qbit, o);
        put(kb + 2, o);
      }
    }
  };
  switch (b) {
    case 3: planes(std::integral_constant<int, 3>{}); break;
    case 4: planes(std::integral_constant<int, 4>{}); break;
    case 5: planes(std::integral_constant<int, 5>{}); break;
    case 6: planes(std::integral_constant<int, 6>{}); break;
    case 16:
      for (int kb = par; kb < nkb; kb += 2) {
        uint4 o[4][4];
        pf_gather_f16(fb, kb, g, o);
        put(kb, o);
      }
      break;
    default:
      if (threadIdx.x == 0) atomicExch(L.err, kErrBits);
  }
}

cudaError_t launch_prefill_dump(const DevLayer& L, int e, int m, __half* out, cudaStream_t s) {
  const int R = m < 2 ? L.f : L.d;
  size_t smem = 0;
  cudaError_t err = window_smem((const void*)prefill_dump_kernel, Pf<2>::TAB_AT + 32 * 1024, smem);
  if (err != cudaSuccess) return err;
  prefill_dump_kernel<<<(R + PF_BM - 1) / PF_BM, 128, smem, s>>>(L, e, m, out);
  return cudaGetLastError();
}

static int env_tokens(const char* name, int dflt) {
  const char* s = getenv(name);
  const int v = s ? atoi(s) : dflt;
  // the persistent decode kernels track at most kSyncChunks chunks of 16 tokens per group
  return v < 0 ? 0 : v > kSyncChunks * 16 ? kSyncChunks * 16 : v;
}

// Routed experts with more tokens than this use the tensor-core GEMM (read per
// call).  Wide experts (ffn >= 4096: at least 32 row tiles of 128 per matrix)
// fill the GPU with GEMM tiles from 33 tokens on -- once the batch gives the
// experts more than 32 tokens on average; at up to 32 on average the few
// experts above 32 stay on the decode kernel up to 64 tokens, and a batch
// that no expert can push past 64 launches no GEMM at all (measured on the
// Mixtral-shaped layer: at 128 tokens 0.129 -> 0.151 of the HBM roofline; at
// 256, where most experts hold 33..90 tokens, 32 stays better, 0.934 against
// 1.161 ms).  Narrow ones in batches of up to 64 tokens stay on the decode
// kernel up to 64 tokens (a lone GEMM expert of a few row tiles would run
// after it, nearly alone on the GPU); in larger batches many experts cross 32
// tokens and their GEMM tiles fill the GPU -- unless the batch spreads over
// 128 experts or more at no more than 32 slots per expert on average, where
// the few that cross are too few to: those stay on the decode kernel up to
// 128 tokens (measured on the 128-expert layer: at 128 tokens 0.124 -> 0.151
// of the HBM roofline; at 8192, where most experts are large, 32 stays
// better, 0.271 against 0.259 of the bf16 peak).
int decode_max_tokens(int ffn, int T, int E, int K) {
  const bool sparse = (long long)T * K <= 32LL * E;  // at most 32 slots per expert on average
  const int thr = ffn >= 4096 ? (sparse ? 64 : 32) : T <= 64 ? 64 : (E >= 128 && sparse) ? 128 : 32;
  return env_tokens("PW_DECODE_MAX_TOK", thr);
}

// The shared FFN (every token of the batch) uses the tensor-core GEMM above this batch size.
int decode_max_tokens_shared() { return env_tokens("PW_DECODE_MAX_TOK_SHARED", 256); }

namespace {
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once.
EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}
}  // namespace

cudaError_t launch_prefill(const DevLayer& L, int mode, int phase, const __half* act, const int* offsets,
                           int n_slots, int min_tokens, __half* h, float* y, cudaStream_t s) {
  PfParams Q;
  Q.L = L;
  Q.mode = mode;
  Q.act = act;
  Q.offsets = offsets;
  Q.n_slots = n_slots;
  Q.min_tokens = min_tokens;
  Q.h = h;
  Q.y = y;
  // activation tensor [n_slots][K] fp16, boxes of 64 columns x 256 rows, 128-byte swizzle
  const int fe = mode == 0 ? L.f : L.fs;
  const int K = phase == 0 ? L.d : fe;
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)n_slots};
  const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)PF_BK, (cuuint32_t)PF_BN};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(act), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int grid = sm_count();
  cudaError_t e;
  if (phase == 0) {
    size_t smem = 0;
    e = window_smem((const void*)ffn_prefill_kernel<2>, Pf<2>::END, smem);
    if (e != cudaSuccess) return e;
    ffn_prefill_kernel<2><<<grid, Pf<2>::THREADS, smem, s>>>(Q, map);
  } else {
    e = ensure_smem((const void*)ffn_prefill_kernel<1>, Pf<1>::SMEM);
    if (e != cudaSuccess) return e;
    ffn_prefill_kernel<1><<<grid, Pf<1>::THREADS, Pf<1>::SMEM, s>>>(Q, map);
  }
  return cudaGetLastError();
}

}  // namespace pw
