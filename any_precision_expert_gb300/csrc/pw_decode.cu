// Persistent decode-side expert FFN: gate/up and down for every routed expert
// with few tokens (3, 4, 5, 6 bits or its fp16 page) and for the fp16 shared
// FFN, in at most two launches (one for 4..6-bit experts, one for the rest).
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): an expert at
// bitwidth b streams only its top b bit-planes, found through the per-expert
// page table, and looks every code up in the row's LUT; a fallback expert
// streams its fp16 page.  Decode batches route a few tokens to each expert, so
// the time goes into streaming weights.
//
// A CTA (four warps) takes one work item at a time and stages the item's
// token rows (up to 32) once into shared memory (K-blocks of 384 columns,
// double-buffered, rows XOR-swizzled for conflict-free ldmatrix).  Weights
// stream through per-warp cp.async rings addressed through the page table.
// Item shapes:
//  - block item (3-bit experts, fp16 pages, shared FFN): (group, phase,
//    32-token chunk, four 16-row tiles), one tile per warp over the whole
//    reduction.  3-bit codes are decoded with byte permutes from register
//    LUTs.
//  - split item (4, 5, 6-bit experts, own launch): (group, phase, 32-token
//    chunk, one tile); warps 0-1 stream gate and 2-3 up (all four for down)
//    over interleaved 128-column units and look codes up in one CTA-wide LUT
//    table (per-lane copies of the row pair g / g+8, so no bank conflicts).
// The weights feed mma.sync m16n8k16 (weights as A, tokens as B, fp32
// accumulation).  Gate/up writes h = silu(g) * u in fp16, down writes y in
// fp32.
//
// CTAs of a launch claim items from one counter in a fixed order: every gate/up item
// (phase 0) before every down item (phase 1); inside a phase the shared FFN
// first, then fp16, 3-bit and 4..6-bit experts.  A down item waits until all
// gate/up tiles of its (group, chunk) are done; those items were claimed
// earlier by running CTAs and never wait, so every wait ends.  The waits are
// bounded anyway: past the limit the kernel records a timeout in the layer's
// error word and carries on.  The phase counters are returned to zero by the
// last down tile of each (group, chunk) and the claim counter by the last CTA
// to leave, so the next launch (or graph replay) starts from zero.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "pw_gemv.cuh"

namespace pw {

constexpr int kCtaThreads = 128;
constexpr int kCtaWarps = kCtaThreads / 32;           // tiles of a block item
constexpr int kTabBytes = 64 * 256;                   // LUT table of a split item (b <= 6, two matrices)
constexpr long long kSpinLimit = 1ll << 22;           // polls of a phase counter (about a second)

// Geometry of the two kernels: items take up to 32 tokens (a weight tile is
// streamed and decoded once for up to 32 tokens).  The 3-bit / fp16 kernel
// stages 256-column K-blocks and runs three CTAs per SM (at most 168
// registers a thread); the 4..6-bit kernel stages 384-column K-blocks, holds
// a LUT table and runs two.
template <bool SPLIT>
struct Geo {
  static constexpr int TOK = 32;                          // tokens per item
  static constexpr int NTM = TOK / 8;                     // mma n-tiles per item
  static constexpr int SCOLS = SPLIT ? 384 : 256;         // columns of one staged K-block
  static constexpr int HALF = TOK * SCOLS * 2;            // bytes of one K-block buffer
  static constexpr int RB = SPLIT ? 10 * 1024 : 9 * 1024;  // cp.async weight ring of one warp
  static constexpr int BLOCKS = SPLIT ? 2 : 3;            // CTAs per SM
  static constexpr int SMEM = 2 * HALF + (SPLIT ? kTabBytes : 0) + kCtaWarps * RB;
};

// Weight units streamed by a warp: one matrix of
//   KIND_F16: one fp16 chunk (64 columns), 4 x 16 B per lane;
//   KIND_PB: half a plane group (2 chunks, 128 columns) of B-bit words, 8 B per lane and plane.
enum { KIND_F16 = 1, KIND_PB = 2 };

template <int KIND, int B, int RB>
struct Unit {
  static constexpr int COLS = KIND == KIND_F16 ? 64 : 128;
  static constexpr int LANE_BYTES = KIND == KIND_F16 ? 4 * 16 : B * 8;
  static constexpr int SLOT = LANE_BYTES * 32;
  static constexpr int R = RB / SLOT > 8 ? 8 : RB / SLOT;  // ring depth
  static_assert(RB / SLOT >= 3, "ring too shallow");
};

struct UniParams {
  DevLayer L;
  const __half* x;     // [T][d] input of the shared FFN, or null (no shared group)
  const __half* xp;    // [n_slots][d] routed input rows, or null (no routed groups)
  const int* offsets;  // [E+1] slot offsets of the experts
  int T;
  int bit_mask;        // routed bitwidths taken: bit 0 -> 3 bits, bit 1 -> fp16 page, bit 2 -> 4..6 bits
  int max_tokens;      // routed experts with more tokens are left to the tensor-core GEMM
  __half* h;           // [n_slots][f]
  __half* hs;          // [T][fs]
  float* y;            // [n_slots][d]
  float* ys;           // [T][d]
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Wait until at most n (clamped to 7) of this thread's newest cp.async groups are pending.
__device__ __forceinline__ void cp_wait_dyn(int n) {
  switch (n < 7 ? n : 7) {
    case 0: cp_wait<0>(); break;
    case 1: cp_wait<1>(); break;
    case 2: cp_wait<2>(); break;
    case 3: cp_wait<3>(); break;
    case 4: cp_wait<4>(); break;
    case 5: cp_wait<5>(); break;
    case 6: cp_wait<6>(); break;
    default: cp_wait<7>(); break;
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte offset of 16-byte piece j (8 columns) of token row r in a staged K-block.
template <class G>
__device__ __forceinline__ uint32_t slab_off(int r, int j) {
  return (uint32_t)(r * (G::SCOLS * 2) + ((j ^ (r & 7)) << 4));
}

// Copy K-block kb of the item's token rows into a slab buffer (all threads).
template <class G>
__device__ __forceinline__ void stage_kblock(const __half* act, const int* s_tok, int rows, int K, int kb,
                                             uint32_t buf) {
  const int c0 = kb * G::SCOLS;
  const int ppr = min(G::SCOLS, K - c0) >> 3;  // 16-byte pieces per row
  const int n = rows * ppr;
  for (int p = threadIdx.x; p < n; p += kCtaThreads) {
    const int r = p / ppr, j = p - r * ppr;
    cp_async16(buf + slab_off<G>(r, j), act + (size_t)s_tok[r] * K + c0 + j * 8);
  }
}

// B fragments of mma step s (16 columns at column kc + 16 s of its K-block)
// for the n-tiles: one ldmatrix.x4 per pair of n-tiles (b0, b1 of each).
// Rows past the item's tokens hold stale data; their n-tiles are not used.
template <class G>
__device__ __forceinline__ void slab_bstep(uint32_t buf, int kc, int s, int NT, uint32_t (&bf)[G::NTM][2]) {
  const int lane = threadIdx.x & 31;
  const int mat = lane >> 3;
  const int j = (kc >> 3) + 2 * s + (mat & 1);
#pragma unroll
  for (int nt0 = 0; nt0 < G::NTM; nt0 += 2) {
    if (nt0 < NT) {
      const int r = (nt0 + (mat >> 1)) * 8 + (lane & 7);
      ldsm_x4(buf + slab_off<G>(r, j), bf[nt0][0], bf[nt0][1], bf[nt0 + 1][0], bf[nt0 + 1][1]);
    }
  }
}

// Decode mma step s of one chunk of B-bit codes into the A fragment through
// the CTA's LUT table: entry (v, matrix m, lane) at byte v*256 + m*128 +
// 4*lane holds LUT[row g][v] in its low and LUT[row g+8][v] in its high half
// (g = lane / 4).  lbm = m*128 + 4*lane.  Plane masking as in decode_step_lut.
template <int B>
__device__ __forceinline__ void decode_step_tab(const uint32_t (&w)[B], const int s, uint32_t tab, uint32_t lbm,
                                                uint32_t (&a)[4]) {
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
    const uint32_t sel = 0x5504u | ((uint32_t)k << 4);
    const uint32_t e0 = lds32(tab + prmt(R[0], lbm, sel));
    const uint32_t e1 = lds32(tab + prmt(R[1], lbm, sel));
    const int reg = (k == 0) ? 0 : (k == 1) ? 2 : (k == 2) ? 1 : 3;
    a[reg] = prmt(e0, e1, (k >> 1) ? 0x7632u : 0x5410u);
  }
}

// LUT table of a split item: both matrices of tile tau at bitwidth B.
template <int B, int NM>
__device__ __forceinline__ void build_tab(const DevLayer& L, int e, int tau, unsigned char* tab) {
  constexpr int V = 1 << B;
  constexpr int RUNS = V / 8;  // 8-entry runs per LUT row
  constexpr int UNITS = NM * 8 * RUNS;
  for (int u = threadIdx.x; u < UNITS; u += kCtaThreads) {
    const int mi = u / (8 * RUNS), g = (u / RUNS) % 8, v0 = (u % RUNS) * 8;
    const __half* lr = lut_rows(L, e, NM == 2 ? mi : 2, B, tau * kTileRows);
    const uint4 lo = *reinterpret_cast<const uint4*>(lr + g * V + v0);
    const uint4 hi = *reinterpret_cast<const uint4*>(lr + (g + 8) * V + v0);
    const uint32_t l4[4] = {lo.x, lo.y, lo.z, lo.w}, h4[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t pair = prmt(l4[i >> 1], h4[i >> 1], (i & 1) ? 0x7632u : 0x5410u);
      *reinterpret_cast<uint4*>(tab + (v0 + i) * 256 + mi * 128 + g * 16) = make_uint4(pair, pair, pair, pair);
    }
  }
}

// Weight sources of one warp's K loop.
template <int NM>
struct WSrc {
  const char* p[NM][6];  // plane tiles (KIND_PB) or the fp16 tile in p[m][0]
  uint32_t lut3[NM][2][4];
};

// K loop of one warp: units u = u0, u0 + ustride, ... of one tile (unit u =
// (column block u / NM, matrix u % NM)).  Every warp of the CTA runs it for
// the same item and passes the same K-block barriers; the token rows of
// K-block kb are staged at the start of K-block kb - 1.
template <class G, int KIND, int B, int NM>
__device__ __forceinline__ void kloop(const WSrc<NM>& src, int K, int NT, int u0, int ustride, uint32_t ring,
                                      uint32_t slab, uint32_t tab, const __half* act, const int* s_tok,
                                      float (&acc)[NM][G::NTM][4]) {
  using U = Unit<KIND, B, G::RB>;
  static_assert(G::SCOLS % U::COLS == 0, "units must not straddle K-blocks");
  constexpr int R = U::R;
  const int lane = threadIdx.x & 31;
  const int rows = NT * 8;
  const int nk = K / 64, GR = nk / 4, rem = nk % 4;
  const int ncb = (K + U::COLS - 1) / U::COLS;  // column blocks
  const int nu = ncb * NM;
  const int mine = u0 < nu ? (nu - u0 + ustride - 1) / ustride : 0;
  const int kbs = (K + G::SCOLS - 1) / G::SCOLS;

  auto issue = [&](int i) {
    const int u = u0 + i * ustride, cb = u / NM, mi = u % NM;
    const uint32_t slot = ring + (i % R) * U::SLOT;
    const char* const* pp = (NM == 1 || mi == 0) ? src.p[0] : src.p[NM - 1];
    if constexpr (KIND == KIND_F16) {
#pragma unroll
      for (int s = 0; s < 4; ++s)
        cp_async16(slot + (s * 32 + lane) * 16, pp[0] + ((size_t)(cb * 4 + s) * 32 + lane) * 16);
    } else {
      const int gamma = cb >> 1, j = cb & 1;
      if (gamma < GR) {
        const size_t off = (size_t)(gamma * 128 + lane * 4 + 2 * j) * 4;
#pragma unroll
        for (int p = 0; p < B; ++p) cp_async8(slot + (p * 32 + lane) * 8, pp[p] + off);
      } else {
        const int cnt = min(2, rem - 2 * j);
        const size_t off = (size_t)(GR * 128 + lane * rem + 2 * j) * 4;
#pragma unroll
        for (int p = 0; p < B; ++p)
          for (int k = 0; k < cnt; ++k) cp_async4(slot + (p * 32 + lane) * 8 + 4 * k, pp[p] + off + 4 * k);
      }
    }
  };

  // K-blocks 0 and 1 go with the first ring group
  stage_kblock<G>(act, s_tok, rows, K, 0, slab);
  if (kbs > 1) stage_kblock<G>(act, s_tok, rows, K, 1, slab + G::HALF);
  int since_stage = 0;  // groups committed after the newest staging group
#pragma unroll
  for (int i = 0; i < R - 1; ++i) {
    if (i < mine) issue(i);
    cp_commit();
    if (i > 0) ++since_stage;
  }
  int kb_cur = -1;
  auto advance_to = [&](int kb) {
    while (kb_cur < kb) {
      ++kb_cur;
      cp_wait_dyn(since_stage);  // this thread's copies of K-block kb_cur have landed
      __syncthreads();           // ... and everyone's; K-block kb_cur - 1 is no longer read
      if (kb_cur >= 1 && kb_cur + 1 < kbs) {
        stage_kblock<G>(act, s_tok, rows, K, kb_cur + 1, slab + ((kb_cur + 1) & 1) * G::HALF);
        cp_commit();
        since_stage = 0;
      }
    }
  };

#pragma unroll 1
  for (int i = 0; i < mine; ++i) {
    if (i + R - 1 < mine) issue(i + R - 1);
    cp_commit();
    ++since_stage;
    const int u = u0 + i * ustride, cb = u / NM, mi = u % NM;
    const int kb = (cb * U::COLS) / G::SCOLS;
    advance_to(kb);
    cp_wait<R - 1>();  // unit i has landed
    const uint32_t buf = slab + (kb & 1) * G::HALF;
    const int kc0 = (cb * U::COLS) % G::SCOLS;
    const uint32_t slot = ring + (i % R) * U::SLOT;
    // the matrix is fixed for the whole unit: branch once, then fully
    // unrolled chunks of independent decode + mma chains
    auto compute = [&](auto tag) {
      constexpr int m = decltype(tag)::value;
      if constexpr (KIND == KIND_F16) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t bf[G::NTM][2];
          slab_bstep<G>(buf, kc0, s, NT, bf);
          const uint4 v = lds128(slot + (s * 32 + lane) * 16);
          const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int nt = 0; nt < G::NTM; ++nt)
            if (nt < NT) mma16816(acc[m][nt], a, bf[nt][0], bf[nt][1]);
        }
      } else {
        uint32_t w[B][2];
#pragma unroll
        for (int p = 0; p < B; ++p) {
          const uint2 v = lds64(slot + (p * 32 + lane) * 8);
          w[p][0] = v.x;
          w[p][1] = v.y;
        }
        const int nch = (cb >> 1) < GR ? 2 : min(2, rem - 2 * (cb & 1));
        auto chunk = [&](int c) {
          uint32_t wc[B];
#pragma unroll
          for (int p = 0; p < B; ++p) wc[p] = c ? w[p][1] : w[p][0];
          // decode the chunk's four steps first (independent chains), then the mma's
          uint32_t a[4][4];
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            if constexpr (B == 3) decode_step_prmt3(wc, s, src.lut3[m], a[s]);
            else decode_step_tab<B>(wc, s, tab, m * 128 + lane * 4, a[s]);
          }
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            uint32_t bf[G::NTM][2];
            slab_bstep<G>(buf, kc0 + c * 64, s, NT, bf);
#pragma unroll
            for (int nt = 0; nt < G::NTM; ++nt)
              if (nt < NT) mma16816(acc[m][nt], a[s], bf[nt][0], bf[nt][1]);
          }
        };
        if constexpr (B == 3) {
          // register-LUT decode is short: both chunks unrolled (eight independent chains)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            if (c < nch) chunk(c);
        } else {
          // table lookups: the two chunks share one copy of the code (instruction-cache footprint)
#pragma unroll 1
          for (int c = 0; c < 2; ++c)
            if (c < nch) chunk(c);
        }
      }
    };
    if (NM == 1 || mi == 0) compute(std::integral_constant<int, 0>{});
    else compute(std::integral_constant<int, NM - 1>{});
  }
  advance_to(kbs - 1);
  cp_wait<0>();
}

// Epilogue of one tile: C fragment element (row g / g+8, token nt*8 + 2t + {0,1}).
template <int NM, int NTM>
__device__ __forceinline__ void tile_store(const float (&acc)[NM][NTM][4], int tau, int row0, int ntok, int ld,
                                           __half* h, float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NTM; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = nt * 8 + 2 * t + (r & 1);
      const int row = tau * kTileRows + g + 8 * (r >> 1);
      if (j < ntok) {
        if constexpr (NM == 2)
          h[(size_t)(row0 + j) * ld + row] = __float2half_rn(silu_f(acc[0][nt][r]) * acc[1][nt][r]);
        else
          y[(size_t)(row0 + j) * ld + row] = acc[0][nt][r];
      }
    }
}

struct ItemArgs {
  const __half* act;  // token rows of this phase
  int e;              // expert (routed)
  bool sh;            // shared FFN
  int K, NT, row0, ntok, ld;
  __half* h;
  float* y;
};

// Block item: warp w computes tile tau + w over the whole reduction.
template <int NM, int B>
__device__ __forceinline__ void block_item(const DevLayer& L, const ItemArgs& A, int tau, uint32_t ring,
                                           uint32_t slab, const int* s_tok) {
  using G = Geo<false>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tau += warp;
  float acc[NM][G::NTM][4] = {};
  WSrc<NM> src;
#pragma unroll
  for (int mi = 0; mi < NM; ++mi) {
    const int m = NM == 2 ? mi : 2;
    if constexpr (B == 16) {
      src.p[mi][0] = A.sh ? reinterpret_cast<const char*>(L.shared16[m]) + (size_t)tau * 32 * A.K
                          : tile_addr(L, A.e, m, kPlanes, tau);
    } else {
#pragma unroll
      for (int p = 0; p < 3; ++p) src.p[mi][p] = tile_addr(L, A.e, m, p, tau);
      const __half* lr = lut_rows(L, A.e, m, 3, tau * kTileRows);
      load_lut3(lr + (lane >> 2) * 8, src.lut3[mi][0]);
      load_lut3(lr + ((lane >> 2) + 8) * 8, src.lut3[mi][1]);
    }
  }
  if constexpr (B == 16) kloop<G, KIND_F16, 16, NM>(src, A.K, A.NT, 0, 1, ring, slab, 0u, A.act, s_tok, acc);
  else kloop<G, KIND_PB, 3, NM>(src, A.K, A.NT, 0, 1, ring, slab, 0u, A.act, s_tok, acc);
  tile_store<NM, G::NTM>(acc, tau, A.row0, A.ntok, A.ld, A.h, A.y);
}

// Split item: the four warps share tile tau.  For gate/up, warps 0-1 stream
// the gate matrix and warps 2-3 the up matrix (interleaved 128-column units),
// so every warp runs the one-matrix loop; partial sums are added in warp order.
template <int NM, int B>
__device__ __forceinline__ void split_item(const DevLayer& L, const ItemArgs& A, int tau, uint32_t ring,
                                           uint32_t slab, unsigned char* tab_ptr, const int* s_tok) {
  using G = Geo<true>;
  constexpr int kNT = G::NTM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  build_tab<B, NM>(L, A.e, tau, tab_ptr);  // ordered before use by the first K-block barrier
  const int mi = NM == 2 ? warp >> 1 : 0;  // this warp's matrix (index into the item's NM)
  float acc[1][kNT][4] = {};
  WSrc<1> src;
#pragma unroll
  for (int p = 0; p < 6; ++p) src.p[0][p] = p < B ? tile_addr(L, A.e, NM == 2 ? mi : 2, p, tau) : nullptr;
  // the LUT table column of this warp's matrix: unit u of the one-matrix loop is matrix 0
  const uint32_t tab = smem_u32(tab_ptr) + mi * 128;
  if (NM == 2) kloop<G, KIND_PB, B, 1>(src, A.K, A.NT, warp & 1, 2, ring, slab, tab, A.act, s_tok, acc);
  else kloop<G, KIND_PB, B, 1>(src, A.K, A.NT, warp, kCtaWarps, ring, slab, tab, A.act, s_tok, acc);
  __syncthreads();  // the staged rows are no longer read
  float4* red = reinterpret_cast<float4*>(__cvta_shared_to_generic(slab));
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
    red[(warp * kNT + nt) * 32 + lane] = make_float4(acc[0][nt][0], acc[0][nt][1], acc[0][nt][2], acc[0][nt][3]);
  __syncthreads();
  if (warp == 0) {
    constexpr int WPM = kCtaWarps / NM;  // warps per matrix
    float sum[NM][kNT][4];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        float4 v = red[((m * WPM) * kNT + nt) * 32 + lane];
#pragma unroll
        for (int w = 1; w < WPM; ++w) {
          const float4 o = red[((m * WPM + w) * kNT + nt) * 32 + lane];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        sum[m][nt][0] = v.x;
        sum[m][nt][1] = v.y;
        sum[m][nt][2] = v.z;
        sum[m][nt][3] = v.w;
      }
    tile_store<NM, kNT>(sum, tau, A.row0, A.ntok, A.ld, A.h, A.y);
  }
}

__device__ __forceinline__ bool is_split(int b) { return b >= 4 && b <= 6; }

// SPLIT = false: block items (3-bit and fp16 experts, shared FFN); SPLIT = true:
// split items (4, 5, 6-bit experts).  Two instantiations keep each set of
// paths in its own register allocation; their groups are disjoint, so they
// share the layer's phase counters and use separate claim counters.
template <bool SPLIT>
__global__ void __launch_bounds__(kCtaThreads, Geo<SPLIT>::BLOCKS) ffn_cta_kernel(UniParams P) {
  using G = Geo<SPLIT>;
  extern __shared__ __align__(128) unsigned char smem_uni[];
  __shared__ int s_base[kMaxExperts + 1];   // first input row of each group
  __shared__ int s_n[kMaxExperts + 1];      // tokens of each group
  __shared__ short s_b[kMaxExperts + 1];    // bitwidth of each group
  __shared__ short s_ord[kMaxExperts + 1];  // groups in claim order
  __shared__ int s_pref[2][kMaxExperts + 2];
  __shared__ int s_ng, s_it;
  __shared__ int s_tok[G::TOK];

  const DevLayer& L = P.L;
  const int E = L.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* const q = L.sync + (SPLIT ? 2 : 0);           // claim counter, CTA exit counter
  int* const done0 = L.sync + kSyncHeader;           // [E+1][kSyncChunks] gate/up tiles done
  int* const done1 = done0 + (E + 1) * kSyncChunks;  // [E+1][kSyncChunks] down tiles done

  for (int g = tid; g <= E; g += kCtaThreads) {
    int base = 0, n = 0, b = 16;
    if (g < E) {
      if (P.offsets) {
        base = P.offsets[g];
        n = P.offsets[g + 1] - base;
        b = L.bits[g];
        const bool take = SPLIT ? is_split(b) && (P.bit_mask & 4)
                                : (b == 3 && (P.bit_mask & 1)) || (b == 16 && (P.bit_mask & 2));
        if (!take || n > P.max_tokens) n = 0;
      }
    } else if (P.x && !SPLIT) {
      n = P.T;
    }
    s_base[g] = base;
    s_n[g] = n;
    s_b[g] = (short)b;
  }
  __syncthreads();
  if (warp == 0) {
    // claim order: shared FFN, fp16 experts, 3-bit experts, 4..6-bit experts
    int ng = 0;
    for (int pass = 0; pass < 4; ++pass) {
      for (int g0 = 0; g0 <= E; g0 += 32) {
        const int g = g0 + lane;
        bool in = false;
        if (g <= E && s_n[g] > 0) {
          const int b = s_b[g];
          in = pass == 0 ? g == E : g == E ? false : pass == 1 ? b == 16 : pass == 2 ? b == 3 : is_split(b);
        }
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (in) s_ord[ng + __popc(m & ((1u << lane) - 1))] = (short)g;
        ng += __popc(m);
      }
    }
    for (int ph = 0; ph < 2; ++ph) {
      int run = 0;
      for (int k0 = 0; k0 < ng; k0 += 32) {
        const int k = k0 + lane;
        int c = 0;
        if (k < ng) {
          const int g = s_ord[k];
          const int fe = g == E ? L.fs : L.f;
          const int tiles = ph == 0 ? fe / kTileRows : L.d / kTileRows;
          const int per_chunk = SPLIT ? tiles : tiles / kCtaWarps;
          c = ((s_n[g] + G::TOK - 1) / G::TOK) * per_chunk;
        }
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (k < ng) s_pref[ph][k] = run + incl - c;
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) s_pref[ph][ng] = run;
    }
    if (lane == 0) s_ng = ng;
  }
  const uint32_t slab = smem_u32(smem_uni);
  unsigned char* const tab_ptr = smem_uni + 2 * G::HALF;  // split items only
  const uint32_t ring = slab + 2 * G::HALF + (SPLIT ? kTabBytes : 0) + warp * G::RB;

  for (;;) {
    if (tid == 0) s_it = atomicAdd(q, 1);
    __syncthreads();  // also: the previous item no longer reads shared memory
    const int ng = s_ng;
    const int total0 = s_pref[0][ng];
    const int it = s_it;
    if (it >= total0 + s_pref[1][ng]) break;
    const int phase = it >= total0 ? 1 : 0;
    const int* pref = s_pref[phase];
    const int li = phase ? it - total0 : it;
    int lo = 0, hi = ng;  // pref[lo] <= li < pref[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pref[mid] <= li) lo = mid; else hi = mid;
    }
    const int g = s_ord[lo];
    const bool sh = g == E;
    const int b = s_b[g];
    const int n = s_n[g];
    const int nch = (n + G::TOK - 1) / G::TOK;
    const int local = li - pref[lo];
    const int blk = local / nch, chunk = local % nch;  // chunks of one tile (block) are claimed together
    const int fe = sh ? L.fs : L.f;
    const int tiles = phase == 0 ? fe / kTileRows : L.d / kTileRows;
    const int sidx = g * kSyncChunks + chunk;

    ItemArgs A;
    A.e = g;
    A.sh = sh;
    A.row0 = s_base[g] + chunk * G::TOK;
    A.ntok = min(G::TOK, n - chunk * G::TOK);
    A.NT = (A.ntok + 7) >> 3;
    A.K = phase == 0 ? L.d : fe;
    A.act = phase == 0 ? (sh ? P.x : P.xp) : (sh ? P.hs : P.h);
    A.ld = phase == 0 ? fe : L.d;
    A.h = sh ? P.hs : P.h;
    A.y = sh ? P.ys : P.y;

    if (tid < G::TOK) s_tok[tid] = A.row0 + min(tid, A.ntok - 1);
    if (phase == 1 && tid == 0) {  // h of this chunk must be complete
      const int need = fe / kTileRows;
      long long spins = 0;
      while (ld_acquire(done0 + sidx) < need) {
        if (++spins > kSpinLimit) {
          atomicExch(L.err, 1);
          break;
        }
        __nanosleep(100);
      }
    }
    __syncthreads();
    if constexpr (SPLIT) {
      const int tau = blk;
      if (phase == 0) {
        switch (b) {
          case 4: split_item<2, 4>(L, A, tau, ring, slab, tab_ptr, s_tok); break;
          case 5: split_item<2, 5>(L, A, tau, ring, slab, tab_ptr, s_tok); break;
          default: split_item<2, 6>(L, A, tau, ring, slab, tab_ptr, s_tok); break;
        }
      } else {
        switch (b) {
          case 4: split_item<1, 4>(L, A, tau, ring, slab, tab_ptr, s_tok); break;
          case 5: split_item<1, 5>(L, A, tau, ring, slab, tab_ptr, s_tok); break;
          default: split_item<1, 6>(L, A, tau, ring, slab, tab_ptr, s_tok); break;
        }
      }
    } else {
      const int tau = blk * kCtaWarps;
      if (phase == 0) {
        if (b == 16) block_item<2, 16>(L, A, tau, ring, slab, s_tok);
        else block_item<2, 3>(L, A, tau, ring, slab, s_tok);
      } else {
        if (b == 16) block_item<1, 16>(L, A, tau, ring, slab, s_tok);
        else block_item<1, 3>(L, A, tau, ring, slab, s_tok);
      }
    }
    __syncthreads();  // every tile of the item is stored
    if (tid == 0) {
      const int done_tiles = SPLIT ? 1 : kCtaWarps;
      __threadfence();
      if (phase == 0) {
        atomicAdd(done0 + sidx, done_tiles);
      } else if (atomicAdd(done1 + sidx, done_tiles) == tiles - done_tiles) {
        // the last down tiles of this (group, chunk) clear both counters
        atomicExch(done0 + sidx, 0);
        atomicExch(done1 + sidx, 0);
      }
    }
  }

  if (tid == 0) {
    __threadfence();
    if (atomicAdd(q + 1, 1) == (int)gridDim.x - 1) {  // last CTA out: no claims remain
      atomicExch(q, 0);
      atomicExch(q + 1, 0);
    }
  }
}

cudaError_t launch_uni(const DevLayer& L, const __half* x, const __half* x_perm, const int* offsets, int T,
                       int bit_mask, int max_tokens, float split_share, __half* h, __half* hs, float* y, float* ys,
                       cudaStream_t s) {
  if (max_tokens > kSyncChunks * 16 || (x && T > kSyncChunks * 16)) return cudaErrorInvalidValue;
  UniParams P;
  P.L = L;
  P.x = x;
  P.xp = x_perm;
  P.offsets = offsets;
  P.T = T;
  P.bit_mask = bit_mask;
  P.max_tokens = max_tokens;
  P.h = h;
  P.hs = hs;
  P.y = y;
  P.ys = ys;
  const bool split = (bit_mask & 4) != 0, block = (bit_mask & 3) || x;
  cudaError_t e;
  // The two kernels have disjoint groups and claim counters.  When the
  // 4..6-bit experts hold a small share of the weight bytes, their kernel runs
  // on the layer's side stream next to the other one (its latency-bound items
  // overlap the weight streaming); when they hold most of the bytes it needs
  // the whole GPU, and the kernels run one after the other.
  const bool fork = split && block && L.side_stream && split_share < 0.3f;
  cudaStream_t ss = fork ? static_cast<cudaStream_t>(L.side_stream) : s;
  if (fork) {
    if ((e = cudaEventRecord(static_cast<cudaEvent_t>(L.ev_fork), s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss, static_cast<cudaEvent_t>(L.ev_fork), 0)) != cudaSuccess) return e;
  }
  if (split) {
    using G = Geo<true>;
    if ((e = ensure_smem((const void*)ffn_cta_kernel<true>, G::SMEM)) != cudaSuccess) return e;
    // side by side: one CTA per SM, so every SM keeps room for a CTA of the
    // other kernel (whose grid fills the rest of the GPU as these CTAs leave)
    const int grid = sm_count() * (fork ? 1 : G::BLOCKS);
    ffn_cta_kernel<true><<<grid, kCtaThreads, G::SMEM, ss>>>(P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (block) {
    using G = Geo<false>;
    if ((e = ensure_smem((const void*)ffn_cta_kernel<false>, G::SMEM)) != cudaSuccess) return e;
    ffn_cta_kernel<false><<<sm_count() * G::BLOCKS, kCtaThreads, G::SMEM, s>>>(P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (fork) {
    if ((e = cudaEventRecord(static_cast<cudaEvent_t>(L.ev_join), ss)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(L.ev_join), 0)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pw
