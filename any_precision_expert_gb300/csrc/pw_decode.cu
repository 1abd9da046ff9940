// Persistent decode-side expert FFN: one launch runs gate/up and down for
// every routed expert at 3 bits or on its fp16 page, and the fp16 shared FFN.
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): an expert at
// bitwidth b streams only its top b bit-planes, found through the per-expert
// page table, and looks every code up in the row's LUT; a fallback expert
// streams its fp16 page.  Decode batches route a few tokens to each expert, so
// the time goes into streaming weights.
//
// Work item = (group, phase, 16-token chunk, block of four 16-row output
// tiles); a group is a routed expert or the shared FFN.  A CTA of four warps
// takes one item: the chunk's activations are staged once into shared memory
// (K-blocks of 1024 columns, double-buffered, XOR-swizzled rows) and each
// warp streams one tile's weights through its own cp.async ring, reading the
// token fragments from the staged block with ldmatrix.  3-bit codes are
// decoded with byte permutes from register LUTs; the fp16 weights feed
// mma.sync m16n8k16 (weights as A, tokens as B, fp32 accumulation).  Gate/up
// writes h = silu(g) * u in fp16, down writes y in fp32.
//
// CTAs claim items from one counter in a fixed order: every gate/up item
// (phase 0) before every down item (phase 1); inside a phase the shared FFN
// first, then fp16 experts, then 3-bit experts (longest items first).  A down
// item waits until all gate/up tiles of its (group, chunk) are done; those
// items were claimed earlier by running CTAs and never wait, so every wait
// ends.  The waits are bounded anyway: past the limit the kernel records a
// timeout in the layer's error word and carries on.  The phase counters are
// returned to zero by the last down block of each (group, chunk) and the
// claim counter by the last CTA to leave, so the next launch (or graph
// replay) starts from zero.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "pw_gemv.cuh"

namespace pw {

constexpr int kCtaThreads = 128;
constexpr int kCtaWarps = kCtaThreads / 32;          // = tiles per item
constexpr int kCtaBlocksPerSm = 2;
constexpr int kSlabCols = 1024;                      // columns of one staged K-block
constexpr int kSlabRows = kTok;                      // token rows of the staged block
constexpr int kSlabHalf = kSlabRows * kSlabCols * 2; // bytes of one K-block buffer
constexpr int kRingBytes = 8 * 1024;                 // cp.async weight ring of one warp
constexpr int kCtaSmem = 2 * kSlabHalf + kCtaWarps * kRingBytes;
constexpr long long kSpinLimit = 1ll << 22;          // polls of a phase counter (about a second)

// Weight units: one matrix of a plane group (4 chunks) of 3-bit words, or one
// matrix of one fp16 chunk.  Ring depth = slots that fit the warp's ring; at
// most one more than the units of a K-block (the staging of the next K-block
// is then complete when its first unit is).
constexpr int kSlot3 = 3 * 32 * 16;
constexpr int kSlot16 = 4 * 32 * 16;
constexpr int kRing3 = kRingBytes / kSlot3 < 5 ? kRingBytes / kSlot3 : 5;
constexpr int kRing16 = kRingBytes / kSlot16;
static_assert(kRing3 >= 2 && kRing16 >= 2, "ring too small");

struct UniParams {
  DevLayer L;
  const __half* x;     // [T][d] input of the shared FFN, or null (no shared group)
  const __half* xp;    // [n_slots][d] routed input rows, or null (no routed groups)
  const int* offsets;  // [E+1] slot offsets of the experts
  int T;
  int bit_mask;        // routed bitwidths taken: bit 0 -> 3 bits, bit 1 -> fp16 page
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

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte offset of 16-byte piece j (8 columns) of token row r in a staged K-block.
__device__ __forceinline__ uint32_t slab_off(int r, int j) {
  return (uint32_t)(r * (kSlabCols * 2) + ((j ^ (r & 7)) << 4));
}

// Copy K-block kb of the item's token rows into a slab buffer (all threads).
__device__ __forceinline__ void stage_kblock(const __half* act, const int* s_tok, int rows, int K, int kb,
                                             uint32_t buf) {
  const int c0 = kb * kSlabCols;
  const int ppr = min(kSlabCols, K - c0) >> 3;  // 16-byte pieces per row
  const int n = rows * ppr;
  for (int p = threadIdx.x; p < n; p += kCtaThreads) {
    const int r = p / ppr, j = p - r * ppr;
    cp_async16(buf + slab_off(r, j), act + (size_t)s_tok[r] * K + c0 + j * 8);
  }
}

// B fragments of one 64-column chunk (column kc of its K-block) for the n-tiles.
__device__ __forceinline__ void slab_bfrag(uint32_t buf, int kc, int NT, uint32_t (&bf)[kNT][4][2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    if (nt < NT) {
      const int r = nt * 8 + (lane & 7);
      const int j0 = (kc >> 3) + (lane >> 3);
      ldsm_x4(buf + slab_off(r, j0), bf[nt][0][0], bf[nt][0][1], bf[nt][1][0], bf[nt][1][1]);
      ldsm_x4(buf + slab_off(r, j0 + 4), bf[nt][2][0], bf[nt][2][1], bf[nt][3][0], bf[nt][3][1]);
    }
  }
}

// Ring-slot wait at unit i, the K-block barrier and the staging of the next
// K-block.  Returns the slab buffer of unit i's K-block.
__device__ __forceinline__ uint32_t kblock_step(int i, int upb, int K, const __half* act, const int* s_tok,
                                                int rows, uint32_t slab) {
  const int kb = i / upb;
  if (i % upb == 0) {
    __syncthreads();  // everyone's copies of K-block kb landed; K-block kb-1 is no longer read
    if (kb >= 1 && (kb + 1) * kSlabCols < K) {
      stage_kblock(act, s_tok, rows, K, kb + 1, slab + ((kb + 1) & 1) * kSlabHalf);
      cp_commit();
    }
  }
  return slab + (kb & 1) * kSlabHalf;
}

// K loop of one warp over 3-bit plane groups: unit u = (group u / NM, matrix u % NM).
template <int NM>
__device__ __forceinline__ void cta_planes3(const char* const (&base)[NM][3], int K, int NT,
                                            const uint32_t (&lut3)[NM][2][4], uint32_t ring, uint32_t slab,
                                            const __half* act, const int* s_tok, int rows,
                                            float (&acc)[NM][kNT][4]) {
  constexpr int R = kRing3;
  const int lane = threadIdx.x & 31;
  const int nk = K / 64, G = nk / 4, rem = nk % 4, NG = G + (rem ? 1 : 0);
  const int nu = NG * NM, upb = (kSlabCols / 256) * NM;
  auto issue = [&](int u) {
    const int gamma = u / NM, mi = u % NM;
    const uint32_t slot = ring + (u % R) * kSlot3;
    const char* bp[3];
#pragma unroll
    for (int p = 0; p < 3; ++p) bp[p] = (NM == 1 || mi == 0) ? base[0][p] : base[NM - 1][p];
    if (gamma < G) {
      const size_t off = (size_t)(gamma * 128 + lane * 4) * 4;
#pragma unroll
      for (int p = 0; p < 3; ++p) cp_async16(slot + (p * 32 + lane) * 16, bp[p] + off);
    } else {
      const size_t off = (size_t)(G * 128 + lane * rem) * 4;
#pragma unroll
      for (int p = 0; p < 3; ++p)
        for (int k = 0; k < rem; ++k) cp_async4(slot + (p * 32 + lane) * 16 + 4 * k, bp[p] + off + 4 * k);
    }
  };
#pragma unroll
  for (int i = 0; i < R - 1; ++i) {
    if (i < nu) issue(i);
    cp_commit();
  }
  for (int i = 0; i < nu; ++i) {
    if (i + R - 1 < nu) issue(i + R - 1);
    cp_commit();
    cp_wait<R - 1>();
    const uint32_t buf = kblock_step(i, upb, K, act, s_tok, rows, slab);
    const int gamma = i / NM, mi = i % NM;
    const uint32_t slot = ring + (i % R) * kSlot3;
    uint32_t w[3][4];
#pragma unroll
    for (int p = 0; p < 3; ++p) {
      const uint4 v = lds128(slot + (p * 32 + lane) * 16);
      w[p][0] = v.x;
      w[p][1] = v.y;
      w[p][2] = v.z;
      w[p][3] = v.w;
    }
    const int nch = gamma < G ? 4 : rem;
    const int kc0 = (gamma % (kSlabCols / 256)) * 256;
    // the matrix is fixed for the whole unit: branch once, then four fully
    // unrolled chunks of independent decode + mma chains
    auto compute = [&](auto tag) {
      constexpr int m = decltype(tag)::value;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c < nch) {
          uint32_t bf[kNT][4][2];
          slab_bfrag(buf, kc0 + c * 64, NT, bf);
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t wc[3] = {w[0][c], w[1][c], w[2][c]};
            uint32_t a[4];
            decode_step_prmt3(wc, s, lut3[m], a);
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
              if (nt < NT) mma16816(acc[m][nt], a, bf[nt][s][0], bf[nt][s][1]);
          }
        }
      }
    };
    if (NM == 1 || mi == 0) compute(std::integral_constant<int, 0>{});
    else compute(std::integral_constant<int, NM - 1>{});
  }
  cp_wait<0>();
}

// K loop of one warp over fp16 chunks: unit u = (chunk u / NM, matrix u % NM).
template <int NM>
__device__ __forceinline__ void cta_f16(const char* const (&b16)[NM], int K, int NT, uint32_t ring, uint32_t slab,
                                        const __half* act, const int* s_tok, int rows, float (&acc)[NM][kNT][4]) {
  constexpr int R = kRing16;
  const int lane = threadIdx.x & 31;
  const int nk = K / 64;
  const int nu = nk * NM, upb = (kSlabCols / 64) * NM;
  auto issue = [&](int u) {
    const int kappa = u / NM, mi = u % NM;
    const uint32_t slot = ring + (u % R) * kSlot16;
#pragma unroll
    for (int s = 0; s < 4; ++s)
      cp_async16(slot + (s * 32 + lane) * 16,
                 ((NM == 1 || mi == 0) ? b16[0] : b16[NM - 1]) + ((size_t)(kappa * 4 + s) * 32 + lane) * 16);
  };
#pragma unroll
  for (int i = 0; i < R - 1; ++i) {
    if (i < nu) issue(i);
    cp_commit();
  }
  uint32_t bf[kNT][4][2];
  for (int i = 0; i < nu; ++i) {
    if (i + R - 1 < nu) issue(i + R - 1);
    cp_commit();
    cp_wait<R - 1>();
    const uint32_t buf = kblock_step(i, upb, K, act, s_tok, rows, slab);
    const int kappa = i / NM, mi = i % NM;
    if (mi == 0) slab_bfrag(buf, (kappa % (kSlabCols / 64)) * 64, NT, bf);
    const uint32_t slot = ring + (i % R) * kSlot16;
    auto compute = [&](auto tag) {
      constexpr int m = decltype(tag)::value;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint4 v = lds128(slot + (s * 32 + lane) * 16);
        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          if (nt < NT) mma16816(acc[m][nt], a, bf[nt][s][0], bf[nt][s][1]);
      }
    };
    if (NM == 1 || mi == 0) compute(std::integral_constant<int, 0>{});
    else compute(std::integral_constant<int, NM - 1>{});
  }
  cp_wait<0>();
}

// Epilogue of one tile: C fragment element (row g / g+8, token nt*8 + 2t + {0,1}).
template <int NM>
__device__ __forceinline__ void tile_store(const float (&acc)[NM][kNT][4], int tau, int row0, int ntok, int ld,
                                           __half* h, float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
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

// One warp's tile of an item.
template <int NM, int B>
__device__ __forceinline__ void cta_tile(const DevLayer& L, const __half* act, int e, bool sh, int tau, int K,
                                         int NT, int row0, int ntok, int ld, __half* h, float* y, uint32_t ring,
                                         uint32_t slab, const int* s_tok) {
  const int lane = threadIdx.x & 31;
  const int rows = NT * 8;
  float acc[NM][kNT][4] = {};
  if constexpr (B == 16) {
    const char* b16[NM];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi) {
      const int m = NM == 2 ? mi : 2;
      b16[mi] = sh ? reinterpret_cast<const char*>(L.shared16[m]) + (size_t)tau * 32 * K
                   : tile_addr(L, e, m, kPlanes, tau);
    }
    cta_f16<NM>(b16, K, NT, ring, slab, act, s_tok, rows, acc);
  } else {
    const char* base[NM][3];
    uint32_t lut3[NM][2][4];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi) {
      const int m = NM == 2 ? mi : 2;
#pragma unroll
      for (int p = 0; p < 3; ++p) base[mi][p] = tile_addr(L, e, m, p, tau);
      const __half* lr = lut_rows(L, e, m, 3, tau * kTileRows);
      load_lut3(lr + (lane >> 2) * 8, lut3[mi][0]);
      load_lut3(lr + ((lane >> 2) + 8) * 8, lut3[mi][1]);
    }
    cta_planes3<NM>(base, K, NT, lut3, ring, slab, act, s_tok, rows, acc);
  }
  tile_store<NM>(acc, tau, row0, ntok, ld, h, y);
}

__global__ void __launch_bounds__(kCtaThreads, kCtaBlocksPerSm) ffn_uni_kernel(UniParams P) {
  extern __shared__ __align__(128) unsigned char smem_uni[];
  __shared__ int s_base[kMaxExperts + 1];  // first input row of each group
  __shared__ int s_n[kMaxExperts + 1];     // tokens of each group
  __shared__ short s_b[kMaxExperts + 1];   // bitwidth of each group
  __shared__ short s_ord[kMaxExperts + 1]; // groups in claim order
  __shared__ int s_pref[2][kMaxExperts + 2];
  __shared__ int s_ng, s_it;
  __shared__ int s_tok[kSlabRows];

  const DevLayer& L = P.L;
  const int E = L.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* const q = L.sync;                              // claim counter, CTA exit counter
  int* const done0 = L.sync + kSyncHeader;            // [E+1][kSyncChunks] gate/up tile blocks done
  int* const done1 = done0 + (E + 1) * kSyncChunks;   // [E+1][kSyncChunks] down tile blocks done

  for (int g = tid; g <= E; g += kCtaThreads) {
    int base = 0, n = 0, b = 16;
    if (g < E) {
      if (P.offsets) {
        base = P.offsets[g];
        n = P.offsets[g + 1] - base;
        b = L.bits[g];
        const bool take = (b == 3 && (P.bit_mask & 1)) || (b == 16 && (P.bit_mask & 2));
        if (!take || n > P.max_tokens) n = 0;
      }
    } else if (P.x) {
      n = P.T;
    }
    s_base[g] = base;
    s_n[g] = n;
    s_b[g] = (short)b;
  }
  __syncthreads();
  if (warp == 0) {
    // claim order: shared FFN, fp16 experts, 3-bit experts
    int ng = 0;
    for (int pass = 0; pass < 3; ++pass) {
      for (int g0 = 0; g0 <= E; g0 += 32) {
        const int g = g0 + lane;
        bool in = false;
        if (g <= E && s_n[g] > 0) in = pass == 0 ? g == E : pass == 1 ? (g < E && s_b[g] == 16) : s_b[g] == 3;
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
          c = ((s_n[g] + kTok - 1) / kTok) * (tiles / kCtaWarps);
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
  const uint32_t ring = slab + 2 * kSlabHalf + warp * kRingBytes;

  for (;;) {
    if (tid == 0) s_it = atomicAdd(q, 1);
    __syncthreads();  // also: the previous item no longer reads the slab or s_tok
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
    const int n = s_n[g];
    const int nch = (n + kTok - 1) / kTok;
    const int local = li - pref[lo];
    const int blk = local / nch, chunk = local % nch;  // chunks of one tile block are claimed together
    const int row0 = s_base[g] + chunk * kTok;
    const int ntok = min(kTok, n - chunk * kTok);
    const int NT = (ntok + 7) >> 3;
    const int fe = sh ? L.fs : L.f;
    const int K = phase == 0 ? L.d : fe;
    const int tiles = phase == 0 ? fe / kTileRows : L.d / kTileRows;
    const int b = s_b[g];
    const int sidx = g * kSyncChunks + chunk;
    const int tau = blk * kCtaWarps + warp;
    const __half* act = phase == 0 ? (sh ? P.x : P.xp) : (sh ? P.hs : P.h);

    if (tid < kSlabRows) s_tok[tid] = row0 + min(tid, ntok - 1);
    if (phase == 1 && tid == 0) {  // h of this chunk must be complete
      const int need = fe / kTileRows / kCtaWarps;
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
    stage_kblock(act, s_tok, NT * 8, K, 0, slab);
    if (K > kSlabCols) stage_kblock(act, s_tok, NT * 8, K, 1, slab + kSlabHalf);
    if (phase == 0) {
      __half* ho = sh ? P.hs : P.h;
      if (b == 16) cta_tile<2, 16>(L, act, g, sh, tau, K, NT, row0, ntok, fe, ho, nullptr, ring, slab, s_tok);
      else cta_tile<2, 3>(L, act, g, sh, tau, K, NT, row0, ntok, fe, ho, nullptr, ring, slab, s_tok);
    } else {
      float* yo = sh ? P.ys : P.y;
      if (b == 16) cta_tile<1, 16>(L, act, g, sh, tau, K, NT, row0, ntok, L.d, nullptr, yo, ring, slab, s_tok);
      else cta_tile<1, 3>(L, act, g, sh, tau, K, NT, row0, ntok, L.d, nullptr, yo, ring, slab, s_tok);
    }
    __syncthreads();  // every tile of the block is stored
    if (tid == 0) {
      __threadfence();
      if (phase == 0) {
        atomicAdd(done0 + sidx, 1);
      } else if (atomicAdd(done1 + sidx, 1) == tiles / kCtaWarps - 1) {
        // the last down block of this (group, chunk) clears both counters
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
                       int bit_mask, int max_tokens, __half* h, __half* hs, float* y, float* ys, cudaStream_t s) {
  if (max_tokens > kSyncChunks * kTok) return cudaErrorInvalidValue;
  if (x && T > kSyncChunks * kTok) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem((const void*)ffn_uni_kernel, kCtaSmem);
  if (e != cudaSuccess) return e;
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
  ffn_uni_kernel<<<sm_count() * kCtaBlocksPerSm, kCtaThreads, kCtaSmem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace pw
