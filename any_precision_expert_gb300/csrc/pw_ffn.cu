// Grouped expert SwiGLU FFN for decode-sized batches, reading bit-planes
// through the per-expert page table.
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): each expert weight
// is an any-precision code stored as bit-planes plus a LUT; at bitwidth b only
// the top b planes are read, so bytes scale with b/16 of fp16.
//
// Work item = (expert, 32-token chunk, block of `rw` 16-row output tiles).  The
// 8 warps of a CTA cover the block: 8/rw warps per tile split the reduction
// into units (256-column plane groups, or 64-column chunks of fp16 pages) and
// are reduced through shared memory when 8/rw > 1.  Every lane streams its own
// weight words with cp.async into a private ring of shared memory, three units
// ahead of the one it decodes, so a warp keeps several kilobytes in flight
// without spending registers.  Codes are decoded with masks and one rotation
// per four codes; 3-bit codes are looked up with byte permutes from LUT
// registers, 4..6-bit codes in per-lane shared-memory LUT copies; the fp16
// weights feed mma.sync m16n8k16 (weights as A, tokens as B, fp32
// accumulation).  Activations are read through L1 so the warps of a block
// share them.  rw is the largest of 8, 4, 2, 1 that still gives every CTA an
// item (and whose LUT tables fit in 64 KB).  Two kernel classes: b in {3, 16}
// (no tables, two CTAs per SM) and b in {4, 5, 6} (tables).  Phase 0 computes
// gate and up for the same rows and writes h = silu(g) * u (fp16); phase 1
// computes down and writes y (fp32).  Items are derived on the device from the
// expert offsets, so no host synchronisation is needed.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>

#include "pw_gemv.cuh"

namespace pw {

constexpr int kFfnThreads = 256;
constexpr int kFfnWarps = kFfnThreads / 32;
constexpr int kTabBudget = 64 * 1024;  // LUT tables of one item (table class)
constexpr int kTabBytes = 64 * 256;    // LUT table of one 16-row tile of one matrix at b = 6

// Kernel classes: 0 = 3-bit codes (register LUT), 1 = 4, 5, 6 bits (shared-memory
// LUTs), 2 = fp16 pages.  Separate kernels keep each path's registers apart.
__host__ __device__ constexpr bool in_class(int b, int cls) {
  return cls == 0 ? b == 3 : cls == 2 ? b == 16 : (b >= 4 && b <= 6);
}

template <int NM, int CLS>
struct Dec {
  static constexpr int RING = CLS == 1 ? 2 : 3;  // units in flight per lane
  static constexpr int UNIT = CLS == 0 ? NM * 3 * 16 : CLS == 2 ? NM * 4 * 16 : NM * 6 * 16;  // bytes per lane
  static constexpr int WARP_RING = RING * UNIT * 32;
  static constexpr int TABS = CLS == 1 ? kTabBudget : 0;
  static constexpr int RED = kFfnWarps * NM * kNT * 32 * 16;
  static constexpr int RINGS = kFfnWarps * WARP_RING > RED ? kFfnWarps * WARP_RING : RED;
  static constexpr int SMEM = TABS + RINGS;
  static constexpr int MIN_BLOCKS = CLS == 1 ? 1 : 2;
};

struct FfnParams {
  DevLayer L;
  int mode;              // 0: routed experts, 1: shared fp16 FFN
  int phase;             // 0: gate+up -> h, 1: down -> y
  const __half* act;     // phase 0: x rows [slots][d]; phase 1: h rows [slots][fe]
  const int* offsets;    // routed: [E+1]
  int n_slots;
  int max_tokens;        // experts with more tokens are left to the tensor-core GEMM
  __half* h;             // [slots][fe]
  float* y;              // [slots][d]
};

// Largest number of 16-row tiles per item whose LUT tables fit the budget.
__device__ __forceinline__ int rw_cap(int b, int NM) {
  if (b == 3 || b == 16) return 8;
  return min(8, kTabBudget / (NM * (1 << b) * 256));
}

// Per-lane LUT tables (layout of build_lut_table) of the ntl tiles and NM
// matrices of one item, table q = tile * NM + matrix.  Every thread first loads
// its (at most two) 16-byte runs of eight LUT entries, then writes them out, so
// the item pays one global-load latency instead of one per table and entry.
template <int B, int NM>
__device__ __forceinline__ void build_item_tables(const DevLayer& L, int e, int phase, int tile0, int ntl,
                                                  unsigned char* smem, int tid) {
  constexpr int V = 1 << B;
  constexpr int RUNS = V / 8;              // 16-byte runs per LUT row
  constexpr int PER_TABLE = 16 * RUNS;     // runs per 16-row table
  constexpr int MAX_PER_THREAD = (kTabBudget / (V * 256)) * PER_TABLE / kFfnThreads;
  static_assert(MAX_PER_THREAD >= 1 && MAX_PER_THREAD <= 2, "table build sized for two runs per thread");
  const int units = ntl * NM * PER_TABLE;
  uint4 v[MAX_PER_THREAD];
#pragma unroll
  for (int k = 0; k < MAX_PER_THREAD; ++k) {
    const int u = tid + k * kFfnThreads;
    if (u < units) {
      const int q = u / PER_TABLE, w = u % PER_TABLE;
      const int m = phase == 0 ? q % NM : 2;
      const int rg = w / RUNS, v0 = (w % RUNS) * 8;
      const __half* lr = lut_rows(L, e, m, B, (tile0 + q / NM) * kTileRows);
      v[k] = *reinterpret_cast<const uint4*>(lr + rg * V + v0);
    }
  }
#pragma unroll
  for (int k = 0; k < MAX_PER_THREAD; ++k) {
    const int u = tid + k * kFfnThreads;
    if (u < units) {
      const int q = u / PER_TABLE, w = u % PER_TABLE;
      const int rg = w / RUNS, v0 = (w % RUNS) * 8;
      uint4* tab = reinterpret_cast<uint4*>(smem + (size_t)q * V * 256);
      const uint32_t wv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t val = (wv[i >> 1] >> (16 * (i & 1))) & 0xffffu;
        const uint32_t dup = val | (val << 16);
        tab[((v0 + i) * 256 + rg * 16) / 16] = make_uint4(dup, dup, dup, dup);
      }
    }
  }
}

template <int NM, int CLS>
__global__ void __launch_bounds__(kFfnThreads, Dec<NM, CLS>::MIN_BLOCKS) ffn_decode_kernel(FfnParams P) {
  using D = Dec<NM, CLS>;
  extern __shared__ __align__(16) unsigned char smem_ffn[];
  __shared__ int s_pref[kMaxExperts + 1];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_bits[kMaxExperts];
  __shared__ short s_ord[kMaxExperts];  // experts of the class, by bitwidth then index
  __shared__ int s_rw, s_ne;

  const DevLayer& L = P.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool routed = P.mode == 0;
  const int E = routed ? L.E : 1;
  const int fe = routed ? L.f : L.fs;               // FFN width of this call
  const int K = P.phase == 0 ? L.d : fe;            // reduction length
  const int tiles = P.phase == 0 ? fe / kTileRows : L.d / kTileRows;

  if (routed) {
    for (int i = tid; i <= E; i += kFfnThreads) s_off[i] = P.offsets[i];
    for (int i = tid; i < E; i += kFfnThreads) s_bits[i] = L.bits[i];
  } else if (tid == 0) {
    s_off[0] = 0;
    s_off[1] = P.n_slots;
    s_bits[0] = 16;
  }
  __syncthreads();
  if (warp == 0) {
    // items at the largest tile-block size that still feeds every CTA
    auto count = [&](int e, int RW) {
      const int n = s_off[e + 1] - s_off[e];
      if (n == 0 || n > P.max_tokens || !in_class(s_bits[e], CLS)) return 0;
      const int rw = min(RW, rw_cap(s_bits[e], NM));
      return ((n + kTok - 1) / kTok) * ((tiles + rw - 1) / rw);
    };
    int RW = 8;
    for (; RW > 1; RW >>= 1) {
      int tot = 0;
      for (int e = lane; e < E; e += 32) tot += count(e, RW);
#pragma unroll
      for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      if (tot >= (int)gridDim.x) break;
    }
    // experts ordered by bitwidth, so that the CTAs running at the same time
    // mostly execute the decode path of one bitwidth
    int ne = 0;
    for (int b = 3; b <= 16; ++b) {
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool in = e < E && s_bits[e] == b && count(e, RW) > 0;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (in) s_ord[ne + __popc(m & ((1u << lane) - 1))] = (short)e;
        ne += __popc(m);
      }
    }
    int run = 0;
    for (int k0 = 0; k0 < ne; k0 += 32) {
      const int k = k0 + lane;
      const int c = k < ne ? count(s_ord[k], RW) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (k < ne) s_pref[k] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_pref[ne] = run;
      s_ne = ne;
      s_rw = RW;
    }
  }
  __syncthreads();
  const int ne = s_ne;
  const int total = s_pref[ne];
  const int RW = s_rw;

  const uint32_t tab0 = smem_u32(smem_ffn);
  const uint32_t rings = tab0 + D::TABS;
  const uint32_t ring = rings + warp * D::WARP_RING;
  float* red = reinterpret_cast<float*>(smem_ffn + D::TABS);  // aliases the rings after the K loop

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int lo = 0, hi = ne;  // find k with s_pref[k] <= item < s_pref[k+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid] <= item) lo = mid; else hi = mid;
    }
    const int e = s_ord[lo];
    const int b = s_bits[e];
    const int n_e = s_off[e + 1] - s_off[e];
    const int nch = (n_e + kTok - 1) / kTok;
    const int local = item - s_pref[lo];
    // token chunks of one tile block are adjacent, so their weight re-reads hit L2
    const int blk = local / nch, chunk = local % nch;
    const int rw = min(RW, rw_cap(b, NM));
    const int wpt = kFfnWarps / rw;                 // warps per tile
    const int tile0 = blk * rw;
    const int ntl = min(rw, tiles - tile0);         // tiles in this item
    const int jt = warp / wpt, kpart = warp % wpt;  // this warp's tile and reduction part
    const bool active = jt < ntl;
    const int tau = tile0 + (active ? jt : 0);
    const int slot0 = s_off[e] + chunk * kTok;
    const int ntok = min(kTok, s_off[e + 1] - slot0);
    const int NT = (ntok + 7) >> 3;
    const uint32_t tstride = CLS == 1 ? (uint32_t)(1 << b) * 256u : 0u;
    (void)routed;

    if (CLS == 1) {  // per-lane LUT copies of every (tile, matrix) of the item
      switch (b) {
        case 4: build_item_tables<4, NM>(L, e, P.phase, tile0, ntl, smem_ffn, tid); break;
        case 5: build_item_tables<5, NM>(L, e, P.phase, tile0, ntl, smem_ffn, tid); break;
        default: build_item_tables<6, NM>(L, e, P.phase, tile0, ntl, smem_ffn, tid); break;
      }
      __syncthreads();
    }

    float acc[NM][kNT][4];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mi][nt][r] = 0.f;

    if (active) {
      // B-fragment row offsets: token n = nt*8 + g (clamped into the item), column 2t
      int rowoff[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int tok = min(nt * 8 + (lane >> 2), ntok - 1);
        rowoff[nt] = (slot0 + tok) * K + 2 * (lane & 3);
      }
      if constexpr (CLS == 2) {
        const char* b16[NM];
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          const int m = P.phase == 0 ? mi : 2;
          b16[mi] = routed ? tile_addr(L, e, m, kPlanes, tau)
                           : reinterpret_cast<const char*>(L.shared16[m]) + (size_t)tau * 32 * K;
        }
        warp_f16<NM, D::RING>(P.act, b16, K, kpart, wpt, rowoff, NT, ring, acc);
      } else {
        constexpr int PB = CLS == 0 ? 3 : 6;  // plane pointers this class can use
        const char* base[NM][PB];
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          const int m = P.phase == 0 ? mi : 2;
#pragma unroll
          for (int p = 0; p < PB; ++p) base[mi][p] = p < b ? tile_addr(L, e, m, p, tau) : nullptr;
        }
        uint32_t lut3[NM][2][4];
        const uint32_t tab = tab0 + (uint32_t)(jt * NM) * tstride;
        if constexpr (CLS == 0) {
#pragma unroll
          for (int mi = 0; mi < NM; ++mi) {
            const int m = P.phase == 0 ? mi : 2;
            const __half* lr = lut_rows(L, e, m, 3, tau * kTileRows);
            load_lut3(lr + (lane >> 2) * 8, lut3[mi][0]);
            load_lut3(lr + ((lane >> 2) + 8) * 8, lut3[mi][1]);
          }
          warp_planes<3, NM, D::RING, PB>(P.act, base, K, kpart, wpt, rowoff, NT, lut3, tab, tstride, ring, acc);
        } else {
          switch (b) {
            case 4: warp_planes<4, NM, D::RING, PB>(P.act, base, K, kpart, wpt, rowoff, NT, lut3, tab, tstride, ring, acc); break;
            case 5: warp_planes<5, NM, D::RING, PB>(P.act, base, K, kpart, wpt, rowoff, NT, lut3, tab, tstride, ring, acc); break;
            default: warp_planes<6, NM, D::RING, PB>(P.act, base, K, kpart, wpt, rowoff, NT, lut3, tab, tstride, ring, acc); break;
          }
        }
      }
    }

    // epilogue: C fragment (row g / g+8, token nt*8 + 2t + {0,1})
    const int g = lane >> 2, t = lane & 3;
    if (wpt == 1) {
      if (active) {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int j = nt * 8 + 2 * t + (r & 1);
            const int row = tau * kTileRows + g + 8 * (r >> 1);
            if (j < ntok) {
              if (NM == 2)
                P.h[(size_t)(slot0 + j) * fe + row] = __float2half_rn(silu_f(acc[0][nt][r]) * acc[NM - 1][nt][r]);
              else
                P.y[(size_t)(slot0 + j) * L.d + row] = acc[0][nt][r];
            }
          }
      }
    } else {
      __syncthreads();  // every warp is done with its ring
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          reinterpret_cast<float4*>(red)[((warp * NM + mi) * kNT + nt) * 32 + lane] =
              make_float4(acc[mi][nt][0], acc[mi][nt][1], acc[mi][nt][2], acc[mi][nt][3]);
      __syncthreads();
      // element (tile j, token jj, row r): sum the wpt partials of tile j
      for (int idx = tid; idx < ntl * kTok * kTileRows; idx += kFfnThreads) {
        const int jtile = idx / (kTok * kTileRows), rest = idx % (kTok * kTileRows);
        const int jj = rest >> 4, r = rest & 15;
        if (jj >= ntok) continue;
        const int nt = jj >> 3, j8 = jj & 7;
        const int ln = 4 * (r & 7) + (j8 >> 1);
        const int reg = 2 * (r >> 3) + (j8 & 1);
        float sum[NM];
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          float v = 0.f;
          for (int w = jtile * wpt; w < (jtile + 1) * wpt; ++w)
            v += red[(((w * NM + mi) * kNT + nt) * 32 + ln) * 4 + reg];
          sum[mi] = v;
        }
        const int row = (tile0 + jtile) * kTileRows + r;
        if (NM == 2)
          P.h[(size_t)(slot0 + jj) * fe + row] = __float2half_rn(silu_f(sum[0]) * sum[NM - 1]);
        else
          P.y[(size_t)(slot0 + jj) * L.d + row] = sum[0];
      }
    }
    __syncthreads();
  }
}


template <int NM, int CLS>
static cudaError_t launch_decode_class(const FfnParams& P, int grid_per_sm, cudaStream_t s) {
  using D = Dec<NM, CLS>;
  cudaError_t e = ensure_smem((const void*)ffn_decode_kernel<NM, CLS>, D::SMEM);
  if (e != cudaSuccess) return e;
  ffn_decode_kernel<NM, CLS><<<sm_count() * grid_per_sm, kFfnThreads, D::SMEM, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_moe_ffn(const DevLayer& L, const __half* x_perm, const int* offsets, int n_slots, float* y_perm,
                           __half* h, const __half* x_sh, int T, float* y_sh, __half* hs, int class_mask,
                           cudaStream_t s) {
  // Experts with at most `thr` tokens take the decode kernels; larger ones the
  // tcgen05 GEMM.  No expert can have more tokens than the batch, and the
  // shared FFN sees every token.
  const int thr = decode_max_tokens();
  const bool routed = offsets != nullptr && n_slots > 0;
  const bool big = T > thr;
  const bool shared_decode = x_sh != nullptr && T > 0 && !big;
  cudaError_t e;
  if (routed && (class_mask & 2)) {  // 4, 5, 6-bit experts: CTA-level kernel with LUT tables
    FfnParams P;
    P.L = L;
    P.mode = 0;
    P.offsets = offsets;
    P.n_slots = n_slots;
    P.max_tokens = big ? thr : INT_MAX;
    P.h = h;
    P.y = y_perm;
    for (int phase = 0; phase < 2; ++phase) {
      P.phase = phase;
      P.act = phase == 0 ? x_perm : h;
      e = phase == 0 ? launch_decode_class<2, 1>(P, Dec<2, 1>::MIN_BLOCKS, s)
                     : launch_decode_class<1, 1>(P, Dec<1, 1>::MIN_BLOCKS, s);
      if (e != cudaSuccess) return e;
    }
  }
  const int bit_mask = routed ? ((class_mask & 1) ? 1 : 0) | ((class_mask & 4) ? 2 : 0) : 0;
  if (bit_mask || shared_decode) {
    e = launch_uni(L, shared_decode ? x_sh : nullptr, bit_mask ? x_perm : nullptr, bit_mask ? offsets : nullptr, T,
                   bit_mask, big ? thr : T, h, hs, y_perm, y_sh, s);
    if (e != cudaSuccess) return e;
  }
  for (int phase = 0; phase < 2; ++phase) {
    if (routed && big) {
      e = launch_prefill(L, 0, phase, phase == 0 ? x_perm : h, offsets, n_slots, thr, h, y_perm, s);
      if (e != cudaSuccess) return e;
    }
  }
  for (int phase = 0; phase < 2; ++phase) {
    if (x_sh != nullptr && T > 0 && big) {
      e = launch_prefill(L, 1, phase, phase == 0 ? x_sh : hs, nullptr, T, thr, hs, y_sh, s);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// debug: dequantise one matrix of one expert with the production decode path
// ---------------------------------------------------------------------------

template <int B>
__device__ void debug_tile_planes(const DevLayer& L, int e, int m, int tau, int C, uint32_t tab, __half* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = C / 64, G = nk / 4, rem = nk % 4;
  const int g = lane >> 2, t = lane & 3;
  for (int kappa = warp; kappa < nk; kappa += kFfnWarps) {
    const int gamma = kappa / 4, i = kappa % 4;
    const size_t off = gamma < G ? (size_t)(gamma * 128 + lane * 4 + i) * 4 : (size_t)(G * 128 + lane * rem + i) * 4;
    uint32_t w[B];
#pragma unroll
    for (int p = 0; p < B; ++p) w[p] = *reinterpret_cast<const uint32_t*>(tile_addr(L, e, m, p, tau) + off);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4];
      decode_step_lut<B>(w, s, tab, lane * 4, 128 + lane * 4, a);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = tau * 16 + g + 8 * (r & 1);
        const int col = kappa * 64 + s * 16 + 2 * t + 8 * (r >> 1);
        *reinterpret_cast<uint32_t*>(out + (size_t)row * C + col) = a[r];
      }
    }
  }
}

__global__ void __launch_bounds__(kFfnThreads) debug_dequant_kernel(DevLayer L, int e, int m, __half* out) {
  extern __shared__ __align__(16) unsigned char smem_dbg[];
  const int tau = blockIdx.x;
  const int C = m < 2 ? L.d : L.f;
  const int b = L.bits[e];
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem_dbg);
  if (b <= 6) {
    const __half* lr = lut_rows(L, e, m, b, tau * 16);
    switch (b) {
      case 3: build_lut_table<3>(lr, tab, threadIdx.x, kFfnThreads); break;
      case 4: build_lut_table<4>(lr, tab, threadIdx.x, kFfnThreads); break;
      case 5: build_lut_table<5>(lr, tab, threadIdx.x, kFfnThreads); break;
      default: build_lut_table<6>(lr, tab, threadIdx.x, kFfnThreads); break;
    }
  }
  __syncthreads();
  const uint32_t ts = smem_u32(tab);
  switch (b) {
    case 3: debug_tile_planes<3>(L, e, m, tau, C, ts, out); break;
    case 4: debug_tile_planes<4>(L, e, m, tau, C, ts, out); break;
    case 5: debug_tile_planes<5>(L, e, m, tau, C, ts, out); break;
    case 6: debug_tile_planes<6>(L, e, m, tau, C, ts, out); break;
    case 16: {
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      const int g = lane >> 2, t = lane & 3;
      const char* base = tile_addr(L, e, m, kPlanes, tau);
      for (int kappa = warp; kappa < C / 64; kappa += kFfnWarps)
        for (int s = 0; s < 4; ++s) {
          const uint4 A = *reinterpret_cast<const uint4*>(base + ((size_t)(kappa * 4 + s) * 32 + lane) * 16);
          const uint32_t a[4] = {A.x, A.y, A.z, A.w};
          for (int r = 0; r < 4; ++r) {
            const int row = tau * 16 + g + 8 * (r & 1);
            const int col = kappa * 64 + s * 16 + 2 * t + 8 * (r >> 1);
            *reinterpret_cast<uint32_t*>(out + (size_t)row * C + col) = a[r];
          }
        }
      break;
    }
    default:
      if (threadIdx.x == 0) atomicExch(L.err, 3);
  }
}

cudaError_t launch_debug_dequant(const DevLayer& L, int e, int m, __half* out, cudaStream_t s) {
  const int R = m < 2 ? L.f : L.d;
  cudaError_t err = ensure_smem((const void*)debug_dequant_kernel, kTabBytes);
  if (err != cudaSuccess) return err;
  debug_dequant_kernel<<<R / 16, kFfnThreads, kTabBytes, s>>>(L, e, m, out);
  return cudaGetLastError();
}

}  // namespace pw
