// Grouped expert SwiGLU FFN for decode-sized batches, reading bit-planes
// through the per-expert page table.
//
// PagedWeight (zhichai.net/topic/178446964, "核心洞察"): each expert weight is
// an any-precision code stored as bit-planes plus a LUT; at bitwidth b only the
// top b planes exist for the kernel, so bytes read scale with b/16 of fp16.
//
// Work item = (expert, 32-token chunk, 16-row tile of the output).  A CTA of 8
// warps splits the reduction dimension into groups of four 64-column chunks;
// each lane loads one 16-byte word run per plane per group (coalesced, read
// once), turns the planes into codes with masks and rotations, looks the codes
// up in a per-lane copy of the tile's LUT in shared memory, and feeds the fp16
// weights straight into mma.sync m16n8k16 (weights as A, tokens as B).  Phase
// 0 computes gate and up for the same rows and writes h = silu(g) * u (fp16);
// phase 1 computes down and writes y (fp32).  The item list is derived on the
// device from the expert offsets, so no host synchronisation is needed.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>

#include "pw_device.cuh"

namespace pw {

constexpr int kFfnThreads = 256;
constexpr int kFfnWarps = kFfnThreads / 32;
constexpr int kTok = 32;            // tokens per work item
constexpr int kNT = kTok / 8;       // mma n-tiles per item
constexpr int kTabBytes = 64 * 256; // LUT table of one matrix at b <= 6

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

template <int NM>
__device__ __forceinline__ void store_partials(float* red, int warp, int lane, const float (&acc)[NM][kNT][4]) {
#pragma unroll
  for (int mi = 0; mi < NM; ++mi)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
      reinterpret_cast<float4*>(red)[((warp * NM + mi) * kNT + nt) * 32 + lane] =
          make_float4(acc[mi][nt][0], acc[mi][nt][1], acc[mi][nt][2], acc[mi][nt][3]);
}

// Main loop of one item for a bit-plane expert at bitwidth B.
template <int B, int NM>
__device__ __forceinline__ void item_planes(const FfnParams& P, const char* const* s_base, uint32_t tab0, int K,
                                            const int (&rowoff)[kNT], int NT, float (&acc)[NM][kNT][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / 64, G = nk / 4, rem = nk % 4, NG = G + (rem ? 1 : 0);
  const uint32_t lb0 = lane * 4, lb1 = 128 + lane * 4;
  const __half* act = P.act;
  for (int gamma = warp; gamma < NG; gamma += kFfnWarps) {
    uint32_t wv[NM][B][4];
    const bool full = gamma < G;
    const int nch = full ? 4 : rem;
    if (full) {
      const size_t off = (size_t)(gamma * 128 + lane * 4) * 4;
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int p = 0; p < B; ++p) {
          const uint4 v = ldg_stream(s_base[mi * kPlanes + p] + off);
          wv[mi][p][0] = v.x;
          wv[mi][p][1] = v.y;
          wv[mi][p][2] = v.z;
          wv[mi][p][3] = v.w;
        }
    } else {
      const size_t off = (size_t)(G * 128 + lane * rem) * 4;
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int p = 0; p < B; ++p)
#pragma unroll
          for (int i = 0; i < 4; ++i) wv[mi][p][i] = i < rem ? ldg_stream32(s_base[mi * kPlanes + p] + off + 4 * i) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i >= nch) break;
      const int kappa = 4 * gamma + i;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int col = kappa * 64 + s * 16;
        uint32_t bf[kNT][2];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          if (nt < NT) {
            const __half* xp = act + rowoff[nt] + col;
            bf[nt][0] = *reinterpret_cast<const uint32_t*>(xp);
            bf[nt][1] = *reinterpret_cast<const uint32_t*>(xp + 8);
          }
        }
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          uint32_t w[B];
#pragma unroll
          for (int p = 0; p < B; ++p) w[p] = wv[mi][p][i];
          uint32_t a[4];
          decode_step_lut<B>(w, s, tab0 + mi * kTabBytes, lb0, lb1, a);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
            if (nt < NT) mma16816(acc[mi][nt], a, bf[nt][0], bf[nt][1]);
        }
      }
    }
  }
}

// Main loop of one item for fp16 weights (fallback pages or the shared FFN).
template <int NM>
__device__ __forceinline__ void item_f16(const FfnParams& P, const char* const* s_base16, int K,
                                         const int (&rowoff)[kNT], int NT, float (&acc)[NM][kNT][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / 64;
  const __half* act = P.act;
  // chunks are split across warps in the same groups of four as the planes
  const int G = nk / 4, rem = nk % 4, NG = G + (rem ? 1 : 0);
  for (int gamma = warp; gamma < NG; gamma += kFfnWarps) {
    const int nch = gamma < G ? 4 : rem;
    for (int i = 0; i < nch; ++i) {
      const int kappa = 4 * gamma + i;
      uint4 A[NM][4];
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int s = 0; s < 4; ++s)
          A[mi][s] = ldg_stream(s_base16[mi] + ((size_t)(kappa * 4 + s) * 32 + lane) * 16);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int col = kappa * 64 + s * 16;
        uint32_t bf[kNT][2];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          if (nt < NT) {
            const __half* xp = act + rowoff[nt] + col;
            bf[nt][0] = *reinterpret_cast<const uint32_t*>(xp);
            bf[nt][1] = *reinterpret_cast<const uint32_t*>(xp + 8);
          }
        }
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          const uint32_t a[4] = {A[mi][s].x, A[mi][s].y, A[mi][s].z, A[mi][s].w};
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
            if (nt < NT) mma16816(acc[mi][nt], a, bf[nt][0], bf[nt][1]);
        }
      }
    }
  }
}

template <int NM>
__global__ void __launch_bounds__(kFfnThreads, 2) ffn_decode_kernel(FfnParams P) {
  extern __shared__ __align__(16) unsigned char smem_ffn[];
  __shared__ int s_pref[kMaxExperts + 1];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_bits[kMaxExperts];
  __shared__ const char* s_base[NM * kPlanes];
  __shared__ const char* s_base16[NM];

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
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int c = 0;
      if (e < E) {
        const int n = s_off[e + 1] - s_off[e];
        c = n <= P.max_tokens ? ((n + kTok - 1) / kTok) * tiles : 0;
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

  float* red = reinterpret_cast<float*>(smem_ffn + NM * kTabBytes);
  const uint32_t tab0 = smem_u32(smem_ffn);

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int lo = 0, hi = E;  // find e with s_pref[e] <= item < s_pref[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid] <= item) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = item - s_pref[e];
    const int tau = local % tiles, chunk = local / tiles;
    const int slot0 = s_off[e] + chunk * kTok;
    const int ntok = min(kTok, s_off[e + 1] - slot0);
    const int NT = (ntok + 7) >> 3;
    const int b = s_bits[e];

    if (tid < NM * kPlanes) {
      const int mi = tid / kPlanes, p = tid % kPlanes;
      const int m = P.phase == 0 ? mi : 2;
      s_base[tid] = (routed && p < b && b <= 6) ? tile_addr(L, e, m, p, tau) : nullptr;
    }
    if (tid < NM) {
      const int m = P.phase == 0 ? tid : 2;
      if (routed)
        s_base16[tid] = b == 16 ? tile_addr(L, e, m, kPlanes, tau) : nullptr;
      else
        s_base16[tid] = reinterpret_cast<const char*>(L.shared16[m]) + (size_t)tau * 32 * K;
    }
    if (b <= 6) {
      for (int mi = 0; mi < NM; ++mi) {
        const int m = P.phase == 0 ? mi : 2;
        uint32_t* tab = reinterpret_cast<uint32_t*>(smem_ffn + mi * kTabBytes);
        const __half* lr = lut_rows(L, e, m, b, tau * kTileRows);
        switch (b) {
          case 3: build_lut_table<3>(lr, tab, tid, kFfnThreads); break;
          case 4: build_lut_table<4>(lr, tab, tid, kFfnThreads); break;
          case 5: build_lut_table<5>(lr, tab, tid, kFfnThreads); break;
          default: build_lut_table<6>(lr, tab, tid, kFfnThreads); break;
        }
      }
    }
    __syncthreads();

    // B-fragment row offsets: token n = nt*8 + g (clamped into the item), column 2t
    int rowoff[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int tok = min(nt * 8 + (lane >> 2), ntok - 1);
      rowoff[nt] = (slot0 + tok) * K + 2 * (lane & 3);
    }
    float acc[NM][kNT][4];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mi][nt][r] = 0.f;

    switch (b) {
      case 3: item_planes<3, NM>(P, s_base, tab0, K, rowoff, NT, acc); break;
      case 4: item_planes<4, NM>(P, s_base, tab0, K, rowoff, NT, acc); break;
      case 5: item_planes<5, NM>(P, s_base, tab0, K, rowoff, NT, acc); break;
      case 6: item_planes<6, NM>(P, s_base, tab0, K, rowoff, NT, acc); break;
      case 16: item_f16<NM>(P, s_base16, K, rowoff, NT, acc); break;
      default:
        if (tid == 0) atomicExch(L.err, 3);
        break;
    }
    store_partials<NM>(red, warp, lane, acc);
    __syncthreads();

    // cross-warp reduction and epilogue: element (token j, row r) of the tile
    for (int idx = tid; idx < kTok * kTileRows; idx += kFfnThreads) {
      const int j = idx >> 4, r = idx & 15;
      if (j >= ntok) continue;
      const int nt = j >> 3, jj = j & 7;
      const int ln = 4 * (r & 7) + (jj >> 1);
      const int reg = 2 * (r >> 3) + (jj & 1);
      float sum[NM];
#pragma unroll
      for (int mi = 0; mi < NM; ++mi) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kFfnWarps; ++w) v += red[(((w * NM + mi) * kNT + nt) * 32 + ln) * 4 + reg];
        sum[mi] = v;
      }
      const int row = tau * kTileRows + r;
      if (NM == 2) {
        const float hv = silu_f(sum[0]) * sum[NM - 1];
        P.h[(size_t)(slot0 + j) * fe + row] = __float2half_rn(hv);
      } else {
        P.y[(size_t)(slot0 + j) * L.d + row] = sum[0];
      }
    }
    __syncthreads();
  }
}


cudaError_t launch_ffn(const DevLayer& L, int mode, const __half* x, const int* offsets, int n_slots, float* y,
                       __half* h_ws, cudaStream_t s) {
  // Experts with at most `thr` tokens take the mma.sync GEMV path; larger
  // ones the tcgen05 GEMM.  No expert can have more tokens than the batch.
  const int T = mode == 0 ? n_slots / L.K : n_slots;
  const int thr = decode_max_tokens();
  const bool big = T > thr;
  FfnParams P;
  P.L = L;
  P.mode = mode;
  P.offsets = offsets;
  P.n_slots = n_slots;
  P.max_tokens = big ? thr : INT_MAX;
  P.h = h_ws;
  P.y = y;
  const int grid = sm_count() * 2;
  const size_t smem0 = 2 * kTabBytes + (size_t)kFfnWarps * 2 * kNT * 32 * 16;
  const size_t smem1 = 1 * kTabBytes + (size_t)kFfnWarps * 1 * kNT * 32 * 16;
  cudaError_t e = ensure_smem((const void*)ffn_decode_kernel<2>, smem0);
  if (e != cudaSuccess) return e;
  e = ensure_smem((const void*)ffn_decode_kernel<1>, smem1);
  if (e != cudaSuccess) return e;
  P.phase = 0;
  P.act = x;
  ffn_decode_kernel<2><<<grid, kFfnThreads, smem0, s>>>(P);
  if (big) {
    e = launch_prefill(L, mode, 0, x, offsets, n_slots, thr, h_ws, y, s);
    if (e != cudaSuccess) return e;
  }
  P.phase = 1;
  P.act = h_ws;
  ffn_decode_kernel<1><<<grid, kFfnThreads, smem1, s>>>(P);
  if (big) {
    e = launch_prefill(L, mode, 1, h_ws, offsets, n_slots, thr, h_ws, y, s);
    if (e != cudaSuccess) return e;
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
