// Router top-K, stable permutation, weighted combine and the bitwidth write.
//
// Routing and the combine are the standard MoE gate around PagedWeight's
// experts (write-up zhichai.net/topic/178446964, "三层感知" names the router's
// per-expert routing statistics); the permutation groups the (token, k) slots
// by expert so each expert streams its planes once per batch.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "pw_device.cuh"
#include "pw_route.cuh"

namespace pw {

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

cudaError_t ensure_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[std::make_pair(kernel, dev)];
  if (have >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

cudaError_t window_smem(const void* kernel, uint32_t end, size_t& bytes) {
  static std::mutex mu;
  static std::map<const void*, size_t> known;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(kernel);
    if (it != known.end()) {
      bytes = it->second;
      return ensure_smem(kernel, bytes);
    }
  }
  cudaFuncAttributes fa{};
  int dev = 0, rsv = 0;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e != cudaSuccess) return e;
  bytes = (size_t)end + 128 - (size_t)rsv - fa.sharedSizeBytes;
  {
    std::lock_guard<std::mutex> lock(mu);
    known[kernel] = bytes;
  }
  return ensure_smem(kernel, bytes);
}

// ---------------------------------------------------------------------------
// bitwidth word (the stream-ordered commit of a precision change)
// ---------------------------------------------------------------------------

__global__ void set_bits_kernel(int* bits, int e, int b) { bits[e] = b; }

// Word j of canary i holds 0xC0DE0000 | i << 8 | j.
__global__ void canary_kernel(char* ws, Canaries c, int* err, bool fill) {
  const int i = blockIdx.x, j = threadIdx.x;
  if (i >= c.n || j >= kCanaryBytes / 4) return;
  uint32_t* w = reinterpret_cast<uint32_t*>(ws + c.off[i]) + j;
  const uint32_t v = 0xC0DE0000u | (uint32_t)i << 8 | (uint32_t)j;
  if (fill) *w = v;
  else if (*w != v) atomicExch(err, kErrCanary);
}

cudaError_t launch_canaries(char* ws, const Canaries& c, int* err, bool fill, cudaStream_t s) {
  if (c.n <= 0) return cudaSuccess;
  canary_kernel<<<c.n, kCanaryBytes / 4, 0, s>>>(ws, c, err, fill);
  return cudaGetLastError();
}

cudaError_t launch_set_bits(int* bits, int e, int b, cudaStream_t s) {
  set_bits_kernel<<<1, 1, 0, s>>>(bits, e, b);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// router: logits, softmax over E, top-K (ties to the lower index)
// ---------------------------------------------------------------------------

constexpr int kRouteThreads = 512;

template <int kRouteTok>  // tokens per CTA
__global__ void __launch_bounds__(kRouteThreads) route_kernel(DevLayer L, const __half* __restrict__ x,
                                                              const __half* __restrict__ wr,
                                                              const float* __restrict__ bias, int T,
                                                              int* __restrict__ idx, float* __restrict__ wout,
                                                              int* __restrict__ counts) {
  extern __shared__ uint4 smem_route[];
  const int d = L.d, E = L.E, K = L.K;
  const int d8 = d / 8;
  uint4* xs = smem_route;                                         // [kRouteTok][d/8]
  float* logit = reinterpret_cast<float*>(xs + kRouteTok * d8);   // [kRouteTok][E]
  const int t0 = blockIdx.x * kRouteTok;
  const int nt = min(kRouteTok, T - t0);
  const uint4* x4 = reinterpret_cast<const uint4*>(x) + (size_t)t0 * d8;
  for (int i = threadIdx.x; i < nt * d8; i += blockDim.x) xs[i] = x4[i];
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work unit = (four experts, one 1024-column slice of d), order of the sums
  // in pw_route.cuh: a lane loads its four 16-byte pieces of the four W_r rows
  // at once (one memory round trip per unit) and the warps share the units.
  const int ns = route_slices(d);
  const int nb = (E + kRouteEB - 1) / kRouteEB;
  float* part = logit + kRouteTok * E;  // [ns][kRouteTok][E]
  for (int u = warp; u < nb * ns; u += kRouteThreads / 32) {
    const int e0 = (u / ns) * kRouteEB, sl = u % ns;
    uint4 wv[kRouteEB][kRoutePieces];
    route_load_w(wr, d8, E, e0, sl, lane, wv);
    float acc[kRouteEB][kRouteTok];
#pragma unroll
    for (int q = 0; q < kRouteEB; ++q)
#pragma unroll
      for (int t = 0; t < kRouteTok; ++t) acc[q][t] = 0.f;
#pragma unroll
    for (int i = 0; i < kRoutePieces; ++i) {
      const int c = (sl * kRoutePieces + i) * 32 + lane;
      if (c < d8) {
#pragma unroll
        for (int t = 0; t < kRouteTok; ++t) {
          if (t < nt) {
            const uint4 xv = xs[t * d8 + c];
#pragma unroll
            for (int q = 0; q < kRouteEB; ++q) acc[q][t] += dot8(wv[q][i], xv);
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRouteEB; ++q)
#pragma unroll
      for (int t = 0; t < kRouteTok; ++t) {
        const float v = route_warp_sum(acc[q][t]);
        if (lane == 0 && t < nt && e0 + q < E) part[((size_t)sl * kRouteTok + t) * E + e0 + q] = v;
      }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nt * E; i += kRouteThreads) {
    const int t = i / E, e = i % E;
    float v = bias ? bias[e] : 0.f;
    for (int sl = 0; sl < ns; ++sl) v += part[((size_t)sl * kRouteTok + t) * E + e];
    logit[t * E + e] = v;
  }
  __syncthreads();

  if (warp < nt) {
    const int t = t0 + warp;
    route_select(logit + warp * E, E, K, L.renorm, idx + (size_t)t * K, wout + (size_t)t * K, counts);
  }
}

template <int TPC>
static cudaError_t launch_route_tpc(const DevLayer& L, const __half* x, const __half* wr, const float* bias, int T,
                                   int* idx, float* w, int* counts, cudaStream_t s) {
  const int ns = route_slices(L.d);
  const size_t smem = (size_t)TPC * L.d * sizeof(__half) + (size_t)(1 + ns) * TPC * L.E * sizeof(float);
  cudaError_t e = ensure_smem((const void*)route_kernel<TPC>, smem);
  if (e != cudaSuccess) return e;
  route_kernel<TPC><<<(T + TPC - 1) / TPC, kRouteThreads, smem, s>>>(L, x, wr, bias, T, idx, w, counts);
  return cudaGetLastError();
}

cudaError_t launch_route(const DevLayer& L, const __half* x, const __half* wr, const float* bias, int T, int* idx,
                         float* w, int* counts, cudaStream_t s) {
  // small batches: one token per CTA so the router's weight rows are read by
  // many SMs in parallel; large batches: eight tokens per CTA to reuse them
  const int per_sm = T / sm_count();
  if (per_sm < 2) return launch_route_tpc<1>(L, x, wr, bias, T, idx, w, counts, s);
  if (per_sm < 8) return launch_route_tpc<2>(L, x, wr, bias, T, idx, w, counts, s);
  if (per_sm < 32) return launch_route_tpc<4>(L, x, wr, bias, T, idx, w, counts, s);
  return launch_route_tpc<8>(L, x, wr, bias, T, idx, w, counts, s);
}

// ---------------------------------------------------------------------------
// stable permutation: per-chunk histograms, then ranked scatter
// ---------------------------------------------------------------------------

constexpr int kPermChunk = 1024;
constexpr int kPermThreads = 256;

size_t permute_ws_bytes(int S, int E) {
  const int nblk = (S + kPermChunk - 1) / kPermChunk;
  return (size_t)(nblk > 0 ? nblk : 1) * E * sizeof(int);
}

__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(DevLayer L, const int* __restrict__ idx, int S,
                                                                 int* __restrict__ hist) {
  __shared__ int h[kMaxExperts];
  const int E = L.E;
  for (int i = threadIdx.x; i < E; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * kPermChunk, s1 = min(S, s0 + kPermChunk);
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    const int e = idx[s];
    if ((unsigned)e < (unsigned)E)
      atomicAdd(&h[e], 1);
    else
      atomicExch(L.err, kErrRouting);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[blockIdx.x * E + i] = h[i];
}

__global__ void __launch_bounds__(kPermThreads) perm_scatter_kernel(DevLayer L, const int* __restrict__ idx, int S,
                                                                    const int* __restrict__ hist, int nblk,
                                                                    int* __restrict__ offsets,
                                                                    int* __restrict__ perm_src,
                                                                    int* __restrict__ inv_slot) {
  __shared__ int base[kMaxExperts], run[kMaxExperts], scan[kMaxExperts];
  __shared__ int wcnt[kPermThreads / 32][kMaxExperts];
  const int E = L.E, K = L.K, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // bucket starts (exclusive scan of the totals) and this chunk's base per expert;
  // with a single chunk (hist == nullptr) the chunk counts its own slots
  int pre = 0, tot = 0;
  if (hist == nullptr) {
    for (int i = tid; i < E; i += blockDim.x) scan[i] = 0;
    __syncthreads();
    for (int sl = tid; sl < S; sl += blockDim.x) {
      const int e = idx[sl];
      if ((unsigned)e < (unsigned)E) atomicAdd(&scan[e], 1);
      else atomicExch(L.err, kErrRouting);
    }
    __syncthreads();
    if (tid < E) tot = scan[tid];
    __syncthreads();
  } else if (tid < E) {
    for (int c = 0; c < nblk; ++c) {
      const int v = hist[c * E + tid];
      tot += v;
      if (c < (int)blockIdx.x) pre += v;
    }
  }
  if (tid < E) scan[tid] = tot;
  __syncthreads();
  // Hillis-Steele inclusive scan over E <= 256 entries
  for (int o = 1; o < kMaxExperts; o <<= 1) {
    int v = 0;
    if (tid < E && tid >= o) v = scan[tid - o];
    __syncthreads();
    if (tid < E) scan[tid] += v;
    __syncthreads();
  }
  if (tid < E) {
    const int start = scan[tid] - tot;
    base[tid] = start + pre;
    run[tid] = 0;
    if (blockIdx.x == 0) offsets[tid] = start;
  }
  if (blockIdx.x == 0 && tid == 0) offsets[E] = S;
  __syncthreads();

  const int s0 = blockIdx.x * kPermChunk;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < kPermChunk / kPermThreads; ++r) {
    for (int i = tid; i < (kPermThreads / 32) * kMaxExperts; i += kPermThreads) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int slot = s0 + r * kPermThreads + tid;
    const bool valid = slot < S;
    int e = valid ? idx[slot] : -1;
    if ((unsigned)e >= (unsigned)E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int prior = 0;
      for (int w = 0; w < warp; ++w) prior += wcnt[w][e];
      const int pos = base[e] + run[e] + prior + rank;
      perm_src[pos] = slot / K;
      inv_slot[slot] = pos;
    }
    __syncthreads();
    if (tid < E) {
      int add = 0;
      for (int w = 0; w < kPermThreads / 32; ++w) add += wcnt[w][tid];
      run[tid] += add;
    }
    __syncthreads();
  }

}

// x_perm[i] = x[perm_src[i]]: one thread per 16-byte piece.
__global__ void __launch_bounds__(256) perm_gather_kernel(const int* __restrict__ perm_src, int S, int d8,
                                                          const uint4* __restrict__ x, uint4* __restrict__ x_perm) {
  const long long k = (long long)blockIdx.x * 256 + threadIdx.x;
  if (k >= (long long)S * d8) return;
  const int i = (int)(k / d8), c = (int)(k % d8);
  x_perm[(size_t)i * d8 + c] = x[(size_t)perm_src[i] * d8 + c];
}

cudaError_t launch_permute(const DevLayer& L, const int* idx, int T, const __half* x, int* offsets, int* perm_src,
                           int* inv_slot, __half* x_perm, int* hist_ws, cudaStream_t s) {
  const int S = T * L.K;
  if (S == 0) {
    cudaError_t e = cudaMemsetAsync(offsets, 0, sizeof(int) * (L.E + 1), s);
    return e;
  }
  const int nblk = (S + kPermChunk - 1) / kPermChunk;
  if (nblk == 1) {
    perm_scatter_kernel<<<1, kPermThreads, 0, s>>>(L, idx, S, nullptr, 1, offsets, perm_src, inv_slot);
  } else {
    perm_hist_kernel<<<nblk, kPermThreads, 0, s>>>(L, idx, S, hist_ws);
    perm_scatter_kernel<<<nblk, kPermThreads, 0, s>>>(L, idx, S, hist_ws, nblk, offsets, perm_src, inv_slot);
  }
  if (x_perm) {
    const long long pieces = (long long)S * (L.d / 8);
    perm_gather_kernel<<<(unsigned)((pieces + 255) / 256), 256, 0, s>>>(
        perm_src, S, L.d / 8, reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(x_perm));
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// weighted combine: y[t] = sum_k w[t,k] y_perm[inv_slot[t*K+k]] (+ y_shared[t])
// ---------------------------------------------------------------------------

constexpr int kCombThreads = 128;

__global__ void __launch_bounds__(kCombThreads) combine_kernel(DevLayer L, const float* __restrict__ y_perm,
                                                               const int* __restrict__ inv_slot,
                                                               const float* __restrict__ w, int T,
                                                               const float* __restrict__ y_shared,
                                                               __half* __restrict__ y) {
  const int t = blockIdx.x;
  const int d = L.d, K = L.K;
  const int c4 = blockIdx.y * kCombThreads + threadIdx.x;  // float4 column index
  if (c4 * 4 >= d) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < K; ++k) {
    const float wk = w[(size_t)t * K + k];
    int slot = inv_slot[(size_t)t * K + k];
    if ((unsigned)slot >= (unsigned)(T * K)) {  // not a slot of this batch: flagged, read slot 0
      atomicExch(L.err, kErrOffsets);
      slot = 0;
    }
    const float4 v = reinterpret_cast<const float4*>(y_perm + (size_t)slot * d)[c4];
    acc.x = fmaf(wk, v.x, acc.x);
    acc.y = fmaf(wk, v.y, acc.y);
    acc.z = fmaf(wk, v.z, acc.z);
    acc.w = fmaf(wk, v.w, acc.w);
  }
  if (y_shared) {
    const float4 v = reinterpret_cast<const float4*>(y_shared + (size_t)t * d)[c4];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
  uint2 out;
  out.x = *reinterpret_cast<uint32_t*>(&lo);
  out.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(y + (size_t)t * d)[c4] = out;
}

cudaError_t launch_combine(const DevLayer& L, const float* y_perm, const int* inv_slot, const float* w, int T,
                           const float* y_shared, __half* y, cudaStream_t s) {
  const dim3 grid(T, (L.d / 4 + kCombThreads - 1) / kCombThreads);
  combine_kernel<<<grid, kCombThreads, 0, s>>>(L, y_perm, inv_slot, w, T, y_shared, y);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// planner signals: routing mass and prompt residual per expert (write-up
// "内存的饥饿游戏", section 三层感知: routing statistics and the
// routing-weighted input norm)
// ---------------------------------------------------------------------------

constexpr int kStatThreads = 256;

// ||x[t]||_2 for every token, one warp per token; lanes add strided
// 8-element pieces, then a fixed butterfly: deterministic.
__global__ void __launch_bounds__(kStatThreads) token_norm_kernel(const __half* __restrict__ x, int T, int d,
                                                                 float* __restrict__ norms) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kStatThreads / 32) + warp;
  if (t >= T) return;
  const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  float acc = 0.f;
  for (int j = lane; j < d / 8; j += 32) {
    const uint4 v = row[j];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      acc = fmaf(f.x, f.x, acc);
      acc = fmaf(f.y, f.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) norms[t] = sqrtf(acc);
}

// One CTA per expert: thread i adds the slots i, i + 256, ... routed to the
// expert, then the CTA sums the threads in a fixed tree.
__global__ void __launch_bounds__(kStatThreads) expert_stats_kernel(const int* __restrict__ idx,
                                                                   const float* __restrict__ w,
                                                                   const float* __restrict__ norms, int S, int K,
                                                                   float* __restrict__ mass,
                                                                   float* __restrict__ resid) {
  __shared__ float sm[kStatThreads / 32], sr[kStatThreads / 32];
  const int e = blockIdx.x;
  float m = 0.f, r = 0.f;
  for (int i = threadIdx.x; i < S; i += kStatThreads) {
    if (idx[i] == e) {
      const float wi = w[i];
      m += wi;
      r = fmaf(wi, norms[i / K], r);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m += __shfl_xor_sync(0xffffffffu, m, o);
    r += __shfl_xor_sync(0xffffffffu, r, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[warp] = m;
    sr[warp] = r;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tm = 0.f, tr = 0.f;
    for (int k = 0; k < kStatThreads / 32; ++k) {
      tm += sm[k];
      tr += sr[k];
    }
    mass[e] = tm;
    resid[e] = tr;
  }
}

cudaError_t launch_route_stats(const DevLayer& L, const __half* x, const int* idx, const float* w, int T,
                               float* mass, float* resid, float* norms, cudaStream_t s) {
  if (T > 0) {
    token_norm_kernel<<<(T + kStatThreads / 32 - 1) / (kStatThreads / 32), kStatThreads, 0, s>>>(x, T, L.d, norms);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  expert_stats_kernel<<<L.E, kStatThreads, 0, s>>>(idx, w, norms, T * L.K, L.K, mass, resid);
  return cudaGetLastError();
}

}  // namespace pw
