// Expert-FFN dispatch of one layer call, and the debug dequantiser.
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): each expert weight
// is an any-precision code stored as bit-planes plus a LUT; at bitwidth b only
// the top b planes are read, so bytes scale with b/16 of fp16.  Experts with
// few tokens (decode) go to the persistent bit-plane GEMV kernel (pw_decode.cu)
// together with the shared FFN; experts with more tokens than the threshold go
// to the tcgen05 grouped GEMM (pw_prefill.cu).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pw_device.cuh"

namespace pw {

constexpr int kDbgThreads = 256;
constexpr int kTabBytes = 64 * 256;  // LUT table of one 16-row tile of one matrix at b = 6

cudaError_t launch_moe_ffn(const DevLayer& L, const __half* x_perm, const int* offsets, int n_slots, float* y_perm,
                           __half* h, const __half* x_sh, int T, float* y_sh, __half* hs, int class_mask,
                           cudaStream_t s) {
  // Experts with at most `thr` tokens take the decode kernels; larger ones the
  // tcgen05 GEMM.  No expert can have more tokens than the batch, and the
  // shared FFN sees every token.
  const int thr = decode_max_tokens(L.f, T, L.E, L.K);
  const bool routed = offsets != nullptr && n_slots > 0;
  const bool big = T > thr;
  const bool shared_decode = x_sh != nullptr && T > 0 && T <= decode_max_tokens_shared();
  cudaError_t e;
  const int bit_mask =
      routed ? ((class_mask & 1) ? 1 : 0) | ((class_mask & 4) ? 2 : 0) | ((class_mask & 2) ? 4 : 0) : 0;
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
    if (x_sh != nullptr && T > 0 && !shared_decode) {
      e = launch_prefill(L, 1, phase, phase == 0 ? x_sh : hs, nullptr, T, 0, hs, y_sh, s);
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
  for (int kappa = warp; kappa < nk; kappa += (kDbgThreads / 32)) {
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

__global__ void __launch_bounds__(kDbgThreads) debug_dequant_kernel(DevLayer L, int e, int m, __half* out) {
  extern __shared__ __align__(16) unsigned char smem_dbg[];
  const int tau = blockIdx.x;
  const int C = m < 2 ? L.d : L.f;
  const int b = L.bits[e];
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem_dbg);
  if (b <= 6) {
    const __half* lr = lut_rows(L, e, m, b, tau * 16);
    switch (b) {
      case 3: build_lut_table<3>(lr, tab, threadIdx.x, kDbgThreads); break;
      case 4: build_lut_table<4>(lr, tab, threadIdx.x, kDbgThreads); break;
      case 5: build_lut_table<5>(lr, tab, threadIdx.x, kDbgThreads); break;
      default: build_lut_table<6>(lr, tab, threadIdx.x, kDbgThreads); break;
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
      for (int kappa = warp; kappa < C / 64; kappa += (kDbgThreads / 32))
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
      if (threadIdx.x == 0) atomicExch(L.err, kErrBits);
  }
}

cudaError_t launch_debug_dequant(const DevLayer& L, int e, int m, __half* out, cudaStream_t s) {
  const int R = m < 2 ? L.f : L.d;
  cudaError_t err = ensure_smem((const void*)debug_dequant_kernel, kTabBytes);
  if (err != cudaSuccess) return err;
  debug_dequant_kernel<<<R / 16, kDbgThreads, kTabBytes, s>>>(L, e, m, out);
  return cudaGetLastError();
}

}  // namespace pw
