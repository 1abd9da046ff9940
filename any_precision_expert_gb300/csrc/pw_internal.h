// Internal declarations shared by the host runtime and the CUDA kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw.h"

namespace pw {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kPlanes = 6;           // planes of the 6-bit parent code
constexpr int kTileRows = 16;        // rows per stored tile
constexpr int kChunkCols = 64;       // columns per stored chunk
constexpr int kSyncHeader = 32;      // claim and exit counters of the persistent decode kernels
constexpr int kSyncChunks = 64;      // 16-token chunks per group tracked by its phase counters

// Values of a layer's device error word (0 = clear).  A timeout reads back as
// PW_ERR_TIMEOUT, every other value as PW_ERR_DEVICE_CHECK.
constexpr int kErrTimeout = 1;       // a bounded wait gave up
constexpr int kErrRouting = 2;       // an expert index outside [0, E) in a routing result
constexpr int kErrBits = 3;          // a bitwidth word outside {3, 4, 5, 6, 16}
constexpr int kErrOffsets = 4;       // slot offsets not monotone in [0, T*K], or a slot index out of range
constexpr int kErrLayout = 5;        // a kernel's shared-memory window cannot hold its buffer layout
constexpr int kErrCanary = 6;        // a workspace canary changed (a write past a scratch region)

#ifdef __CUDACC__
#define PW_HD __host__ __device__
#else
#define PW_HD
#endif

// 1024-column slices of d in the router's sums (pw_route.cuh).
PW_HD inline int route_slices(int d) { return (d / 8 + 127) / 128; }

// Tokens of a fused layer step (the router runs inside its launch; per-token
// counters live in the sync header).
constexpr int kFusedMaxTokens = 16;

// Words of a layer's sync area: header, then gate/up and down tile counters
// for every (group, chunk), a group being a routed expert or the shared FFN.
inline size_t sync_words(int E) { return kSyncHeader + 2 * (size_t)(E + 1) * kSyncChunks; }

// Per-layer parameter block handed to kernels by value.  All pointers are
// device addresses inside the layer's resident pool run.
struct DevLayer {
  int d, f, E, K, renorm, fs;
  int pmax;      // virtual pages per plane block (expert, plane)
  int pmax16;    // virtual pages per fp16 block (expert)
  int tmax;      // row stride of the tile maps
  const int* bits;                      // [E] current bitwidth
  const unsigned long long* plane_pt;   // [E][6][pmax] page base addresses
  const unsigned long long* f16_pt;     // [E][pmax16]
  const uint2* tmap;                    // [3][tmax] plane tile -> (vpage, byte offset)
  const uint2* tmap16;                  // [3][tmax] fp16 tile -> (vpage, byte offset)
  const unsigned long long* lut_base;   // [E] LUT block of each expert
  unsigned lut_off[3][4];               // byte offset of LUT_b (b = 3 + i) of matrix m
  const __half* shared16[3];            // packed fp16 shared FFN (gate, up, down) or null
  int* err;                             // device error word
  int* sync;                            // [sync_words(E)] zero between launches
  long long spin_limit;                 // polls before a bounded wait of the decode kernel gives up
  int wait_bias;                        // testing: added to the count a down item waits for (0 normally)
  int nblk;                             // decode-kernel configuration for this layer (nblk_for)
};

// Polls of a phase counter before the decode kernel gives up (about a second).
constexpr long long kDefaultSpinPolls = 1ll << 22;

// Scratch carved out of the caller's workspace for one hot-path call.
struct FfnScratch {
  __half* h;        // [n_slots][ffn] fp16 activations between gate/up and down
};

int sm_count();
// Opt a kernel into `bytes` of dynamic shared memory (once per kernel and device).
cudaError_t ensure_smem(const void* kernel, size_t bytes);
// Dynamic shared memory for a kernel whose buffers sit at fixed addresses of
// its CTA's shared-memory window, up to `end`: the dynamic part starts after
// the reserved and static bytes (plus 128 for the base's alignment).
cudaError_t window_smem(const void* kernel, uint32_t end, size_t& bytes);

cudaError_t launch_set_bits(int* bits, int e, int b, cudaStream_t s);
// Workspace canaries (debug bounds): kCanaryBytes after each scratch region,
// filled with a pattern before a call and checked after it.
constexpr int kCanaryBytes = 256;
constexpr int kMaxCanaries = 16;
struct Canaries {
  unsigned long long off[kMaxCanaries];  // byte offsets in the workspace
  int n;
};
// fill: write the pattern; else check it, flagging kErrCanary in err[0] on a difference.
cudaError_t launch_canaries(char* ws, const Canaries& c, int* err, bool fill, cudaStream_t s);
cudaError_t launch_route(const DevLayer& L, const __half* x, const __half* wr, const float* bias,
                         int T, int* idx, float* w, int* counts, cudaStream_t s);
size_t permute_ws_bytes(int S, int E);
cudaError_t launch_permute(const DevLayer& L, const int* idx, int T, const __half* x,
                           int* offsets, int* perm_src, int* inv_slot, __half* x_perm,
                           int* hist_ws, cudaStream_t s);
// Expert FFN of one layer call.  Routed experts over permuted slots when
// offsets is non-null (x_perm, y_perm, h [n_slots][ffn]); the shared fp16 FFN
// over all T tokens when x_sh is non-null (y_sh, hs [T][shared_ffn]).
// class_mask: bit 0 routed 3-bit experts may occur, bit 1 4..6-bit ones, bit 2
// fp16 pages.
cudaError_t launch_moe_ffn(const DevLayer& L, const __half* x_perm, const int* offsets, int n_slots, float* y_perm,
                           __half* h, const __half* x_sh, int T, float* y_sh, __half* hs, int class_mask,
                           cudaStream_t s);
// Persistent decode kernel for routed 3-bit / fp16 / 4..6-bit experts
// (bit_mask bits 0 / 1 / 2) with at most max_tokens tokens and, when x is
// non-null, the shared FFN.
cudaError_t launch_uni(const DevLayer& L, const __half* x, const __half* x_perm, const int* offsets, int T,
                       int bit_mask, int max_tokens, __half* h, __half* hs, float* y, float* ys, cudaStream_t s);
// Fused decode step for T tokens (at most kFusedMaxTokens): the router,
// per-expert offsets from its idx, the expert FFN of every group (routed rows
// staged straight from x) and the shared FFN, then the weighted combine into
// y.  Every expert must be decode-sized (T at most the decode token
// thresholds).
// The router runs in the same launch: idx / w are written, rpart holds
// [T][route_slices(d)][E] floats of its partial sums.
cudaError_t launch_layer_fused(const DevLayer& L, const __half* x, const __half* wr, const float* bias, int* idx,
                               float* w, float* rpart, int T, __half* h, __half* hs, float* y_perm, float* ys,
                               __half* y, int* offsets_out, cudaStream_t s);
int decode_max_tokens(int ffn, int T, int E, int K);
int decode_max_tokens_shared();
cudaError_t launch_prefill(const DevLayer& L, int mode, int phase, const __half* act, const int* offsets,
                           int n_slots, int min_tokens, __half* h, float* y, cudaStream_t s);
// Routing mass and prompt residual per expert (norms: T floats of scratch).
cudaError_t launch_route_stats(const DevLayer& L, const __half* x, const int* idx, const float* w, int T,
                               float* mass, float* resid, float* norms, cudaStream_t s);
cudaError_t launch_combine(const DevLayer& L, const float* y_perm, const int* inv_slot,
                           const float* w, int T, const float* y_shared, __half* y, cudaStream_t s);
cudaError_t launch_debug_dequant(const DevLayer& L, int e, int m, __half* out, cudaStream_t s);
// The decoded weights of expert e's matrix m as the decode kernel's K loop
// (launch_decode_dump, in either LUT-table configuration) or the prefill
// kernel's dequant warps (launch_prefill_dump) produce them.
cudaError_t launch_decode_dump(const DevLayer& L, int e, int m, bool lane_tables, __half* out, cudaStream_t s);
// Decode-kernel configuration of a layer: 2 (per-lane LUT tables, two CTAs per
// SM) or 3 (row-pair tables, three CTAs per SM).
int nblk_for(const DevLayer& L);
// The configuration expected to be faster for a layer whose expert weights
// hold bytes[0..4] at fp16 / 6 / 5 / 4 / 3 bits, experts of ffn rows (host side).
int decode_nblk(const double (&bytes)[5], int ffn);
cudaError_t launch_prefill_dump(const DevLayer& L, int e, int m, __half* out, cudaStream_t s);

// Host-side checks shared by the expert-FFN entry points: validates the
// arguments of a routed FFN call for T tokens and returns the layer's kernel
// parameters, the decode kernel classes it needs and the bytes of h scratch.
pw_status ffn_call_args(pw_layer_t layer, const void* x_perm, const int32_t* offsets, int T, const float* y_perm,
                        DevLayer* dev, int* class_mask, size_t* h_bytes);
// Records a CUDA error for pw_last_cuda_error and returns PW_ERR_CUDA.
pw_status record_cuda_error(cudaError_t e);

}  // namespace pw
