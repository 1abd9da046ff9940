/*
 * pw.h - C ABI of the GB300 routed any-precision MoE expert layer.
 *
 * The method: PagedWeight (Yang, Zhao, Dasgupta, Misailovic; write-up at
 * zhichai.net/topic/178446964).  Section "核心洞察" of that page: every expert
 * weight is an any-precision code kept as bit-planes plus a lookup table
 * (LUT), switchable among 3, 4, 5, 6 bits or a 16-bit fallback, and the planes
 * are managed like pages so that an expert's precision can be lowered by
 * detaching planes.  Section "安全边界与异步搬运": changes commit at a "safe
 * boundary".  The second write-up (time-frame.cloud, "方法与技术路线") adds a
 * "virtual page table" through which kernels read the weights.
 *
 * This header exposes one MoE layer's hot path on one GPU:
 *   pw_route_topk -> pw_permute -> pw_expert_ffn_bitplane (+ pw_shared_ffn, or both
 *   in one pw_moe_ffn)
 *   -> pw_combine,   and   pw_set_expert_bitwidth.
 * pw_moe_forward runs the whole chain in one call (one fused persistent
 * kernel, router included, for decode-sized batches; the separate kernels
 * above otherwise).
 * pw_route_stats and pw_plan_bitwidths give the signals and the per-expert
 * bitwidth plan that pw_set_expert_bitwidth then applies.
 *
 * Conventions for every function
 *  - Return value: pw_status.  Arguments are validated on the host before any
 *    work is enqueued; a failed check has no side effects.
 *  - "device" pointers are CUDA device memory owned by the caller (e.g. torch
 *    tensors); "host" pointers are ordinary host memory owned by the caller.
 *    The library never allocates device memory: weights, LUTs and its small
 *    tables live in a pool carved from a caller-provided device buffer.
 *  - Hot-path calls are asynchronous on the given stream (a cudaStream_t passed
 *    as void*, NULL = legacy default stream) and never synchronise it.
 *  - Matrices are row-major and "out x in": gate [ffn][d], up [ffn][d],
 *    down [d][ffn]; a row is an output channel.
 *  - fp16 data is passed as raw IEEE binary16 (uint16_t / void*).
 *  - Shapes: d and ffn (and shared_ffn) must be multiples of 64, n_experts in
 *    [1, 256], top_k in [1, min(8, n_experts)]; token counts T in [0, 2^20]
 *    (PW_ERR_INVALID_ARG outside).
 *  - A layer handle is not thread-safe: use one host thread per handle.
 */
#ifndef PW_H
#define PW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PW_OK = 0,
  PW_ERR_INVALID_ARG = 1,   /* bad pointer, size, index or bitwidth */
  PW_ERR_UNSUPPORTED = 2,   /* valid request the library cannot serve (shape, mode) */
  PW_ERR_OOM = 3,           /* pool or workspace too small */
  PW_ERR_NOT_RESIDENT = 4,  /* raising precision needs planes no longer in the pool */
  PW_ERR_CUDA = 5,          /* a CUDA call failed; see pw_last_cuda_error */
  PW_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up (device error word) */
  PW_ERR_DEVICE_CHECK = 7   /* a device-side bounds check fired (device error word) */
} pw_status;

typedef struct pw_pool_s* pw_pool_t;
typedef struct pw_layer_s* pw_layer_t;

/* Human-readable name of a status. */
const char* pw_status_str(pw_status s);

/* The cudaError_t value behind the most recent PW_ERR_CUDA on this thread. */
pw_status pw_last_cuda_error(int* cuda_err);

/* ---------------------------------------------------------------------------
 * Page pool
 * ---------------------------------------------------------------------------
 * A pool hands out fixed-size pages of a caller-provided device buffer.  Pages
 * hold bit-planes and fp16 fallback pages (paged, freed when an expert's
 * precision drops); LUTs, the page table itself and the shared FFN are
 * "resident" allocations taken from the end of the buffer.
 *   dev_base   device pointer, 256-byte aligned; must outlive the pool.
 *   bytes      usable size of the buffer.
 *   page_bytes page size: multiple of 64 KiB, at least 64 KiB (2 MiB usual).
 */
pw_status pw_pool_create(void* dev_base, size_t bytes, size_t page_bytes, pw_pool_t* out);
pw_status pw_pool_destroy(pw_pool_t pool);   /* all layers on it must be destroyed first */

/*
 * A pool whose page table is the GPU's own virtual memory (the "virtual page
 * table" of the second write-up, section 方法与技术路线; stable virtual
 * addresses per expert as in the third page's PagedTensor).  The caller
 * allocates the physical pages with the CUDA driver's virtual memory
 * management -- one cuMemCreate allocation of exactly page_bytes per page,
 * pinned device memory on `device` -- and passes their handles
 * (CUmemGenericAllocationHandle); the caller keeps ownership and releases
 * them (cuMemRelease) after pw_pool_destroy.  The library allocates no
 * physical memory: every layer on the pool reserves one virtual range
 * (cuMemAddressReserve) with a fixed sub-range per (expert, plane) block and
 * maps a block's pages into it (cuMemMap, cuMemSetAccess read/write for
 * `device`) while the block holds them.  So an expert's plane addresses --
 * and the device page table the kernels read -- never change: lowering
 * precision still moves no data and changes no mapping; a block's pages are
 * unmapped (cuMemUnmap) only when they are handed to another block, after
 * the lowering's safe boundary has passed, or when the expert is reloaded or
 * the layer destroyed (both synchronise first).  Everything else -- the
 * hot-path calls, pw_set_expert_bitwidth, pw_prefetch_expert, CUDA graphs --
 * works as on an ordinary pool.
 *   handles     host array of n_pages handles (copied)
 *   page_bytes  a multiple of 2 MiB (the allocation granularity)
 *   device      the CUDA device the handles live on (current for the calls)
 * PW_ERR_UNSUPPORTED when the driver offers no virtual memory management;
 * PW_ERR_CUDA when a mapping fails (the failed call has no effect).
 */
pw_status pw_pool_create_vmm(const unsigned long long* handles, size_t n_pages, size_t page_bytes, int device,
                             pw_pool_t* out);

typedef struct {
  size_t total_pages, free_pages, mapped_pages, reclaimable_pages;
  size_t resident_bytes, page_bytes;
} pw_pool_stats;
pw_status pw_pool_get_stats(pw_pool_t pool, pw_pool_stats* out);

/* ---------------------------------------------------------------------------
 * Layer lifecycle (setup; not on the timed path; may synchronise the stream)
 * ------------------------------------------------------------------------- */
typedef struct {
  int d;            /* hidden size, multiple of 64 */
  int ffn;          /* expert FFN size, multiple of 64 */
  int n_experts;    /* routed experts E, 1..256 */
  int top_k;        /* K, 1..min(8, E) */
  int renormalize;  /* 1: the K kept router weights are rescaled to sum 1 */
  int shared_ffn;   /* size of an always-on fp16 shared FFN, 0 = none */
} pw_layer_desc;

pw_status pw_layer_create(pw_pool_t pool, const pw_layer_desc* desc, pw_layer_t* out);
pw_status pw_layer_destroy(pw_layer_t layer);  /* returns every page and resident block */

/*
 * Upload one expert and map it at `bits` (3, 4, 5, 6 or 16).
 *   code6[m]   host uint8 [rows][cols] 6-bit parent codes (values 0..63) of
 *              matrix m = 0 gate, 1 up, 2 down.  Plane p holds bit (5 - p);
 *              planes 0..min(bits,6)-1 are packed and paged (all six when
 *              bits == 16, so that lowering from 16 moves no data).
 *   lut[m][i]  host fp16 [rows][2^(i+3)]: LUT_b for b = i + 3, all four kept
 *              resident (the dequantised weight is LUT_b[row][code6 >> (6-b)]).
 *   w16[m]     host fp16 [rows][cols] fallback page, required iff bits == 16,
 *              else may be NULL (then the expert can never be raised to 16).
 * Re-loading an expert first releases its previous pages.  A load the pool
 * cannot hold, counting the pages that release would free, returns
 * PW_ERR_OOM and leaves the expert and the pool as they were.
 * Synchronises `stream` before returning (host buffers may be freed after).
 */
pw_status pw_layer_load_expert(pw_layer_t layer, int e, int bits,
                               const uint8_t* const code6[3],
                               const uint16_t* const lut[3][4],
                               const uint16_t* const w16[3], void* stream);

/*
 * Give expert e of `layer` a copy of expert e_src of `src` at bitwidth `bits`
 * (planes 0..bits-1, or all six planes and the fp16 page for 16), together
 * with its LUTs, by device-to-device copies in stream order.  Both layers
 * must have the same d and ffn and pools with the same page size (the pools
 * may differ).  Every copied block must be one the source reads at its
 * current bitwidth (PW_ERR_NOT_RESIDENT otherwise; a lowered expert's
 * reclaimable planes are not copied).  Like pw_layer_load_expert it
 * synchronises the stream first, replaces whatever expert e held and returns
 * after the copies are done.  Setup call (e.g. building many layers from one
 * uploaded set of experts); not for the hot path.
 */
pw_status pw_layer_copy_expert(pw_layer_t layer, int e, pw_layer_t src, int e_src, int bits, void* stream);

/* Upload the fp16 shared FFN: w16[0] gate [shared_ffn][d], w16[1] up, w16[2] down [d][shared_ffn]. */
pw_status pw_layer_load_shared(pw_layer_t layer, const uint16_t* const w16[3], void* stream);

/* ---------------------------------------------------------------------------
 * Hot path
 * ------------------------------------------------------------------------- */

/*
 * Router (PagedWeight write-up, "三层感知", routing statistics; the router
 * itself is the standard MoE gate).  For each token t:
 *   l = W_r x_t + bias (fp32 accumulation of fp16 products),
 *   p = softmax(l) over all E experts,
 *   idx[t][0..K) = the K largest l, descending, exact ties to the lower index,
 *   w[t][k] = p[idx[t][k]], divided by their sum when renormalize is set.
 *   x       device fp16 [T][d]          wr  device fp16 [E][d]
 *   bias    device fp32 [E] or NULL     idx device int32 [T][K]   w device fp32 [T][K]
 *   expert_count  device int32 [E] or NULL: if given, incremented by the number
 *           of (t, k) slots routed to each expert ("routing mass" counters);
 *           the caller zeroes it.
 * T may be 0 (nothing is launched).
 */
pw_status pw_route_topk(pw_layer_t layer, const void* x, const void* wr, const float* bias,
                        int T, int32_t* idx, float* w, int32_t* expert_count, void* stream);

/*
 * Stable permutation of the S = T*K slots (flat index t*K + k) by expert:
 * inside an expert's bucket the slots keep ascending flat order.
 * The write-ups do not describe this step.  Their method runs each expert's
 * FFN over the tokens routed to it ("核心洞察"), and grouping the routed
 * (token, k) slots by expert is what gives every expert those tokens as one
 * contiguous batch; the definition above (a stable counting sort) is this
 * library's, chosen so the result is unique and deterministic.
 *   offsets  device int32 [E+1]: bucket e is [offsets[e], offsets[e+1])
 *   perm_src device int32 [S]:   token of each sorted slot
 *   inv_slot device int32 [S]:   sorted position of flat slot t*K + k
 *   x        device fp16 [T][d] and x_perm device fp16 [S][d]: if both are
 *            non-NULL, x_perm[i] = x[perm_src[i]].
 *   ws       device scratch of at least pw_workspace_size() bytes,
 *            16-byte aligned.
 * Deterministic (no atomics decide any order).
 */
pw_status pw_permute(pw_layer_t layer, const int32_t* idx, int T, const void* x,
                     int32_t* offsets, int32_t* perm_src, int32_t* inv_slot, void* x_perm,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * Routed expert SwiGLU FFN over the permuted slots (write-up "内存的饥饿游戏",
 * section 核心洞察: each expert weight is an any-precision code stored as
 * bit-planes plus a per-row LUT; an expert at b bits reads only its top b
 * planes, and a 16-bit expert its fp16 page).  For each expert e with
 * tokens (bucket of `offsets`) at its current bitwidth b_e:
 *   W = LUT_b[row][code_b] built from planes 0..b-1 only (planes >= b are never
 *       read), or the fp16 page when b_e == 16,
 *   h = silu(W_gate x) * (W_up x)   (fp32 accumulation; h rounded to fp16),
 *   y_perm[slot] = W_down h          (fp32).
 *   x_perm  device fp16 [T*K][d]     offsets device int32 [E+1]
 *   y_perm  device fp32 [T*K][d]
 *   ws      device scratch of at least pw_workspace_size(T) bytes, 16-byte
 *           aligned (the h activations are carved out of it)
 * offsets must be monotone in [0, T*K]; the kernels clamp a bad table to the
 * slot rows and flag the layer's device error word (pw_layer_check_device
 * then returns PW_ERR_DEVICE_CHECK), so nothing outside x_perm, y_perm and ws
 * is touched.
 */
pw_status pw_expert_ffn_bitplane(pw_layer_t layer, const void* x_perm, const int32_t* offsets,
                                 int T, float* y_perm, void* ws, size_t ws_bytes, void* stream);

/*
 * Same computation as pw_expert_ffn_bitplane, for callers that cannot
 * allocate device memory when they run the layer -- e.g. a serving engine that
 * has given all of HBM to its weight pool and KV cache and permits no further
 * cudaMalloc, or a host program that only passes in pre-allocated inputs and
 * outputs.  The paper has no counterpart; it is an addition of this library.
 *
 * Instead of a caller workspace the call uses one fixed array of 8 MiB in the
 * library's own device memory (every GPU that loads the library holds it until
 * the process exits), so T * top_k * ffn * 2 bytes must not exceed 8 MiB
 * (PW_ERR_OOM otherwise; nothing is launched).  No device memory is allocated
 * by this call.  Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept for the life of the
 * process: no device reset (cudaDeviceReset) may come between calls on that
 * device.  All calls share the array: calls whose
 * kernels overlap on the GPU (different streams, or different layers run
 * concurrently) race on it, so serialise them.  Nothing in it has to start at
 * zero; it keeps the last call's data.
 */
pw_status pw_expert_ffn_bitplane_noalloc(pw_layer_t layer, const void* x_perm, const int32_t* offsets,
                                         int T, float* y_perm, void* stream);

/*
 * fp16 shared FFN on all T tokens: y_shared [T][d] fp32 (layers with
 * shared_ffn > 0).  ws: pw_workspace_size(T) bytes, 16-byte aligned.
 */
pw_status pw_shared_ffn(pw_layer_t layer, const void* x, int T, float* y_shared,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * pw_expert_ffn_bitplane and, for layers with a shared FFN, pw_shared_ffn in
 * one call: decode-sized work of both runs in one persistent kernel, so the
 * shared FFN's weight stream overlaps the routed experts'.  Same results as
 * the two calls.  x [T][d] and y_shared [T][d] are ignored (may be NULL) when
 * the layer has no shared FFN.  ws must hold pw_workspace_size(T) bytes and
 * be 16-byte aligned.
 *
 * The FFN calls of one layer keep progress counters in the layer's device
 * state: run them on one stream (they may not overlap on the GPU).
 */
pw_status pw_moe_ffn(pw_layer_t layer, const void* x, const void* x_perm, const int32_t* offsets,
                     int T, float* y_perm, float* y_shared, void* ws, size_t ws_bytes, void* stream);

/*
 * Weighted combine:
 *   y[t] = sum_{k<K} w[t][k] * y_perm[inv_slot[t*K+k]]  (+ y_shared[t])
 * summed in k order in fp32, rounded to fp16.  The shared FFN output is added
 * unweighted.  y_shared may be NULL.  y device fp16 [T][d].
 * The write-ups do not describe this step either: it is the output of a
 * routed MoE layer, each token's experts weighted by its router weights (the
 * gate that "三层感知" reads its routing statistics from).  The k order and
 * fp32 sum are this library's, for a deterministic result.  An inv_slot entry
 * outside [0, T*K) is read as slot 0 and flags the layer's device error word.
 */
pw_status pw_combine(pw_layer_t layer, const float* y_perm, const int32_t* inv_slot,
                     const float* w, int T, const float* y_shared, void* y, void* stream);

/*
 * Change one expert's precision (write-up "核心洞察": lower the least
 * sensitive experts under KV-cache pressure; "安全边界与异步搬运": commit at a
 * safe boundary).
 * Lowering b -> b' moves no weight data: the device bitwidth word is written
 * in stream order (kernels enqueued later read only planes < b'), and the pages
 * of planes b'..b-1 (and the fp16 page when leaving 16) become reclaimable.
 * They are handed to other owners only after an event recorded here has
 * completed, i.e. after every kernel enqueued before this call is done.
 * Raising succeeds only while every needed page is still reclaimable
 * (otherwise PW_ERR_NOT_RESIDENT and nothing changes).  Never synchronises.
 */
pw_status pw_set_expert_bitwidth(pw_layer_t layer, int e, int bits, void* stream);

/*
 * Bring back the blocks expert e needs at `bits` without changing its
 * bitwidth yet (write-up "安全边界与异步搬运": planes move in the background
 * and the change commits later at a safe boundary).  Blocks still on the
 * reclaim queue are taken off it (their data is intact).  Blocks that are
 * gone get free pages (or reclaimable ones whose safe boundary has passed;
 * the call waits for it if it must) and their data is copied from host
 * memory on `copy_stream`, followed by the expert's page-table rows (entries
 * of the planes the current bitwidth reads keep their values; kernels never
 * read planes at or above it).  A later pw_set_expert_bitwidth raise on any
 * stream waits for these copies before it commits.
 *   planes_host[m][p]  plane p of matrix m as packed by pw_pack_planes
 *                      (uint32 [R*C/32]); read for the missing planes only
 *                      (others may be NULL; the whole array may be NULL when
 *                      nothing is missing)
 *   w16_host[m]        fp16 page of matrix m as packed by pw_pack_f16; read
 *                      when bits == 16 and the fp16 block is missing
 * Host buffers should be pinned for the copies to be asynchronous, and must
 * stay valid until they complete.  PW_ERR_INVALID_ARG when a needed host
 * array is NULL; PW_ERR_OOM (no change) when the pool has no room.
 */
pw_status pw_prefetch_expert(pw_layer_t layer, int e, int bits, const uint32_t* const planes_host[3][6],
                             const uint16_t* const w16_host[3], void* copy_stream);

/*
 * pw_prefetch_expert followed by the raise pw_set_expert_bitwidth(e, bits,
 * stream): `stream` waits for the copies and then writes the bitwidth word,
 * so kernels enqueued on `stream` after this call read the new bitwidth and
 * kernels enqueued before it keep the old one.  bits must be above the
 * current bitwidth (16 above 6; PW_ERR_INVALID_ARG otherwise).  To keep the
 * wait off the compute stream, prefetch a step ahead and raise later.
 */
pw_status pw_raise_expert_async(pw_layer_t layer, int e, int bits, const uint32_t* const planes_host[3][6],
                                const uint16_t* const w16_host[3], void* copy_stream, void* stream);

/* Host mirror of an expert's current bitwidth (0 if not loaded). */
pw_status pw_get_expert_bitwidth(pw_layer_t layer, int e, int* bits);

/*
 * How a batch of T tokens is split between the kernels (host only; no GPU
 * needed).  The pages fix no such split: it is this library's choice of
 * where the bit-plane GEMV stops paying and the tensor-core GEMM starts,
 * set by measurement.
 *   routed_max: routed experts with more tokens than this run on the
 *     tcgen05 GEMM, the others on the decode kernel;
 *   shared_max: the shared FFN runs on the GEMM when T exceeds this;
 *   fused: 1 when pw_moe_forward takes its one-launch fused step.
 * The environment overrides the kernels read (PW_DECODE_MAX_TOK,
 * PW_DECODE_MAX_TOK_SHARED) apply here too.  PW_ERR_INVALID_ARG for a null
 * pointer, T < 0 or a descriptor with non-positive sizes.
 */
pw_status pw_decode_plan(const pw_layer_desc* desc, int T, int* routed_max, int* shared_max, int* fused);

/* Scratch bytes that pw_permute / pw_expert_ffn_bitplane / pw_shared_ffn need for T tokens. */
pw_status pw_workspace_size(pw_layer_t layer, int T, size_t* bytes);

/*
 * The whole layer for T tokens in one call.  For decode batches of at most
 * 16 tokens (T also within the decode token thresholds and T*K <= 512): one
 * persistent kernel that routes (its CTAs share the router's sums; the last
 * one to finish a token's sums selects its experts, and every CTA waits,
 * bounded, until all tokens are routed), permutes, runs every expert's FFN
 * and the shared FFN and combines (the permutation is never written out:
 * routed rows are read from x through the routing result).  Otherwise
 * pw_route_topk, pw_permute, pw_moe_ffn and pw_combine.  Both ways give the
 * same idx, w and y, bit for bit, as those separate calls: the router adds
 * its fp32 sums in one fixed order, every expert-FFN item is computed the
 * same way and the fused combine adds the k terms in the same order.
 *   x   device fp16 [T][d]   wr device fp16 [E][d]   bias device fp32 [E] or NULL
 *   idx device int32 [T][K], w device fp32 [T][K]: the routing (outputs)
 *   y   device fp16 [T][d] (output)
 *   ws  device scratch of at least pw_moe_forward_workspace_size(T) bytes
 * Asynchronous on `stream`; run the calls of one layer on one stream.
 * Errors (checked before anything is enqueued): PW_ERR_INVALID_ARG for
 * T < 0, a null pointer (T > 0), x / wr / y / ws not 16-byte aligned, an
 * expert never loaded, or a shared FFN declared but not loaded; PW_ERR_OOM
 * when ws_bytes is below the workspace size; PW_ERR_CUDA when a launch
 * fails.  T = 0 enqueues nothing.
 */
pw_status pw_moe_forward(pw_layer_t layer, const void* x, const void* wr, const float* bias, int T,
                         int32_t* idx, float* w, void* y, void* ws, size_t ws_bytes, void* stream);
pw_status pw_moe_forward_workspace_size(pw_layer_t layer, int T, size_t* bytes);

/* ---------------------------------------------------------------------------
 * Quality-aware bitwidth planning (PagedWeight write-up "内存的饥饿游戏",
 * sections 三层感知 and 安全边界与异步搬运; budget M_w = M_total - M_kv and
 * the greedy approximation from "动态量化优化MoE模型服务", 方法与技术路线).
 * ------------------------------------------------------------------------- */

/*
 * Online signals of the planner for one routed batch (the router's outputs):
 *   mass[e]  = sum of w[t][k] over the slots with idx[t][k] == e
 *              ("routing mass": protects busy experts),
 *   resid[e] = sum of w[t][k] * ||x[t]||_2 over the same slots
 *              ("prompt residual": the routing-weighted input norm).
 *   x     device fp16 [T][d]      idx device int32 [T][K]   w device fp32 [T][K]
 *   mass, resid  device fp32 [E], overwritten.
 *   ws    device scratch of at least 4*T bytes (token norms).
 * fp32 accumulation in a fixed order: deterministic.  T may be 0 (zeros).
 */
pw_status pw_route_stats(pw_layer_t layer, const void* x, const int32_t* idx, const float* w, int T,
                         float* mass, float* resid, void* ws, size_t ws_bytes, void* stream);

/*
 * Pool bytes one expert of this layer holds at bitwidth `bits` (3..6: that
 * many plane blocks; 16: the fp16 block and all six plane blocks, so that
 * lowering from 16 moves no data).  Host only; the planner's size table.
 */
pw_status pw_expert_resident_bytes(pw_layer_t layer, int bits, uint64_t* bytes);

/*
 * Staged greedy bitwidth plan under a byte budget (host only, no layer).
 *   sens    host [E][4]  offline damage of each expert at 3, 4, 5, 6 bits
 *                        (0 at 16); any non-negative scale
 *   mass    host [E] or NULL, resid host [E] or NULL (pw_route_stats; NULL
 *                        switches the factor off)
 *   floors  host [E] or NULL (3): lowest bitwidth allowed per expert
 *   ceils   host [E] or NULL (16): highest (the plan starts there)
 *   sizes   host [E][5]  bytes of each expert at 16, 6, 5, 4, 3 bits
 *   budget  bytes the experts may hold (M_w = M_total - M_kv - fixed)
 *   bits    host [E] out: the plan;  used  host out: its bytes
 * Expert weight = (mass_e / sum mass) * ((resid_e / mass_e) / (sum resid /
 * sum mass)) (1 / E and 1 when a signal is NULL; ratio 1 for an expert
 * without mass); damage(e, b) = weight_e * sens[e][b].  Stages lower the
 * levels 16 -> 6 -> 5 -> 4 -> 3 one at a time, never below a floor; inside a
 * stage, while over budget, the expert whose next step down costs the least
 * damage per byte saved moves (ties: lower index).  Sums run in index order
 * in double.  Returns PW_ERR_OOM (bits = floors, *used their bytes) when even
 * the floors exceed the budget; PW_ERR_INVALID_ARG for bad arguments
 * (E < 1, negative values, floors not in {3,4,5,6,16} or above ceils).
 */
pw_status pw_plan_bitwidths(int E, const double* sens, const double* mass, const double* resid,
                            const int* floors, const int* ceils, const uint64_t* sizes, uint64_t budget,
                            int* bits, uint64_t* used);

/*
 * Reads (synchronously) and clears the layer's device error word, set by
 * bounded device-side waits or bounds checks of earlier launches.
 * PW_OK if nothing was flagged, else PW_ERR_TIMEOUT / PW_ERR_DEVICE_CHECK.
 */
pw_status pw_layer_check_device(pw_layer_t layer, void* stream);

/*
 * Workspace canaries (debug bounds) for one layer.  When on, the sizes that
 * pw_moe_forward_workspace_size and pw_workspace_size report include a
 * 256-byte block after every scratch region; pw_moe_forward and pw_moe_ffn
 * fill those blocks with a fixed pattern before their kernels and check the
 * pattern after them (both stream-ordered, on the call's stream), flagging a
 * changed word -- a write past a scratch region -- in the layer's device error
 * word (PW_ERR_DEVICE_CHECK from pw_layer_check_device).  Workspaces must be
 * sized after the setting changes (PW_ERR_OOM otherwise).  Off by default;
 * PW_DEBUG_BOUNDS=1 in the environment turns it on for layers created
 * afterwards.  With PW_NVTX=1 the hot-path calls also open NVTX ranges named
 * after the call (for a profiler's timeline).
 */
pw_status pw_layer_set_debug_bounds(pw_layer_t layer, int on);

/*
 * Check, on the stream, the canaries of a whole-layer workspace laid out for
 * T tokens (as pw_moe_forward lays it out); the result lands in the layer's
 * device error word.  PW_ERR_INVALID_ARG when debug bounds are off,
 * PW_ERR_OOM when ws_bytes is below that layout's size.
 */
pw_status pw_debug_check_workspace(pw_layer_t layer, int T, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Host utilities and debugging
 * ------------------------------------------------------------------------- */

/*
 * Pack 6-bit codes [R][C] (host) into six plane arrays planes_out[p] of
 * R*C/32 uint32 words each (plane p = bit 5-p), in the stored word order:
 *   tile = r / 16, chunk = c / 64; g = r%16 % 8, rowsel = r%16 / 8;
 *   s = c%64 / 16, colhalf = c%16 / 8, t = c%8 / 2, h = c % 2;
 *   lane = 4g + t, k = 2 rowsel + colhalf, q = 8k + 4h + s;
 *   plane p keeps the bit at position (q + 5 - p) mod 32 of word
 *   tile*(C/64)*32 + [group*128 + 4*lane + i] for chunk 4*group + i of a full
 *   group of four chunks, or [G*128 + r*lane + i] in a final group of r < 4 chunks.
 */
pw_status pw_pack_planes(const uint8_t* code6, int R, int C, uint32_t* const planes_out[6]);

/*
 * Pack an fp16 matrix [R][C] into the stored fp16-page order: half index
 * (((tile*(C/64) + chunk)*4 + s)*32 + lane)*8 + 2a + h with a = rowsel + 2 colhalf.
 */
pw_status pw_pack_f16(const uint16_t* w, int R, int C, uint16_t* out);

/*
 * Debug: write expert e's matrix m (0 gate, 1 up, 2 down) at its current
 * bitwidth, dequantised, into out (device fp16 [rows][cols]).  A plain
 * reference decoder: the planes are read through the page table and every
 * code is looked up in a per-lane LUT table (the layout of the stored words
 * and tables, not the kernels' own loops; pw_debug_dequant_kernel below dumps
 * those).
 */
pw_status pw_debug_dequant(pw_layer_t layer, int e, int m, void* out, void* stream);

/*
 * Debug: the same dump, produced by the FFN kernels' own code paths:
 *   PW_KERNEL_DECODE   the decode kernel's K loop (its cp.async ring through
 *                      the page table, 3-bit register-LUT byte permutes,
 *                      4..6-bit shared-memory LUT table, fp16 fragments) with
 *                      each decoded A fragment written out instead of
 *                      multiplied, in the configuration this layer's FFN
 *                      calls use;
 *   PW_KERNEL_DECODE_ROW_TABLES, PW_KERNEL_DECODE_LANE_TABLES  the same K loop
 *                      in a given configuration: 4..6-bit tables shared by
 *                      the lanes of a row pair (layers with ffn < 4096), or
 *                      one copy per lane (ffn >= 4096);
 *   PW_KERNEL_PREFILL  the tcgen05 GEMM's dequant warps (plane loads, LUT
 *                      set-up and decode) writing rows instead of the
 *                      swizzled shared-memory tile.
 * out device fp16 [rows][cols], 16-byte aligned.  Section 核心洞察 of the
 * write-up fixes the value: W = LUT_b[row][code6 >> (6 - b)], or the fp16
 * page at 16 bits.
 */
enum { PW_KERNEL_DECODE = 0, PW_KERNEL_PREFILL = 1, PW_KERNEL_DECODE_ROW_TABLES = 2,
       PW_KERNEL_DECODE_LANE_TABLES = 3 };
pw_status pw_debug_dequant_kernel(pw_layer_t layer, int e, int m, int kernel, void* out, void* stream);

/* Debug: device address of virtual page `vpage` of expert e's plane p (p = 6: fp16 page), or 0. */
pw_status pw_debug_page_address(pw_layer_t layer, int e, int p, int vpage, uint64_t* addr);

/*
 * Testing hook: host-simulated device (call before creating any pool).  The
 * pool buffer is then host memory, uploads are memcpy, events complete only
 * when pw_testing_complete_events() is called, and every compute entry point
 * returns PW_ERR_UNSUPPORTED.  Used to test pool / page-table bookkeeping on
 * machines without a GPU.  enable = 0 restores normal operation.
 */
pw_status pw_testing_host_sim(int enable);
pw_status pw_testing_complete_events(void);

/*
 * Testing hook: pages mapped and unmapped so far by a virtual-memory pool
 * (pw_pool_create_vmm).  In host-sim mode such a pool simulates the physical
 * pages with one shared memory file and maps them with mmap, so the same
 * bookkeeping and the bytes behind every virtual address can be checked on
 * machines without a GPU.
 */
pw_status pw_testing_vmm_counts(pw_pool_t pool, uint64_t* maps, uint64_t* unmaps);

/*
 * Testing hook for the bounded waits of the decode kernel: a down item waits
 * (polling a counter) until every gate/up tile of its token chunk is done,
 * and the fused step waits for every down item before its combine.
 *   polls        polls before such a wait gives up (0 restores the default,
 *                about a second); the kernel then sets the layer's device
 *                error word, carries on and returns its counters to zero,
 *                and pw_layer_check_device reports PW_ERR_TIMEOUT.
 *   never_ready  1: down items wait for one tile more than exist (a count
 *                nothing reaches), so every such wait runs out; 0: normal.
 * Affects launches enqueued after the call, for this layer only.
 */
pw_status pw_testing_wait_limit(pw_layer_t layer, long long polls, int never_ready);

#ifdef __cplusplus
}
#endif
#endif /* PW_H */
