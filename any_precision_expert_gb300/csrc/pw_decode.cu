// Persistent decode-side expert FFN: gate/up and down for every routed expert
// with few tokens (3, 4, 5, 6 bits or its fp16 page) and for the fp16 shared
// FFN, in one launch.
//
// PagedWeight (write-up "内存的饥饿游戏", section 核心洞察): an expert at
// bitwidth b streams only its top b bit-planes, found through the per-expert
// page table, and looks every code up in the row's LUT; a fallback expert
// streams its fp16 page.  Decode batches route a few tokens to each expert, so
// the time goes into streaming weights.
//
// A CTA (four warps) takes one work item at a time: (group, phase, 32-token
// chunk, two gate/up tiles or one to four down tiles).  It stages the item's
// distinct token rows once into shared memory (double-buffered K-blocks of
// 256 columns, or 512 / 1024 for one or two token tiles; rows XOR-swizzled
// for conflict-free ldmatrix), and every warp streams one matrix of one
// 16-row tile through its own cp.async ring, addressed through the page table
// (gate/up: warps 0-1 the gate rows of the two tiles, warps 2-3 their up rows,
// which reach the gate warps through shared memory for SwiGLU).  Down items of
// groups with few tokens and a long reduction split each tile's reduction
// over two or four warps (interleaved units, partial sums added in warp
// order), so that their chains stay short.  Codes become weights by
//  - 3 bits: byte permutes from register LUTs (whole plane groups, 16 B per
//    lane and plane);
//  - 4, 5, 6 bits: lookups in the warp's LUT table in shared memory (row
//    pair g / g+8 per 32-bit entry); one code path for the three bitwidths;
//  - fp16 pages: stored in mma fragment order, used as they are.
// The weights feed mma.sync m16n8k16 (weights as A, tokens as B, fp32
// accumulation).  Gate/up writes h = silu(g) * u in fp16, down writes y in
// fp32.  Each weight kind has a single copy of its loop body (the kernel's
// instruction footprint stays small).
//
// Fused layer step (FUSED): given the router's output, the kernel also does
// the permutation and the combine -- every CTA sorts the (at most 512) slots
// by expert in shared memory itself (stable: ascending flat order inside an
// expert), routed rows are staged straight from x, and when every down item
// is done the CTAs add y[t] = sum_k w[t][k] y_perm[slot(t, k)] (+ the shared
// FFN) in k order, as the separate combine does.
//
// CTAs claim items from one counter in a fixed order: groups in the order
// shared FFN, fp16, 4..6-bit, 3-bit experts; a group's down items (phase 1)
// follow about one wave of CTAs after its gate/up items (phase 0), so that
// long down items start early.  A down item waits until all gate/up tiles of
// its (group, chunk) are done; those items were claimed earlier by running
// CTAs and never wait, so every wait ends.  The waits are
// bounded anyway: past the limit the kernel records a timeout in the layer's
// error word and carries on.  The phase counters are returned to zero by the
// last down tile of each (group, chunk) and the claim counter by the last CTA
// to leave, so the next launch (or graph replay) starts from zero.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "pw_gemv.cuh"
#include "pw_route.cuh"

namespace pw {

constexpr int kCtaThreads = 128;
constexpr int kCtaWarps = kCtaThreads / 32;
constexpr int kFusedSlots = 512;             // routed slots (T * K) of a fused layer step

// Items take up to 32 tokens (a weight tile is streamed and decoded once for
// up to 32 tokens).  Shared memory: two K-block buffers of token rows, a LUT
// table and a weight ring per warp.
struct Geo {
  static constexpr int TOK = 32;                // tokens per item
  static constexpr int NTM = TOK / 8;           // mma n-tiles per item
  static constexpr int SCOLS = 256;             // columns of one staged K-block at 32 tokens
  static constexpr int HALF = TOK * SCOLS * 2;  // bytes of one K-block buffer
};

// The kernel's two configurations, which differ in the 4..6-bit LUT table:
//   NBLK = 3: three CTAs per SM; one table per warp shared by the lanes of a
//     row pair (entry (v, g) = LUT[g][v] | LUT[g+8][v] << 16 at byte 32 v + 4 g,
//     2 KB at 6 bits); the four lanes of a row can collide on a bank;
//   NBLK = 2: two CTAs per SM; every lane its own copy of its two rows (entry
//     (v, lane) at byte 128 v + 4 lane, 8 KB at 6 bits): the 32 lookups of a
//     warp never collide on a bank, at two thirds of the resident warps.
// Measured: the second is 12% faster on experts of ffn 14336 at 64 tokens and
// 12% slower on the Qwen-shaped layer (few 4..6-bit experts, where the
// warps matter more); layers with ffn >= 4096 take it (nblk_for).
//
// NBLK = 2 places its buffers at fixed addresses of the CTA's shared-memory
// window, so that one byte permute forms a lookup's whole address
// (decode_step_px): the four warps' rings from the dynamic base, K-block
// buffer 0 at 48 KB, the LUT tables at 64 KB (entry (v, warp w, lane l) at
// 64 KB + 512 v + 256 (w / 2) + 128 (w % 2) + 4 l), K-block buffer 1 at 96 KB,
// the window's end at 112 KB.  The kernel checks at entry that its window
// holds this layout (kErrLayout otherwise, before anything else is touched).
template <int NBLK>
struct Cfg {
  static constexpr bool LANE = NBLK == 2;              // per-lane LUT tables
  static constexpr int BLOCKS = NBLK;                  // CTAs per SM
  static constexpr int TABW = LANE ? 64 * 32 * 4 : 64 * 8 * 4;  // LUT table of one warp (b <= 6)
  static constexpr int TSHIFT = LANE ? 7 : 5;          // log2 of the table's stride per code
  static constexpr int RB = LANE ? 10 * 1024 : 7 * 1024;  // cp.async weight ring of one warp
  static constexpr int SMEM = 2 * Geo::HALF + kCtaWarps * (TABW + RB);  // NBLK = 3: one contiguous block
  static constexpr uint32_t SLAB0 = 48 * 1024;         // NBLK = 2: fixed addresses
  static constexpr uint32_t TAB_AT = 64 * 1024;
  static constexpr uint32_t SDELTA = LANE ? 48 * 1024 : Geo::HALF;  // K-block buffer 1 - buffer 0
  static constexpr uint32_t END = 112 * 1024;
  static_assert(!LANE || (SLAB0 + Geo::HALF <= TAB_AT && TAB_AT + kCtaWarps * TABW == SLAB0 + SDELTA &&
                          SLAB0 + SDELTA + Geo::HALF == END),
                "fixed layout of the per-lane-table configuration");
};

// Weight units streamed by a warp (one matrix of its tile):
//   KIND_F16: 64 columns of the fp16 page, 4 x 16 B per lane (ring depth 3);
//   KIND_PB: half a plane group (2 chunks, 128 columns), 8 B per lane and plane
//     (4..6 bits with the three-CTA configuration's 7 KB rings);
//   KIND_PG: a whole plane group (4 chunks, 256 columns), 16 B per lane and plane
//     (3 bits; 4..6 bits with the two-CTA configuration's 10 KB rings).
enum { KIND_F16 = 1, KIND_PB = 2, KIND_PG = 3 };
constexpr int kF16Steps = 4;  // mma steps (16 columns each) of one fp16 unit

template <int KIND, int B, int RB>
struct Unit {
  static constexpr int COLS = KIND == KIND_F16 ? 16 * kF16Steps : KIND == KIND_PB ? 128 : 256;
  static constexpr int LANE_BYTES = KIND == KIND_F16 ? kF16Steps * 16 : KIND == KIND_PB ? B * 8 : B * 16;
  static constexpr int SLOT = LANE_BYTES * 32;
  static constexpr int R = RB / SLOT > 8 ? 8 : RB / SLOT;  // ring depth
  static_assert(RB / SLOT >= 3, "ring too shallow");
  static_assert(Geo::SCOLS % COLS == 0, "units must not straddle K-blocks");
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
  // fused layer step only: the kernel routes, the routing result replaces
  // offsets / x_perm, and the kernel ends with the weighted combine
  const __half* wr;    // [E][d] router weight
  const float* bias;   // [E] router bias, or null
  float* rpart;        // [T][route_slices(d)][E] partial sums of the router
  int* idx;            // [T][K] experts of each token (written by the router)
  float* wk;           // [T][K] routing weights (written by the router)
  __half* yout;        // [T][d] layer output
  int* offsets_out;    // [E+1] slot offsets (written by CTA 0), or null
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
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

// log2 of the columns of one staged K-block for an item of ntok token rows:
// the 16 KB buffer holds the rows rounded up to a power of two, from 32 rows
// of 256 columns to one row of 8192, so items with few tokens pass few
// K-block barriers (a 4096-column reduction at one token: none).
__device__ __forceinline__ int kblock_log2(int ntok) {
  const int r = ntok <= 1 ? 0 : 32 - __clz(ntok - 1);  // log2 of the rows
  return 13 - r;
}
static_assert(Geo::SCOLS == 256 && Geo::HALF == 32 * 256 * 2, "kblock_log2 assumes 16 KB K-block buffers");

// Byte offset of 16-byte piece j (8 columns) of token row r in a staged
// K-block whose rows are rs bytes apart.
__device__ __forceinline__ uint32_t slab_off(int r, int j, int rs) {
  return (uint32_t)(r * rs + ((j ^ (r & 7)) << 4));
}

// Copy K-block kb (kbw columns) of the item's srows distinct token rows into
// a slab buffer (all threads).
__device__ __forceinline__ void stage_kblock(const __half* act, const int* s_tok, int srows, int K, int kb, int kbw,
                                             uint32_t buf) {
  const int c0 = kb * kbw;
  const int ppr = min(kbw, K - c0) >> 3;  // 16-byte pieces per row
  if (ppr == (kbw >> 3) && ppr <= kCtaThreads) {
    // whole K-block (ppr a power of two): each thread keeps one piece column
    const int lg = __ffs(ppr) - 1;
    const int j = threadIdx.x & (ppr - 1), rstep = kCtaThreads >> lg;
    const __half* src = act + c0 + j * 8;
#pragma unroll 4
    for (int r = threadIdx.x >> lg; r < srows; r += rstep)
      cp_async16(buf + slab_off(r, j, kbw * 2), src + (size_t)s_tok[r] * K);
    return;
  }
  if (ppr == (kbw >> 3)) {
    // whole K-block wider than the CTA (few rows): rows one by one
    for (int r = 0; r < srows; ++r) {
      const __half* src = act + (size_t)s_tok[r] * K + c0;
      for (int j = threadIdx.x; j < ppr; j += kCtaThreads) cp_async16(buf + slab_off(r, j, kbw * 2), src + j * 8);
    }
    return;
  }
  const int n = srows * ppr;
  for (int p = threadIdx.x; p < n; p += kCtaThreads) {
    const int r = p / ppr, j = p - r * ppr;
    cp_async16(buf + slab_off(r, j, kbw * 2), act + (size_t)s_tok[r] * K + c0 + j * 8);
  }
}

// This lane's ldmatrix row of each pair of n-tiles in a staged K-block, fixed
// for a whole K loop: off = r * rs (row r = token (2 i + mat / 2) * 8 + lane %
// 8, rows past the staged ones reading the last one) and x16 = (r % 8 ^ mat %
// 2) * 16, the swizzle of the row's 16-byte pieces.  Since every step starts
// at a multiple of 64 columns, piece 2 s + mat % 2 of step s sits at byte
// 2 kc + ((32 s) ^ x16) of the row.
struct BRows {
  uint32_t off[Geo::NTM / 2];
  uint32_t x16[Geo::NTM / 2];
};

__device__ __forceinline__ BRows slab_brows(int srows, int rs) {
  const int lane = threadIdx.x & 31, mat = lane >> 3;
  BRows o;
#pragma unroll
  for (int i = 0; i < Geo::NTM / 2; ++i) {
    const int r = min((2 * i + (mat >> 1)) * 8 + (lane & 7), srows - 1);
    o.off[i] = (uint32_t)(r * rs);
    o.x16[i] = (uint32_t)(((r & 7) ^ (mat & 1)) << 4);
  }
  return o;
}

// B fragments of mma step s (16 columns at column kc + 16 s of its K-block,
// kc a multiple of 64) for the n-tiles: one ldmatrix.x4 per pair of n-tiles
// (b0, b1 of each).  Rows past the staged ones read the last staged row;
// their results are not stored.
__device__ __forceinline__ void slab_bstep(uint32_t buf, int kc, int s, int NT, const BRows& br,
                                           uint32_t (&bf)[Geo::NTM][2]) {
  const uint32_t row0 = buf + 2 * (uint32_t)kc;
#pragma unroll
  for (int nt0 = 0; nt0 < Geo::NTM; nt0 += 2) {
    if (nt0 < NT)
      ldsm_x4(row0 + br.off[nt0 / 2] + (br.x16[nt0 / 2] ^ (uint32_t)(32 * s)), bf[nt0][0], bf[nt0][1],
              bf[nt0 + 1][0], bf[nt0 + 1][1]);
  }
}

__device__ __forceinline__ void mma_tiles(float (&acc)[Geo::NTM][4], const uint32_t (&a)[4],
                                          const uint32_t (&bf)[Geo::NTM][2], int NT) {
#pragma unroll
  for (int nt = 0; nt < Geo::NTM; ++nt)
    if (nt < NT) mma16816(acc[nt], a, bf[nt][0], bf[nt][1]);
}

// The warp's LUT table for one 16-row tile at bitwidth b (4..6): lr = the
// tile's LUT_b rows (16 x 2^b fp16, row-major); layouts in Cfg.
template <int NBLK>
__device__ __forceinline__ void build_tab_warp(const __half* lr, int b, uint32_t tab) {
  const int V = 1 << b, lane = threadIdx.x & 31;
  if constexpr (Cfg<NBLK>::LANE) {
    // each lane writes its own copy of rows g and g + 8, eight entries per
    // pair of 16-byte loads, at the fixed addresses of decode_step_px
    const int g = lane >> 2, warp = threadIdx.x >> 5;
    const uint32_t at = Cfg<NBLK>::TAB_AT + (warp >> 1) * 256 + (warp & 1) * 128 + lane * 4;
    for (int v0 = 0; v0 < V; v0 += 8) {
      const uint4 lo = *reinterpret_cast<const uint4*>(lr + g * V + v0);
      const uint4 hi = *reinterpret_cast<const uint4*>(lr + (g + 8) * V + v0);
      const uint32_t l4[4] = {lo.x, lo.y, lo.z, lo.w}, h4[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        sts32(at + (v0 + j) * 512, prmt(l4[j >> 1], h4[j >> 1], (j & 1) ? 0x7632u : 0x5410u));
    }
  } else {
    for (int i = lane; i < V; i += 32) {  // (row pair g, run of 8 entries from v0)
      const int g = i & 7, v0 = (i >> 3) * 8;
      const uint4 lo = *reinterpret_cast<const uint4*>(lr + g * V + v0);
      const uint4 hi = *reinterpret_cast<const uint4*>(lr + (g + 8) * V + v0);
      const uint32_t l4[4] = {lo.x, lo.y, lo.z, lo.w}, h4[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        sts32(tab + ((v0 + j) * 8 + g) * 4, prmt(l4[j >> 1], h4[j >> 1], (j & 1) ? 0x7632u : 0x5410u));
    }
  }
  __syncwarp();
}

// Destination of a dump of the decoded weights (the debug path): the A
// fragments of a tile are written to out[row][col] instead of feeding the mma.
struct Dump {
  __half* out;  // [rows][ld] fp16
  int ld;       // columns of the matrix
  int row0;     // first row of the warp's tile
  bool store;   // false: run the loop (barriers) but write nothing
};

// A fragment of mma step at column col: a0 row g cols 2t.., a1 row g+8, a2 row
// g cols 2t+8.., a3 row g+8 cols 2t+8.. (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void dump_frag(const Dump& D, const uint32_t (&a)[4], int col) {
  if (!D.store) return;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    *reinterpret_cast<uint32_t*>(D.out + (size_t)(D.row0 + g + 8 * (r & 1)) * D.ld + col + 2 * t + 8 * (r >> 1)) =
        a[r];
}

// Weight sources of one warp's K loop.
struct WSrc {
  const char* p[kPlanes];  // plane tiles, or the fp16 tile in p[0]
  uint32_t lut3[2][4];     // 3 bits: register LUTs of rows g and g + 8
  uint32_t tabl;           // 4..6 bits: this lane's base in the warp's LUT table (Cfg)
  uint32_t qbit;           // NBLK = 2: the warp's table parity (decode_step_px)
};

// K loop of one warp over the units cb = u0, u0 + us, ... of its tile (unit
// cb = columns cb * COLS ...).  Every warp of the CTA runs it for the same
// item and passes the same K-block barriers; the ntok distinct token rows of
// K-block kb are staged at the start of K-block kb - 1.  B: 16 (fp16), 3, 4, 5
// or 6.  pre() runs once the first weight units are in flight.
template <int KIND, int B, int NBLK, bool DUMP = false, class Pre>
__device__ __forceinline__ void kloop(const WSrc& src, int K, int NT, int ntok, int u0, int us, uint32_t ring,
                                      uint32_t slab, const __half* act, const int* s_tok,
                                      float (&acc)[Geo::NTM][4], Pre&& pre, const Dump* dump = nullptr) {
  using G = Geo;
  using U = Unit<KIND, B, Cfg<NBLK>::RB>;
  constexpr int R = U::R;
  const int lane = threadIdx.x & 31;
  const int lkb = kblock_log2(ntok), kbw = 1 << lkb, rs = kbw * 2;
  const int nk = K / 64, GR = nk / 4, rem = nk % 4;
  const int nu = (K + U::COLS - 1) / U::COLS;
  const int mine = u0 < nu ? (nu - u0 + us - 1) / us : 0;
  const int kbs = (K + kbw - 1) / kbw;
  const BRows br = slab_brows(ntok, rs);

  auto issue = [&](int i) {
    const int cb = u0 + i * us;
    const uint32_t slot = ring + (i % R) * U::SLOT;
    if constexpr (KIND == KIND_F16) {
#pragma unroll
      for (int s = 0; s < kF16Steps; ++s)
        cp_async16(slot + (s * 32 + lane) * 16, src.p[0] + ((size_t)(cb * kF16Steps + s) * 32 + lane) * 16);
    } else if constexpr (KIND == KIND_PG) {
      if (cb < GR) {
        const size_t off = (size_t)(cb * 128 + lane * 4) * 4;
#pragma unroll
        for (int p = 0; p < B; ++p) cp_async16(slot + (p * 32 + lane) * 16, src.p[p] + off);
      } else {
        const size_t off = (size_t)(GR * 128 + lane * rem) * 4;
#pragma unroll
        for (int p = 0; p < B; ++p)
          for (int k = 0; k < rem; ++k) cp_async4(slot + (p * 32 + lane) * 16 + 4 * k, src.p[p] + off + 4 * k);
      }
    } else {
      const int gamma = cb >> 1, j = cb & 1;
      if (gamma < GR) {
        const size_t off = (size_t)(gamma * 128 + lane * 4 + 2 * j) * 4;
#pragma unroll
        for (int p = 0; p < B; ++p) cp_async8(slot + (p * 32 + lane) * 8, src.p[p] + off);
      } else {
        const int cnt = min(2, rem - 2 * j);
        const size_t off = (size_t)(GR * 128 + lane * rem + 2 * j) * 4;
#pragma unroll
        for (int p = 0; p < B; ++p)
          for (int k = 0; k < cnt; ++k) cp_async4(slot + (p * 32 + lane) * 8 + 4 * k, src.p[p] + off + 4 * k);
      }
    }
  };

  // K-blocks 0 and 1 go with the first ring group
  stage_kblock(act, s_tok, ntok, K, 0, kbw, slab);
  if (kbs > 1) stage_kblock(act, s_tok, ntok, K, 1, kbw, slab + Cfg<NBLK>::SDELTA);
  int since_stage = 0;  // groups committed after the newest staging group
#pragma unroll
  for (int i = 0; i < R - 1; ++i) {
    if (i < mine) issue(i);
    cp_commit();
    if (i > 0) ++since_stage;
  }
  pre();
  int kb_cur = -1;
  auto advance_to = [&](int kb) {
    while (kb_cur < kb) {
      ++kb_cur;
      cp_wait_dyn(since_stage);  // this thread's copies of K-block kb_cur have landed
      __syncthreads();           // ... and everyone's; K-block kb_cur - 1 is no longer read
      if (kb_cur >= 1 && kb_cur + 1 < kbs) {
        stage_kblock(act, s_tok, ntok, K, kb_cur + 1, kbw, slab + ((kb_cur + 1) & 1) * Cfg<NBLK>::SDELTA);
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
    const int cb = u0 + i * us;
    const int kb = (cb * U::COLS) >> lkb;
    advance_to(kb);
    cp_wait<R - 1>();  // unit cb has landed
    const uint32_t buf = slab + (kb & 1) * Cfg<NBLK>::SDELTA;
    const int kc0 = (cb * U::COLS) & (kbw - 1);
    const uint32_t slot = ring + (i % R) * U::SLOT;
    if constexpr (KIND == KIND_F16) {
#pragma unroll
      for (int s = 0; s < kF16Steps; ++s) {
        const uint4 v = lds128(slot + (s * 32 + lane) * 16);
        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
        if constexpr (DUMP) {
          dump_frag(*dump, a, (kb << lkb) + kc0 + 16 * s);
        } else {
          uint32_t bf[G::NTM][2];
          slab_bstep(buf, kc0, s, NT, br, bf);
          mma_tiles(acc, a, bf, NT);
        }
      }
    } else {
      // 3 bits: the unit's words of every plane in one 16-byte load per
      // plane, chunks unrolled; 4..6 bits: each chunk reads its own word of
      // every plane (no selects between chunk words)
      constexpr int W = KIND == KIND_PG ? 4 : 2;  // words (chunks) per lane and plane
      uint32_t w[B][W];
      if constexpr (B == 3) {
#pragma unroll
        for (int p = 0; p < B; ++p) {
          const uint4 v = lds128(slot + (p * 32 + lane) * 16);
          w[p][0] = v.x;
          w[p][1] = v.y;
          w[p][2] = v.z;
          w[p][3] = v.w;
        }
      }
      const int nch = W == 4 ? (cb < GR ? 4 : rem) : (cb >> 1) < GR ? 2 : min(2, rem - 2 * (cb & 1));
      // the four mma steps of chunk c into A fragments a[s]
      auto decode = [&](int c, uint32_t (&a)[4][4]) {
        uint32_t wc[B];
#pragma unroll
        for (int p = 0; p < B; ++p) {
          if constexpr (B == 3) wc[p] = c == 0 ? w[p][0] : c == 1 ? w[p][1] : c == 2 ? w[p][2] : w[p][3];
          else wc[p] = lds32(slot + (p * 32 + lane) * (4 * W) + 4 * c);
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if constexpr (B == 3) decode_step_prmt3(wc, s, src.lut3, a[s]);
          else if constexpr (Cfg<NBLK>::LANE) decode_step_px<B>(wc, s, src.qbit, src.tabl, a[s]);
          else decode_step_rt<B, Cfg<NBLK>::TSHIFT>(wc, s, src.tabl, a[s]);
        }
      };
      auto mma = [&](int c, const uint32_t (&a)[4][4]) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if constexpr (DUMP) {
            dump_frag(*dump, a[s], (kb << lkb) + kc0 + c * 64 + 16 * s);
          } else {
            uint32_t bf[G::NTM][2];
            slab_bstep(buf, kc0 + c * 64, s, NT, br, bf);
            mma_tiles(acc, a[s], bf, NT);
          }
        }
      };
      // decode a chunk's four steps first (independent chains), then its mma's
      auto chunk = [&](int c) {
        uint32_t a[4][4];
        decode(c, a);
        mma(c, a);
      };
      if constexpr (B == 3) {
        // register-LUT decode is short: the unit's chunks unrolled (independent chains)
#pragma unroll
        for (int c = 0; c < W; ++c)
          if (c < nch) chunk(c);
      } else if constexpr (Cfg<NBLK>::LANE) {
        // table lookups, two chunks at a time: twice the independent chains
        // for the two resident warps per scheduler (registers allow it here)
        int c = 0;
#pragma unroll 1
        for (; c + 1 < nch; c += 2) {
          uint32_t a0[4][4], a1[4][4];
          decode(c, a0);
          decode(c + 1, a1);
          mma(c, a0);
          mma(c + 1, a1);
        }
        if (c < nch) chunk(c);
      } else {
        // table lookups: the chunks share one copy of the code
#pragma unroll 1
        for (int c = 0; c < nch; ++c) chunk(c);
      }
    }
  }
  advance_to(kbs - 1);
  cp_wait<0>();
}

// K loop of one warp over two 16-row tiles of 3-bit codes at once (wide
// gate/up items of the per-lane-table configuration): the ring holds both
// tiles' plane groups side by side, so the tiles share every staged K-block
// and every B fragment, and each chunk decodes two independent tiles.  Same
// staging, ring discipline and decode (byte permutes from register LUTs) as
// kloop; DUMP writes both tiles' A fragments instead of feeding the mma.
template <int NBLK, bool DUMP = false>
__device__ __forceinline__ void kloop3w(const WSrc (&src)[2], int K, int NT, int ntok, uint32_t ring, uint32_t slab,
                                        const __half* act, const int* s_tok, float (&acc)[2][Geo::NTM][4],
                                        const Dump* dump = nullptr) {
  using G = Geo;
  constexpr int SLOT = 2 * 3 * 16 * 32;  // both tiles' three planes, 16 bytes per lane each
  constexpr int R = Cfg<NBLK>::RB / SLOT > 8 ? 8 : Cfg<NBLK>::RB / SLOT;
  static_assert(R >= 3, "ring too shallow");
  const int lane = threadIdx.x & 31;
  const int lkb = kblock_log2(ntok), kbw = 1 << lkb, rs = kbw * 2;
  const int nk = K / 64, GR = nk / 4, rem = nk % 4;
  const int nu = (K + 255) / 256;
  const int kbs = (K + kbw - 1) / kbw;
  const BRows br = slab_brows(ntok, rs);

  auto issue = [&](int cb) {
    const uint32_t slot = ring + (cb % R) * SLOT;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (cb < GR) {
        const size_t off = (size_t)(cb * 128 + lane * 4) * 4;
#pragma unroll
        for (int p = 0; p < 3; ++p) cp_async16(slot + ((j * 3 + p) * 32 + lane) * 16, src[j].p[p] + off);
      } else {
        const size_t off = (size_t)(GR * 128 + lane * rem) * 4;
#pragma unroll
        for (int p = 0; p < 3; ++p)
          for (int k = 0; k < rem; ++k)
            cp_async4(slot + ((j * 3 + p) * 32 + lane) * 16 + 4 * k, src[j].p[p] + off + 4 * k);
      }
    }
  };

  stage_kblock(act, s_tok, ntok, K, 0, kbw, slab);
  if (kbs > 1) stage_kblock(act, s_tok, ntok, K, 1, kbw, slab + Cfg<NBLK>::SDELTA);
  int since_stage = 0;
#pragma unroll
  for (int i = 0; i < R - 1; ++i) {
    if (i < nu) issue(i);
    cp_commit();
    if (i > 0) ++since_stage;
  }
  int kb_cur = -1;
  auto advance_to = [&](int kb) {
    while (kb_cur < kb) {
      ++kb_cur;
      cp_wait_dyn(since_stage);
      __syncthreads();
      if (kb_cur >= 1 && kb_cur + 1 < kbs) {
        stage_kblock(act, s_tok, ntok, K, kb_cur + 1, kbw, slab + ((kb_cur + 1) & 1) * Cfg<NBLK>::SDELTA);
        cp_commit();
        since_stage = 0;
      }
    }
  };

#pragma unroll 1
  for (int cb = 0; cb < nu; ++cb) {
    if (cb + R - 1 < nu) issue(cb + R - 1);
    cp_commit();
    ++since_stage;
    const int kb = (cb * 256) >> lkb;
    advance_to(kb);
    cp_wait<R - 1>();  // unit cb has landed
    const uint32_t buf = slab + (kb & 1) * Cfg<NBLK>::SDELTA;
    const int kc0 = (cb * 256) & (kbw - 1);
    const uint32_t slot = ring + (cb % R) * SLOT;
    uint32_t w[2][3][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        const uint4 v = lds128(slot + ((j * 3 + p) * 32 + lane) * 16);
        w[j][p][0] = v.x;
        w[j][p][1] = v.y;
        w[j][p][2] = v.z;
        w[j][p][3] = v.w;
      }
    const int nch = cb < GR ? 4 : rem;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c >= nch) break;
      uint32_t a[2][4][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t wc[3] = {w[j][0][c], w[j][1][c], w[j][2][c]};
#pragma unroll
        for (int s = 0; s < 4; ++s) decode_step_prmt3(wc, s, src[j].lut3, a[j][s]);
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if constexpr (DUMP) {
          dump_frag(dump[0], a[0][s], (kb << lkb) + kc0 + c * 64 + 16 * s);
          dump_frag(dump[1], a[1][s], (kb << lkb) + kc0 + c * 64 + 16 * s);
        } else {
          uint32_t bf[G::NTM][2];
          slab_bstep(buf, kc0 + c * 64, s, NT, br, bf);
          mma_tiles(acc[0], a[0][s], bf, NT);
          mma_tiles(acc[1], a[1][s], bf, NT);
        }
      }
    }
  }
  advance_to(kbs - 1);
  cp_wait<0>();
}

// Epilogue of one tile: C fragment element (row g / g+8, token nt*8 + 2t + {0,1}).
// Gate/up: h = silu(gate) * up in fp16; down: y in fp32.
__device__ __forceinline__ void tile_store_h(const float (&gt)[Geo::NTM][4], const float (&up)[Geo::NTM][4], int tau,
                                             int row0, int ntok, int ld, __half* h) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < Geo::NTM; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = nt * 8 + 2 * t + (r & 1);
      const int row = tau * kTileRows + g + 8 * (r >> 1);
      if (j < ntok) h[(size_t)(row0 + j) * ld + row] = __float2half_rn(silu_f(gt[nt][r]) * up[nt][r]);
    }
}

__device__ __forceinline__ void tile_store_y(const float (&acc)[Geo::NTM][4], int tau, int row0, int ntok, int ld,
                                             float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < Geo::NTM; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = nt * 8 + 2 * t + (r & 1);
      const int row = tau * kTileRows + g + 8 * (r >> 1);
      if (j < ntok) y[(size_t)(row0 + j) * ld + row] = acc[nt][r];
    }
}

// Weight sources of tile t of matrix m (expert e, or the shared FFN) for one
// warp: page-table addresses of its planes or fp16 tile, and for 3 bits the
// register LUTs of the lane's rows.  Returns the tile's LUT_B rows, from which
// a 4..6-bit warp builds its shared table (null otherwise).  B: 16, 3, 4, 5, 6.
template <int B, int NBLK>
__device__ __forceinline__ const __half* tile_src(const DevLayer& L, int e, bool sh, int m, int t, int K,
                                                  uint32_t tab, WSrc& src) {
  const int lane = threadIdx.x & 31;
  if constexpr (B == 16) {
    src.p[0] = sh ? reinterpret_cast<const char*>(L.shared16[m]) + (size_t)t * 32 * K : tile_addr(L, e, m, kPlanes, t);
    return nullptr;
  } else if constexpr (B == 3) {
#pragma unroll
    for (int p = 0; p < 3; ++p) src.p[p] = tile_addr(L, e, m, p, t);
    const __half* lr = lut_rows(L, e, m, 3, t * kTileRows);
    load_lut3(lr + (lane >> 2) * 8, src.lut3[0]);
    load_lut3(lr + ((lane >> 2) + 8) * 8, src.lut3[1]);
    return nullptr;
  } else {
#pragma unroll
    for (int p = 0; p < kPlanes; ++p) src.p[p] = p < B ? tile_addr(L, e, m, p, t) : nullptr;
    if constexpr (Cfg<NBLK>::LANE) {
      const int warp = threadIdx.x >> 5;
      src.tabl = Cfg<NBLK>::TAB_AT + (warp & 1) * 128 + lane * 4;
      src.qbit = (warp >> 1) ? 0x01010101u : 0u;
    } else {
      src.tabl = tab + (lane >> 2) * 4;
    }
    return lut_rows(L, e, m, B, t * kTileRows);
  }
}

struct ItemArgs {
  const __half* act;  // token rows of this phase
  int e;              // expert (routed)
  bool sh;            // shared FFN
  int b;              // bitwidth
  int K, NT, row0, ntok, ld;
  __half* h;
  float* y;
};

// One item.  Gate/up (NM = 2): warps 0-1 stream the gate rows of tiles tau
// and tau + 1, warps 2-3 their up rows.  Down (NM = 1): S warps share each
// tile (S = 1: warp w takes tile tau + w; S = 2: tiles tau, tau + 1; S = 4:
// tile tau), slice k of a tile taking every S-th unit from unit k.  Partial
// and up sums go through shared memory to the first warp of each tile, which
// adds them in warp order and stores.  B: 16 (fp16 page), 3, 4, 5 or 6.
template <int B, int NBLK>
__device__ __forceinline__ void block_item(const DevLayer& L, const ItemArgs& A, int NM, int S, int tau,
                                           uint32_t ring, uint32_t slab, uint32_t tab, const int* s_tok) {
  constexpr int kNT = Geo::NTM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = NM == 2 ? warp & 1 : warp;  // warp index within its matrix
  const int t = tau + q / S;                 // this warp's tile
  const int slice = q % S;
  const int m = NM == 2 ? warp >> 1 : 2;     // and matrix
  float acc[kNT][4] = {};
  WSrc src;
  const __half* lr = tile_src<B, NBLK>(L, A.e, A.sh, m, t, A.K, tab, src);
  if constexpr (B == 16) {
    kloop<KIND_F16, 16, NBLK>(src, A.K, A.NT, A.ntok, slice, S, ring, slab, A.act, s_tok, acc, [] {});
  } else if constexpr (B == 3) {
    kloop<KIND_PG, 3, NBLK>(src, A.K, A.NT, A.ntok, slice, S, ring, slab, A.act, s_tok, acc, [] {});
  } else {
    kloop<Cfg<NBLK>::LANE ? KIND_PG : KIND_PB, B, NBLK>(src, A.K, A.NT, A.ntok, slice, S, ring, slab, A.act,
                                                          s_tok, acc, [&] { build_tab_warp<NBLK>(lr, B, tab); });
  }
  if (NM == 1 && S == 1) {
    tile_store_y(acc, t, A.row0, A.ntok, A.ld, A.y);
    return;
  }
  __syncthreads();  // the staged rows are no longer read
  float4* red = reinterpret_cast<float4*>(__cvta_shared_to_generic(slab));
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
    red[(warp * kNT + nt) * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  __syncthreads();
  if (slice != 0 || m == 1) return;
  // warp order: slices of the tile's (gate) rows, then of its up rows
  auto add = [&](float (&sum)[kNT][4], int w) {
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const float4 v = red[(w * kNT + nt) * 32 + lane];
      sum[nt][0] += v.x;
      sum[nt][1] += v.y;
      sum[nt][2] += v.z;
      sum[nt][3] += v.w;
    }
  };
  for (int k = 1; k < S; ++k) add(acc, warp + k);
  if (NM == 1) {
    tile_store_y(acc, t, A.row0, A.ntok, A.ld, A.y);
  } else {
    float up[kNT][4] = {};
    for (int k = 0; k < S; ++k) add(up, 2 + warp + k);
    tile_store_h(acc, up, t, A.row0, A.ntok, A.ld, A.h);
  }
}

// Wide gate/up item of 3-bit codes (per-lane-table configuration): tiles
// tau .. tau + 3; warp q = 0, 1 streams the gate rows of tiles tau + 2q and
// tau + 2q + 1 (kloop3w), warps 2-3 their up rows; up sums reach the gate
// warps through shared memory for SwiGLU.
template <int NBLK>
__device__ __forceinline__ void block_item3w(const DevLayer& L, const ItemArgs& A, int tau, uint32_t ring,
                                             uint32_t slab, const int* s_tok) {
  constexpr int kNT = Geo::NTM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = warp >> 1, t0 = tau + 2 * (warp & 1);
  WSrc src[2];
  tile_src<3, NBLK>(L, A.e, A.sh, m, t0, A.K, 0, src[0]);
  tile_src<3, NBLK>(L, A.e, A.sh, m, t0 + 1, A.K, 0, src[1]);
  float acc[2][kNT][4] = {};
  kloop3w<NBLK>(src, A.K, A.NT, A.ntok, ring, slab, A.act, s_tok, acc);
  __syncthreads();  // the staged rows are no longer read
  float4* red = reinterpret_cast<float4*>(__cvta_shared_to_generic(slab));
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
      red[((warp * 2 + j) * kNT + nt) * 32 + lane] =
          make_float4(acc[j][nt][0], acc[j][nt][1], acc[j][nt][2], acc[j][nt][3]);
  __syncthreads();
  if (m == 1) return;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float up[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const float4 v = red[(((2 + warp) * 2 + j) * kNT + nt) * 32 + lane];
      up[nt][0] = v.x;
      up[nt][1] = v.y;
      up[nt][2] = v.z;
      up[nt][3] = v.w;
    }
    tile_store_h(acc[j], up, t0 + j, A.row0, A.ntok, A.ld, A.h);
  }
}

// Gate/up items of a 3-bit group are wide (four tiles) in the per-lane-table
// configuration when the group's tiles come in fours.
template <int NBLK>
__device__ __forceinline__ bool wide3(int b, int tiles) {
  return Cfg<NBLK>::LANE && b == 3 && (tiles & 3) == 0;
}

// Warps sharing one down tile for a group of n tokens with reduction length
// K: reductions of 4096 columns or more are split in four (up to 8 tokens,
// 1024-column K-blocks) or two (up to 16 tokens, 512-column K-blocks), so
// every K-block still gives each warp of a tile a share of whole units.
// Only batches of at most 16 tokens (SPLITK) split; larger ones fill the GPU
// with whole tiles and run a kernel without the split paths.
template <bool SPLITK>
__device__ __forceinline__ int down_split(int n, int K) {
  return !SPLITK || K < 4096 || n > 16 ? 1 : n > 8 ? 2 : 4;
}

__device__ __forceinline__ bool is_tab(int b) { return b >= 4 && b <= 6; }

// Shared-memory addresses of this warp's buffers (Cfg).  NBLK = 2 checks
// that its fixed layout lies inside the CTA's window; false (after flagging
// kErrLayout) when it does not.
template <int NBLK>
__device__ __forceinline__ bool cta_layout(const unsigned char* dyn_base, int* err, uint32_t& slab, uint32_t& tab,
                                           uint32_t& ring) {
  using CF = Cfg<NBLK>;
  const int warp = threadIdx.x >> 5;
  const uint32_t o = smem_u32(dyn_base);
  if constexpr (CF::LANE) {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (o + kCtaWarps * CF::RB > CF::SLAB0 || o + dyn < CF::END) {
      if (threadIdx.x == 0) atomicExch(err, kErrLayout);
      return false;
    }
    slab = CF::SLAB0;
    tab = CF::TAB_AT;
    ring = o + warp * CF::RB;
  } else {
    slab = o;
    tab = o + 2 * Geo::HALF + warp * CF::TABW;
    ring = o + 2 * Geo::HALF + kCtaWarps * CF::TABW + warp * CF::RB;
  }
  return true;
}

template <bool SPLITK, bool FUSED, int NBLK>
__global__ void __launch_bounds__(kCtaThreads, NBLK) ffn_cta_kernel(UniParams P) {
  using G = Geo;
  using CF = Cfg<NBLK>;
  extern __shared__ __align__(128) unsigned char smem_uni[];
  __shared__ int s_base[kMaxExperts + 1];   // first input row of each group
  __shared__ int s_n[kMaxExperts + 1];      // tokens of each group
  __shared__ short s_b[kMaxExperts + 1];    // bitwidth of each group
  __shared__ short s_ord[kMaxExperts + 1];  // groups in claim order
  __shared__ int s_pref[2][kMaxExperts + 2];  // claim position of each group's gate/up and down segment
  __shared__ short s_ins[kMaxExperts + 1];
  __shared__ int s_ng, s_it, s_total, s_total1;
  __shared__ int s_tok[G::TOK];
  __shared__ int s_pos[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  __shared__ short s_perm[FUSED ? kFusedSlots : 1];  // fused: token of each sorted slot
  __shared__ int s_last;

  const DevLayer& L = P.L;
  const int E = L.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // sync header: [0] item claims, [1] CTAs out, [4] down items done, [5]
  // route items claimed, [6] tokens routed, [8..8+T) route items done per token
  int* const q = L.sync;
  int* const done0 = L.sync + kSyncHeader;           // [E+1][kSyncChunks] gate/up tiles done
  int* const done1 = done0 + (E + 1) * kSyncChunks;  // [E+1][kSyncChunks] down tiles done

  uint32_t slab, tab, ring;  // K-block buffer 0, this warp's LUT table and weight ring
  if (!cta_layout<NBLK>(smem_uni, L.err, slab, tab, ring)) return;  // uniform: nothing touched yet

  const int n_slots = P.T * L.K;  // routed slots (fused step)
  if constexpr (FUSED) {
    // The router (sums in the order of pw_route.cuh, so idx and w equal the
    // router kernel's bit for bit).  Items (token t, four units of (4
    // experts, 1024-column slice)) are claimed from a counter, one unit per
    // warp; the CTA that completes a token's last item adds its slice sums
    // and selects its experts.  Every CTA then waits (bounded) until all
    // tokens are routed: the items were claimed by running CTAs that wait on
    // nothing, so the wait ends.
    {
      const int d8 = L.d / 8, ns = route_slices(L.d), nb = (E + kRouteEB - 1) / kRouteEB;
      const int nunits = nb * ns, ngroups = (nunits + kCtaWarps - 1) / kCtaWarps;
      const int total = P.T * ngroups;
      int* const rclaim = q + 5;  // route items claimed
      int* const rdone = q + 6;   // tokens routed
      int* const tokcnt = q + 8;  // [T] items done per token
      float* const lg = reinterpret_cast<float*>(smem_uni);  // [E] logits of a token being finished
      for (;;) {
        if (tid == 0) s_it = atomicAdd(rclaim, 1);
        __syncthreads();
        const int it = s_it;
        if (it >= total) break;
        const int t = it / ngroups, u = (it - t * ngroups) * kCtaWarps + warp;
        if (u < nunits) {
          const int e0 = (u / ns) * kRouteEB, sl = u % ns;
          uint4 wv[kRouteEB][kRoutePieces];
          route_load_w(P.wr, d8, E, e0, sl, lane, wv);
          const uint4* x4 = reinterpret_cast<const uint4*>(P.x) + (size_t)t * d8;
          float acc[kRouteEB] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < kRoutePieces; ++i) {
            const int c = (sl * kRoutePieces + i) * 32 + lane;
            if (c < d8) {
              const uint4 xv = x4[c];
#pragma unroll
              for (int qq = 0; qq < kRouteEB; ++qq) acc[qq] += dot8(wv[qq][i], xv);
            }
          }
#pragma unroll
          for (int qq = 0; qq < kRouteEB; ++qq) {
            const float v = route_warp_sum(acc[qq]);
            if (lane == 0 && e0 + qq < E) P.rpart[((size_t)t * ns + sl) * E + e0 + qq] = v;
          }
        }
        __syncthreads();  // this item's sums are written
        if (tid == 0) {
          __threadfence();
          s_last = atomicAdd(tokcnt + t, 1) == ngroups - 1;
        }
        __syncthreads();
        if (s_last) {
          __threadfence();
          for (int e = tid; e < E; e += kCtaThreads) {
            float v = P.bias ? P.bias[e] : 0.f;
            for (int sl = 0; sl < ns; ++sl) v += __ldcg(P.rpart + ((size_t)t * ns + sl) * E + e);
            lg[e] = v;
          }
          __syncthreads();
          if (warp == 0) route_select(lg, E, L.K, L.renorm, P.idx + (size_t)t * L.K, P.wk + (size_t)t * L.K, nullptr);
          if (tid == 0) {  // lane 0 of warp 0 wrote this token's idx / w
            tokcnt[t] = 0;  // back to zero for the next launch
            __threadfence();
            atomicAdd(rdone, 1);
          }
        }
      }
      if (tid == 0) {
        long long spins = 0;
        while (ld_acquire(rdone) < P.T) {
          if (++spins > L.spin_limit) {
            atomicExch(L.err, kErrTimeout);
            break;
          }
          __nanosleep(100);
        }
      }
      __syncthreads();
    }
    // slot counts per expert from the routing result (written in this launch
    // by other CTAs: read through L2), then their prefix
    for (int g = tid; g <= E; g += kCtaThreads) s_n[g] = 0;
    __syncthreads();
    for (int i = tid; i < n_slots; i += kCtaThreads) {
      const int e = __ldcg(P.idx + i);
      if ((unsigned)e < (unsigned)E) atomicAdd(&s_n[e], 1);
      else atomicExch(L.err, kErrRouting);  // not a routing result: the slot is dropped
    }
    __syncthreads();
    if (warp == 0) {
      int run = 0;
      for (int g0 = 0; g0 < E; g0 += 32) {
        const int g = g0 + lane;
        const int c = g < E ? s_n[g] : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (g < E) s_base[g] = run + incl - c;
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncthreads();
    if (blockIdx.x == 0 && P.offsets_out)
      for (int g = tid; g <= E; g += kCtaThreads) P.offsets_out[g] = g < E ? s_base[g] : n_slots;
    // token of every sorted slot (stable: ascending flat order inside an
    // expert), one warp, 32 slots at a time; s_pref[0] holds the running
    // position of each expert meanwhile
    if (warp == 0) {
      constexpr int kBatches = kFusedSlots / 32;
      int ev[kBatches];  // every slot's expert, loaded at once (one memory round trip)
#pragma unroll
      for (int b = 0; b < kBatches; ++b) {
        const int j = b * 32 + lane;
        ev[b] = j < n_slots ? min(max(__ldcg(P.idx + j), 0), E - 1) : -1 - lane;
      }
      for (int g = lane; g < E; g += 32) s_pref[0][g] = s_base[g];
      __syncwarp();
#pragma unroll
      for (int b = 0; b < kBatches; ++b) {
        if (b * 32 < n_slots) {
          const int j = b * 32 + lane, e = ev[b];
          const unsigned same = __match_any_sync(0xffffffffu, e);
          if (j < n_slots) {
            const int pos = s_pref[0][e] + __popc(same & ((1u << lane) - 1));
            if (pos < kFusedSlots) s_perm[pos] = (short)(j / L.K);
          }
          __syncwarp();
          if (j < n_slots && (same & ((1u << lane) - 1)) == 0) s_pref[0][e] += __popc(same);
          __syncwarp();
        }
      }
    }
    __syncthreads();
  }
  for (int g = tid; g <= E; g += kCtaThreads) {
    int base = 0, n = 0, b = 16;
    if (g < E) {
      if (FUSED) {
        base = s_base[g];
        n = s_n[g];
        b = L.bits[g];
      } else if (P.offsets) {
        // the caller's bucket, clamped to the slot rows [0, T*K): a bad table
        // flags the layer's error word and nothing is read or written outside
        const int o0 = P.offsets[g], o1 = P.offsets[g + 1];
        base = min(max(o0, 0), n_slots);
        n = min(max(o1, base), n_slots) - base;
        if (o0 < 0 || o1 < o0 || o1 > n_slots) atomicExch(L.err, kErrOffsets);
        b = L.bits[g];
        const bool take = (b == 3 && (P.bit_mask & 1)) || (b == 16 && (P.bit_mask & 2)) ||
                          (is_tab(b) && (P.bit_mask & 4));
        if (!take || n > P.max_tokens) n = 0;
      }
    } else if (P.x && L.fs) {  // the shared FFN (x doubles as the routed input of a fused step)
      n = P.T;
    }
    s_base[g] = base;
    s_n[g] = n;
    s_b[g] = (short)b;
  }
  __syncthreads();
  if (warp == 0) {
    // claim order: shared FFN, fp16 experts, 4..6-bit experts, 3-bit experts
    int ng = 0;
    for (int pass = 0; pass < 4; ++pass) {
      for (int g0 = 0; g0 <= E; g0 += 32) {
        const int g = g0 + lane;
        bool in = false;
        if (g <= E && s_n[g] > 0) {
          const int b = s_b[g];
          in = pass == 0 ? g == E : g == E ? false : pass == 1 ? b == 16 : pass == 2 ? is_tab(b) : b == 3;
        }
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (in) s_ord[ng + __popc(m & ((1u << lane) - 1))] = (short)g;
        ng += __popc(m);
      }
    }
    __syncwarp();
    for (int ph = 0; ph < 2; ++ph) {
      int run = 0;
      for (int k0 = 0; k0 < ng; k0 += 32) {
        const int k = k0 + lane;
        int c = 0;
        if (k < ng) {
          const int g = s_ord[k];
          const int fe = g == E ? L.fs : L.f;
          const int tiles = ph == 0 ? fe / kTileRows : L.d / kTileRows;
          const int per_item = ph == 0 ? (wide3<NBLK>(s_b[g], tiles) ? 4 : 2)
                                       : kCtaWarps / down_split<SPLITK>(s_n[g], fe);
          c = ((s_n[g] + G::TOK - 1) / G::TOK) * (tiles / per_item);
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
    // s_pref[ph] holds prefix counts C_ph of the segments.  The down segment
    // of group k goes in front of the first gate/up segment that starts at
    // least two waves (2 gridDim.x items) of gate/up items after the end of
    // k's own gate/up segment, or after all of them; so down items never
    // precede their gate/up items, and those are usually done when they are
    // claimed (measured against one wave: Mixtral-shaped layer at 64 tokens
    // 0.521 -> 0.513 ms, the Qwen-shaped one unchanged).
    __syncwarp();
    constexpr int kPer = (kMaxExperts + 1 + 31) / 32;
    const int wave = 2 * (int)gridDim.x;
    int ins[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int k = lane + 32 * i;
      ins[i] = ng;
      if (k < ng) {
        const int target = s_pref[0][k + 1] + wave;
        int lo = k + 1, hi = ng;  // first j in [k + 1, ng] with C_0[j] >= target
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (s_pref[0][mid] >= target) hi = mid; else lo = mid + 1;
        }
        ins[i] = lo;
        s_ins[k] = (short)lo;
      }
    }
    __syncwarp();
    int p0[kPer], p1[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int k = lane + 32 * i;
      p0[i] = p1[i] = 0;
      if (k < ng) {
        p1[i] = s_pref[0][ins[i]] + s_pref[1][k];
        int lo = 0, hi = ng;  // down segments placed in front of gate/up segment k
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (s_ins[mid] <= k) lo = mid + 1; else hi = mid;
        }
        p0[i] = s_pref[0][k] + s_pref[1][lo];
      }
    }
    const int total = s_pref[0][ng] + s_pref[1][ng];
    const int total1 = s_pref[1][ng];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int k = lane + 32 * i;
      if (k < ng) {
        s_pref[0][k] = p0[i];
        s_pref[1][k] = p1[i];
      }
    }
    if (lane == 0) {
      s_ng = ng;
      s_total = total;
      s_total1 = total1;
    }
  }
  for (;;) {
    if (tid == 0) s_it = atomicAdd(q, 1);
    __syncthreads();  // also: the previous item no longer reads shared memory
    const int ng = s_ng;
    const int it = s_it;
    if (it >= s_total) break;
    // the segment holding item it: the latest segment start at or before it
    int sk[2];
#pragma unroll
    for (int ph = 0; ph < 2; ++ph) {
      int lo = -1, hi = ng - 1;  // last k with s_pref[ph][k] <= it (-1: none)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pref[ph][mid] <= it) lo = mid; else hi = mid - 1;
      }
      sk[ph] = lo;
    }
    const int phase = sk[1] >= 0 && s_pref[1][sk[1]] > s_pref[0][sk[0]] ? 1 : 0;
    const int lo = phase ? sk[1] : sk[0];
    const int g = s_ord[lo];
    const bool sh = g == E;
    const int b = s_b[g];
    const int n = s_n[g];
    const int nch = (n + G::TOK - 1) / G::TOK;
    const int local = it - s_pref[phase][lo];
    const int blk = local / nch, chunk = local % nch;  // chunks of one tile block are claimed together
    const int fe = sh ? L.fs : L.f;
    const int tiles = phase == 0 ? fe / kTileRows : L.d / kTileRows;
    const int sidx = g * kSyncChunks + chunk;
    const int S = phase == 0 ? 1 : down_split<SPLITK>(n, fe);  // warps per tile
    const bool wide = phase == 0 && wide3<NBLK>(b, tiles);
    const int per_item = phase == 0 ? (wide ? 4 : 2) : kCtaWarps / S;  // tiles of one item

    ItemArgs A;
    A.e = g;
    A.sh = sh;
    A.b = b;
    A.row0 = s_base[g] + chunk * G::TOK;
    A.ntok = min(G::TOK, n - chunk * G::TOK);
    A.NT = (A.ntok + 7) >> 3;
    A.K = phase == 0 ? L.d : fe;
    A.act = phase == 0 ? (sh || FUSED ? P.x : P.xp) : (sh ? P.hs : P.h);
    A.ld = phase == 0 ? fe : L.d;
    A.h = sh ? P.hs : P.h;
    A.y = sh ? P.ys : P.y;

    if (FUSED && phase == 0 && !sh) {
      if (tid < A.ntok) s_tok[tid] = s_perm[min(A.row0 + tid, kFusedSlots - 1)];  // tokens of the item's slots
    } else if (tid < A.ntok) {
      s_tok[tid] = A.row0 + tid;
    }
    if (phase == 1 && tid == 0) {  // h of this chunk must be complete
      const int need = fe / kTileRows + L.wait_bias;
      long long spins = 0;
      while (ld_acquire(done0 + sidx) < need) {
        if (++spins > L.spin_limit) {
          atomicExch(L.err, kErrTimeout);
          break;
        }
        __nanosleep(100);
      }
    }
    __syncthreads();
    const int tau = blk * per_item;
    const int NM = phase == 0 ? 2 : 1;
    switch (b) {
      case 16: block_item<16, NBLK>(L, A, NM, S, tau, ring, slab, tab, s_tok); break;
      case 3:
        if constexpr (CF::LANE) {
          if (wide) {
            block_item3w<NBLK>(L, A, tau, ring, slab, s_tok);
            break;
          }
        }
        block_item<3, NBLK>(L, A, NM, S, tau, ring, slab, tab, s_tok);
        break;
      case 4: block_item<4, NBLK>(L, A, NM, S, tau, ring, slab, tab, s_tok); break;
      case 5: block_item<5, NBLK>(L, A, NM, S, tau, ring, slab, tab, s_tok); break;
      default: block_item<6, NBLK>(L, A, NM, S, tau, ring, slab, tab, s_tok); break;
    }
    __syncthreads();  // every tile of the item is stored
    if (tid == 0) {
      const int done_tiles = per_item;
      __threadfence();
      if (phase == 0) {
        atomicAdd(done0 + sidx, done_tiles);
      } else {
        if (atomicAdd(done1 + sidx, done_tiles) == tiles - done_tiles) {
          // the last down tiles of this (group, chunk) clear both counters
          atomicExch(done0 + sidx, 0);
          atomicExch(done1 + sidx, 0);
        }
        if (FUSED) atomicAdd(q + 4, 1);
      }
    }
  }

  if constexpr (FUSED) {
    // combine once every down item is done (all were claimed, none waits on a later one)
    if (tid == 0) {
      long long spins = 0;
      while (ld_acquire(q + 4) < s_total1) {
        if (++spins > L.spin_limit) {
          atomicExch(L.err, kErrTimeout);
          break;
        }
        __nanosleep(100);
      }
    }
    __syncthreads();
    const int K = L.K, d4 = L.d / 4;
    for (int t = blockIdx.x; t < P.T; t += gridDim.x) {
      for (int k = warp; k < K; k += kCtaWarps) {
        // sorted slot of (t, k): the one slot of token t in expert e's bucket
        const int flat = t * K + k, e = min(max(__ldcg(P.idx + flat), 0), E - 1);
        const int lo = s_base[e], hi = min(lo + s_n[e], kFusedSlots);
        int pos = lo;
        for (int p0 = lo; p0 < hi; p0 += 32) {
          const int pp = p0 + lane;
          const unsigned m = __ballot_sync(0xffffffffu, pp < hi && s_perm[pp] == t);
          if (m) {
            pos = p0 + __ffs(m) - 1;
            break;
          }
        }
        if (lane == 0) {
          s_pos[k] = pos;
          s_w[k] = __ldcg(P.wk + flat);
        }
      }
      __syncthreads();
      for (int c4 = tid; c4 < d4; c4 += kCtaThreads) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
          const float wkk = s_w[k];
          const float4 v = reinterpret_cast<const float4*>(P.y + (size_t)s_pos[k] * L.d)[c4];
          acc.x = fmaf(wkk, v.x, acc.x);
          acc.y = fmaf(wkk, v.y, acc.y);
          acc.z = fmaf(wkk, v.z, acc.z);
          acc.w = fmaf(wkk, v.w, acc.w);
        }
        if (P.ys) {
          const float4 v = reinterpret_cast<const float4*>(P.ys + (size_t)t * L.d)[c4];
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
        uint2 out;
        out.x = *reinterpret_cast<uint32_t*>(&lo);
        out.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(P.yout + (size_t)t * L.d)[c4] = out;
      }
      __syncthreads();
    }
  }

  if (tid == 0) {
    __threadfence();
    if (atomicAdd(q + 1, 1) == (int)gridDim.x - 1) {  // last CTA out: no claims remain
      atomicExch(q, 0);
      if (FUSED) {
        atomicExch(q + 4, 0);
        atomicExch(q + 5, 0);
        atomicExch(q + 6, 0);
      }
      atomicExch(q + 1, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// Debug: the decoded weights of expert e's matrix m exactly as this kernel
// produces them.  Each warp runs the K loop of one 16-row tile (same ring
// loads through the page table, same LUT set-up and decode routines as an
// item of the FFN kernel) with its A fragments written to out[rows][cols]
// instead of feeding the mma.
// ---------------------------------------------------------------------------
template <int B, int NBLK>
__device__ __forceinline__ void dump_tile(const DevLayer& L, int e, int m, int t, int C, uint32_t ring,
                                          uint32_t slab, uint32_t tab, const int* s_tok, const Dump& D) {
  float acc[Geo::NTM][4] = {};
  WSrc src;
  const __half* lr = tile_src<B, NBLK>(L, e, false, m, t, C, tab, src);
  if constexpr (B == 16) {
    kloop<KIND_F16, 16, NBLK, true>(src, C, 1, 0, 0, 1, ring, slab, D.out, s_tok, acc, [] {}, &D);
  } else if constexpr (B == 3) {
    kloop<KIND_PG, 3, NBLK, true>(src, C, 1, 0, 0, 1, ring, slab, D.out, s_tok, acc, [] {}, &D);
  } else {
    kloop<Cfg<NBLK>::LANE ? KIND_PG : KIND_PB, B, NBLK, true>(src, C, 1, 0, 0, 1, ring, slab, D.out, s_tok, acc,
                                  [&] { build_tab_warp<NBLK>(lr, B, tab); }, &D);
  }
}

template <int NBLK>
__global__ void __launch_bounds__(kCtaThreads) decode_dump_kernel(DevLayer L, int e, int m, __half* out) {
  extern __shared__ __align__(128) unsigned char smem_dump[];
  __shared__ int s_tok[Geo::TOK];
  const int warp = threadIdx.x >> 5;
  const int R = m < 2 ? L.f : L.d, C = m < 2 ? L.d : L.f;
  const int ntile = R / kTileRows;
  const int t = min((int)blockIdx.x * kCtaWarps + warp, ntile - 1);  // spare warps repeat the last tile unstored
  const Dump D{out, C, t * kTileRows, (int)blockIdx.x * kCtaWarps + warp < ntile};
  uint32_t slab, tab, ring;
  if (!cta_layout<NBLK>(smem_dump, L.err, slab, tab, ring)) return;
  if constexpr (Cfg<NBLK>::LANE) {
   if (m < 2 && L.bits[e] == 3 && wide3<NBLK>(3, ntile)) {
    // gate / up at 3 bits: the wide items' two-tile K loop, warp pair index
    // blockIdx.x * 4 + warp (tiles 2i, 2i + 1; spare warps repeat the last pair unstored)
    const int i = (int)blockIdx.x * kCtaWarps + warp, t0 = min(2 * i, ntile - 2);
    const Dump D2[2] = {{out, C, t0 * kTileRows, 2 * i < ntile}, {out, C, (t0 + 1) * kTileRows, 2 * i < ntile}};
    WSrc src[2];
    tile_src<3, NBLK>(L, e, false, m, t0, C, tab, src[0]);
    tile_src<3, NBLK>(L, e, false, m, t0 + 1, C, tab, src[1]);
    float acc[2][Geo::NTM][4] = {};
    kloop3w<NBLK, true>(src, C, 1, 0, ring, slab, out, s_tok, acc, D2);
    return;
   }
  }
  switch (L.bits[e]) {
    case 16: dump_tile<16, NBLK>(L, e, m, t, C, ring, slab, tab, s_tok, D); break;
    case 3: dump_tile<3, NBLK>(L, e, m, t, C, ring, slab, tab, s_tok, D); break;
    case 4: dump_tile<4, NBLK>(L, e, m, t, C, ring, slab, tab, s_tok, D); break;
    case 5: dump_tile<5, NBLK>(L, e, m, t, C, ring, slab, tab, s_tok, D); break;
    case 6: dump_tile<6, NBLK>(L, e, m, t, C, ring, slab, tab, s_tok, D); break;
    default:
      if (threadIdx.x == 0) atomicExch(L.err, kErrBits);
  }
}

// Dynamic shared memory of a launch of fn in configuration NBLK (NBLK = 2:
// its window up to Cfg::END).
template <int NBLK>
static cudaError_t cta_smem(const void* fn, size_t& bytes) {
  if (!Cfg<NBLK>::LANE) {
    bytes = Cfg<NBLK>::SMEM;
    return ensure_smem(fn, bytes);
  }
  return window_smem(fn, Cfg<NBLK>::END, bytes);
}

template <int NBLK>
static cudaError_t launch_decode_dump_cfg(const DevLayer& L, int e, int m, __half* out, cudaStream_t s) {
  const int R = m < 2 ? L.f : L.d;
  size_t smem = 0;
  cudaError_t err = cta_smem<NBLK>((const void*)decode_dump_kernel<NBLK>, smem);
  if (err != cudaSuccess) return err;
  const int ntile = R / kTileRows;
  decode_dump_kernel<NBLK><<<(ntile + kCtaWarps - 1) / kCtaWarps, kCtaThreads, smem, s>>>(L, e, m, out);
  return cudaGetLastError();
}

cudaError_t launch_decode_dump(const DevLayer& L, int e, int m, bool lane_tables, __half* out, cudaStream_t s) {
  return lane_tables ? launch_decode_dump_cfg<2>(L, e, m, out, s) : launch_decode_dump_cfg<3>(L, e, m, out, s);
}

// The configuration a layer's decode launches take (Cfg), chosen by the host
// per call (DevLayer::nblk, decode_nblk) -- both compute every item alike,
// so the choice only moves time.  PW_DECODE_NBLK=2 or 3 (read per call)
// overrides it.
int nblk_for(const DevLayer& L) {
  const char* s = getenv("PW_DECODE_NBLK");
  if (s && (s[0] == '2' || s[0] == '3') && s[1] == 0) return s[0] - '0';
  return L.nblk == 2 ? 2 : 3;
}

// Measured on one GB300 (Mixtral-shaped layer, every expert at one bitwidth,
// 64 tokens), as fractions of the HBM roofline, three CTAs / two CTAs per
// SM: fp16 pages 0.86 / 0.83, 6 bits 0.18 / 0.26, 5 bits 0.16 / 0.23, 4 bits
// 0.14 / 0.19, 3 bits 0.20 / 0.20 (wide 3-bit items in the second).  The
// per-lane tables win on 4..6-bit lookups and lose a third of the resident
// warps everywhere else; for a layer with experts of ffn >= 4096 rows the
// choice compares the time each configuration would take for the layer's
// bytes (bytes / fraction; bytes: fp16, 6, 5, 4, 3 bits).  Narrower experts
// get few tokens each and short items, where the resident warps matter
// more: measured, two CTAs per SM cost the Qwen-shaped layer (ffn 1408) 11%
// at 64 tokens and tie on the 128-expert one (ffn 704), so those take three.
int decode_nblk(const double (&bytes)[5], int ffn) {
  if (ffn < 4096) return 3;
  static constexpr double f3[5] = {0.86, 0.18, 0.16, 0.14, 0.20};
  static constexpr double f2[5] = {0.83, 0.26, 0.23, 0.19, 0.20};
  double t3 = 0, t2 = 0;
  for (int i = 0; i < 5; ++i) {
    t3 += bytes[i] / f3[i];
    t2 += bytes[i] / f2[i];
  }
  return t2 < t3 ? 2 : 3;
}

template <bool FUSED, int NBLK>
static cudaError_t launch_cta_cfg(const UniParams& P, int T, cudaStream_t s) {
  // The split paths depend on the batch size only, so a routed call, a shared
  // call and the combined call compute every item the same way.
  const bool splitk = T <= 16;
  const void* fn = splitk ? (const void*)ffn_cta_kernel<true, FUSED, NBLK>
                          : (const void*)ffn_cta_kernel<false, FUSED, NBLK>;
  size_t smem = 0;
  cudaError_t e;
  if ((e = cta_smem<NBLK>(fn, smem)) != cudaSuccess) return e;
  const int grid = sm_count() * NBLK;
  if (splitk) ffn_cta_kernel<true, FUSED, NBLK><<<grid, kCtaThreads, smem, s>>>(P);
  else ffn_cta_kernel<false, FUSED, NBLK><<<grid, kCtaThreads, smem, s>>>(P);
  return cudaGetLastError();
}

template <bool FUSED>
static cudaError_t launch_cta(const UniParams& P, int T, cudaStream_t s) {
  return nblk_for(P.L) == 2 ? launch_cta_cfg<FUSED, 2>(P, T, s) : launch_cta_cfg<FUSED, 3>(P, T, s);
}

cudaError_t launch_uni(const DevLayer& L, const __half* x, const __half* x_perm, const int* offsets, int T,
                       int bit_mask, int max_tokens, __half* h, __half* hs, float* y, float* ys, cudaStream_t s) {
  if (max_tokens > kSyncChunks * 16 || (x && T > kSyncChunks * 16)) return cudaErrorInvalidValue;
  if (!bit_mask && !x) return cudaSuccess;
  UniParams P{};
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
  return launch_cta<false>(P, T, s);
}

cudaError_t launch_layer_fused(const DevLayer& L, const __half* x, const __half* wr, const float* bias, int* idx,
                               float* w, float* rpart, int T, __half* h, __half* hs, float* y_perm, float* ys,
                               __half* y, int* offsets_out, cudaStream_t s) {
  static_assert(8 + kFusedMaxTokens <= kSyncHeader, "per-token router counters must fit the sync header");
  if (T < 1 || T > kFusedMaxTokens || T * L.K > kFusedSlots) return cudaErrorInvalidValue;
  UniParams P{};
  P.L = L;
  P.x = x;
  P.T = T;
  P.bit_mask = 7;
  P.max_tokens = T;
  P.h = h;
  P.hs = L.fs ? hs : nullptr;
  P.y = y_perm;
  P.ys = L.fs ? ys : nullptr;
  P.wr = wr;
  P.bias = bias;
  P.rpart = rpart;
  P.idx = idx;
  P.wk = w;
  P.yout = y;
  P.offsets_out = offsets_out;
  return launch_cta<true>(P, T, s);
}

}  // namespace pw
