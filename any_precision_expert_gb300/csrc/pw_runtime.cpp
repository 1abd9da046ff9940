// Host runtime: status codes, the page pool, the per-expert page table, layer
// lifecycle, bitwidth changes and argument validation for the hot-path calls.
//
// PagedWeight (zhichai.net/topic/178446964, "核心洞察") keeps each expert's
// bit-planes as pages so that precision can be lowered by detaching the low
// planes; "安全边界与异步搬运" commits changes at a safe boundary.  Here:
//  * a pool of fixed-size pages carved from one caller-owned device buffer;
//  * a plane block = plane p of gate/up/down of one expert, paged with no
//    16-row tile straddling a page; an fp16 block = the expert's fp16 page;
//  * the device page table holds the page base addresses of every block;
//  * lowering only rewrites the device bitwidth word (stream ordered) and moves
//    the freed blocks to a reclaim queue guarded by a CUDA event (the safe
//    boundary); raising re-maps blocks that are still intact.
#include <cuda.h>  // driver API types of the virtual-memory calls (looked up at run time)
#include <nvtx3/nvToolsExt.h>  // header-only NVTX ranges (no-ops unless a tool is attached)
#include <sys/mman.h>
#include <unistd.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <set>
#include <vector>

#include "pw_internal.h"

using namespace pw;

struct pw_pool_s;
struct pw_layer_s;

namespace {

thread_local int g_last_cuda = 0;
bool g_sim = false;                // host-simulated device (tests without a GPU)
uint64_t g_sim_issued = 0, g_sim_done = 0;

pw_status cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return PW_ERR_CUDA;
}

#define PW_CUDA(call)                                  \
  do {                                                 \
    cudaError_t _e = (call);                           \
    if (_e != cudaSuccess) return cuda_fail(_e);       \
  } while (0)

#define PW_TRY(call)                                   \
  do {                                                 \
    pw_status _s = (call);                             \
    if (_s != PW_OK) return _s;                        \
  } while (0)

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Ranges of the hot-path calls, when PW_NVTX=1 (read once) and a tool listens.
struct NvtxRange {
  static bool on() {
    static const bool v = [] {
      const char* e = getenv("PW_NVTX");
      return e && e[0] == '1';
    }();
    return v;
  }
  explicit NvtxRange(const char* name) {
    if (on()) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on()) nvtxRangePop();
  }
};

pw_status dev_h2d(void* dst, const void* src, size_t n, cudaStream_t s) {
  if (n == 0) return PW_OK;
  if (g_sim) {
    memcpy(dst, src, n);
    return PW_OK;
  }
  PW_CUDA(cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s));
  return PW_OK;
}

pw_status dev_d2d(void* dst, const void* src, size_t n, cudaStream_t s) {
  if (n == 0) return PW_OK;
  if (g_sim) {
    memcpy(dst, src, n);
    return PW_OK;
  }
  PW_CUDA(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, s));
  return PW_OK;
}

pw_status dev_zero(void* dst, size_t n, cudaStream_t s) {
  if (n == 0) return PW_OK;
  if (g_sim) {
    memset(dst, 0, n);
    return PW_OK;
  }
  PW_CUDA(cudaMemsetAsync(dst, 0, n, s));
  return PW_OK;
}

pw_status dev_sync(cudaStream_t s) {
  if (g_sim) return PW_OK;
  PW_CUDA(cudaStreamSynchronize(s));
  return PW_OK;
}

// CUDA virtual memory management (driver API), looked up once.  The library
// reserves virtual address ranges and maps the caller's physical pages into
// them; it never creates or releases physical memory.
struct VmmApi {
  CUresult (*reserve)(CUdeviceptr*, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
  CUresult (*release_va)(CUdeviceptr, size_t) = nullptr;
  CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long) = nullptr;
  CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
  CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc*, size_t) = nullptr;
  bool ok = false;
};

const VmmApi& vmm_api() {
  static VmmApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    auto get = [](const char* name, void** fn) {
      cudaDriverEntryPointQueryResult q;
      return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
             q == cudaDriverEntryPointSuccess && *fn != nullptr;
    };
    api.ok = get("cuMemAddressReserve", reinterpret_cast<void**>(&api.reserve)) &&
             get("cuMemAddressFree", reinterpret_cast<void**>(&api.release_va)) &&
             get("cuMemMap", reinterpret_cast<void**>(&api.map)) &&
             get("cuMemUnmap", reinterpret_cast<void**>(&api.unmap)) &&
             get("cuMemSetAccess", reinterpret_cast<void**>(&api.set_access));
  });
  return api;
}

// The safe boundary of one bitwidth change.
struct Event {
  cudaEvent_t ev = nullptr;
  uint64_t seq = 0;
  ~Event() {
    if (ev) cudaEventDestroy(ev);
  }
  bool done() const {
    if (g_sim) return seq <= g_sim_done;
    return cudaEventQuery(ev) == cudaSuccess;
  }
  void wait() const {
    if (!g_sim) cudaEventSynchronize(ev);
  }
};

pw_status make_event(cudaStream_t s, std::shared_ptr<Event>* out) {
  auto ev = std::make_shared<Event>();
  if (g_sim) {
    ev->seq = ++g_sim_issued;
  } else {
    PW_CUDA(cudaEventCreateWithFlags(&ev->ev, cudaEventDisableTiming));
    cudaError_t e = cudaEventRecord(ev->ev, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  *out = ev;
  return PW_OK;
}

enum BlockState { B_NONE = 0, B_MAPPED = 1, B_RECLAIM = 2 };

struct Block {
  BlockState st = B_NONE;
  char* va = nullptr;             // virtual-memory pools: the block's fixed address range
  std::vector<int> pages;         // physical page ids, indexed by virtual page
  std::shared_ptr<Event> ev;      // set while reclaimable
  std::shared_ptr<Event> ready;   // set while an asynchronous upload into the block may be in flight
  uint64_t fifo_key = 0;
};

}  // namespace

struct pw_pool_s {
  char* base = nullptr;
  size_t bytes = 0, page_bytes = 0, npages = 0;
  // virtual-memory pools: page p is the caller's physical allocation
  // handles[p], visible only where it is mapped (host-sim: a memfd page)
  bool vmm = false;
  int device = 0;
  std::vector<unsigned long long> handles;
  int sim_fd = -1;
  uint64_t n_map = 0, n_unmap = 0;
  std::set<int> free_pages;                 // ordered: paged blocks take the lowest ids
  std::vector<uint8_t> kind;                // 0 free, 1 paged, 2 resident
  std::map<uint64_t, Block*> reclaim;       // oldest first
  uint64_t fifo_counter = 0;
  size_t mapped_pages = 0, reclaim_pages = 0, resident_bytes = 0;
  int n_layers = 0;

  char* page_addr(int p) const { return base + (size_t)p * page_bytes; }

  // Map physical page p at va (one page, read/write for the pool's device).
  pw_status vmm_map(char* va, int p) {
    if (g_sim) {
      if (mmap(va, page_bytes, PROT_READ | PROT_WRITE, MAP_SHARED | MAP_FIXED, sim_fd, (off_t)p * page_bytes) ==
          MAP_FAILED)
        return PW_ERR_UNSUPPORTED;
    } else {
      const VmmApi& a = vmm_api();
      const CUdeviceptr d = reinterpret_cast<CUdeviceptr>(va);
      if (a.map(d, page_bytes, 0, handles[p], 0) != CUDA_SUCCESS) return PW_ERR_CUDA;
      CUmemAccessDesc acc{};
      acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
      acc.location.id = device;
      acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
      if (a.set_access(d, page_bytes, &acc, 1) != CUDA_SUCCESS) {
        a.unmap(d, page_bytes);
        return PW_ERR_CUDA;
      }
    }
    ++n_map;
    return PW_OK;
  }
  void vmm_unmap(char* va) {
    if (g_sim)
      mmap(va, page_bytes, PROT_NONE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_FIXED | MAP_NORESERVE, -1, 0);
    else
      vmm_api().unmap(reinterpret_cast<CUdeviceptr>(va), page_bytes);
    ++n_unmap;
  }
  // Reserve / free a virtual range of n pages (no physical memory).
  char* vmm_reserve(size_t n) {
    const size_t len = n * page_bytes;
    if (g_sim) {
      void* p = mmap(nullptr, len, PROT_NONE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_NORESERVE, -1, 0);
      return p == MAP_FAILED ? nullptr : static_cast<char*>(p);
    }
    CUdeviceptr d = 0;
    if (vmm_api().reserve(&d, len, page_bytes, 0, 0) != CUDA_SUCCESS) return nullptr;
    return reinterpret_cast<char*>(d);
  }
  void vmm_free(char* va, size_t n) {
    if (!va) return;
    if (g_sim) munmap(va, n * page_bytes);
    else vmm_api().release_va(reinterpret_cast<CUdeviceptr>(va), n * page_bytes);
  }

  void to_reclaim(Block& b, std::shared_ptr<Event> ev) {
    b.st = B_RECLAIM;
    b.ev = std::move(ev);
    b.fifo_key = ++fifo_counter;
    reclaim[b.fifo_key] = &b;
    mapped_pages -= b.pages.size();
    reclaim_pages += b.pages.size();
  }
  void remap(Block& b) {  // reclaimable -> mapped (raise)
    reclaim.erase(b.fifo_key);
    b.ev.reset();
    b.st = B_MAPPED;
    reclaim_pages -= b.pages.size();
    mapped_pages += b.pages.size();
  }
  void release(Block& b) {  // any state -> none, pages back to the free set
    if (b.st == B_RECLAIM) {
      reclaim.erase(b.fifo_key);
      reclaim_pages -= b.pages.size();
    } else if (b.st == B_MAPPED) {
      mapped_pages -= b.pages.size();
    }
    // virtual-memory pools unmap here, the only place a block gives up its
    // pages: after its safe boundary (reuse) or a synchronize (reload, destroy)
    if (vmm && b.st != B_NONE)
      for (size_t v = 0; v < b.pages.size(); ++v) vmm_unmap(b.va + v * page_bytes);
    for (int p : b.pages) {
      kind[p] = 0;
      free_pages.insert(p);
    }
    b.pages.clear();
    b.ev.reset();
    b.ready.reset();
    b.st = B_NONE;
  }
  // Whether take_pages may give up reclaimable block b (on a real device it
  // waits for the block's safe-boundary event; in host-sim mode pending
  // blocks are skipped).
  static bool reusable(const Block& b) { return !g_sim || b.ev->done(); }
  // Pages a take could use now: the free ones and those of reusable
  // reclaimable blocks.  Callers that take several blocks check their total
  // against this first, so that a request that cannot be met gives up no
  // reclaimable block.
  size_t reusable_pages() const {
    size_t n = free_pages.size();
    for (auto& kv : reclaim)
      if (reusable(*kv.second)) n += kv.second->pages.size();
    return n;
  }
  // Take n pages for a new mapped block.  Reclaimable blocks are given up
  // oldest first, and only once they are reusable.
  pw_status take_pages(size_t n, std::vector<int>* out) {
    if (reusable_pages() < n) return PW_ERR_OOM;
    while (free_pages.size() < n) {
      Block* victim = nullptr;
      for (auto& kv : reclaim)
        if (reusable(*kv.second)) {
          victim = kv.second;
          break;
        }
      if (!victim) return PW_ERR_OOM;
      victim->ev->wait();
      release(*victim);
    }
    out->clear();
    for (size_t i = 0; i < n; ++i) {
      int p = *free_pages.begin();
      free_pages.erase(free_pages.begin());
      kind[p] = 1;
      out->push_back(p);
    }
    mapped_pages += n;
    return PW_OK;
  }
  // n contiguous pages from the top of the buffer for resident data.
  int take_resident(size_t n) {
    if (n == 0 || n > npages) return -1;
    for (long top = (long)npages - 1; top >= (long)n - 1; --top) {
      bool ok = true;
      for (long i = top; i > top - (long)n; --i)
        if (kind[i] != 0) {
          ok = false;
          top = i;  // skip past the occupied page
          break;
        }
      if (ok) {
        int first = (int)(top - (long)n + 1);
        for (size_t i = 0; i < n; ++i) {
          kind[first + i] = 2;
          free_pages.erase(first + (int)i);
        }
        resident_bytes += n * page_bytes;
        return first;
      }
    }
    return -1;
  }
  void give_back_resident(int first, size_t n) {
    for (size_t i = 0; i < n; ++i) {
      kind[first + i] = 0;
      free_pages.insert(first + (int)i);
    }
    resident_bytes -= n * page_bytes;
  }
};

struct pw_layer_s {
  pw_pool_s* pool = nullptr;
  pw_layer_desc desc{};
  int R[3], C[3];
  int tmax = 0, pmax = 0, pmax16 = 0;
  std::vector<uint2> tmap, tmap16;           // [3][tmax]
  size_t lut_block_bytes = 0;
  unsigned lut_off[3][4];
  int res_first = -1;
  size_t res_npages = 0;
  char* res_base = nullptr;
  char* va = nullptr;    // virtual-memory pools: the layer's reserved range
  size_t va_pages = 0;
  // device tables (inside the resident run)
  int* d_bits = nullptr;
  int* d_err = nullptr;
  int* d_sync = nullptr;
  unsigned long long* d_plane_pt = nullptr;
  unsigned long long* d_f16_pt = nullptr;
  uint2* d_tmap = nullptr;
  uint2* d_tmap16 = nullptr;
  unsigned long long* d_lut_base = nullptr;
  char* d_luts = nullptr;
  __half* d_shared[3] = {nullptr, nullptr, nullptr};
  // host mirrors
  std::vector<int> bits;                     // 0 = not loaded
  std::vector<Block> planes;                 // [E][6]
  std::vector<Block> f16;                    // [E]
  std::vector<unsigned long long> h_plane_pt, h_f16_pt;
  bool shared_loaded = false;
  long long spin_limit = kDefaultSpinPolls;  // see pw_testing_wait_limit
  // workspace canaries (pw_layer_set_debug_bounds; PW_DEBUG_BOUNDS=1 turns them on for new layers)
  bool debug_bounds = [] {
    const char* e = getenv("PW_DEBUG_BOUNDS");
    return e && e[0] == '1';
  }();
  int wait_bias = 0;

  Block& plane(int e, int p) { return planes[(size_t)e * kPlanes + p]; }

  DevLayer dev() const {
    DevLayer L{};
    L.d = desc.d;
    L.f = desc.ffn;
    L.E = desc.n_experts;
    L.K = desc.top_k;
    L.renorm = desc.renormalize;
    L.fs = desc.shared_ffn;
    L.pmax = pmax;
    L.pmax16 = pmax16;
    L.tmax = tmax;
    L.bits = d_bits;
    L.plane_pt = d_plane_pt;
    L.f16_pt = d_f16_pt;
    L.tmap = d_tmap;
    L.tmap16 = d_tmap16;
    L.lut_base = d_lut_base;
    memcpy(L.lut_off, lut_off, sizeof(lut_off));
    for (int m = 0; m < 3; ++m) L.shared16[m] = shared_loaded ? d_shared[m] : nullptr;
    L.err = d_err;
    L.sync = d_sync;
    L.spin_limit = spin_limit;
    L.wait_bias = wait_bias;
    // decode-kernel configuration from the bytes the experts hold at their
    // current bitwidths (and the fp16 shared FFN)
    double by[5] = {3.0 * desc.d * desc.shared_ffn * 2, 0, 0, 0, 0};  // fp16, 6, 5, 4, 3 bits
    const double per_bit = 3.0 * desc.d * desc.ffn / 8;
    for (int b : bits) {
      if (b == 16) by[0] += per_bit * 16;
      else if (b >= 3 && b <= 6) by[7 - b] += per_bit * b;
    }
    L.nblk = decode_nblk(by, desc.ffn);
    return L;
  }
};

namespace {

// Lay tiles of the three matrices one after another into virtual pages, never
// letting a tile straddle a page.  Returns the number of virtual pages used.
int build_tile_map(const int R[3], const int C[3], size_t tile_bytes_per_col, size_t page_bytes,
                   int tmax, std::vector<uint2>* map) {
  map->assign((size_t)3 * tmax, make_uint2(0, 0));
  size_t vpage = 0, off = 0;
  for (int m = 0; m < 3; ++m) {
    const size_t tb = tile_bytes_per_col * (size_t)C[m];
    if (tb > page_bytes) return -1;
    for (int tau = 0; tau < R[m] / kTileRows; ++tau) {
      if (off + tb > page_bytes) {
        ++vpage;
        off = 0;
      }
      (*map)[(size_t)m * tmax + tau] = make_uint2((unsigned)vpage, (unsigned)off);
      off += tb;
    }
  }
  return (int)vpage + 1;
}

bool valid_bits(int b) { return b == 3 || b == 4 || b == 5 || b == 6 || b == 16; }

pw_status check_layer(pw_layer_t l) { return l ? PW_OK : PW_ERR_INVALID_ARG; }

// The stream-ordered write of a bitwidth word: a stream memory operation
// (cuStreamWriteValue32: the GPU's front end performs it in stream order, no
// kernel launch between the caller's kernels), or a one-thread kernel where
// the driver does not offer it.
using WriteValue32 = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
WriteValue32 write_value32() {
  static WriteValue32 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WriteValue32>(p);
  });
  return fn;
}

pw_status write_bits(pw_layer_t l, int e, int b, cudaStream_t s) {
  if (g_sim) {
    l->d_bits[e] = b;
    return PW_OK;
  }
  if (WriteValue32 fn = write_value32())
    if (fn(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(l->d_bits + e), (cuuint32_t)b,
           CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS)
      return PW_OK;
  PW_CUDA(launch_set_bits(l->d_bits, e, b, s));
  return PW_OK;
}

// Address of virtual page v of block b: its fixed virtual range in a
// virtual-memory pool, else the physical page's address in the buffer.
char* blk_addr(const pw_layer_s* l, const Block& b, int v) {
  return l->pool->vmm ? b.va + (size_t)v * l->pool->page_bytes : l->pool->page_addr(b.pages[v]);
}

// Give block b its pages (mapped at its virtual range in a virtual-memory pool).
pw_status attach_block(pw_layer_t l, Block& b, std::vector<int> pages) {
  b.pages = std::move(pages);
  b.st = B_MAPPED;
  if (l->pool->vmm)
    for (size_t v = 0; v < b.pages.size(); ++v) PW_TRY(l->pool->vmm_map(b.va + v * l->pool->page_bytes, b.pages[v]));
  return PW_OK;
}

pw_status upload_pt_rows(pw_layer_t l, int e, cudaStream_t s) {
  const size_t prow = (size_t)kPlanes * l->pmax;
  PW_TRY(dev_h2d(l->d_plane_pt + (size_t)e * prow, l->h_plane_pt.data() + (size_t)e * prow,
                 prow * sizeof(unsigned long long), s));
  PW_TRY(dev_h2d(l->d_f16_pt + (size_t)e * l->pmax16, l->h_f16_pt.data() + (size_t)e * l->pmax16,
                 (size_t)l->pmax16 * sizeof(unsigned long long), s));
  return PW_OK;
}

// Copy a block image (virtual pages) page by page to its physical pages.
pw_status upload_block(pw_layer_t l, const Block& b, const std::vector<char>& img, cudaStream_t s) {
  const size_t pb = l->pool->page_bytes;
  for (size_t v = 0; v < b.pages.size(); ++v) {
    const size_t n = std::min(pb, img.size() - v * pb);
    PW_TRY(dev_h2d(blk_addr(l, b, (int)v), img.data() + v * pb, n, s));
  }
  return PW_OK;
}

// Pages for the blocks an expert at `bits` reads: np plane blocks, plus the
// fp16 block at 16 bits (pages[np]).  All or nothing: a request the pool
// cannot meet is refused before any reclaimable block is given up.
pw_status take_expert_pages(pw_layer_t l, int bits, std::vector<std::vector<int>>* pages) {
  pw_pool_s* pool = l->pool;
  const int np = bits == 16 ? kPlanes : bits;
  if (pool->reusable_pages() < (size_t)np * l->pmax + (bits == 16 ? (size_t)l->pmax16 : 0)) return PW_ERR_OOM;
  pages->assign(np + 1, {});
  auto give_back = [&](int upto) {
    for (int q = 0; q < upto; ++q)
      for (int pg : (*pages)[q]) {
        pool->kind[pg] = 0;
        pool->free_pages.insert(pg);
        pool->mapped_pages--;
      }
  };
  for (int p = 0; p < np; ++p) {
    pw_status st = pool->take_pages(l->pmax, &(*pages)[p]);
    if (st != PW_OK) {
      give_back(p);
      return st;
    }
  }
  if (bits == 16) {
    pw_status st = pool->take_pages(l->pmax16, &(*pages)[np]);
    if (st != PW_OK) {
      give_back(np);
      return st;
    }
  }
  return PW_OK;
}

// Whether expert e could be (re)placed at `bits` once its current blocks are
// released: release frees its mapped blocks and its reclaimable ones not yet
// reusable, on top of what the pool can already hand out.  Load and copy ask
// this before releasing anything, so a refused request leaves e as it was.
bool fits_after_release(pw_layer_t l, int e, int bits) {
  size_t avail = l->pool->reusable_pages();
  auto add = [&](const Block& b) {
    if (b.st == B_MAPPED || (b.st == B_RECLAIM && !pw_pool_s::reusable(b))) avail += b.pages.size();
  };
  for (int p = 0; p < kPlanes; ++p) add(l->plane(e, p));
  add(l->f16[e]);
  const int np = bits == 16 ? kPlanes : bits;
  return avail >= (size_t)np * l->pmax + (bits == 16 ? (size_t)l->pmax16 : 0);
}

// The layer's resident run back to the pool (and, in a virtual-memory pool,
// its mappings and its reserved range).
void release_resident(pw_layer_t l) {
  pw_pool_s* pool = l->pool;
  if (pool->vmm && l->va) {
    for (size_t i = 0; i < l->res_npages; ++i) pool->vmm_unmap(l->va + i * pool->page_bytes);
    pool->vmm_free(l->va, l->va_pages);
    l->va = nullptr;
  }
  pool->give_back_resident(l->res_first, l->res_npages);
}

void release_expert(pw_layer_t l, int e) {
  for (int p = 0; p < kPlanes; ++p) l->pool->release(l->plane(e, p));
  l->pool->release(l->f16[e]);
  l->bits[e] = 0;
}

}  // namespace

// ---------------------------------------------------------------------------
// status
// ---------------------------------------------------------------------------

extern "C" const char* pw_status_str(pw_status s) {
  switch (s) {
    case PW_OK: return "PW_OK";
    case PW_ERR_INVALID_ARG: return "PW_ERR_INVALID_ARG";
    case PW_ERR_UNSUPPORTED: return "PW_ERR_UNSUPPORTED";
    case PW_ERR_OOM: return "PW_ERR_OOM";
    case PW_ERR_NOT_RESIDENT: return "PW_ERR_NOT_RESIDENT";
    case PW_ERR_CUDA: return "PW_ERR_CUDA";
    case PW_ERR_TIMEOUT: return "PW_ERR_TIMEOUT";
    case PW_ERR_DEVICE_CHECK: return "PW_ERR_DEVICE_CHECK";
  }
  return "PW_ERR_UNKNOWN";
}

extern "C" pw_status pw_last_cuda_error(int* cuda_err) {
  if (!cuda_err) return PW_ERR_INVALID_ARG;
  *cuda_err = g_last_cuda;
  return PW_OK;
}

extern "C" pw_status pw_testing_host_sim(int enable) {
  g_sim = enable != 0;
  return PW_OK;
}

extern "C" pw_status pw_testing_wait_limit(pw_layer_t l, long long polls, int never_ready) {
  if (!l || polls < 0 || (never_ready != 0 && never_ready != 1)) return PW_ERR_INVALID_ARG;
  l->spin_limit = polls == 0 ? kDefaultSpinPolls : polls;
  l->wait_bias = never_ready;
  return PW_OK;
}

extern "C" pw_status pw_testing_complete_events(void) {
  g_sim_done = g_sim_issued;
  return PW_OK;
}

// ---------------------------------------------------------------------------
// pool
// ---------------------------------------------------------------------------

extern "C" pw_status pw_pool_create(void* dev_base, size_t bytes, size_t page_bytes, pw_pool_t* out) {
  if (!dev_base || !out || (reinterpret_cast<uintptr_t>(dev_base) & 255)) return PW_ERR_INVALID_ARG;
  if (page_bytes < (64u << 10) || page_bytes % (64u << 10)) return PW_ERR_INVALID_ARG;
  if (bytes < page_bytes) return PW_ERR_OOM;
  auto* p = new pw_pool_s();
  p->base = static_cast<char*>(dev_base);
  p->bytes = bytes;
  p->page_bytes = page_bytes;
  p->npages = bytes / page_bytes;
  p->kind.assign(p->npages, 0);
  for (size_t i = 0; i < p->npages; ++i) p->free_pages.insert((int)i);
  *out = p;
  return PW_OK;
}

extern "C" pw_status pw_pool_create_vmm(const unsigned long long* handles, size_t n_pages, size_t page_bytes,
                                        int device, pw_pool_t* out) {
  if (!handles || !out || n_pages == 0 || n_pages > (size_t)1 << 30) return PW_ERR_INVALID_ARG;
  if (page_bytes == 0 || page_bytes % (2u << 20)) return PW_ERR_INVALID_ARG;  // whole 2 MiB granules
  if (device < 0) return PW_ERR_INVALID_ARG;
  auto p = std::make_unique<pw_pool_s>();
  p->vmm = true;
  p->device = device;
  p->page_bytes = page_bytes;
  p->npages = n_pages;
  p->bytes = n_pages * page_bytes;
  p->handles.assign(handles, handles + n_pages);
  if (g_sim) {
    // host simulation of the physical pages: one shared memory file, page p
    // at offset p * page_bytes, mapped into reserved ranges with mmap
    p->sim_fd = memfd_create("pw_vmm_pool", 0);
    if (p->sim_fd < 0) return PW_ERR_UNSUPPORTED;
    if (ftruncate(p->sim_fd, (off_t)p->bytes) != 0) {
      close(p->sim_fd);
      return PW_ERR_UNSUPPORTED;
    }
  } else if (!vmm_api().ok) {
    return PW_ERR_UNSUPPORTED;
  }
  p->kind.assign(p->npages, 0);
  for (size_t i = 0; i < p->npages; ++i) p->free_pages.insert((int)i);
  *out = p.release();
  return PW_OK;
}

extern "C" pw_status pw_pool_destroy(pw_pool_t pool) {
  if (!pool) return PW_ERR_INVALID_ARG;
  if (pool->n_layers) return PW_ERR_INVALID_ARG;
  if (pool->sim_fd >= 0) close(pool->sim_fd);
  delete pool;
  return PW_OK;
}

extern "C" pw_status pw_testing_vmm_counts(pw_pool_t pool, uint64_t* maps, uint64_t* unmaps) {
  if (!pool || !maps || !unmaps) return PW_ERR_INVALID_ARG;
  *maps = pool->n_map;
  *unmaps = pool->n_unmap;
  return PW_OK;
}

extern "C" pw_status pw_pool_get_stats(pw_pool_t pool, pw_pool_stats* out) {
  if (!pool || !out) return PW_ERR_INVALID_ARG;
  out->total_pages = pool->npages;
  out->free_pages = pool->free_pages.size();
  out->mapped_pages = pool->mapped_pages;
  out->reclaimable_pages = pool->reclaim_pages;
  out->resident_bytes = pool->resident_bytes;
  out->page_bytes = pool->page_bytes;
  return PW_OK;
}

// ---------------------------------------------------------------------------
// layer lifecycle
// ---------------------------------------------------------------------------

extern "C" pw_status pw_layer_create(pw_pool_t pool, const pw_layer_desc* desc, pw_layer_t* out) {
  if (!pool || !desc || !out) return PW_ERR_INVALID_ARG;
  const pw_layer_desc& D = *desc;
  if (D.d <= 0 || D.ffn <= 0 || D.d % 64 || D.ffn % 64) return PW_ERR_INVALID_ARG;
  if (D.n_experts < 1 || D.n_experts > kMaxExperts) return PW_ERR_INVALID_ARG;
  if (D.top_k < 1 || D.top_k > kMaxTopK || D.top_k > D.n_experts) return PW_ERR_INVALID_ARG;
  if (D.renormalize != 0 && D.renormalize != 1) return PW_ERR_INVALID_ARG;
  if (D.shared_ffn < 0 || D.shared_ffn % 64) return PW_ERR_INVALID_ARG;
  if (D.d > 16384 || D.ffn > 32768 || D.shared_ffn > 32768) return PW_ERR_UNSUPPORTED;

  auto l = std::make_unique<pw_layer_s>();
  l->pool = pool;
  l->desc = D;
  const int E = D.n_experts;
  l->R[0] = l->R[1] = D.ffn;
  l->C[0] = l->C[1] = D.d;
  l->R[2] = D.d;
  l->C[2] = D.ffn;
  l->tmax = std::max(D.ffn, D.d) / kTileRows;
  l->pmax = build_tile_map(l->R, l->C, 2, pool->page_bytes, l->tmax, &l->tmap);
  l->pmax16 = build_tile_map(l->R, l->C, 32, pool->page_bytes, l->tmax, &l->tmap16);
  if (l->pmax < 0 || l->pmax16 < 0) return PW_ERR_UNSUPPORTED;  // page too small for one tile

  size_t lb = 0;
  for (int m = 0; m < 3; ++m)
    for (int i = 0; i < 4; ++i) {
      l->lut_off[m][i] = (unsigned)lb;
      lb += (size_t)l->R[m] * (1u << (i + 3)) * 2;
    }
  l->lut_block_bytes = align_up(lb, 256);

  // resident run: small tables, LUT blocks, shared FFN
  size_t off = 0;
  auto carve = [&](size_t n) {
    size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  const size_t o_bits = carve(sizeof(int) * E);
  const size_t o_err = carve(16);
  const size_t o_sync = carve(sizeof(int) * sync_words(E));
  const size_t o_ppt = carve(sizeof(unsigned long long) * (size_t)E * kPlanes * l->pmax);
  const size_t o_fpt = carve(sizeof(unsigned long long) * (size_t)E * l->pmax16);
  const size_t o_tmap = carve(sizeof(uint2) * 3 * (size_t)l->tmax);
  const size_t o_tmap16 = carve(sizeof(uint2) * 3 * (size_t)l->tmax);
  const size_t o_lutb = carve(sizeof(unsigned long long) * E);
  const size_t o_luts = carve(l->lut_block_bytes * E);
  size_t o_sh[3] = {0, 0, 0};
  if (D.shared_ffn) {
    o_sh[0] = carve((size_t)D.shared_ffn * D.d * 2);
    o_sh[1] = carve((size_t)D.shared_ffn * D.d * 2);
    o_sh[2] = carve((size_t)D.d * D.shared_ffn * 2);
  }
  l->res_npages = (off + pool->page_bytes - 1) / pool->page_bytes;
  l->res_first = pool->take_resident(l->res_npages);
  if (l->res_first < 0) return PW_ERR_OOM;
  if (pool->vmm) {
    // one reserved range per layer: the resident run, then a fixed range per
    // block (expert e, plane p: pmax pages; its fp16 block: pmax16 pages).
    // A block's pages are mapped into its range while it holds them, so its
    // addresses (and the device page table) never change.
    const size_t per_expert = (size_t)kPlanes * l->pmax + l->pmax16;
    l->va_pages = l->res_npages + (size_t)E * per_expert;
    l->va = pool->vmm_reserve(l->va_pages);
    pw_status st = l->va ? PW_OK : (g_sim ? PW_ERR_UNSUPPORTED : PW_ERR_CUDA);
    size_t mapped = 0;
    for (; st == PW_OK && mapped < l->res_npages; ++mapped)
      st = pool->vmm_map(l->va + mapped * pool->page_bytes, l->res_first + (int)mapped);
    if (st != PW_OK) {
      for (size_t i = 0; i + 1 < mapped; ++i) pool->vmm_unmap(l->va + i * pool->page_bytes);
      pool->vmm_free(l->va, l->va_pages);
      pool->give_back_resident(l->res_first, l->res_npages);
      return st;
    }
    l->res_base = l->va;
  } else {
    l->res_base = pool->page_addr(l->res_first);
  }
  char* rb = l->res_base;
  l->d_bits = reinterpret_cast<int*>(rb + o_bits);
  l->d_err = reinterpret_cast<int*>(rb + o_err);
  l->d_sync = reinterpret_cast<int*>(rb + o_sync);
  l->d_plane_pt = reinterpret_cast<unsigned long long*>(rb + o_ppt);
  l->d_f16_pt = reinterpret_cast<unsigned long long*>(rb + o_fpt);
  l->d_tmap = reinterpret_cast<uint2*>(rb + o_tmap);
  l->d_tmap16 = reinterpret_cast<uint2*>(rb + o_tmap16);
  l->d_lut_base = reinterpret_cast<unsigned long long*>(rb + o_lutb);
  l->d_luts = rb + o_luts;
  for (int m = 0; m < 3; ++m) l->d_shared[m] = D.shared_ffn ? reinterpret_cast<__half*>(rb + o_sh[m]) : nullptr;

  l->bits.assign(E, 0);
  l->planes.resize((size_t)E * kPlanes);
  l->f16.resize(E);
  if (pool->vmm) {
    const size_t pb = pool->page_bytes, per_expert = (size_t)kPlanes * l->pmax + l->pmax16;
    for (int e = 0; e < E; ++e) {
      char* ev = l->va + (l->res_npages + (size_t)e * per_expert) * pb;
      for (int p = 0; p < kPlanes; ++p) l->plane(e, p).va = ev + (size_t)p * l->pmax * pb;
      l->f16[e].va = ev + (size_t)kPlanes * l->pmax * pb;
    }
  }
  l->h_plane_pt.assign((size_t)E * kPlanes * l->pmax, 0ull);
  l->h_f16_pt.assign((size_t)E * l->pmax16, 0ull);
  std::vector<unsigned long long> lutb(E);
  for (int e = 0; e < E; ++e)
    lutb[e] = reinterpret_cast<unsigned long long>(l->d_luts + (size_t)e * l->lut_block_bytes);

  cudaStream_t s = nullptr;
  pw_status st = PW_OK;
  if (st == PW_OK) st = dev_zero(rb, o_ppt, s);  // bits, error word, sync area
  if (st == PW_OK) st = dev_zero(l->d_plane_pt, (o_tmap - o_ppt), s);
  if (st == PW_OK) st = dev_h2d(l->d_tmap, l->tmap.data(), sizeof(uint2) * l->tmap.size(), s);
  if (st == PW_OK) st = dev_h2d(l->d_tmap16, l->tmap16.data(), sizeof(uint2) * l->tmap16.size(), s);
  if (st == PW_OK) st = dev_h2d(l->d_lut_base, lutb.data(), sizeof(unsigned long long) * E, s);
  if (st == PW_OK) st = dev_sync(s);
  if (st != PW_OK) {
    release_resident(l.get());
    return st;
  }
  pool->n_layers++;
  *out = l.release();
  return PW_OK;
}

extern "C" pw_status pw_layer_destroy(pw_layer_t l) {
  PW_TRY(check_layer(l));
  if (!g_sim) cudaDeviceSynchronize();
  for (int e = 0; e < l->desc.n_experts; ++e) release_expert(l, e);
  release_resident(l);
  l->pool->n_layers--;
  delete l;
  return PW_OK;
}

extern "C" pw_status pw_layer_load_expert(pw_layer_t l, int e, int bits, const uint8_t* const code6[3],
                                          const uint16_t* const lut[3][4], const uint16_t* const w16[3],
                                          void* stream) {
  PW_TRY(check_layer(l));
  if (e < 0 || e >= l->desc.n_experts || !valid_bits(bits) || !code6 || !lut) return PW_ERR_INVALID_ARG;
  for (int m = 0; m < 3; ++m) {
    if (!code6[m]) return PW_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (!lut[m][i]) return PW_ERR_INVALID_ARG;
    if (bits == 16 && (!w16 || !w16[m])) return PW_ERR_INVALID_ARG;
  }
  cudaStream_t s = as_stream(stream);
  pw_pool_s* pool = l->pool;
  if (!fits_after_release(l, e, bits)) return PW_ERR_OOM;  // expert e stays as it was
  // kernels still reading the old pages must finish before they are reused
  PW_TRY(dev_sync(s));
  release_expert(l, e);

  const int np = bits == 16 ? kPlanes : bits;
  std::vector<std::vector<int>> pages;
  PW_TRY(take_expert_pages(l, bits, &pages));

  // pack and upload planes
  const size_t pb = pool->page_bytes;
  std::vector<std::vector<char>> img(np, std::vector<char>((size_t)l->pmax * pb, 0));
  for (int m = 0; m < 3; ++m) {
    const int R = l->R[m], C = l->C[m];
    const size_t nw = (size_t)R * C / 32;
    std::vector<uint32_t> packed((size_t)kPlanes * nw);
    uint32_t* outs[6];
    for (int p = 0; p < 6; ++p) outs[p] = packed.data() + p * nw;
    PW_TRY(pw_pack_planes(code6[m], R, C, outs));
    const size_t tb = 2 * (size_t)C;  // bytes of one 16-row tile of one plane
    for (int tau = 0; tau < R / kTileRows; ++tau) {
      const uint2 loc = l->tmap[(size_t)m * l->tmax + tau];
      for (int p = 0; p < np; ++p)
        memcpy(img[p].data() + (size_t)loc.x * pb + loc.y, outs[p] + (size_t)tau * (tb / 4), tb);
    }
  }
  for (int p = 0; p < np; ++p) {
    Block& b = l->plane(e, p);
    PW_TRY(attach_block(l, b, pages[p]));
    PW_TRY(upload_block(l, b, img[p], s));
    for (int v = 0; v < l->pmax; ++v)
      l->h_plane_pt[((size_t)e * kPlanes + p) * l->pmax + v] = reinterpret_cast<unsigned long long>(blk_addr(l, b, v));
  }
  img.clear();
  if (bits == 16) {
    std::vector<char> im((size_t)l->pmax16 * pb, 0);
    for (int m = 0; m < 3; ++m) {
      const int R = l->R[m], C = l->C[m];
      std::vector<uint16_t> packed((size_t)R * C);
      PW_TRY(pw_pack_f16(w16[m], R, C, packed.data()));
      const size_t tb = 32 * (size_t)C;
      for (int tau = 0; tau < R / kTileRows; ++tau) {
        const uint2 loc = l->tmap16[(size_t)m * l->tmax + tau];
        memcpy(im.data() + (size_t)loc.x * pb + loc.y, packed.data() + (size_t)tau * (tb / 2), tb);
      }
    }
    Block& b = l->f16[e];
    PW_TRY(attach_block(l, b, pages[np]));
    PW_TRY(upload_block(l, b, im, s));
    for (int v = 0; v < l->pmax16; ++v)
      l->h_f16_pt[(size_t)e * l->pmax16 + v] = reinterpret_cast<unsigned long long>(blk_addr(l, b, v));
  }
  // LUTs (all four bitwidths stay resident)
  char* lb = l->d_luts + (size_t)e * l->lut_block_bytes;
  for (int m = 0; m < 3; ++m)
    for (int i = 0; i < 4; ++i)
      PW_TRY(dev_h2d(lb + l->lut_off[m][i], lut[m][i], (size_t)l->R[m] * (1u << (i + 3)) * 2, s));
  PW_TRY(upload_pt_rows(l, e, s));
  PW_TRY(write_bits(l, e, bits, s));
  PW_TRY(dev_sync(s));
  l->bits[e] = bits;
  return PW_OK;
}

extern "C" pw_status pw_layer_copy_expert(pw_layer_t l, int e, pw_layer_t src, int e_src, int bits,
                                          void* stream) {
  PW_TRY(check_layer(l));
  PW_TRY(check_layer(src));
  if (e < 0 || e >= l->desc.n_experts || e_src < 0 || e_src >= src->desc.n_experts || !valid_bits(bits))
    return PW_ERR_INVALID_ARG;
  if (l == src && e == e_src) return PW_ERR_INVALID_ARG;
  if (l->desc.d != src->desc.d || l->desc.ffn != src->desc.ffn || l->pool->page_bytes != src->pool->page_bytes)
    return PW_ERR_INVALID_ARG;
  if (src->bits[e_src] == 0) return PW_ERR_INVALID_ARG;
  const int np = bits == 16 ? kPlanes : bits;
  // only blocks the source reads at its current bitwidth: reclaimable ones
  // could be handed to the copy itself
  for (int p = 0; p < np; ++p)
    if (src->plane(e_src, p).st != B_MAPPED) return PW_ERR_NOT_RESIDENT;
  if (bits == 16 && src->f16[e_src].st != B_MAPPED) return PW_ERR_NOT_RESIDENT;

  cudaStream_t s = as_stream(stream);
  if (!fits_after_release(l, e, bits)) return PW_ERR_OOM;  // expert e stays as it was
  PW_TRY(dev_sync(s));  // kernels still reading the old pages must finish before they are reused
  release_expert(l, e);
  std::vector<std::vector<int>> pages;
  PW_TRY(take_expert_pages(l, bits, &pages));
  const size_t pb = l->pool->page_bytes;
  // same shapes give the same tile maps: copy page by page
  for (int p = 0; p < np; ++p) {
    Block& b = l->plane(e, p);
    const Block& sb = src->plane(e_src, p);
    PW_TRY(attach_block(l, b, pages[p]));
    for (int v = 0; v < l->pmax; ++v) {
      PW_TRY(dev_d2d(blk_addr(l, b, v), blk_addr(src, sb, v), pb, s));
      l->h_plane_pt[((size_t)e * kPlanes + p) * l->pmax + v] = reinterpret_cast<unsigned long long>(blk_addr(l, b, v));
    }
  }
  if (bits == 16) {
    Block& b = l->f16[e];
    const Block& sb = src->f16[e_src];
    PW_TRY(attach_block(l, b, pages[np]));
    for (int v = 0; v < l->pmax16; ++v) {
      PW_TRY(dev_d2d(blk_addr(l, b, v), blk_addr(src, sb, v), pb, s));
      l->h_f16_pt[(size_t)e * l->pmax16 + v] = reinterpret_cast<unsigned long long>(blk_addr(l, b, v));
    }
  }
  PW_TRY(dev_d2d(l->d_luts + (size_t)e * l->lut_block_bytes, src->d_luts + (size_t)e_src * src->lut_block_bytes,
                 l->lut_block_bytes, s));
  PW_TRY(upload_pt_rows(l, e, s));
  PW_TRY(write_bits(l, e, bits, s));
  PW_TRY(dev_sync(s));
  l->bits[e] = bits;
  return PW_OK;
}

extern "C" pw_status pw_layer_load_shared(pw_layer_t l, const uint16_t* const w16[3], void* stream) {
  PW_TRY(check_layer(l));
  if (l->desc.shared_ffn == 0) return PW_ERR_INVALID_ARG;
  if (!w16 || !w16[0] || !w16[1] || !w16[2]) return PW_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  const int d = l->desc.d, fs = l->desc.shared_ffn;
  const int R[3] = {fs, fs, d}, C[3] = {d, d, fs};
  for (int m = 0; m < 3; ++m) {
    std::vector<uint16_t> packed((size_t)R[m] * C[m]);
    PW_TRY(pw_pack_f16(w16[m], R[m], C[m], packed.data()));
    PW_TRY(dev_h2d(l->d_shared[m], packed.data(), packed.size() * 2, s));
    PW_TRY(dev_sync(s));
  }
  l->shared_loaded = true;
  return PW_OK;
}

// ---------------------------------------------------------------------------
// bitwidth changes (the paging mechanism)
// ---------------------------------------------------------------------------

extern "C" pw_status pw_set_expert_bitwidth(pw_layer_t l, int e, int bits, void* stream) {
  PW_TRY(check_layer(l));
  if (e < 0 || e >= l->desc.n_experts || !valid_bits(bits)) return PW_ERR_INVALID_ARG;
  const int cur = l->bits[e];
  if (cur == 0) return PW_ERR_INVALID_ARG;  // never loaded
  if (cur == bits) return PW_OK;
  const int need = bits == 16 ? kPlanes : bits;
  // every block the new bitwidth reads must still hold its data
  for (int p = 0; p < need; ++p)
    if (l->plane(e, p).st == B_NONE) return PW_ERR_NOT_RESIDENT;
  if (bits == 16 && l->f16[e].st == B_NONE) return PW_ERR_NOT_RESIDENT;

  cudaStream_t s = as_stream(stream);
  NvtxRange range("pw_set_expert_bitwidth");
  // blocks filled by an asynchronous upload: the commit waits for the copies
  auto await_upload = [&](Block& b) -> pw_status {
    if (b.ready) {
      if (!g_sim) PW_CUDA(cudaStreamWaitEvent(s, b.ready->ev, 0));
      b.ready.reset();
    }
    return PW_OK;
  };
  for (int p = 0; p < need; ++p) PW_TRY(await_upload(l->plane(e, p)));
  if (bits == 16) PW_TRY(await_upload(l->f16[e]));
  PW_TRY(write_bits(l, e, bits, s));
  // raise: re-map still-intact blocks (their page-table entries never changed)
  for (int p = 0; p < need; ++p)
    if (l->plane(e, p).st == B_RECLAIM) l->pool->remap(l->plane(e, p));
  if (bits == 16 && l->f16[e].st == B_RECLAIM) l->pool->remap(l->f16[e]);
  // lower: blocks no longer read become reclaimable after the safe boundary
  std::vector<Block*> drop;
  for (int p = need; p < kPlanes; ++p)
    if (l->plane(e, p).st == B_MAPPED) drop.push_back(&l->plane(e, p));
  if (bits != 16 && l->f16[e].st == B_MAPPED) drop.push_back(&l->f16[e]);
  if (!drop.empty()) {
    std::shared_ptr<Event> ev;
    PW_TRY(make_event(s, &ev));
    for (Block* b : drop) l->pool->to_reclaim(*b, ev);
  }
  l->bits[e] = bits;
  return PW_OK;
}

namespace {

pw_status dev_h2d_on(void* dst, const void* src, size_t n, cudaStream_t s) { return dev_h2d(dst, src, n, s); }

// Copy the tiles of one block image from a packed host array: tiles of matrix
// m are consecutive in the packed array and, page by page, in the block; runs
// of tiles that stay inside one page go as one copy.
pw_status upload_tiles(pw_layer_t l, const Block& b, const std::vector<uint2>& map, int m, const char* host,
                       size_t tile_bytes, cudaStream_t s) {
  const int ntiles = l->R[m] / kTileRows;
  int tau = 0;
  while (tau < ntiles) {
    const uint2 loc = map[(size_t)m * l->tmax + tau];
    int run = 1;
    while (tau + run < ntiles) {
      const uint2 nx = map[(size_t)m * l->tmax + tau + run];
      if (nx.x != loc.x || nx.y != loc.y + run * tile_bytes) break;
      ++run;
    }
    PW_TRY(dev_h2d_on(blk_addr(l, b, (int)loc.x) + loc.y, host + (size_t)tau * tile_bytes,
                      (size_t)run * tile_bytes, s));
    tau += run;
  }
  return PW_OK;
}

}  // namespace

extern "C" pw_status pw_prefetch_expert(pw_layer_t l, int e, int bits, const uint32_t* const planes_host[3][6],
                                        const uint16_t* const w16_host[3], void* copy_stream) {
  PW_TRY(check_layer(l));
  if (e < 0 || e >= l->desc.n_experts || !valid_bits(bits)) return PW_ERR_INVALID_ARG;
  if (l->bits[e] == 0) return PW_ERR_INVALID_ARG;  // never loaded
  NvtxRange range("pw_prefetch_expert");
  const int need = bits == 16 ? kPlanes : bits;
  // the host data of every block that is gone
  std::vector<int> missing;
  for (int p = 0; p < need; ++p)
    if (l->plane(e, p).st == B_NONE) {
      for (int m = 0; m < 3; ++m)
        if (!planes_host || !planes_host[m][p]) return PW_ERR_INVALID_ARG;
      missing.push_back(p);
    }
  const bool f16_missing = bits == 16 && l->f16[e].st == B_NONE;
  if (f16_missing)
    for (int m = 0; m < 3; ++m)
      if (!w16_host || !w16_host[m]) return PW_ERR_INVALID_ARG;

  pw_pool_s* pool = l->pool;
  cudaStream_t cs = as_stream(copy_stream);
  // refuse a request the pool cannot meet before anything changes: the
  // expert's own intact blocks are held below, so their pages do not count
  size_t own = 0;
  for (int p = 0; p < need; ++p)
    if (l->plane(e, p).st == B_RECLAIM && pw_pool_s::reusable(l->plane(e, p))) own += l->plane(e, p).pages.size();
  if (bits == 16 && l->f16[e].st == B_RECLAIM && pw_pool_s::reusable(l->f16[e])) own += l->f16[e].pages.size();
  const size_t want = missing.size() * (size_t)l->pmax + (f16_missing ? (size_t)l->pmax16 : 0);
  if (pool->reusable_pages() - own < want) return PW_ERR_OOM;
  // still-intact blocks are held (re-mapped) so that they cannot be handed out
  // before the raise; they hold their data already
  std::vector<Block*> held;
  for (int p = 0; p < need; ++p)
    if (l->plane(e, p).st == B_RECLAIM) {
      pool->remap(l->plane(e, p));
      held.push_back(&l->plane(e, p));
    }
  if (bits == 16 && l->f16[e].st == B_RECLAIM) {
    pool->remap(l->f16[e]);
    held.push_back(&l->f16[e]);
  }
  std::vector<std::vector<int>> pages(missing.size() + 1);
  size_t taken = 0;
  for (size_t i = 0; i < missing.size(); ++i, ++taken)
    if (pool->take_pages(l->pmax, &pages[i]) != PW_OK) break;
  bool ok = taken == missing.size();
  if (ok && f16_missing) ok = pool->take_pages(l->pmax16, &pages[missing.size()]) == PW_OK;
  if (!ok) {
    for (size_t i = 0; i < taken; ++i)
      for (int pg : pages[i]) {
        pool->kind[pg] = 0;
        pool->free_pages.insert(pg);
        pool->mapped_pages--;
      }
    if (!held.empty()) {  // back to the reclaim queue, releasable at once
      std::shared_ptr<Event> ev;
      if (make_event(cs, &ev) == PW_OK)
        for (Block* b : held) pool->to_reclaim(*b, ev);
    }
    return PW_ERR_OOM;
  }
  if (missing.empty() && !f16_missing) return PW_OK;
  // copies on the copy stream, then the page-table rows (entries the current
  // bitwidth reads keep their values; kernels never read planes >= bits[e])
  for (size_t i = 0; i < missing.size(); ++i) {
    const int p = missing[i];
    Block& b = l->plane(e, p);
    PW_TRY(attach_block(l, b, pages[i]));
    for (int m = 0; m < 3; ++m)
      PW_TRY(upload_tiles(l, b, l->tmap, m, reinterpret_cast<const char*>(planes_host[m][p]),
                          2 * (size_t)l->C[m], cs));
    for (int v = 0; v < l->pmax; ++v)
      l->h_plane_pt[((size_t)e * kPlanes + p) * l->pmax + v] = reinterpret_cast<unsigned long long>(blk_addr(l, b, v));
  }
  if (f16_missing) {
    Block& b = l->f16[e];
    PW_TRY(attach_block(l, b, pages[missing.size()]));
    for (int m = 0; m < 3; ++m)
      PW_TRY(upload_tiles(l, b, l->tmap16, m, reinterpret_cast<const char*>(w16_host[m]), 32 * (size_t)l->C[m],
                          cs));
    for (int v = 0; v < l->pmax16; ++v)
      l->h_f16_pt[(size_t)e * l->pmax16 + v] = reinterpret_cast<unsigned long long>(blk_addr(l, b, v));
  }
  PW_TRY(upload_pt_rows(l, e, cs));
  std::shared_ptr<Event> ready;
  PW_TRY(make_event(cs, &ready));
  for (int p : missing) l->plane(e, p).ready = ready;
  if (f16_missing) l->f16[e].ready = ready;
  return PW_OK;
}

extern "C" pw_status pw_raise_expert_async(pw_layer_t l, int e, int bits, const uint32_t* const planes_host[3][6],
                                           const uint16_t* const w16_host[3], void* copy_stream, void* stream) {
  PW_TRY(check_layer(l));
  if (e < 0 || e >= l->desc.n_experts || !valid_bits(bits)) return PW_ERR_INVALID_ARG;
  const int cur = l->bits[e];
  if (cur == 0) return PW_ERR_INVALID_ARG;
  const int have = cur == 16 ? kPlanes : cur;
  if (bits == cur || (bits != 16 && bits <= have)) return PW_ERR_INVALID_ARG;  // not a raise
  PW_TRY(pw_prefetch_expert(l, e, bits, planes_host, w16_host, copy_stream));
  return pw_set_expert_bitwidth(l, e, bits, stream);
}

extern "C" pw_status pw_get_expert_bitwidth(pw_layer_t l, int e, int* bits) {
  PW_TRY(check_layer(l));
  if (!bits || e < 0 || e >= l->desc.n_experts) return PW_ERR_INVALID_ARG;
  *bits = l->bits[e];
  return PW_OK;
}

// ---------------------------------------------------------------------------
// workspace and hot-path entry points
// ---------------------------------------------------------------------------

namespace {

struct WsLayout {
  size_t perm_off, perm_bytes, h_off, h_bytes, hs_off, hs_bytes, total;
  Canaries can;  // with debug bounds: a canary block after each region
};

// Scratch regions at 256-byte boundaries; with debug bounds each is followed
// by a kCanaryBytes block whose offset is recorded.
struct Carver {
  bool dbg;
  Canaries* can;
  size_t o = 0;
  size_t take(size_t n) {
    const size_t at = o;
    o += align_up(n, 256);
    if (dbg && can->n < kMaxCanaries) {
      can->off[can->n++] = o;
      o += kCanaryBytes;
    }
    return at;
  }
};

WsLayout ws_layout(const pw_layer_s* l, int T) {
  WsLayout w{};
  w.can.n = 0;
  Carver c{l->debug_bounds, &w.can};
  const size_t S = (size_t)T * l->desc.top_k;
  w.perm_bytes = align_up(permute_ws_bytes((int)S, l->desc.n_experts), 256);
  w.perm_off = c.take(w.perm_bytes);
  w.h_bytes = align_up(S * l->desc.ffn * 2, 256);
  w.h_off = c.take(w.h_bytes);
  w.hs_bytes = align_up((size_t)T * l->desc.shared_ffn * 2, 256);
  w.hs_off = c.take(w.hs_bytes);
  w.total = c.o;
  return w;
}


pw_status device_only() { return g_sim ? PW_ERR_UNSUPPORTED : PW_OK; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Token counts past 2^20 are refused: slot counts (T * top_k) then stay well
// inside int and every scratch size inside size_t.
constexpr int kMaxTokens = 1 << 20;
bool bad_tokens(int T) { return T < 0 || T > kMaxTokens; }

pw_status all_loaded(const pw_layer_s* l) {
  for (int b : l->bits)
    if (b == 0) return PW_ERR_INVALID_ARG;
  return PW_OK;
}

pw_status launched(cudaError_t e) { return e == cudaSuccess ? PW_OK : cuda_fail(e); }

// Whether pw_moe_forward takes the one-launch fused step for T tokens: decode
// batches of at most kFusedMaxTokens whose routed experts and shared FFN all
// stay on the decode kernel (measured: 3-5% faster at 1-8 tokens, 1.5%
// slower at 64, where the separate small kernels cost less than the fused
// kernel's final barrier).
bool fused_step(const pw_layer_desc& d, int T) {
  return T <= kFusedMaxTokens && T <= decode_max_tokens(d.ffn, T, d.n_experts, d.top_k) &&
         (d.shared_ffn == 0 || T <= decode_max_tokens_shared()) && T * d.top_k <= 512;
}

// Which decode kernel classes the layer can need: bit 0 for 3-bit experts
// (every loaded expert can be lowered to 3 bits), bit 1 for experts with at
// least four planes still resident (4..6 bits reachable), bit 2 for experts
// whose fp16 page is still resident (16 bits reachable).  A class whose
// bitwidths no expert can reach without a reload is not launched.
int class_mask(const pw_layer_s* l) {
  int m = 0;
  for (int e = 0; e < l->desc.n_experts; ++e) {
    if (l->bits[e] == 0) continue;
    m |= 1;
    if (l->planes[(size_t)e * kPlanes + 3].st != B_NONE) m |= 2;
    if (l->f16[e].st != B_NONE) m |= 4;
  }
  return m;
}

}  // namespace

// Scratch of one whole-layer call (pw_moe_forward): the permutation and the
// routed / shared FFN intermediates, then the hot-path scratch of ws_layout.
struct FwdLayout {
  size_t off_offsets, off_perm_src, off_inv_slot, off_x_perm, off_y_perm, off_ys, off_rpart, off_base, total;
  Canaries can;  // with debug bounds: this layout's and the hot-path scratch's canaries
};

FwdLayout fwd_layout(const pw_layer_s* l, int T) {
  FwdLayout f{};
  f.can.n = 0;
  const size_t S = (size_t)T * l->desc.top_k, d = l->desc.d;
  Carver c{l->debug_bounds, &f.can};
  auto take = [&](size_t n) { return c.take(n); };
  f.off_offsets = take(sizeof(int32_t) * (l->desc.n_experts + 1));
  f.off_perm_src = take(sizeof(int32_t) * S);
  f.off_inv_slot = take(sizeof(int32_t) * S);
  f.off_x_perm = take(2 * S * d);
  f.off_y_perm = take(sizeof(float) * S * d);
  f.off_ys = take(l->desc.shared_ffn ? sizeof(float) * (size_t)T * d : 0);
  // router partial sums of the fused step (batches of at most kFusedMaxTokens)
  f.off_rpart = take(sizeof(float) * (size_t)std::min(T, kFusedMaxTokens) * route_slices(l->desc.d) *
                     l->desc.n_experts);
  f.off_base = c.o;
  const WsLayout W = ws_layout(l, T);
  for (int i = 0; i < W.can.n && f.can.n < kMaxCanaries; ++i) f.can.off[f.can.n++] = f.off_base + W.can.off[i];
  f.total = f.off_base + W.total;
  return f;
}

extern "C" pw_status pw_moe_forward_workspace_size(pw_layer_t l, int T, size_t* bytes) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T) || !bytes) return PW_ERR_INVALID_ARG;
  *bytes = fwd_layout(l, T).total;
  return PW_OK;
}

extern "C" pw_status pw_moe_forward(pw_layer_t l, const void* x, const void* wr, const float* bias, int T,
                                    int32_t* idx, float* w, void* y, void* ws, size_t ws_bytes, void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T)) return PW_ERR_INVALID_ARG;
  const bool sh = l->desc.shared_ffn != 0;
  if (sh && !l->shared_loaded) return PW_ERR_INVALID_ARG;
  if (T == 0) return device_only();
  if (!x || !wr || !idx || !w || !y || !ws) return PW_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(wr) || !aligned16(y) || !aligned16(ws)) return PW_ERR_INVALID_ARG;
  const FwdLayout F = fwd_layout(l, T);
  if (ws_bytes < F.total) return PW_ERR_OOM;
  PW_TRY(all_loaded(l));
  PW_TRY(device_only());
  const DevLayer L = l->dev();
  cudaStream_t s = as_stream(stream);
  char* wsb = static_cast<char*>(ws);
  const WsLayout W = ws_layout(l, T);
  char* base = wsb + F.off_base;
  auto* offsets = reinterpret_cast<int*>(wsb + F.off_offsets);
  auto* y_perm = reinterpret_cast<float*>(wsb + F.off_y_perm);
  auto* ys = sh ? reinterpret_cast<float*>(wsb + F.off_ys) : nullptr;
  auto* h = reinterpret_cast<__half*>(base + W.h_off);
  auto* hs = sh ? reinterpret_cast<__half*>(base + W.hs_off) : nullptr;
  const auto* xh = static_cast<const __half*>(x);
  const auto* wrh = static_cast<const __half*>(wr);
  NvtxRange range("pw_moe_forward");
  if (l->debug_bounds) PW_TRY(launched(launch_canaries(wsb, F.can, L.err, true, s)));
  auto run = [&]() -> pw_status {
    // one fused launch (router, permutation, expert FFN, shared FFN, combine)
    // for small decode batches; both give the same idx, w and y bit for bit
    if (fused_step(l->desc, T))
      return launched(launch_layer_fused(L, xh, wrh, bias, idx, w, reinterpret_cast<float*>(wsb + F.off_rpart), T,
                                         h, hs, y_perm, ys, static_cast<__half*>(y), offsets, s));
    PW_TRY(launched(launch_route(L, xh, wrh, bias, T, idx, w, nullptr, s)));
    auto* perm_src = reinterpret_cast<int*>(wsb + F.off_perm_src);
    auto* inv_slot = reinterpret_cast<int*>(wsb + F.off_inv_slot);
    auto* x_perm = reinterpret_cast<__half*>(wsb + F.off_x_perm);
    PW_TRY(launched(launch_permute(L, idx, T, xh, offsets, perm_src, inv_slot, x_perm,
                                   reinterpret_cast<int*>(base + W.perm_off), s)));
    PW_TRY(launched(launch_moe_ffn(L, x_perm, offsets, T * l->desc.top_k, y_perm, h, sh ? xh : nullptr, T, ys, hs,
                                   class_mask(l), s)));
    return launched(launch_combine(L, y_perm, inv_slot, w, T, ys, static_cast<__half*>(y), s));
  };
  PW_TRY(run());
  if (l->debug_bounds) PW_TRY(launched(launch_canaries(wsb, F.can, L.err, false, s)));
  return PW_OK;
}

extern "C" pw_status pw_layer_set_debug_bounds(pw_layer_t l, int on) {
  PW_TRY(check_layer(l));
  l->debug_bounds = on != 0;
  return PW_OK;
}

extern "C" pw_status pw_debug_check_workspace(pw_layer_t l, int T, void* ws, size_t ws_bytes, void* stream) {
  PW_TRY(check_layer(l));
  if (!l->debug_bounds || bad_tokens(T) || !ws) return PW_ERR_INVALID_ARG;
  const FwdLayout F = fwd_layout(l, T);
  if (ws_bytes < F.total) return PW_ERR_OOM;
  PW_TRY(device_only());
  return launched(launch_canaries(static_cast<char*>(ws), F.can, l->d_err, false, as_stream(stream)));
}

extern "C" pw_status pw_decode_plan(const pw_layer_desc* desc, int T, int* routed_max, int* shared_max,
                                    int* fused) {
  if (!desc || T < 0 || desc->ffn <= 0 || desc->n_experts <= 0 || desc->top_k <= 0 || !routed_max || !shared_max ||
      !fused)
    return PW_ERR_INVALID_ARG;
  *routed_max = decode_max_tokens(desc->ffn, T, desc->n_experts, desc->top_k);
  *shared_max = decode_max_tokens_shared();
  *fused = T > 0 && fused_step(*desc, T) ? 1 : 0;
  return PW_OK;
}

extern "C" pw_status pw_workspace_size(pw_layer_t l, int T, size_t* bytes) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T) || !bytes) return PW_ERR_INVALID_ARG;
  *bytes = ws_layout(l, T).total;
  return PW_OK;
}

extern "C" pw_status pw_route_topk(pw_layer_t l, const void* x, const void* wr, const float* bias, int T,
                                   int32_t* idx, float* w, int32_t* expert_count, void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T)) return PW_ERR_INVALID_ARG;
  if (T > 0 && (!x || !wr || !idx || !w)) return PW_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(x) || !aligned16(wr))) return PW_ERR_INVALID_ARG;
  PW_TRY(device_only());
  if (T == 0) return PW_OK;
  NvtxRange range("pw_route_topk");
  return launched(launch_route(l->dev(), static_cast<const __half*>(x), static_cast<const __half*>(wr), bias, T,
                               idx, w, expert_count, as_stream(stream)));
}

extern "C" pw_status pw_route_stats(pw_layer_t l, const void* x, const int32_t* idx, const float* w, int T,
                                    float* mass, float* resid, void* ws, size_t ws_bytes, void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T) || !mass || !resid) return PW_ERR_INVALID_ARG;
  if (T > 0 && (!x || !idx || !w || !ws)) return PW_ERR_INVALID_ARG;
  if (T > 0 && !aligned16(x)) return PW_ERR_INVALID_ARG;
  if (T > 0 && ws_bytes < (size_t)T * sizeof(float)) return PW_ERR_OOM;
  PW_TRY(device_only());
  return launched(launch_route_stats(l->dev(), static_cast<const __half*>(x), idx, w, T, mass, resid,
                                     static_cast<float*>(ws), as_stream(stream)));
}

extern "C" pw_status pw_expert_resident_bytes(pw_layer_t l, int bits, uint64_t* bytes) {
  PW_TRY(check_layer(l));
  if (!bytes || !valid_bits(bits)) return PW_ERR_INVALID_ARG;
  const uint64_t pb = l->pool->page_bytes;
  const uint64_t planes = (uint64_t)(bits == 16 ? kPlanes : bits) * (uint64_t)l->pmax;
  *bytes = (planes + (bits == 16 ? (uint64_t)l->pmax16 : 0)) * pb;
  return PW_OK;
}

extern "C" pw_status pw_permute(pw_layer_t l, const int32_t* idx, int T, const void* x, int32_t* offsets,
                                int32_t* perm_src, int32_t* inv_slot, void* x_perm, void* ws, size_t ws_bytes,
                                void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T) || !offsets) return PW_ERR_INVALID_ARG;
  if (T > 0 && (!idx || !perm_src || !inv_slot || !ws)) return PW_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr) != (x_perm == nullptr)) return PW_ERR_INVALID_ARG;
  if (T > 0 && x && (!aligned16(x) || !aligned16(x_perm))) return PW_ERR_INVALID_ARG;
  if (T > 0 && !aligned16(ws)) return PW_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(l, T);
  if (T > 0 && ws_bytes < W.perm_off + W.perm_bytes) return PW_ERR_OOM;
  PW_TRY(device_only());
  NvtxRange range("pw_permute");
  char* wsb = static_cast<char*>(ws);
  return launched(launch_permute(l->dev(), idx, T, static_cast<const __half*>(x), offsets, perm_src, inv_slot,
                                 static_cast<__half*>(x_perm), reinterpret_cast<int*>(wsb + W.perm_off),
                                 as_stream(stream)));
}

extern "C" pw_status pw_expert_ffn_bitplane(pw_layer_t l, const void* x_perm, const int32_t* offsets, int T,
                                            float* y_perm, void* ws, size_t ws_bytes, void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T)) return PW_ERR_INVALID_ARG;
  if (T == 0) return device_only();
  if (!x_perm || !offsets || !y_perm || !ws) return PW_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(y_perm) || !aligned16(ws)) return PW_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(l, T);
  if (ws_bytes < W.h_off + W.h_bytes) return PW_ERR_OOM;
  PW_TRY(all_loaded(l));
  PW_TRY(device_only());
  NvtxRange range("pw_expert_ffn_bitplane");
  char* wsb = static_cast<char*>(ws);
  return launched(launch_moe_ffn(l->dev(), static_cast<const __half*>(x_perm), offsets, T * l->desc.top_k, y_perm,
                                 reinterpret_cast<__half*>(wsb + W.h_off), nullptr, T, nullptr, nullptr,
                                 class_mask(l), as_stream(stream)));
}

extern "C" pw_status pw_shared_ffn(pw_layer_t l, const void* x, int T, float* y_shared, void* ws, size_t ws_bytes,
                                   void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T)) return PW_ERR_INVALID_ARG;
  if (l->desc.shared_ffn == 0 || !l->shared_loaded) return PW_ERR_INVALID_ARG;
  if (T == 0) return device_only();
  if (!x || !y_shared || !ws || !aligned16(x) || !aligned16(y_shared) || !aligned16(ws)) return PW_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(l, T);
  if (ws_bytes < W.total) return PW_ERR_OOM;
  PW_TRY(device_only());
  NvtxRange range("pw_shared_ffn");
  char* wsb = static_cast<char*>(ws);
  return launched(launch_moe_ffn(l->dev(), nullptr, nullptr, 0, nullptr, nullptr, static_cast<const __half*>(x), T,
                                 y_shared, reinterpret_cast<__half*>(wsb + W.hs_off), 0, as_stream(stream)));
}

extern "C" pw_status pw_moe_ffn(pw_layer_t l, const void* x, const void* x_perm, const int32_t* offsets, int T,
                                float* y_perm, float* y_shared, void* ws, size_t ws_bytes, void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T)) return PW_ERR_INVALID_ARG;
  const bool sh = l->desc.shared_ffn != 0;
  if (sh && !l->shared_loaded) return PW_ERR_INVALID_ARG;
  if (T == 0) return device_only();
  if (!x_perm || !offsets || !y_perm || !ws) return PW_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(y_perm) || !aligned16(ws)) return PW_ERR_INVALID_ARG;
  if (sh && (!x || !y_shared || !aligned16(x) || !aligned16(y_shared))) return PW_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(l, T);
  if (ws_bytes < W.total) return PW_ERR_OOM;
  PW_TRY(all_loaded(l));
  PW_TRY(device_only());
  NvtxRange range("pw_moe_ffn");
  char* wsb = static_cast<char*>(ws);
  cudaStream_t s = as_stream(stream);
  if (l->debug_bounds) PW_TRY(launched(launch_canaries(wsb, W.can, l->d_err, true, s)));
  PW_TRY(launched(launch_moe_ffn(l->dev(), static_cast<const __half*>(x_perm), offsets, T * l->desc.top_k, y_perm,
                                 reinterpret_cast<__half*>(wsb + W.h_off), sh ? static_cast<const __half*>(x) : nullptr,
                                 T, sh ? y_shared : nullptr, reinterpret_cast<__half*>(wsb + W.hs_off), class_mask(l),
                                 s)));
  if (l->debug_bounds) PW_TRY(launched(launch_canaries(wsb, W.can, l->d_err, false, s)));
  return PW_OK;
}

extern "C" pw_status pw_combine(pw_layer_t l, const float* y_perm, const int32_t* inv_slot, const float* w, int T,
                                const float* y_shared, void* y, void* stream) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T)) return PW_ERR_INVALID_ARG;
  if (T > 0 && (!y_perm || !inv_slot || !w || !y)) return PW_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(y_perm) || !aligned16(y) || (y_shared && !aligned16(y_shared))))
    return PW_ERR_INVALID_ARG;
  PW_TRY(device_only());
  NvtxRange range("pw_combine");
  if (T == 0) return PW_OK;
  return launched(launch_combine(l->dev(), y_perm, inv_slot, w, T, y_shared, static_cast<__half*>(y),
                                 as_stream(stream)));
}

extern "C" pw_status pw_layer_check_device(pw_layer_t l, void* stream) {
  PW_TRY(check_layer(l));
  int err[4] = {0, 0, 0, 0};
  if (g_sim) {
    memcpy(err, l->d_err, sizeof(err));
    memset(l->d_err, 0, sizeof(err));
  } else {
    cudaStream_t s = as_stream(stream);
    PW_CUDA(cudaMemcpyAsync(err, l->d_err, sizeof(err), cudaMemcpyDeviceToHost, s));
    PW_CUDA(cudaStreamSynchronize(s));
    PW_CUDA(cudaMemsetAsync(l->d_err, 0, sizeof(err), s));
    // a kernel that gave up on a wait may have left its counters half-way
    if (err[0] != 0) PW_CUDA(cudaMemsetAsync(l->d_sync, 0, sizeof(int) * sync_words(l->desc.n_experts), s));
    PW_CUDA(cudaStreamSynchronize(s));
  }
  if (err[0] == kErrTimeout) return PW_ERR_TIMEOUT;
  if (err[0] != 0) return PW_ERR_DEVICE_CHECK;
  return PW_OK;
}

extern "C" pw_status pw_debug_dequant(pw_layer_t l, int e, int m, void* out, void* stream) {
  PW_TRY(check_layer(l));
  if (e < 0 || e >= l->desc.n_experts || m < 0 || m > 2 || !out) return PW_ERR_INVALID_ARG;
  if (l->bits[e] == 0) return PW_ERR_INVALID_ARG;
  PW_TRY(device_only());
  return launched(launch_debug_dequant(l->dev(), e, m, static_cast<__half*>(out), as_stream(stream)));
}

extern "C" pw_status pw_debug_dequant_kernel(pw_layer_t l, int e, int m, int kernel, void* out, void* stream) {
  PW_TRY(check_layer(l));
  if (e < 0 || e >= l->desc.n_experts || m < 0 || m > 2 || !out || !aligned16(out)) return PW_ERR_INVALID_ARG;
  if (kernel != PW_KERNEL_DECODE && kernel != PW_KERNEL_PREFILL && kernel != PW_KERNEL_DECODE_ROW_TABLES &&
      kernel != PW_KERNEL_DECODE_LANE_TABLES)
    return PW_ERR_INVALID_ARG;
  if (l->bits[e] == 0) return PW_ERR_INVALID_ARG;
  PW_TRY(device_only());
  const DevLayer L = l->dev();
  auto* o = static_cast<__half*>(out);
  cudaStream_t s = as_stream(stream);
  if (kernel == PW_KERNEL_PREFILL) return launched(launch_prefill_dump(L, e, m, o, s));
  const bool lane = kernel == PW_KERNEL_DECODE ? nblk_for(L) == 2 : kernel == PW_KERNEL_DECODE_LANE_TABLES;
  return launched(launch_decode_dump(L, e, m, lane, o, s));
}

extern "C" pw_status pw_debug_page_address(pw_layer_t l, int e, int p, int vpage, uint64_t* addr) {
  PW_TRY(check_layer(l));
  if (!addr || e < 0 || e >= l->desc.n_experts || p < 0 || p > kPlanes || vpage < 0) return PW_ERR_INVALID_ARG;
  const Block& b = p < kPlanes ? l->planes[(size_t)e * kPlanes + p] : l->f16[e];
  if (b.st == B_NONE || vpage >= (int)b.pages.size()) {
    *addr = 0;
    return PW_OK;
  }
  *addr = reinterpret_cast<uint64_t>(blk_addr(l, b, vpage));
  return PW_OK;
}

// ---------------------------------------------------------------------------
// helpers for other entry points (pw_internal.h)
// ---------------------------------------------------------------------------

pw_status pw::record_cuda_error(cudaError_t e) { return cuda_fail(e); }

pw_status pw::ffn_call_args(pw_layer_t l, const void* x_perm, const int32_t* offsets, int T, const float* y_perm,
                            DevLayer* dev, int* cmask, size_t* h_bytes) {
  PW_TRY(check_layer(l));
  if (bad_tokens(T) || !dev || !cmask || !h_bytes) return PW_ERR_INVALID_ARG;
  if (T == 0) return device_only();
  if (!x_perm || !offsets || !y_perm) return PW_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(y_perm)) return PW_ERR_INVALID_ARG;
  PW_TRY(all_loaded(l));
  PW_TRY(device_only());
  *dev = l->dev();
  *cmask = class_mask(l);
  *h_bytes = (size_t)T * l->desc.top_k * l->desc.ffn * 2;
  return PW_OK;
}
