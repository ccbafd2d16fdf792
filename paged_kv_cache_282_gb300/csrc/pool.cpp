// pool.cpp -- host side of libpkv: block allocator, decode planner, staging,
// timing and every entry point of the C ABI declared in include/pkv.h.
//
// The allocator follows the runtime components of the PagedAttention page
// ("KV Cache 与 PagedAttention：显存复用与长上下文推理", sections PagedAttention
// 的设计, 三大运行时组件 and the copy_on_write sketch): a global free pool of
// 16-token blocks, one block table per sequence, reference counts and a copy
// on the first write to a shared block.  Its determinism rules (initial
// order, front-of-pool reuse, smallest free sequence id, order of frees) are
// fixed here so that tests can replay them exactly.

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <numeric>
#include <set>
#include <string>
#include <vector>

#include "../../include/pkv.h"
#include "pkv_internal.h"

using namespace pkv;

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------

static thread_local std::string g_last_error;

static pkv_status fail(pkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

void pkv::set_error(const char* msg) { g_last_error = msg ? msg : ""; }

// Runs an entry point's body; a C++ exception (a failed host allocation)
// becomes a status instead of crossing the C ABI.
template <class F>
static pkv_status guarded(F&& body) noexcept {
  const char* what = nullptr;
  pkv_status st = PKV_ERR_HOST_MEMORY;
  try {
    return body();
  } catch (const std::bad_alloc&) {
    what = "host memory allocation failed";
  } catch (...) {
    what = "unexpected C++ exception";
    st = PKV_ERR_INVALID_ARG;
  }
  try {
    g_last_error = what;
  } catch (...) {
  }
  return st;
}

#define PKV_CUDA(call)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(PKV_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                  __FILE__, __LINE__);                                                  \
  } while (0)

// ---------------------------------------------------------------------------
// keep-set geometry (which logical blocks a decode must read)
// ---------------------------------------------------------------------------

struct BlockRange {
  int32_t lo, hi;  // logical blocks [lo, hi)
};

static int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Logical block ranges that intersect the keep-set of a decode query at
// position L - 1 (mask semantics in include/pkv.h).
static int keep_ranges(int L, int mode, int S, int W, BlockRange out[2]) {
  if (L <= 0) return 0;
  const int nblk = ceil_div(L, kBlock);
  if (mode == PKV_MASK_FULL) {
    out[0] = {0, nblk};
    return 1;
  }
  if (mode == PKV_MASK_SLIDING) {
    int lo_tok = std::max(0, L - 1 - W);
    out[0] = {lo_tok / kBlock, nblk};
    return 1;
  }
  // sink + window
  if ((int64_t)L <= (int64_t)S + W) {
    out[0] = {0, nblk};
    return 1;
  }
  const int sink_hi = ceil_div(S, kBlock);  // blocks holding the sinks
  const int win_lo = (L - W) / kBlock;      // first block holding the window
  if (S > 0 && W > 0 && sink_hi >= win_lo) {
    out[0] = {0, nblk};
    return 1;
  }
  int n = 0;
  if (S > 0) out[n++] = {0, sink_hi};
  if (W > 0) out[n++] = {win_lo, nblk};
  return n;
}

// ---------------------------------------------------------------------------
// host block allocator
// ---------------------------------------------------------------------------

static uint64_t mix64(uint64_t& s) {  // splitmix64 (Steele, Lea & Flood 2014)
  s += 0x9E3779B97F4A7C15ULL;
  uint64_t z = s;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

struct TablePatch {
  int32_t index, value;  // flat index into the device block table
};

struct HostAllocator {
  int32_t NB = 0, max_seqs = 0, max_blocks = 0;
  std::vector<int32_t> refcount;
  std::vector<int32_t> free_blocks;  // back() is the front of the free pool
  std::vector<std::vector<int32_t>> table;
  std::vector<int32_t> len;
  std::vector<uint8_t> live, holes;
  std::set<int32_t> free_ids;
  int64_t cow_count = 0, n_alloc = 0, n_freed = 0;
  int64_t n_multi = 0;  // blocks held more than once (refcount > 1)
  // queued device-side effects (device pools only: a host-only pool has no
  // device table or blocks to update)
  bool queue = false;
  std::vector<int32_t> pending_cow;  // (src, dst) pairs
  std::vector<TablePatch> pending_patch;
  // duplicate checks of sequence lists: the check's epoch, per sequence id
  std::vector<uint32_t> seen_mark;
  uint32_t seen_epoch = 0;
  // per-block counters of one append's dry run (valid for the current epoch)
  std::vector<uint32_t> drop_mark;
  std::vector<int32_t> drop_count;
  uint32_t drop_epoch = 0;

  // Starts a fresh set of per-block counters (all zero).
  void begin_drops() {
    if (drop_mark.size() != (size_t)NB) {
      drop_mark.assign(NB, 0);
      drop_count.assign(NB, 0);
    }
    if (++drop_epoch == 0) {
      std::fill(drop_mark.begin(), drop_mark.end(), 0);
      drop_epoch = 1;
    }
  }
  int32_t& dropped(int32_t b) {
    if (drop_mark[b] != drop_epoch) {
      drop_mark[b] = drop_epoch;
      drop_count[b] = 0;
    }
    return drop_count[b];
  }
  // per table entry: the position of its last queued patch (valid only for
  // the entries the queue names, which each collapse writes before reading,
  // so the array is never cleared and its untouched pages are never mapped)
  std::unique_ptr<int32_t[]> patch_last;
  size_t patch_last_n = 0;
  // per source block of a swap (device or host block): its destination,
  // valid where move_mark holds the current epoch
  std::vector<uint32_t> move_mark;
  std::vector<int32_t> move_dst;
  uint32_t move_epoch = 0;
  void begin_moves(size_t n_src) {
    if (move_mark.size() < n_src) {
      move_mark.assign(n_src, 0);
      move_dst.assign(n_src, -1);
    }
    if (++move_epoch == 0) {
      std::fill(move_mark.begin(), move_mark.end(), 0);
      move_epoch = 1;
    }
  }
  // per block, for the current wave of copies: 2 * epoch when the block is a
  // source in it, 2 * epoch + 1 when it is a destination
  std::vector<uint32_t> wave_mark;
  uint32_t wave_epoch = 0;

  // The first id that occurs twice in ids[0, n), or -1 (ids must already be
  // valid sequence ids).  Linear in n.
  int32_t first_repeat(int32_t n, const int32_t* ids) {
    if (seen_mark.size() != (size_t)max_seqs) seen_mark.assign(max_seqs, 0);
    if (++seen_epoch == 0) {
      std::fill(seen_mark.begin(), seen_mark.end(), 0);
      seen_epoch = 1;
    }
    for (int32_t i = 0; i < n; ++i) {
      if (seen_mark[ids[i]] == seen_epoch) return ids[i];
      seen_mark[ids[i]] = seen_epoch;
    }
    return -1;
  }

  void init(int32_t nb, int32_t ms, int32_t mb, uint64_t seed, const int32_t* order) {
    NB = nb;
    max_seqs = ms;
    max_blocks = mb;
    refcount.assign(nb, 0);
    n_multi = 0;
    std::vector<int32_t> front_first(nb);
    if (order) {
      std::copy(order, order + nb, front_first.begin());
    } else {
      std::iota(front_first.begin(), front_first.end(), 0);
      if (seed != 0) {
        uint64_t st = seed;
        for (int32_t i = nb - 1; i >= 1; --i) {
          int32_t j = (int32_t)(mix64(st) % (uint64_t)(i + 1));
          std::swap(front_first[i], front_first[j]);
        }
      }
    }
    free_blocks.assign(front_first.rbegin(), front_first.rend());
    table.assign(ms, {});
    len.assign(ms, 0);
    live.assign(ms, 0);
    holes.assign(ms, 0);
    swapped.assign(ms, 0);
    host_table.assign(ms, {});
    free_ids.clear();
    for (int32_t s = 0; s < ms; ++s) free_ids.insert(s);
  }

  bool valid_seq(int32_t s) const { return s >= 0 && s < max_seqs && live[s]; }
  // live and with its blocks on the device (not swapped out)
  bool on_device(int32_t s) const { return valid_seq(s) && !swapped[s]; }

  // CPU swap space: host blocks with their own counts and free pool
  int32_t NH = 0;
  std::vector<int32_t> host_refcount, host_free;  // host_free.back() is the front
  std::vector<std::vector<int32_t>> host_table;
  std::vector<uint8_t> swapped;
  void set_swap_space(int32_t nh) {
    NH = nh;
    host_refcount.assign(nh, 0);
    host_free.resize(nh);
    for (int32_t i = 0; i < nh; ++i) host_free[i] = nh - 1 - i;
  }
  int32_t take_host() {
    const int32_t b = host_free.back();
    host_free.pop_back();
    host_refcount[b] = 1;
    return b;
  }
  void release_host(int32_t b) {
    if (--host_refcount[b] == 0) host_free.push_back(b);
  }

  int32_t take() {
    int32_t b = free_blocks.back();
    free_blocks.pop_back();
    refcount[b] = 1;
    ++n_alloc;
    return b;
  }
  // Undoes the latest take() of b (blocks go back in the reverse order of
  // their takes, which restores the free pool exactly).
  void untake(int32_t b) {
    refcount[b] = 0;
    free_blocks.push_back(b);
    --n_alloc;
  }
  void release(int32_t b) {
    if (refcount[b] == 2) --n_multi;
    if (--refcount[b] == 0) {
      free_blocks.push_back(b);
      ++n_freed;
    }
  }
  void add_ref(int32_t b) {
    if (++refcount[b] == 2) ++n_multi;
  }
  void set_entry(int32_t s, int32_t lb, int32_t v) {
    if ((int32_t)table[s].size() <= lb) table[s].resize(lb + 1, -1);
    table[s][lb] = v;
    if (queue) pending_patch.push_back({s * max_blocks + lb, v});
  }
  // Releases the blocks of s from logical block first_lb on (ascending) and
  // shortens its table there.  Runs of evicted entries (-1), which fill most
  // of a long streaming sequence's table, are skipped eight at a time.  The
  // released entries get -1 patches from logical block patch_from on (the
  // caller sets the ones below it again).
  void drop_from(int32_t s, int32_t first_lb, int32_t patch_from = 0) {
    auto& t = table[s];
    const int32_t n = (int32_t)t.size();
    for (int32_t lb = first_lb; lb < n;) {
      if (lb + 8 <= n) {
        uint64_t w[4];
        memcpy(w, t.data() + lb, sizeof w);
        if ((w[0] & w[1] & w[2] & w[3]) == ~uint64_t(0)) {
          lb += 8;
          continue;
        }
      }
      for (const int32_t e = std::min(n, lb + 8); lb < e; ++lb) {
        const int32_t b = t[lb];
        if (b >= 0) release(b);
        if (queue && b != -1 && lb >= patch_from) pending_patch.push_back({s * max_blocks + lb, -1});
      }
    }
    if (n > first_lb) t.resize(first_lb);
  }
};

// ---------------------------------------------------------------------------
// staging: pinned host slots mirrored by device slots, reused round-robin
// ---------------------------------------------------------------------------

struct StagingSlot {
  char* host = nullptr;
  char* dev = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;    // recorded after the last kernel reading `dev`
  cudaEvent_t copied = nullptr;  // recorded after an upload on the copy stream
  bool pending = false;
};

struct Staging {
  // Enough slots that a step's uploads (plan, per-sequence rows) reuse a slot
  // only well after its kernel has run, so acquire does not stall the host.
  static constexpr int kSlots = 16;
  StagingSlot slot[kSlots];
  int next = 0;

  pkv_status acquire(size_t bytes, StagingSlot** out) {
    StagingSlot& s = slot[next];
    next = (next + 1) % kSlots;
    if (s.pending) {
      PKV_CUDA(cudaEventSynchronize(s.done));
      s.pending = false;
    }
    if (s.cap < bytes) {
      size_t cap = std::max<size_t>(bytes, size_t(1) << 18);
      cap = (cap + 4095) & ~size_t(4095);
      if (s.host) PKV_CUDA(cudaFreeHost(s.host));
      if (s.dev) PKV_CUDA(cudaFree(s.dev));
      s.host = nullptr;
      s.dev = nullptr;
      s.cap = 0;
      PKV_CUDA(cudaHostAlloc((void**)&s.host, cap, cudaHostAllocDefault));
      PKV_CUDA(cudaMalloc((void**)&s.dev, cap));
      s.cap = cap;
    }
    if (!s.done) PKV_CUDA(cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming));
    *out = &s;
    return PKV_OK;
  }
  static pkv_status upload(StagingSlot* s, size_t bytes, cudaStream_t st) {
    if (bytes) PKV_CUDA(cudaMemcpyAsync(s->dev, s->host, bytes, cudaMemcpyHostToDevice, st));
    return PKV_OK;
  }
  // The same copy on the pool's own copy stream, with `st` waiting for it: the
  // copy then overlaps whatever `st` is still running (a decode plan upload
  // overlaps the append kernel before it).  The slot's previous readers have
  // finished (acquire waited for them), so nothing on `st` is overtaken.
  cudaStream_t copy_stream = nullptr;
  pkv_status upload_overlapped(StagingSlot* s, size_t bytes, cudaStream_t st) {
    if (!bytes) return PKV_OK;
    if (!copy_stream) PKV_CUDA(cudaStreamCreateWithFlags(&copy_stream, cudaStreamNonBlocking));
    if (!s->copied) PKV_CUDA(cudaEventCreateWithFlags(&s->copied, cudaEventDisableTiming));
    PKV_CUDA(cudaMemcpyAsync(s->dev, s->host, bytes, cudaMemcpyHostToDevice, copy_stream));
    PKV_CUDA(cudaEventRecord(s->copied, copy_stream));
    PKV_CUDA(cudaStreamWaitEvent(st, s->copied, 0));
    return PKV_OK;
  }
  static pkv_status release(StagingSlot* s, cudaStream_t st) {
    PKV_CUDA(cudaEventRecord(s->done, st));
    s->pending = true;
    return PKV_OK;
  }
  void destroy() {
    if (copy_stream) cudaStreamSynchronize(copy_stream);
    for (auto& s : slot) {
      if (s.pending) cudaEventSynchronize(s.done);
      if (s.host) cudaFreeHost(s.host);
      if (s.dev) cudaFree(s.dev);
      if (s.done) cudaEventDestroy(s.done);
      if (s.copied) cudaEventDestroy(s.copied);
      s = StagingSlot{};
    }
    if (copy_stream) cudaStreamDestroy(copy_stream);
    copy_stream = nullptr;
  }
};

// ---------------------------------------------------------------------------
// per-kernel event timing
// ---------------------------------------------------------------------------

struct Timing {
  int32_t mask = 0;  // bit k: bracket launches of kernel id k with events
  std::vector<cudaEvent_t> spare;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> marks[PKV_KERNEL_COUNT];

  cudaEvent_t get() {
    if (!spare.empty()) {
      cudaEvent_t e = spare.back();
      spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void destroy() {
    for (auto& v : marks)
      for (auto& pr : v) {
        cudaEventDestroy(pr.first);
        cudaEventDestroy(pr.second);
      }
    for (auto e : spare) cudaEventDestroy(e);
    spare.clear();
    for (auto& v : marks) v.clear();
  }
};

// ---------------------------------------------------------------------------
// the pool
// ---------------------------------------------------------------------------

namespace {
struct PlanCache;  // the decode planner's reusable buffers
void destroy_plan_cache(PlanCache* c);
struct PlanCacheDeleter {
  void operator()(PlanCache* c) const { destroy_plan_cache(c); }
};
}  // namespace

struct pkv_pool {
  pkv_pool_config cfg{};
  bool device = false;
  pkv_pool_buffers buf{};
  HostAllocator alloc;
  Staging staging;
  Timing timing;
  int64_t launches = 0;
  int device_id = 0, num_sms = 0;
  int tc_warps_per_cta = 0, tc_ctas_per_sm = 0;    // one sequence per warp
  int tc2_warps_per_cta = 0, tc2_ctas_per_sm = 0;  // up to two sequences over shared blocks
  int cascade = 1;  // 0: off; 1: sequence pairs; 2: group prefixes (multi-query kernel)
  size_t tc_smem = 0;
  CUtensorMap tmap_k{}, tmap_v{};
  bool tc_path = false;
  const float* k_channel = nullptr;  // per-channel scales [Hk][D] (device, borrowed), FP8 / INT8 only
  const float* v_channel = nullptr;
  int G = 1;   // query heads per kv head
  int HG = 1;  // kv heads per unit of the tensor-core decode (the planner's kv heads hold HG each)
  uint64_t wait_limit_ns = 4000000000ull;  // bound of the decode kernel's waits
  int32_t starve_warp = -1;                // one-shot wait-expiry test hook
  bool starve_select = false;              // one-shot wait-expiry test hook of the selection
  bool general_plan = false;               // test hook: plan every decode on the general path
  // Vectors reused by every decode plan: fresh ones each call would spend
  // most of the planning time faulting in new pages.
  std::unique_ptr<PlanCache, PlanCacheDeleter> plan_cache;
  // CPU swap space (host pointers and their device-mapped addresses)
  bool swap_space = false;
  void *host_k = nullptr, *host_v = nullptr;
  float *host_ks = nullptr, *host_vs = nullptr;
  void *host_k_dev = nullptr, *host_v_dev = nullptr;
  float *host_ks_dev = nullptr, *host_vs_dev = nullptr;
};

namespace {

template <class F>
pkv_status launch(pkv_pool* p, int kernel, cudaStream_t st, F&& fn) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool timed = (p->timing.mask >> kernel) & 1;
  if (timed) {
    a = p->timing.get();
    b = p->timing.get();
    PKV_CUDA(cudaEventRecord(a, st));
  }
  cudaError_t e = fn();
  if (e != cudaSuccess) {
    if (timed) {  // the pair goes back unused
      p->timing.spare.push_back(a);
      p->timing.spare.push_back(b);
    }
    return fail(PKV_ERR_CUDA, "kernel %d launch failed: %s", kernel, cudaGetErrorString(e));
  }
  ++p->launches;
  if (timed) {
    PKV_CUDA(cudaEventRecord(b, st));
    p->timing.marks[kernel].push_back({a, b});
  }
  return PKV_OK;
}

int elem_bytes(int kv_dtype) { return kv_dtype == PKV_KV_FP32 ? 4 : kv_dtype == PKV_KV_BF16 ? 2 : 1; }
// FP8 and INT8 pools keep one fp32 scale per (token, kv head) for K and V
bool has_scales(int kv_dtype) { return kv_dtype == PKV_KV_FP8_E4M3 || kv_dtype == PKV_KV_INT8; }

pkv_status check_config(const pkv_pool_config* c) {
  if (!c) return fail(PKV_ERR_INVALID_ARG, "config is NULL");
  if (c->block_size != kBlock) return fail(PKV_ERR_UNSUPPORTED, "block_size must be 16");
  if (c->num_blocks < 0 || c->max_seqs <= 0 || c->max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_blocks, max_seqs and max_blocks_per_seq must be positive");
  if ((int64_t)c->max_seqs * c->max_blocks_per_seq >= (int64_t(1) << 31))
    return fail(PKV_ERR_UNSUPPORTED, "block table larger than 2^31 entries");
  if ((int64_t)c->max_blocks_per_seq * kBlock >= (int64_t(1) << 31))
    return fail(PKV_ERR_UNSUPPORTED, "max_blocks_per_seq too large");
  if (c->n_heads <= 0 || c->n_kv_heads <= 0 || c->n_heads % c->n_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "n_heads must be a positive multiple of n_kv_heads");
  int G = c->n_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(PKV_ERR_UNSUPPORTED, "group size %d not in {1,2,4,8}", G);
  if (c->kv_dtype != PKV_KV_FP32 && c->kv_dtype != PKV_KV_BF16 && c->kv_dtype != PKV_KV_FP8_E4M3 &&
      c->kv_dtype != PKV_KV_INT8)
    return fail(PKV_ERR_INVALID_ARG, "unknown kv_dtype %d", c->kv_dtype);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", c->head_dim);
  if ((int64_t)c->num_blocks * c->n_kv_heads * kBlock >= (int64_t(1) << 31))
    return fail(PKV_ERR_UNSUPPORTED, "pool too large for 32-bit row coordinates");
  if (c->free_order) {
    std::vector<uint8_t> seen(c->num_blocks, 0);
    for (int32_t i = 0; i < c->num_blocks; ++i) {
      int32_t b = c->free_order[i];
      if (b < 0 || b >= c->num_blocks || seen[b]) return fail(PKV_ERR_INVALID_ARG, "free_order is not a permutation");
      seen[b] = 1;
    }
  }
  return PKV_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

// kv heads per unit of the tensor-core decode for this pool (1 unless the
// pool's kv heads split evenly into tc_head_group-sized units).
int unit_heads(const pkv_pool_config& c, int G) {
  if (c.kv_dtype == PKV_KV_FP32) return 1;
  const int hg = tc_head_group(c.kv_dtype, G, c.head_dim);
  return hg > 1 && c.n_kv_heads % hg == 0 ? hg : 1;
}

pkv_status make_tensor_map(CUtensorMap* m, void* base, const pkv_pool_config& c, int hg) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    PKV_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q));
    if (q != cudaDriverEntryPointSuccess || !ptr) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    fn = (EncodeTiledFn)ptr;
  }
  const bool fp8 = elem_bytes(c.kv_dtype) == 1;  // FP8 or INT8 codes
  const int es = fp8 ? 1 : 2;
  const uint64_t rows = (uint64_t)c.num_blocks * c.n_kv_heads * kBlock;
  const int row_bytes = c.head_dim * es;
  // 2-D view with 128-byte box rows and the 128-byte swizzle.  Rows of at
  // least 128 bytes: rows = (block, kv head, slot), columns = head_dim
  // elements, one box = 16 rows x 128 bytes (64 bf16 or 128 one-byte codes).
  // 64-byte rows (one-byte codes, head_dim 64): two slots per 128-byte row,
  // one box = the 8 rows of a (block, kv head) chunk.  A decode unit of hg
  // adjacent kv heads takes hg chunks in one box.
  const bool pair_rows = row_bytes < 128;
  cuuint64_t dims[2] = {(cuuint64_t)(pair_rows ? 128 : c.head_dim), (cuuint64_t)(pair_rows ? rows / 2 : rows)};
  cuuint64_t strides[1] = {(cuuint64_t)(pair_rows ? 128 : row_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)((pair_rows ? kBlock / 2 : kBlock) * hg)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PKV_OK;
}

// Several queued changes of one table entry collapse to the last one (the
// kernels that apply patches do so in parallel); the kept patches stay in
// queue order.
std::vector<TablePatch> dedup_patches(HostAllocator& A, const std::vector<TablePatch>& q) {
  const size_t entries = (size_t)A.max_seqs * A.max_blocks;
  if (A.patch_last_n != entries) {
    A.patch_last.reset(new int32_t[entries]);
    A.patch_last_n = entries;
  }
  for (size_t i = 0; i < q.size(); ++i) A.patch_last[q[i].index] = (int32_t)i;
  std::vector<TablePatch> out;
  out.reserve(q.size());
  for (size_t i = 0; i < q.size(); ++i)
    if (A.patch_last[q[i].index] == (int32_t)i) out.push_back(q[i]);
  return out;
}

// The queued copies must give what running them one by one in queue order
// gives, and the copies of one launch run in any order.  So the queue is cut
// into waves that run in order, each free of conflicts: within a wave no
// copy reads a block that another writes (a source that is an earlier
// copy's destination, or a destination that is an earlier copy's source)
// and no two copies write one block.  A block freed after it was queued as
// a source can come back as a later copy's destination.  Returns the first
// copy of each wave and, last, the number of copies.
std::vector<size_t> cow_waves(HostAllocator& A) {
  const size_t ncow = A.pending_cow.size() / 2;
  std::vector<size_t> start{0};
  if (ncow) {
    if (A.wave_mark.size() != (size_t)A.NB) A.wave_mark.assign(A.NB, 0);
    auto next_wave = [&A]() {
      if (++A.wave_epoch >= (1u << 31)) {
        std::fill(A.wave_mark.begin(), A.wave_mark.end(), 0);
        A.wave_epoch = 1;
      }
    };
    next_wave();
    for (size_t k = 0; k < ncow; ++k) {
      const int32_t src = A.pending_cow[2 * k], dst = A.pending_cow[2 * k + 1];
      const uint32_t as_src = 2 * A.wave_epoch, as_dst = as_src + 1;
      if (A.wave_mark[src] == as_dst || A.wave_mark[dst] == as_src || A.wave_mark[dst] == as_dst) {
        start.push_back(k);
        next_wave();
      }
      A.wave_mark[src] = 2 * A.wave_epoch;
      A.wave_mark[dst] = 2 * A.wave_epoch + 1;
    }
  }
  start.push_back(ncow);
  return start;
}

// Flushes queued copy-on-write copies and, unless the caller applies them
// itself (the append kernel does), the queued block-table patches.
// patches_unique: the caller knows no table entry is queued twice.
pkv_status flush_pending(pkv_pool* p, cudaStream_t st, bool with_patches = true, bool patches_unique = false) {
  HostAllocator& A = p->alloc;
  if (A.pending_cow.empty() && (A.pending_patch.empty() || !with_patches)) return PKV_OK;
  // Table patches: several changes to one entry collapse to the last one (the
  // patch kernel applies its list in parallel).
  std::vector<TablePatch> collapsed;
  if (with_patches && !patches_unique) collapsed = dedup_patches(A, A.pending_patch);
  const std::vector<TablePatch>& patches = !with_patches || !patches_unique ? collapsed : A.pending_patch;
  // COW copies in waves of independent copies
  const std::vector<size_t> wave_start = cow_waves(A);
  const size_t ncow = A.pending_cow.size() / 2, npatch = patches.size();
  const size_t cow_bytes = ncow * 2 * sizeof(int32_t), patch_off = (cow_bytes + 255) & ~size_t(255);
  const size_t bytes = patch_off + npatch * sizeof(TablePatch);
  StagingSlot* s;
  if (pkv_status r = p->staging.acquire(bytes, &s)) return r;
  if (ncow) memcpy(s->host, A.pending_cow.data(), cow_bytes);
  if (npatch) memcpy(s->host + patch_off, patches.data(), npatch * sizeof(TablePatch));
  if (pkv_status r = Staging::upload(s, bytes, st)) return r;
  const auto& c = p->cfg;
  if (ncow) {
    const size_t blk_bytes = (size_t)c.n_kv_heads * kBlock * c.head_dim * elem_bytes(c.kv_dtype);
    const size_t scl = has_scales(c.kv_dtype) ? (size_t)c.n_kv_heads * kBlock : 0;
    for (size_t w = 0; w + 1 < wave_start.size(); ++w) {
      const size_t k0 = wave_start[w], k1 = wave_start[w + 1];
      if (k1 == k0) continue;
      if (pkv_status r = launch(p, PKV_KERNEL_COW_COPY, st, [&] {
            return launch_cow_copy((const int32_t*)s->dev + 2 * k0, (int)(k1 - k0), p->buf.k_pool, p->buf.v_pool,
                                   p->buf.k_scale, p->buf.v_scale, blk_bytes, scl, st);
          }))
        return r;
    }
  }
  if (npatch) {
    if (pkv_status r = launch(p, PKV_KERNEL_TABLE_PATCH, st, [&] {
          return launch_table_patch((const int32_t*)(s->dev + patch_off), (int)npatch, p->buf.block_tables, st);
        }))
      return r;
  }
  if (pkv_status r = Staging::release(s, st)) return r;
  A.pending_cow.clear();
  if (with_patches) A.pending_patch.clear();
  return PKV_OK;
}

pkv_status check_seq_list(const pkv_pool* p, int32_t n, const int32_t* ids) {
  if (n < 0) return fail(PKV_ERR_INVALID_ARG, "n_seqs < 0");
  if (n > 0 && !ids) return fail(PKV_ERR_INVALID_ARG, "seq_ids is NULL");
  for (int32_t i = 0; i < n; ++i)
    if (!p->alloc.on_device(ids[i]))
      return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live or is swapped out", ids[i]);
  return PKV_OK;
}

bool valid_mask(int mode, int S, int W) {
  if (mode == PKV_MASK_FULL) return true;
  if (mode == PKV_MASK_SLIDING) return W >= 0;
  if (mode == PKV_MASK_SINK_WINDOW) return S >= 0 && W >= 0;
  return false;
}

}  // namespace

// ---------------------------------------------------------------------------
// decode planning
// ---------------------------------------------------------------------------

namespace {

constexpr int kMinUnitsPerWarp = 4;

struct Plan {
  std::vector<int32_t> warp_begin;  // per physical warp slot (cta * warps_per_cta + warp)
  std::vector<Piece> pieces;        // grouped by physical warp slot
  std::vector<CombineItem> combine;
  std::vector<EmptyItem> empty;
  int total_warps = 0;  // physical warp slots = ctas * warps_per_cta
  int ctas = 0;
  int n_partials = 0;
  int nq = 1;  // 2: pieces may carry a second sequence (the two-sequence kernel)
  std::vector<PrefixItem> prefix_items;  // the multi-query kernel's work (group prefixes)
  std::vector<PrefixMember> prefix_members;
};

struct Seg {
  int32_t b, g, lo, hi;  // batch index, kv head, logical blocks [lo, hi)
  int32_t b1;            // >= 0: a second sequence over the same physical blocks
  int32_t stream_from;   // blocks from this one on are read once (Piece::stream_from)
};

struct PlanRun {
  size_t begin, end;  // pieces [begin, end)
  bool record0;       // the first sequence writes a partial record
};

struct PlanCache {
  Plan plan;
  std::vector<Seg> segs;
  std::vector<int64_t> bg_units;
  std::vector<int32_t> piece_warp, first_partial, n_part, item_of, cursor;
  std::vector<PlanRun> runs;
  std::vector<size_t> vstart;
  std::vector<Piece> ordered;
  std::vector<char> blob;
  struct BgRecord {
    int32_t vfirst, first_partial, flags;
  };
  struct WarpStartRec {
    int64_t unit;
    int32_t seg, seg_off;
  };
  std::vector<BgRecord> bg_rec;
  std::vector<WarpStartRec> warp_start;
  struct SegRecord {
    int32_t v0, runs, rec0, rec1;
  };
  std::vector<SegRecord> seg_rec;
  struct SegPiece {
    Piece piece;  // the fields every piece of the segment shares
    int32_t first_partial, vfirst;
    bool run_continues;
  };
  std::vector<SegPiece> seg_piece;
};

void destroy_plan_cache(PlanCache* c) { delete c; }

PlanCache& plan_cache(pkv_pool* p) {
  if (!p->plan_cache) p->plan_cache.reset(new PlanCache());
  return *p->plan_cache;
}

int warps_per_cta(const pkv_pool* p, int nq) {
  return std::max(1, nq == 2 ? p->tc2_warps_per_cta : p->tc_warps_per_cta);
}

int max_total_warps(const pkv_pool* p, int nq = 1) {
  const int ctas = nq == 2 ? p->tc2_ctas_per_sm : p->tc_ctas_per_sm;
  return std::max(1, p->num_sms * std::max(1, ctas) * warps_per_cta(p, nq));
}

// Upper bound of partial records (and pieces) of one decode call.
size_t max_pieces(const pkv_pool* p, int32_t n_seqs, int32_t num_splits) {
  const size_t nbg = (size_t)n_seqs * (p->cfg.n_kv_heads / p->HG);
  const size_t a = 2 * nbg + (size_t)max_total_warps(p) + 1;
  const size_t b = nbg * (size_t)std::max(1, num_splits) + nbg + 1;
  // shared-prefix plans: 3 segments per sequence pair and kv head, a record
  // for each sequence of a run, and up to kMaxPrefixSplit group-prefix records
  const size_t c = 2 * (2 * nbg + (size_t)max_total_warps(p, 2)) + 4 * nbg + 2;
  return std::max(std::max(a, b), c);
}

// Shared-prefix planning for decode over whole keep-sets.  Blocks are shared
// only through forks and replaced only at the tail (append, copy-on-write,
// truncate) or all at once (compaction), so two sequences that hold the same
// physical block at logical index k share every block before it as well:
// sharing is a prefix of the tables.

// Leading full blocks that rows x and y share, among the first lim: the last
// equal entry by bisection, checked by memcmp (a mismatch inside the found
// prefix, never expected, falls back to the exact scan).
int32_t shared_blocks(const int32_t* x, const int32_t* y, int32_t from, int32_t lim) {
  if (lim <= from) return from;
  int32_t c = from, hi = lim;
  if (x[lim - 1] == y[lim - 1]) {
    c = lim;
  } else {
    while (c < hi) {  // entries below c equal; entry hi - 1 differs (or hi = lim)
      const int32_t mid = (c + hi) / 2;
      if (x[mid] == y[mid]) c = mid + 1; else hi = mid;
    }
  }
  if (c > 0 && (memcmp(x, y, (size_t)c * sizeof(int32_t)) != 0 || x[0] < 0))
    c = (int32_t)(std::mismatch(x, x + c, y).first - x);
  return c;
}

// Groups of at least kMinGroupMembers sequences sharing their first
// kMinGroupBlocks (or more) full blocks: the group's common prefix is read
// once per CTA by the multi-query kernel (BF16 pools).
constexpr int kMinGroupMembers = 4, kMinGroupBlocks = 8;
constexpr int kMaxPrefixSplit = 4;  // records per (sequence, kv head) from its group prefix

struct PrefixGroup {
  std::vector<int32_t> members;  // batch indices, ascending
  int32_t shared;                // common full blocks
};

std::vector<PrefixGroup> find_prefix_groups(const pkv_pool* p, int32_t n, const int32_t* ids) {
  std::vector<PrefixGroup> groups;
  if (p->cfg.kv_dtype != PKV_KV_BF16 || p->cfg.head_dim != 128) return groups;  // the multi-query kernel's shapes
  const auto& A = p->alloc;
  auto full = [&](int32_t b) { return A.len[ids[b]] / kBlock; };
  auto row = [&](int32_t b) { return A.table[ids[b]].data(); };
  std::vector<std::pair<int32_t, int32_t>> keyed;  // (first block, batch index)
  for (int32_t b = 0; b < n; ++b)
    if (full(b) >= kMinGroupBlocks && row(b)[0] >= 0) keyed.push_back({row(b)[0], b});
  std::sort(keyed.begin(), keyed.end());
  for (size_t i = 0; i < keyed.size();) {
    size_t j = i;
    while (j < keyed.size() && keyed[j].first == keyed[i].first) ++j;
    if (j - i >= (size_t)kMinGroupMembers) {
      PrefixGroup gr;
      const int32_t x = keyed[i].second;
      int32_t c = full(x);
      for (size_t k = i; k < j; ++k) {
        gr.members.push_back(keyed[k].second);
        if (k > i) c = std::min(c, shared_blocks(row(x), row(keyed[k].second), 0, std::min(c, full(keyed[k].second))));
      }
      gr.shared = c;
      if (c >= kMinGroupBlocks) groups.push_back(std::move(gr));
    }
    i = j;
  }
  return groups;
}

// Pairs of sequences that share blocks past their group prefix (base[b]
// blocks, 0 outside groups): first those whose last full blocks coincide
// (they share every full block), then those with the same first block past
// the base.  Pairs form only between sequences with the same base.  Returns
// (b0, b1, shared blocks) triples (shared counted from block 0).
struct Pairing {
  int32_t b0, b1, shared;
};

std::vector<Pairing> pair_shared_prefixes(const pkv_pool* p, int32_t n, const int32_t* ids,
                                          const std::vector<int32_t>& base) {
  const auto& A = p->alloc;
  auto full = [&](int32_t b) { return A.len[ids[b]] / kBlock; };
  auto row = [&](int32_t b) { return A.table[ids[b]].data(); };
  std::vector<Pairing> pairs;
  std::vector<uint8_t> used(n, 0);
  std::vector<std::pair<std::pair<int64_t, int32_t>, int32_t>> keyed;  // ((key, base), b)
  keyed.reserve(n);
  auto pair_adjacent = [&]() {
    std::sort(keyed.begin(), keyed.end());
    for (size_t i = 0; i + 1 < keyed.size();) {
      if (keyed[i].first != keyed[i + 1].first) {
        ++i;
        continue;
      }
      const int32_t x = keyed[i].second, y = keyed[i + 1].second;
      const int32_t c = shared_blocks(row(x), row(y), 0, std::min(full(x), full(y)));
      if (c > base[x]) {
        pairs.push_back({std::min(x, y), std::max(x, y), c});
        used[x] = used[y] = 1;
        i += 2;
      } else {
        ++i;
      }
    }
  };
  for (int32_t b = 0; b < n; ++b)
    if (full(b) > base[b] && row(b)[full(b) - 1] >= 0)
      keyed.push_back({{((int64_t)full(b) << 32) | row(b)[full(b) - 1], base[b]}, b});
  pair_adjacent();
  keyed.clear();
  for (int32_t b = 0; b < n; ++b)
    if (!used[b] && full(b) > base[b] && row(b)[base[b]] >= 0) keyed.push_back({{row(b)[base[b]], base[b]}, b});
  pair_adjacent();
  return pairs;
}

// Fills plan = the pool's cached plan; the returned reference stays valid
// until the next call.
// The stream-K plan when every piece serves one sequence (no pairs, no group
// prefixes, automatic partition), in one pass over the warps: the same plan
// as the general path below, built without its intermediate piece lists.
// Warp w takes the units [U w / TW, U (w + 1) / TW) of the segment list; a
// (sequence, kv head) whose units span warps vfirst..vlast > vfirst writes
// one partial record per warp, numbered in warp order from its first record;
// each warp's pieces go straight to its physical slot.
// The warp that holds unit u (warp w holds [U w / TW, U (w + 1) / TW)), for
// u that never decreases: the bounds advance by U / TW plus a carry of the
// remainder, without division.
struct WarpCursor {
  int64_t q, r, TW, next, carry;  // next: first unit of warp v + 1
  int32_t v = 0;
  WarpCursor(int64_t U, int64_t tw) : q(U / tw), r(U % tw), TW(tw), next(U / tw), carry(U % tw) {}
  int32_t at(int64_t u) {
    while (next <= u) {
      ++v;
      next += q;
      carry += r;
      if (carry >= TW) {
        carry -= TW;
        ++next;
      }
    }
    return v;
  }
};

void plan_stream_k_single(pkv_pool* p, int32_t n, const int32_t* ids, PlanCache& cache, int TWmax) {
  Plan& plan = cache.plan;
  const int Hk = p->cfg.n_kv_heads / p->HG;  // units of HG kv heads
  const auto& A = p->alloc;
  const std::vector<Seg>& segs = cache.segs;
  const std::vector<int64_t>& bg_units = cache.bg_units;
  const size_t nbg = (size_t)n * Hk;
  int64_t U = 0;
  for (const Seg& sg : segs) U += sg.hi - sg.lo;
  const int TW = (int)std::min<int64_t>(TWmax, (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp);
  // per (sequence, kv head): its first warp, first record and merge item
  // (flags: the merge item << 1, 0 when the output is written directly)
  using BgRec = PlanCache::BgRecord;
  std::vector<BgRec>& bgr = cache.bg_rec;
  bgr.assign(nbg, BgRec{0, -1, 0});
  WarpCursor wc(U, TW);
  int next_partial = 0;
  {
    int64_t off = 0;
    for (size_t bg = 0; bg < nbg; ++bg) {
      const int64_t nu = bg_units[bg];
      if (nu == 0) {
        plan.empty.push_back({(int32_t)(bg / Hk), (int32_t)(bg % Hk)});
        continue;
      }
      const int32_t v0 = wc.at(off), v1 = wc.at(off + nu - 1);
      bgr[bg].vfirst = v0;
      if (v1 > v0) {
        bgr[bg].first_partial = next_partial;
        bgr[bg].flags = (int32_t)plan.combine.size() << 1;
        plan.combine.push_back({(int32_t)(bg / Hk), (int32_t)(bg % Hk), next_partial, v1 - v0 + 1});
        next_partial += v1 - v0 + 1;
      }
      off += nu;
    }
  }
  plan.n_partials = next_partial;
  // each virtual warp's first unit, the segment holding it and its offset there
  std::vector<PlanCache::WarpStartRec>& ws = cache.warp_start;
  ws.resize(TW + 1);
  {
    size_t si = 0;
    int64_t pos = 0;  // first unit of segment si
    const int64_t q = U / TW, r = U % TW;
    int64_t bound = 0, carry = 0;  // first unit of warp v: U v / TW, advanced without division
    for (int v = 0; v <= TW; ++v) {
      while (v < TW && si < segs.size() && pos + (segs[si].hi - segs[si].lo) <= bound) {
        pos += segs[si].hi - segs[si].lo;
        ++si;
      }
      ws[v] = {bound, (int32_t)si, (int32_t)(bound - pos)};
      bound += q;
      carry += r;
      if (carry >= TW) {
        carry -= TW;
        ++bound;
      }
    }
  }
  // per segment: its pieces' common fields, whether the next segment
  // continues the same (sequence, kv head), and its records
  std::vector<PlanCache::SegPiece>& tpl = cache.seg_piece;
  tpl.resize(segs.size());
  for (size_t k = 0; k < segs.size(); ++k) {
    const Seg& sg = segs[k];
    const BgRec& br = bgr[(size_t)sg.b * Hk + sg.g];
    Piece& pc = tpl[k].piece;
    pc.seq_slot = ids[sg.b];
    pc.q_row = sg.b;
    pc.kv_head = sg.g;
    pc.lblk_begin = pc.lblk_end = 0;
    pc.ctx_len = A.len[pc.seq_slot];
    pc.out_index = -1;
    pc.flags = br.flags;
    pc.q_row1 = -1;
    pc.out_index1 = -1;
    pc.item1 = 0;
    pc.stream_from = sg.stream_from;
    tpl[k].first_partial = br.first_partial;
    tpl[k].vfirst = br.vfirst;
    tpl[k].run_continues = k + 1 < segs.size() && segs[k + 1].b == sg.b && segs[k + 1].g == sg.g;
  }
  // physical placement: virtual warp v runs in CTA v % C as its warp v / C;
  // pieces are written in place (at most one per segment plus one per warp)
  const int WPC = warps_per_cta(p, 1);
  const int C = std::max(1, std::min(TW, TWmax / WPC));
  const int slots = TW > 0 ? C * WPC : 0;
  plan.pieces.resize(segs.size() + TW);
  Piece* out = plan.pieces.data();
  size_t np = 0;
  plan.warp_begin.assign(slots + 1, 0);
  int phys = 0;
  for (int cta = 0; cta < C; ++cta)
    for (int wl = 0; wl < WPC; ++wl, ++phys) {
      plan.warp_begin[phys] = (int32_t)np;
      const int v = wl * C + cta;
      if (v >= TW) continue;
      int64_t left = ws[v + 1].unit - ws[v].unit;
      int32_t si = ws[v].seg;
      int32_t lo = segs[si].lo + ws[v].seg_off;
      while (left > 0) {
        const PlanCache::SegPiece& t = tpl[si];
        const int32_t hi = (int32_t)std::min<int64_t>(segs[si].hi, lo + left);
        left -= hi - lo;
        // the run ends with the warp's units or where the next segment is another (sequence, kv head)
        const bool last = left == 0 || !t.run_continues;
        Piece& pc = out[np++];
        pc = t.piece;
        pc.lblk_begin = lo;
        pc.lblk_end = hi;
        if (t.first_partial >= 0) pc.out_index = t.first_partial + (v - t.vfirst);
        if (last) pc.flags |= kPieceLastOfRun;
        if (left > 0) lo = segs[++si].lo;
      }
    }
  plan.pieces.resize(np);
  plan.warp_begin[slots] = (int32_t)np;
  plan.total_warps = slots;
  plan.ctas = TW > 0 ? C : 0;
}

// The same one-pass construction for plans with sequence pairs (whole
// keep-sets, no group prefixes): every (sequence, kv head) has at most one
// pair segment, shared with its partner, and one segment of its own (the
// remainder past the shared blocks, or its whole context).  A segment spans
// the warps v0 .. v0 + runs - 1, one run in each.  A pair segment's runs
// write one record per sequence; a remainder's always do (it never holds
// all of its sequence's units); an unpaired segment's only when it spans
// several warps.  A sequence's records are its pair runs' and then its own
// segment's, in warp order -- the order of the general path.
void plan_stream_k_pairs(pkv_pool* p, int32_t n, const int32_t* ids, PlanCache& cache, int TWmax) {
  Plan& plan = cache.plan;
  const int Hk = p->cfg.n_kv_heads / p->HG;  // units of HG kv heads
  const auto& A = p->alloc;
  const std::vector<Seg>& segs = cache.segs;
  const std::vector<int64_t>& bg_units = cache.bg_units;
  const size_t nbg = (size_t)n * Hk, ns = segs.size();
  int64_t U = 0;
  for (const Seg& sg : segs) U += sg.hi - sg.lo;
  const int TW = (int)std::min<int64_t>(TWmax, (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp);
  WarpCursor wc(U, TW);
  // per segment: first warp, number of runs, and its records' first index
  // for the first and the second sequence
  using SegRec = PlanCache::SegRecord;
  std::vector<SegRec>& sr = cache.seg_rec;
  sr.resize(ns);
  std::vector<int32_t>& pair_runs = cache.cursor;  // per (sequence, kv head): runs of its pair segment
  std::vector<int32_t>& own_runs = cache.n_part;   // runs of its own segment that write records
  pair_runs.assign(nbg, 0);
  own_runs.assign(nbg, 0);
  {
    int64_t off = 0;
    for (size_t k = 0; k < ns; ++k) {
      const Seg& sg = segs[k];
      const int64_t len = sg.hi - sg.lo;
      const int32_t v0 = wc.at(off), runs = wc.at(off + len - 1) - v0 + 1;
      sr[k] = {v0, runs, -1, -1};
      const size_t bg = (size_t)sg.b * Hk + sg.g;
      if (sg.b1 >= 0) {
        pair_runs[bg] = runs;
        pair_runs[(size_t)sg.b1 * Hk + sg.g] = runs;
      } else if (runs > 1 || len != bg_units[bg]) {
        own_runs[bg] = runs;
      }
      off += len;
    }
  }
  std::vector<int32_t>& first_partial = cache.first_partial;
  std::vector<int32_t>& item_of = cache.item_of;
  first_partial.assign(nbg, -1);
  item_of.assign(nbg, -1);
  int next_partial = 0;
  for (size_t bg = 0; bg < nbg; ++bg) {
    const int32_t np = pair_runs[bg] + own_runs[bg];
    if (bg_units[bg] == 0) {
      plan.empty.push_back({(int32_t)(bg / Hk), (int32_t)(bg % Hk)});
    } else if (np > 0) {
      first_partial[bg] = next_partial;
      item_of[bg] = (int32_t)plan.combine.size();
      plan.combine.push_back({(int32_t)(bg / Hk), (int32_t)(bg % Hk), next_partial, np});
      next_partial += np;
    }
  }
  plan.n_partials = next_partial;
  for (size_t k = 0; k < ns; ++k) {
    const Seg& sg = segs[k];
    const size_t bg = (size_t)sg.b * Hk + sg.g;
    if (sg.b1 >= 0) {
      sr[k].rec0 = first_partial[bg];
      sr[k].rec1 = first_partial[(size_t)sg.b1 * Hk + sg.g];
    } else if (own_runs[bg] > 0) {
      sr[k].rec0 = first_partial[bg] + pair_runs[bg];
    }
  }
  // each virtual warp's first unit, the segment holding it and its offset there
  std::vector<PlanCache::WarpStartRec>& ws = cache.warp_start;
  ws.resize(TW + 1);
  {
    size_t si = 0;
    int64_t pos = 0;
    const int64_t q = U / TW, r = U % TW;
    int64_t bound = 0, carry = 0;
    for (int v = 0; v <= TW; ++v) {
      while (v < TW && si < ns && pos + (segs[si].hi - segs[si].lo) <= bound) {
        pos += segs[si].hi - segs[si].lo;
        ++si;
      }
      ws[v] = {bound, (int32_t)si, (int32_t)(bound - pos)};
      bound += q;
      carry += r;
      if (carry >= TW) {
        carry -= TW;
        ++bound;
      }
    }
  }
  // per segment: its pieces' common fields and whether the next segment
  // continues the same run key (sequence, kv head, second sequence)
  std::vector<PlanCache::SegPiece>& tpl = cache.seg_piece;
  tpl.resize(ns);
  for (size_t k = 0; k < ns; ++k) {
    const Seg& sg = segs[k];
    const SegRec& rc = sr[k];
    Piece& pc = tpl[k].piece;
    pc.seq_slot = ids[sg.b];
    pc.q_row = sg.b;
    pc.kv_head = sg.g;
    pc.lblk_begin = pc.lblk_end = 0;
    pc.ctx_len = A.len[pc.seq_slot];
    pc.out_index = -1;
    pc.flags = rc.rec0 >= 0 ? item_of[(size_t)sg.b * Hk + sg.g] << 1 : 0;
    pc.q_row1 = sg.b1;
    pc.out_index1 = -1;
    pc.item1 = sg.b1 >= 0 ? item_of[(size_t)sg.b1 * Hk + sg.g] : 0;
    pc.stream_from = sg.stream_from;
    tpl[k].first_partial = rc.rec0;
    tpl[k].vfirst = rc.v0;
    tpl[k].run_continues =
        k + 1 < ns && segs[k + 1].b == sg.b && segs[k + 1].g == sg.g && segs[k + 1].b1 == sg.b1;
  }
  const int WPC = warps_per_cta(p, 2);
  const int C = std::max(1, std::min(TW, TWmax / WPC));
  const int slots = TW > 0 ? C * WPC : 0;
  plan.pieces.resize(ns + TW);
  Piece* out = plan.pieces.data();
  size_t np = 0;
  plan.warp_begin.assign(slots + 1, 0);
  int phys = 0;
  for (int cta = 0; cta < C; ++cta)
    for (int wl = 0; wl < WPC; ++wl, ++phys) {
      plan.warp_begin[phys] = (int32_t)np;
      const int v = wl * C + cta;
      if (v >= TW) continue;
      int64_t left = ws[v + 1].unit - ws[v].unit;
      int32_t si = ws[v].seg;
      int32_t lo = segs[si].lo + ws[v].seg_off;
      while (left > 0) {
        const PlanCache::SegPiece& t = tpl[si];
        const int32_t hi = (int32_t)std::min<int64_t>(segs[si].hi, lo + left);
        const int32_t j = v - t.vfirst;  // this warp's run of the segment
        left -= hi - lo;
        const bool last = left == 0 || !t.run_continues;
        Piece& pc = out[np++];
        pc = t.piece;
        pc.lblk_begin = lo;
        pc.lblk_end = hi;
        if (t.first_partial >= 0) pc.out_index = t.first_partial + j;
        if (pc.q_row1 >= 0) pc.out_index1 = sr[si].rec1 + j;
        if (last) pc.flags |= kPieceLastOfRun;
        if (left > 0) lo = segs[++si].lo;
      }
    }
  plan.pieces.resize(np);
  plan.warp_begin[slots] = (int32_t)np;
  plan.total_warps = slots;
  plan.ctas = TW > 0 ? C : 0;
}

// The start of the longest tail [x, hi) of the logical blocks [lo, hi) of
// sequence slot s whose every block at most `limit` sequences hold (lo when
// no block of the pool is held twice).  The call reads those blocks once
// (limit 2: a pair's shared blocks, read once for both), so their copies may
// leave L2 first.  Without eviction, sharing is a prefix of the tables and
// this is every such block; an evicted sibling can leave its window blocks
// shared behind blocks that are not, which then keep the default policy.
int32_t stream_from(const pkv_pool* p, int32_t s, int32_t lo, int32_t hi, int32_t limit) {
  if (!PKV_KV_EVICT_FIRST) return INT32_MAX;
  const auto& A = p->alloc;
  if (A.n_multi == 0) return lo;
  const int32_t* t = A.table[s].data();
  int32_t x = hi;
  while (x > lo && (t[x - 1] < 0 || A.refcount[t[x - 1]] <= limit)) --x;
  return x;
}

Plan& build_plan(pkv_pool* p, int32_t n, const int32_t* ids, int mode, int S, int W, int num_splits) {
  const int Hk = p->cfg.n_kv_heads / p->HG;  // units of HG kv heads
  const auto& A = p->alloc;
  PlanCache& cache = plan_cache(p);
  Plan& plan = cache.plan;
  plan.empty.clear();
  plan.total_warps = plan.ctas = plan.n_partials = 0;
  std::vector<Seg>& segs = cache.segs;
  segs.clear();
  std::vector<int64_t>& bg_units = cache.bg_units;
  bg_units.assign((size_t)n * Hk, 0);
  // whole keep-sets (no mask), automatic partition: a prefix shared by a
  // group is read once per CTA of the multi-query kernel; blocks shared by a
  // pair past that are read once by the two-sequence kernel
  std::vector<Pairing> pairs;
  std::vector<PrefixGroup> groups;
  std::vector<int32_t> base(n, 0);
  plan.prefix_items.clear();
  plan.prefix_members.clear();
  if (p->cascade && mode == 0 && num_splits <= 0 && n >= 2) {
    if (p->cascade >= 2) groups = find_prefix_groups(p, n, ids);
    for (const auto& gr : groups)
      for (int32_t b : gr.members) base[b] = gr.shared;
    // Pairs only where no group prefix was taken out: past a group prefix the
    // blocks a pair shares come from DRAM, where the two-sequence kernel
    // (8 warps per SM) is slower than two one-sequence reads, the second of
    // which hits L2.
    if (groups.empty()) pairs = pair_shared_prefixes(p, n, ids, base);
    // pairing alone must save an eighth of the block reads to be worth the
    // two-sequence kernel's lower occupancy
    int64_t saved = 0, total = 0;
    for (int32_t b = 0; b < n; ++b) total += ceil_div(A.len[ids[b]], kBlock);
    for (const auto& pr : pairs) saved += pr.shared - base[pr.b0];
    if (saved * 8 < total) pairs.clear();
  }
  plan.nq = pairs.empty() ? 1 : 2;
  if (!pairs.empty() || !groups.empty()) {
    // each pair's shared segment is followed by the two remainders, so the
    // short remainder runs (and the merges they end with) spread over all
    // warps instead of piling up at the end of the unit list
    std::vector<uint8_t> paired(n, 0);
    auto nblk = [&](int32_t b) { return ceil_div(A.len[ids[b]], kBlock); };
    for (const auto& pr : pairs) {
      paired[pr.b0] = paired[pr.b1] = 1;
      // the pair's shared blocks stream where only the pair holds them
      const int32_t sf_pair = stream_from(p, ids[pr.b0], base[pr.b0], pr.shared, 2);
      const int32_t sf0 = stream_from(p, ids[pr.b0], pr.shared, nblk(pr.b0), 1);
      const int32_t sf1 = stream_from(p, ids[pr.b1], pr.shared, nblk(pr.b1), 1);
      for (int g = 0; g < Hk; ++g) {
        segs.push_back({pr.b0, g, base[pr.b0], pr.shared, pr.b1, sf_pair});
        if (pr.shared < nblk(pr.b0)) segs.push_back({pr.b0, g, pr.shared, nblk(pr.b0), -1, sf0});
        if (pr.shared < nblk(pr.b1)) segs.push_back({pr.b1, g, pr.shared, nblk(pr.b1), -1, sf1});
      }
    }
    for (int32_t b = 0; b < n; ++b) {
      const int32_t sf = paired[b] ? 0 : stream_from(p, ids[b], base[b], nblk(b), 1);
      for (int g = 0; g < Hk; ++g) {
        if (!paired[b] && nblk(b) > base[b]) segs.push_back({b, g, base[b], nblk(b), -1, sf});
        bg_units[(size_t)b * Hk + g] = nblk(b);
      }
    }
    // multi-query items: per group, kv head and tile of up to 128 query rows,
    // the prefix cut into `split` block ranges so the grid covers the GPU
    if (!groups.empty()) {
      const int G = p->G, per_tile = kPrefixRowsPerCta / G;
      int64_t tiles = 0;
      for (const auto& gr : groups) tiles += (int64_t)Hk * ceil_div((int32_t)gr.members.size(), per_tile);
      const int64_t want = 2LL * std::max(1, p->num_sms);
      for (const auto& gr : groups) {
        const int32_t split = (int32_t)std::max<int64_t>(
            1, std::min<int64_t>({(want + tiles - 1) / tiles, (int64_t)kMaxPrefixSplit,
                                  (int64_t)(gr.shared / kMinGroupBlocks)}));
        const int32_t M = (int32_t)gr.members.size();
        for (int g = 0; g < Hk; ++g)
          for (int32_t t0 = 0; t0 < M; t0 += per_tile)
            for (int32_t k = 0; k < split; ++k) {
              PrefixItem it{};
              it.kv_head = g;
              it.table_seq = ids[gr.members[0]];
              it.lblk_begin = (int32_t)((int64_t)gr.shared * k / split);
              it.lblk_end = (int32_t)((int64_t)gr.shared * (k + 1) / split);
              it.member_begin = (int32_t)plan.prefix_members.size();
              it.n_members = std::min(per_tile, M - t0);
              for (int32_t m = 0; m < it.n_members; ++m)
                plan.prefix_members.push_back({gr.members[t0 + m], -1, g, 0});  // item field: kv head for now
              plan.prefix_items.push_back(it);
            }
      }
    }
  } else {
    for (int32_t b = 0; b < n; ++b) {
      BlockRange r[2];
      const int nr = keep_ranges(A.len[ids[b]], mode, S, W, r);
      int32_t sf[2];
      for (int k = 0; k < nr; ++k) sf[k] = stream_from(p, ids[b], r[k].lo, r[k].hi, 1);
      for (int g = 0; g < Hk; ++g)
        for (int k = 0; k < nr; ++k) {
          segs.push_back({b, g, r[k].lo, r[k].hi, -1, sf[k]});
          bg_units[(size_t)b * Hk + g] += r[k].hi - r[k].lo;
        }
    }
  }
  // (the one-pass paths size the piece array themselves: clearing it first
  // would make them zero-fill all of it again)
  plan.combine.clear();
  plan.warp_begin.clear();
  const int TWmax = max_total_warps(p, plan.nq);
  if (!p->general_plan && num_splits <= 0 && plan.nq == 2 && plan.prefix_items.empty() && !segs.empty()) {
    plan_stream_k_pairs(p, n, ids, cache, TWmax);
    return plan;
  }
  if (!p->general_plan && num_splits <= 0 && plan.nq == 1 && plan.prefix_items.empty()) {
    if (!segs.empty()) {
      plan_stream_k_single(p, n, ids, cache, TWmax);
    } else {  // nothing to read: every (sequence, kv head) has an empty keep-set
      plan.pieces.clear();
      for (int32_t b = 0; b < n; ++b)
        for (int g = 0; g < Hk; ++g) plan.empty.push_back({b, g});
      plan.warp_begin.assign(1, 0);
    }
    return plan;
  }
  plan.pieces.clear();
  auto piece_of = [&](const Seg& s, int32_t lo, int32_t hi) {
    Piece pc;
    pc.seq_slot = ids[s.b];
    pc.q_row = s.b;
    pc.kv_head = s.g;
    pc.lblk_begin = lo;
    pc.lblk_end = hi;
    pc.ctx_len = A.len[ids[s.b]];
    pc.out_index = -1;
    pc.flags = 0;
    pc.q_row1 = s.b1;
    pc.out_index1 = -1;
    pc.item1 = 0;
    pc.stream_from = s.stream_from;
    return pc;
  };
  std::vector<int32_t>& piece_warp = cache.piece_warp;  // warp of each piece
  piece_warp.clear();
  if (num_splits <= 0) {
    int64_t U = 0;
    for (auto& s : segs) U += s.hi - s.lo;
    int TW = (int)std::min<int64_t>(TWmax, (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp);
    plan.total_warps = TW;
    if (TW > 0) {
      plan.pieces.reserve(segs.size() + TW);
      piece_warp.reserve(segs.size() + TW);
      // warp w takes units [floor(U w / TW), floor(U (w + 1) / TW)); the
      // bounds advance by U / TW plus a carry of the remainder, no division
      const int64_t q = U / TW, r = U % TW;
      int64_t next = q + (r >= TW ? 1 : 0), carry = r;  // bound of warp 1
      if (carry >= TW) carry -= TW;
      auto step_bound = [&]() {
        carry += r;
        next += q;
        if (carry >= TW) {
          carry -= TW;
          ++next;
        }
      };
      int w = 0;
      int64_t pos = 0;
      for (auto& s : segs) {
        int64_t start = pos, end = pos + (s.hi - s.lo);
        while (start < end) {
          while (next <= start) {
            ++w;
            step_bound();
          }
          const int64_t stop = std::min(end, next);
          plan.pieces.push_back(piece_of(s, s.lo + (int32_t)(start - pos), s.lo + (int32_t)(stop - pos)));
          piece_warp.push_back(w);
          start = stop;
        }
        pos = end;
      }
    }
  } else {
    // exactly num_splits equal parts of each (sequence, kv head) unit list
    struct Part {
      size_t first_piece, n_pieces;
    };
    std::vector<Piece> parts_pieces;
    std::vector<Part> parts;
    size_t si = 0;
    for (int32_t b = 0; b < n; ++b)
      for (int g = 0; g < Hk; ++g) {
        size_t s0 = si;
        while (si < segs.size() && segs[si].b == b && segs[si].g == g) ++si;
        const int64_t nu = bg_units[(size_t)b * Hk + g];
        for (int k = 0; k < num_splits; ++k) {
          int64_t u0 = nu * k / num_splits, u1 = nu * (k + 1) / num_splits;
          if (u1 <= u0) continue;
          Part pt{parts_pieces.size(), 0};
          int64_t off = 0;
          for (size_t j = s0; j < si; ++j) {
            const Seg& s = segs[j];
            int64_t a = std::max(u0, off), e = std::min(u1, off + (s.hi - s.lo));
            if (a < e) {
              parts_pieces.push_back(piece_of(s, s.lo + (int32_t)(a - off), s.lo + (int32_t)(e - off)));
              ++pt.n_pieces;
            }
            off += s.hi - s.lo;
          }
          parts_pieces[parts_pieces.size() - 1].flags |= kPieceLastOfRun;
          parts.push_back(pt);
        }
      }
    // every warp gets the same number of parts (rounds), or one fewer
    const int64_t P = (int64_t)parts.size();
    const int64_t rounds = P > 0 ? (P + TWmax - 1) / TWmax : 0;
    const int TW = rounds > 0 ? (int)((P + rounds - 1) / rounds) : 0;
    plan.total_warps = TW;
    for (int w = 0; w < TW; ++w) {
      const int64_t a = P * w / TW, e = P * (w + 1) / TW;
      for (int64_t k = a; k < e; ++k)
        for (size_t j = 0; j < parts[k].n_pieces; ++j) {
          plan.pieces.push_back(parts_pieces[parts[k].first_piece + j]);
          piece_warp.push_back(w);
        }
    }
  }
  // runs: consecutive pieces of one (b, g) -- or one sequence pair and g --
  // inside one warp; explicit split parts already carry their own run ends
  const size_t np = plan.pieces.size();
  for (size_t k = 0; k < np; ++k) {
    const bool end_of_warp = k + 1 == np || piece_warp[k + 1] != piece_warp[k];
    const bool next_other = k + 1 == np || plan.pieces[k + 1].q_row != plan.pieces[k].q_row ||
                            plan.pieces[k + 1].kv_head != plan.pieces[k].kv_head ||
                            plan.pieces[k + 1].q_row1 != plan.pieces[k].q_row1;
    if (end_of_warp || next_other) plan.pieces[k].flags |= kPieceLastOfRun;
  }
  // partial records: a single-sequence run that covers all units of its
  // (b, g) writes the final output; every other run writes one record per
  // sequence.  Records of one (b, g) are consecutive: counted first, then
  // numbered.
  std::vector<int32_t>& first_partial = cache.first_partial;
  std::vector<int32_t>& n_part = cache.n_part;
  first_partial.assign((size_t)n * Hk, -1);
  n_part.assign((size_t)n * Hk, 0);
  std::vector<PlanRun>& runs = cache.runs;
  runs.clear();
  {
    size_t start = 0;
    int64_t units = 0;
    for (size_t k = 0; k < np; ++k) {
      const Piece& pc = plan.pieces[k];
      units += pc.lblk_end - pc.lblk_begin;
      if (!(pc.flags & kPieceLastOfRun)) continue;
      const bool rec0 = pc.q_row1 >= 0 || units != bg_units[(size_t)pc.q_row * Hk + pc.kv_head];
      runs.push_back({start, k + 1, rec0});
      if (rec0) ++n_part[(size_t)pc.q_row * Hk + pc.kv_head];
      if (pc.q_row1 >= 0) ++n_part[(size_t)pc.q_row1 * Hk + pc.kv_head];
      start = k + 1;
      units = 0;
    }
  }
  for (const PrefixMember& pm : plan.prefix_members) ++n_part[(size_t)pm.q_row * Hk + pm.item];
  int next_partial = 0;
  for (size_t bg = 0; bg < (size_t)n * Hk; ++bg)
    if (n_part[bg] > 0) {
      first_partial[bg] = next_partial;
      next_partial += n_part[bg];
    }
  plan.n_partials = next_partial;
  std::vector<int32_t>& item_of = cache.item_of;
  item_of.assign((size_t)n * Hk, -1);
  for (int32_t b = 0; b < n; ++b)
    for (int g = 0; g < Hk; ++g) {
      const size_t bg = (size_t)b * Hk + g;
      if (bg_units[bg] == 0) {
        plan.empty.push_back({b, g});
      } else if (n_part[bg] > 0) {
        item_of[bg] = (int32_t)plan.combine.size();
        plan.combine.push_back({b, g, first_partial[bg], n_part[bg]});
      }
    }
  std::vector<int32_t>& cursor = cache.cursor;
  cursor = first_partial;
  for (PrefixMember& pm : plan.prefix_members) {
    const size_t bg = (size_t)pm.q_row * Hk + pm.item;
    pm.out_index = cursor[bg]++;
    pm.item = item_of[bg];
  }
  for (const PlanRun& ru : runs) {
    const Piece& pc = plan.pieces[ru.end - 1];
    const size_t bg0 = (size_t)pc.q_row * Hk + pc.kv_head;
    const int32_t idx0 = ru.record0 ? cursor[bg0]++ : -1;
    int32_t idx1 = -1, item1 = 0;
    if (pc.q_row1 >= 0) {
      const size_t bg1 = (size_t)pc.q_row1 * Hk + pc.kv_head;
      idx1 = cursor[bg1]++;
      item1 = item_of[bg1];
    }
    for (size_t j = ru.begin; j < ru.end; ++j) {
      Piece& q = plan.pieces[j];
      q.out_index = idx0;
      if (idx0 >= 0) q.flags |= item_of[bg0] << 1;
      q.out_index1 = idx1;
      q.item1 = item1;
    }
  }

  // Physical placement: virtual warp v runs in CTA v % C as its warp v / C,
  // so that the work is spread over as many SMs as possible.
  const int TW = plan.total_warps;
  const int WPC = warps_per_cta(p, plan.nq);
  const int C = std::max(1, std::min(TW, max_total_warps(p, plan.nq) / WPC));
  std::vector<size_t>& vstart = cache.vstart;
  vstart.assign(TW + 1, 0);
  {
    size_t k = 0;
    for (int v = 0; v < TW; ++v) {
      vstart[v] = k;
      while (k < np && piece_warp[k] == v) ++k;
    }
    vstart[TW] = k;
  }
  std::vector<Piece>& ordered = cache.ordered;
  ordered.resize(np);
  const int slots = TW > 0 ? C * WPC : 0;
  plan.warp_begin.assign(slots + 1, 0);
  size_t filled = 0;
  for (int phys = 0; phys < slots; ++phys) {
    plan.warp_begin[phys] = (int32_t)filled;
    const int v = (phys % WPC) * C + phys / WPC;
    if (v < TW) {
      std::copy(plan.pieces.begin() + vstart[v], plan.pieces.begin() + vstart[v + 1], ordered.begin() + filled);
      filled += vstart[v + 1] - vstart[v];
    }
  }
  plan.warp_begin[slots] = (int32_t)filled;
  plan.pieces.swap(ordered);
  plan.total_warps = slots;
  plan.ctas = TW > 0 ? C : 0;
  return plan;
}

pkv_status check_keep_blocks_present(const pkv_pool* p, int32_t n, const int32_t* ids, int mode, int S, int W) {
  const auto& A = p->alloc;
  for (int32_t b = 0; b < n; ++b) {
    const int32_t s = ids[b];
    if (!A.holes[s]) continue;
    BlockRange r[2];
    const int nr = keep_ranges(A.len[s], mode, S, W, r);
    for (int k = 0; k < nr; ++k)
      for (int32_t lb = r[k].lo; lb < r[k].hi; ++lb)
        if (A.table[s][lb] < 0)
          return fail(PKV_ERR_INVALID_ARG, "sequence %d: block %d of the keep-set was evicted", s, lb);
  }
  return PKV_OK;
}

// Byte layout of an uploaded decode plan: [warp_begin][pieces][merge items]
// [merge counters, zero][empty items], each part 32-byte aligned.
struct PlanLayout {
  size_t wb = 0, pieces = 0, combine = 0, counters = 0, empty = 0, pitems = 0, pmembers = 0, bytes = 0;
};

PlanLayout plan_layout(Plan& pl, int wpc, size_t base) {
  if (pl.total_warps == 0 && !pl.empty.empty()) {  // only empty keep-sets: one CTA writes them
    pl.ctas = 1;
    pl.total_warps = wpc;
    pl.warp_begin.assign(wpc + 1, 0);
  }
  auto up = [](size_t x) { return (x + 31) & ~size_t(31); };
  PlanLayout L;
  L.wb = up(base);
  L.pieces = up(L.wb + pl.warp_begin.size() * sizeof(int32_t));
  L.combine = up(L.pieces + pl.pieces.size() * sizeof(Piece));
  L.counters = up(L.combine + pl.combine.size() * sizeof(CombineItem));
  L.empty = up(L.counters + pl.combine.size() * sizeof(int32_t));
  L.pitems = up(L.empty + pl.empty.size() * sizeof(EmptyItem));
  L.pmembers = up(L.pitems + pl.prefix_items.size() * sizeof(PrefixItem));
  L.bytes = L.pmembers + pl.prefix_members.size() * sizeof(PrefixMember);
  return L;
}

void plan_write(const Plan& pl, const PlanLayout& L, char* host) {
  if (!pl.warp_begin.empty()) memcpy(host + L.wb, pl.warp_begin.data(), pl.warp_begin.size() * sizeof(int32_t));
  if (!pl.pieces.empty()) memcpy(host + L.pieces, pl.pieces.data(), pl.pieces.size() * sizeof(Piece));
  if (!pl.combine.empty()) {
    memcpy(host + L.combine, pl.combine.data(), pl.combine.size() * sizeof(CombineItem));
    memset(host + L.counters, 0, pl.combine.size() * sizeof(int32_t));
  }
  if (!pl.empty.empty()) memcpy(host + L.empty, pl.empty.data(), pl.empty.size() * sizeof(EmptyItem));
  if (!pl.prefix_items.empty()) {
    memcpy(host + L.pitems, pl.prefix_items.data(), pl.prefix_items.size() * sizeof(PrefixItem));
    memcpy(host + L.pmembers, pl.prefix_members.data(), pl.prefix_members.size() * sizeof(PrefixMember));
  }
}

// Launches the tensor-core decode (with its fused merge) over an uploaded plan.
pkv_status launch_tc_plan(pkv_pool* p, cudaStream_t st, const Plan& pl, const PlanLayout& L, const char* dev,
                          const void* q, float scale, int mode, int S, int W, void* out, float* lse, float* logits,
                          int64_t logits_stride, void* partials) {
  if (pl.total_warps == 0 && pl.prefix_items.empty()) return PKV_OK;
  const auto& c = p->cfg;
  DecodeTCParams prm;
  prm.tmap_k = p->tmap_k;
  prm.tmap_v = p->tmap_v;
  prm.k_scale = p->buf.k_scale;
  prm.v_scale = p->buf.v_scale;
  prm.tables = p->buf.block_tables;
  prm.max_blocks = c.max_blocks_per_seq;
  prm.num_blocks = c.num_blocks;
  prm.n_heads = c.n_heads;
  prm.n_kv_heads = c.n_kv_heads;
  prm.q = q;
  prm.out = out;
  prm.lse = lse;
  prm.logits = logits;
  prm.logits_stride = logits_stride;
  prm.pieces = (const Piece*)(dev + L.pieces);
  prm.warp_begin = (const int32_t*)(dev + L.wb);
  prm.total_warps = pl.total_warps;
  prm.partials = (float*)partials;
  prm.combine = (const CombineItem*)(dev + L.combine);
  prm.counters = (int32_t*)(dev + L.counters);
  prm.empty = (const EmptyItem*)(dev + L.empty);
  prm.n_empty = (int32_t)pl.empty.size();
  prm.scale = scale;
  prm.mask_mode = mode;
  prm.num_sinks = S;
  prm.window = W;
  prm.status = p->buf.status;
  prm.wait_limit_ns = p->wait_limit_ns;
  prm.starve_warp = p->starve_warp;
  p->starve_warp = -1;
  prm.prefix_items = (const PrefixItem*)(dev + L.pitems);
  prm.prefix_members = (const PrefixMember*)(dev + L.pmembers);
  prm.n_prefix_items = (int32_t)pl.prefix_items.size();
  prm.k_channel = p->k_channel;
  prm.v_channel = p->v_channel;
  // one-sequence rings: evict-first when no block of the pool is held twice
  // (deciding per unit, as the pair rings do, costs those rings about a
  // quarter more instructions)
  prm.kv_evict_first = PKV_KV_EVICT_FIRST && pl.nq == 1 && p->alloc.n_multi == 0 ? 1 : 0;
  if (prm.n_prefix_items > 0)
    if (pkv_status r = launch(p, PKV_KERNEL_PREFIX, st, [&] { return launch_prefix_decode(p->G, prm, st); })) return r;
  if (pl.total_warps == 0) return PKV_OK;
  return launch(p, PKV_KERNEL_DECODE, st,
                [&] { return launch_decode_tc(c.kv_dtype, p->G, p->HG, pl.nq, c.head_dim, prm, pl.ctas, st); });
}

}  // namespace

// ---------------------------------------------------------------------------
// decode into caller-supplied device regions (used by the static-scratch
// entry point); shares the planner and the launchers, allocates nothing
// ---------------------------------------------------------------------------

int pkv::decode_attn_into(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const void* q, float scale,
                          int32_t mode, int32_t S, int32_t W, int32_t num_splits, void* out, float* lse,
                          float* logits, int64_t logits_stride, void* plan_dev, size_t plan_cap, void* partials_dev,
                          size_t partials_cap) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
    if (p->cfg.kv_dtype == PKV_KV_FP32)
      return fail(PKV_ERR_UNSUPPORTED, "static-scratch decode serves bf16 / fp8 / int8 pools");
    {
      int cur = -1;
      if (cudaGetDevice(&cur) != cudaSuccess || cur != p->device_id)
        return fail(PKV_ERR_INVALID_ARG, "the pool's device (%d) is not the current device (%d)", p->device_id, cur);
    }
    if (pkv_status r = check_seq_list(p, n, ids)) return r;
    if (!valid_mask(mode, S, W)) return fail(PKV_ERR_INVALID_ARG, "invalid mask %d (%d, %d)", mode, S, W);
    if (num_splits < 0) return fail(PKV_ERR_INVALID_ARG, "num_splits < 0");
    if (n > 0 && (!q || !out)) return fail(PKV_ERR_INVALID_ARG, "q / out is NULL");
    HostAllocator& A = p->alloc;
    int32_t maxlen = 0;
    for (int32_t i = 0; i < n; ++i) maxlen = std::max(maxlen, A.len[ids[i]]);
    if (logits && logits_stride < maxlen) return fail(PKV_ERR_INVALID_ARG, "logits_stride < max length");
    if (pkv_status r = check_keep_blocks_present(p, n, ids, mode, S, W)) return r;
    const auto& c = p->cfg;
    cudaStream_t st = (cudaStream_t)stream;

    // queued allocator effects: last value per table entry; copies in waves
    const std::vector<TablePatch> patches = dedup_patches(A, A.pending_patch);
    const size_t ncow = A.pending_cow.size() / 2;
    const std::vector<size_t> waves = cow_waves(A);
    Plan empty_plan;
    Plan& plan = n > 0 ? build_plan(p, n, ids, mode, S, W, num_splits) : empty_plan;
    const size_t pf = (size_t)partial_floats(p->G * p->HG, c.head_dim) * sizeof(float);
    if ((size_t)plan.n_partials * pf > partials_cap)
      return fail(PKV_ERR_WORKSPACE, "needs %zu bytes of partial records, the static scratch holds %zu",
                  (size_t)plan.n_partials * pf, partials_cap);

    // one blob: [cow pairs][patches][plan]
    auto up32 = [](size_t x) { return (x + 31) & ~size_t(31); };
    const size_t cow_off = 0, patch_off = up32(ncow * 2 * sizeof(int32_t));
    const PlanLayout L =
        plan_layout(plan, warps_per_cta(p, plan.nq), patch_off + patches.size() * sizeof(TablePatch));
    const size_t bytes = L.bytes;
    if (bytes > plan_cap)
      return fail(PKV_ERR_WORKSPACE, "needs %zu bytes of plan, the static scratch holds %zu", bytes, plan_cap);
    std::vector<char>& blob = plan_cache(p).blob;
    if (blob.size() < bytes) blob.resize(bytes);
    if (ncow) memcpy(blob.data() + cow_off, A.pending_cow.data(), ncow * 2 * sizeof(int32_t));
    if (!patches.empty()) memcpy(blob.data() + patch_off, patches.data(), patches.size() * sizeof(TablePatch));
    plan_write(plan, L, blob.data());
    char* dev = (char*)plan_dev;
    if (bytes) PKV_CUDA(cudaMemcpyAsync(dev, blob.data(), bytes, cudaMemcpyHostToDevice, st));

    if (ncow) {
      const size_t blk_bytes = (size_t)c.n_kv_heads * kBlock * c.head_dim * elem_bytes(c.kv_dtype);
      const size_t scl = has_scales(c.kv_dtype) ? (size_t)c.n_kv_heads * kBlock : 0;
      for (size_t w = 0; w + 1 < waves.size(); ++w) {
        const size_t k0 = waves[w], k1 = waves[w + 1];
        if (k1 == k0) continue;
        if (pkv_status r = launch(p, PKV_KERNEL_COW_COPY, st, [&] {
              return launch_cow_copy((const int32_t*)(dev + cow_off) + 2 * k0, (int)(k1 - k0), p->buf.k_pool,
                                     p->buf.v_pool, p->buf.k_scale, p->buf.v_scale, blk_bytes, scl, st);
            }))
          return r;
      }
    }
    if (!patches.empty()) {
      if (pkv_status r = launch(p, PKV_KERNEL_TABLE_PATCH, st, [&] {
            return launch_table_patch((const int32_t*)(dev + patch_off), (int)patches.size(), p->buf.block_tables, st);
          }))
        return r;
    }
    A.pending_cow.clear();
    A.pending_patch.clear();
    if (n == 0) return PKV_OK;
    return launch_tc_plan(p, st, plan, L, dev, q, scale, mode, S, W, out, lse, logits, logits_stride, partials_dev);
  });
}

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// CPU swap space
// ---------------------------------------------------------------------------

namespace {

pkv_status map_host(void* h, void** dev, const char* what) {
  *dev = nullptr;
  if (!h) return PKV_OK;
  if ((uintptr_t)h & 15) return fail(PKV_ERR_INVALID_ARG, "%s must be 16-byte aligned", what);
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, h) != cudaSuccess || at.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(PKV_ERR_UNSUPPORTED, "%s is not page-locked host memory", what);
  }
  if (cudaHostGetDevicePointer(dev, h, 0) != cudaSuccess || !*dev) {
    cudaGetLastError();
    return fail(PKV_ERR_UNSUPPORTED, "%s has no device-mapped address", what);
  }
  return PKV_OK;
}

// Swap-out (out) or swap-in of the listed sequences: allocator moves, then the
// block copies on `stream`.
pkv_status swap_move(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, bool out) {
  if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (!p->swap_space) return fail(PKV_ERR_INVALID_ARG, "the pool has no swap space");
  if (n < 0 || (n > 0 && !ids)) return fail(PKV_ERR_INVALID_ARG, "bad sequence list");
  auto& A = p->alloc;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = ids[i];
    if (!A.valid_seq(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live", s);
    if (A.swapped[s] != (out ? 0 : 1))
      return fail(PKV_ERR_INVALID_ARG, "sequence %d is already %s", s, out ? "swapped out" : "on the device");
  }
  if (const int32_t d = A.first_repeat(n, ids); d >= 0)
    return fail(PKV_ERR_INVALID_ARG, "sequence %d listed twice", d);
  // each distinct source block moves once: its destination, once taken,
  // serves every listed sequence that holds it
  A.begin_moves(out ? (size_t)A.NB : (size_t)A.NH);
  size_t need = 0;
  for (int32_t i = 0; i < n; ++i)
    for (int32_t b : out ? A.table[ids[i]] : A.host_table[ids[i]])
      if (b >= 0 && A.move_mark[b] != A.move_epoch) {
        A.move_mark[b] = A.move_epoch;
        A.move_dst[b] = -1;
        ++need;
      }
  const size_t avail = out ? A.host_free.size() : A.free_blocks.size();
  if (need > avail)
    return fail(PKV_ERR_OUT_OF_BLOCKS, "swap-%s needs %zu blocks, %zu free", out ? "out" : "in", need, avail);
  cudaStream_t st = (cudaStream_t)stream;
  // queued copies first: a pending copy-on-write must land before its blocks move
  if (p->device)
    if (pkv_status r = flush_pending(p, st)) return r;
  std::vector<int32_t> pairs;
  pairs.reserve(2 * need);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = ids[i], nb = ceil_div(A.len[s], kBlock);
    std::vector<int32_t> row(nb, -1);
    const std::vector<int32_t>& from = out ? A.table[s] : A.host_table[s];
    for (int32_t lb = 0; lb < nb && lb < (int32_t)from.size(); ++lb) {
      const int32_t b = from[lb];
      if (b < 0) continue;
      int32_t& m = A.move_dst[b];
      if (m < 0) {
        m = out ? A.take_host() : A.take();
        pairs.push_back(b);
        pairs.push_back(m);
      } else if (out) {
        ++A.host_refcount[m];
      } else {
        A.add_ref(m);
      }
      row[lb] = m;
    }
    if (out) {
      A.host_table[s] = row;
    } else {  // the device row is all -1 since the swap-out: patch the blocks only
      A.table[s] = row;
      if (A.queue)
        for (int32_t lb = 0; lb < nb; ++lb)
          if (row[lb] >= 0) A.pending_patch.push_back({s * A.max_blocks + lb, row[lb]});
    }
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = ids[i], nb = ceil_div(A.len[s], kBlock);
    if (out) {
      A.drop_from(s, 0);  // releases the device blocks, ascending; rows become -1
      A.table[s].assign(nb, -1);
      A.swapped[s] = 1;
    } else {
      for (int32_t hb : A.host_table[s])
        if (hb >= 0) A.release_host(hb);
      A.host_table[s].clear();
      A.swapped[s] = 0;
    }
  }
  if (!p->device) return PKV_OK;
  const int npairs = (int)(pairs.size() / 2);
  if (npairs == 0) return PKV_OK;
  const auto& c = p->cfg;
  const size_t blk_bytes = (size_t)c.n_kv_heads * kBlock * c.head_dim * elem_bytes(c.kv_dtype);
  const size_t scl = has_scales(c.kv_dtype) ? (size_t)c.n_kv_heads * kBlock : 0;
  StagingSlot* sl;
  if (pkv_status r = p->staging.acquire(pairs.size() * sizeof(int32_t), &sl)) return r;
  memcpy(sl->host, pairs.data(), pairs.size() * sizeof(int32_t));
  if (pkv_status r = Staging::upload(sl, pairs.size() * sizeof(int32_t), st)) return r;
  if (pkv_status r = launch(p, PKV_KERNEL_SWAP_COPY, st, [&] {
        if (out)
          return launch_block_copy((const int32_t*)sl->dev, npairs, p->buf.k_pool, p->buf.v_pool, p->buf.k_scale,
                                   p->buf.v_scale, p->host_k_dev, p->host_v_dev, p->host_ks_dev, p->host_vs_dev,
                                   blk_bytes, scl, st);
        return launch_block_copy((const int32_t*)sl->dev, npairs, p->host_k_dev, p->host_v_dev, p->host_ks_dev,
                                 p->host_vs_dev, p->buf.k_pool, p->buf.v_pool, p->buf.k_scale, p->buf.v_scale,
                                 blk_bytes, scl, st);
      }))
    return r;
  return Staging::release(sl, st);
}

}  // namespace

extern "C" {

const char* pkv_last_error(void) { return g_last_error.c_str(); }
const char* pkv_version(void) { return "pkv 0.1 (sm_103a)"; }

pkv_status pkv_pool_required_bytes(const pkv_pool_config* cfg, pkv_buffer_sizes* out) {
  return guarded([&]() -> pkv_status {
    if (pkv_status r = check_config(cfg)) return r;
    if (!out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
    const size_t rows = (size_t)cfg->num_blocks * cfg->n_kv_heads * kBlock;
    out->k_pool = out->v_pool = rows * cfg->head_dim * elem_bytes(cfg->kv_dtype);
    out->k_scale = out->v_scale = has_scales(cfg->kv_dtype) ? rows * sizeof(float) : 0;
    out->block_tables = (size_t)cfg->max_seqs * cfg->max_blocks_per_seq * sizeof(int32_t);
    out->status = 4 * sizeof(int32_t);
    return PKV_OK;
  });
}

pkv_status pkv_pool_create(const pkv_pool_config* cfg, const pkv_pool_buffers* buffers, pkv_pool** out) {
  return guarded([&]() -> pkv_status {
    if (!out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (pkv_status r = check_config(cfg)) return r;
    pkv_pool* p = new pkv_pool();
    p->cfg = *cfg;
    p->cfg.free_order = nullptr;
    p->G = cfg->n_heads / cfg->n_kv_heads;
    p->HG = unit_heads(*cfg, p->G);
    p->alloc.init(cfg->num_blocks, cfg->max_seqs, cfg->max_blocks_per_seq, cfg->alloc_seed, cfg->free_order);
    if (buffers) {
      const auto& b = *buffers;
      const bool fp8 = has_scales(cfg->kv_dtype);
      if (!b.k_pool || !b.v_pool || !b.block_tables || !b.status || (fp8 && (!b.k_scale || !b.v_scale))) {
        delete p;
        return fail(PKV_ERR_INVALID_ARG, "a required device buffer is NULL");
      }
      if (((uintptr_t)b.k_pool | (uintptr_t)b.v_pool) & 127) {
        delete p;
        return fail(PKV_ERR_INVALID_ARG, "k_pool / v_pool must be 128-byte aligned");
      }
      if (fp8 && (((uintptr_t)b.k_scale | (uintptr_t)b.v_scale) & 15)) {
        delete p;
        return fail(PKV_ERR_INVALID_ARG, "k_scale / v_scale must be 16-byte aligned");
      }
      p->device = true;
      p->alloc.queue = true;
      p->buf = b;
      auto fail_dev = [&](pkv_status r) {
        p->staging.destroy();
        delete p;
        return r;
      };
      cudaError_t e = cudaGetDevice(&p->device_id);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device_id);
      if (e != cudaSuccess) return fail_dev(fail(PKV_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e)));
      const size_t tbytes = (size_t)cfg->max_seqs * cfg->max_blocks_per_seq * sizeof(int32_t);
      e = cudaMemset(b.block_tables, 0xFF, tbytes);
      if (e == cudaSuccess) e = cudaMemset(b.status, 0, 4 * sizeof(int32_t));
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return fail_dev(fail(PKV_ERR_CUDA, "buffer init failed: %s", cudaGetErrorString(e)));
      if (cfg->kv_dtype != PKV_KV_FP32) {
        p->tc_path = true;
        const int D = cfg->head_dim, hg = p->HG;
        if (pkv_status r = make_tensor_map(&p->tmap_k, b.k_pool, p->cfg, hg)) return fail_dev(r);
        if (pkv_status r = make_tensor_map(&p->tmap_v, b.v_pool, p->cfg, hg)) return fail_dev(r);
        e = decode_tc_prepare(cfg->kv_dtype, p->G, hg, 1, D);
        if (e == cudaSuccess) e = decode_tc_prepare(cfg->kv_dtype, p->G, hg, 2, D);
        if (e == cudaSuccess && cfg->kv_dtype == PKV_KV_BF16 && D == 128) e = prefix_decode_prepare(p->G);
        int occ = 0, occ2 = 0;
        if (e == cudaSuccess) e = decode_tc_occupancy(cfg->kv_dtype, p->G, hg, 1, D, &occ);
        if (e == cudaSuccess) e = decode_tc_occupancy(cfg->kv_dtype, p->G, hg, 2, D, &occ2);
        if (e != cudaSuccess) return fail_dev(fail(PKV_ERR_CUDA, "decode kernel setup failed: %s", cudaGetErrorString(e)));
        // the plan's warps are the kernel's teams (hg warps each)
        p->tc_ctas_per_sm = std::max(1, occ);
        p->tc_warps_per_cta = tc_teams(cfg->kv_dtype, 1, D, hg);
        p->tc2_ctas_per_sm = std::max(1, occ2);
        p->tc2_warps_per_cta = tc_teams(cfg->kv_dtype, 2, D, hg);
        p->tc_smem = tc_smem_bytes(cfg->kv_dtype, 1, D, hg);
      }
    }
    *out = p;
    return PKV_OK;
  });
}

void pkv_pool_destroy(pkv_pool* p) {
  if (!p) return;
  if (p->device) {
    p->staging.destroy();
    p->timing.destroy();
  }
  delete p;
}

pkv_status pkv_seq_add(pkv_pool* p, int32_t* seq_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !seq_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    auto& A = p->alloc;
    if (A.free_ids.empty()) return fail(PKV_ERR_OUT_OF_SEQS, "all %d sequence ids are in use", A.max_seqs);
    int32_t s = *A.free_ids.begin();
    A.free_ids.erase(A.free_ids.begin());
    A.live[s] = 1;
    A.holes[s] = 0;
    A.len[s] = 0;
    A.table[s].clear();
    *seq_out = s;
    return PKV_OK;
  });
}

pkv_status pkv_seq_fork(pkv_pool* p, int32_t src, int32_t* dst_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !dst_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    auto& A = p->alloc;
    if (!A.on_device(src)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live or is swapped out", src);
    int32_t d;
    if (pkv_status r = pkv_seq_add(p, &d)) return r;
    // The new id's device row is all -1 (every release of an entry queued a
    // -1 for it), so only the blocks it shares need table patches.
    const int32_t nblk = ceil_div(A.len[src], kBlock);
    const int32_t* from = A.table[src].data();
    A.table[d].assign(from, from + nblk);
    for (int32_t lb = 0; lb < nblk; ++lb) {
      const int32_t b = from[lb];
      if (b < 0) continue;
      A.add_ref(b);
      if (A.queue) A.pending_patch.push_back({d * A.max_blocks + lb, b});
    }
    A.len[d] = A.len[src];
    A.holes[d] = A.holes[src];
    *dst_out = d;
    return PKV_OK;
  });
}

pkv_status pkv_seq_truncate(pkv_pool* p, int32_t s, int32_t new_len) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    auto& A = p->alloc;
    if (!A.on_device(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live or is swapped out", s);
    if (new_len < 0 || new_len > A.len[s]) return fail(PKV_ERR_INVALID_ARG, "new_len %d outside [0, %d]", new_len, A.len[s]);
    const int32_t keep_blk = ceil_div(new_len, kBlock);
    if (new_len % kBlock && A.table[s][keep_blk - 1] < 0)
      return fail(PKV_ERR_INVALID_ARG, "the new last block of sequence %d was evicted", s);
    A.drop_from(s, keep_blk);
    A.len[s] = new_len;
    return PKV_OK;
  });
}

pkv_status pkv_seq_truncate_many(pkv_pool* p, int32_t n, const int32_t* ids, const int32_t* new_lens) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (n < 0 || (n > 0 && (!ids || !new_lens))) return fail(PKV_ERR_INVALID_ARG, "bad arrays");
    auto& A = p->alloc;
    for (int32_t i = 0; i < n; ++i) {  // validate everything before changing anything
      const int32_t s = ids[i], L = new_lens[i];
      if (!A.on_device(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live or is swapped out", s);
      if (L < 0 || L > A.len[s]) return fail(PKV_ERR_INVALID_ARG, "new_len %d outside [0, %d]", L, A.len[s]);
      if (L % kBlock && A.table[s][ceil_div(L, kBlock) - 1] < 0)
        return fail(PKV_ERR_INVALID_ARG, "the new last block of sequence %d was evicted", s);
    }
    if (const int32_t d = A.first_repeat(n, ids); d >= 0)
      return fail(PKV_ERR_INVALID_ARG, "sequence %d listed twice", d);
    for (int32_t i = 0; i < n; ++i) {
      A.drop_from(ids[i], ceil_div(new_lens[i], kBlock));
      A.len[ids[i]] = new_lens[i];
    }
    return PKV_OK;
  });
}

pkv_status pkv_seq_free(pkv_pool* p, int32_t s) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    auto& A = p->alloc;
    if (A.valid_seq(s) && A.swapped[s]) {  // give back the host blocks, ascending
      for (int32_t hb : A.host_table[s])
        if (hb >= 0) A.release_host(hb);
      A.host_table[s].clear();
      A.table[s].clear();
      A.swapped[s] = 0;
      A.len[s] = 0;
    } else if (pkv_status r = pkv_seq_truncate(p, s, 0)) {
      return r;
    }
    A.live[s] = 0;
    A.holes[s] = 0;
    A.free_ids.insert(s);
    return PKV_OK;
  });
}

pkv_status pkv_seq_evict(pkv_pool* p, int32_t s, int32_t S, int32_t W) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    auto& A = p->alloc;
    if (!A.valid_seq(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live", s);
    if (S < 0 || W < 1) return fail(PKV_ERR_INVALID_ARG, "need num_sinks >= 0 and window >= 1");
    if (A.swapped[s]) return fail(PKV_ERR_INVALID_ARG, "sequence %d is swapped out", s);
    const int32_t L = A.len[s];
    if ((int64_t)L <= (int64_t)S + W) return PKV_OK;
    const int32_t nblk = ceil_div(L, kBlock);
    for (int32_t lb = 0; lb < nblk; ++lb) {
      const int32_t b = A.table[s][lb];
      if (b < 0) continue;
      const int32_t lo = lb * kBlock, hi = std::min(L, lo + kBlock);  // tokens [lo, hi)
      const bool touches_sinks = lo < S;
      const bool touches_window = hi > L - W;
      if (!touches_sinks && !touches_window) {
        A.release(b);
        A.set_entry(s, lb, -1);
        A.holes[s] = 1;
      }
    }
    return PKV_OK;
  });
}

pkv_status pkv_seq_len(const pkv_pool* p, int32_t s, int32_t* len_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !len_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (!p->alloc.valid_seq(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live", s);
    *len_out = p->alloc.len[s];
    return PKV_OK;
  });
}

pkv_status pkv_get_block_table(const pkv_pool* p, int32_t s, int32_t* host_out, int32_t cap, int32_t* n_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !n_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    const auto& A = p->alloc;
    if (!A.valid_seq(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live", s);
    const int32_t n = ceil_div(A.len[s], kBlock);
    *n_out = n;
    if (n > cap || (n > 0 && !host_out)) return fail(PKV_ERR_INVALID_ARG, "capacity %d < %d entries", cap, n);
    for (int32_t i = 0; i < n; ++i) host_out[i] = A.table[s][i];
    return PKV_OK;
  });
}

pkv_status pkv_pool_stats(const pkv_pool* p, pkv_stats* out) {
  return guarded([&]() -> pkv_status {
    if (!p || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    const auto& A = p->alloc;
    out->num_blocks = A.NB;
    out->free_blocks = (int64_t)A.free_blocks.size();
    out->used_blocks = A.NB - out->free_blocks;
    out->shared_blocks = A.n_multi;
    out->active_seqs = A.max_seqs - (int64_t)A.free_ids.size();
    out->cow_copies = A.cow_count;
    out->blocks_allocated = A.n_alloc;
    out->blocks_freed = A.n_freed;
    return PKV_OK;
  });
}

pkv_status pkv_reserve_slots(pkv_pool* p, int32_t n, const int32_t* ids, int32_t T, int64_t* slots_out,
                             int32_t* cow_out, int32_t cow_cap, int32_t* n_cow_out) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (T < 0) return fail(PKV_ERR_INVALID_ARG, "T < 0");
    if (pkv_status r = check_seq_list(p, n, ids)) return r;
    auto& A = p->alloc;
    if (A.first_repeat(n, ids) >= 0) return fail(PKV_ERR_INVALID_ARG, "a sequence appears twice in one append");
    // dry run: count the blocks needed, with the refcount drops earlier
    // copies in this call cause
    int64_t need = 0;
    A.begin_drops();
    for (int32_t i = 0; i < n; ++i) {
      const int32_t s = ids[i];
      if ((int64_t)A.len[s] + T > (int64_t)A.max_blocks * kBlock)
        return fail(PKV_ERR_INVALID_ARG, "sequence %d would exceed max_blocks_per_seq", s);
      for (int32_t t = 0; t < T; ++t) {
        const int32_t pos = A.len[s] + t;
        if (pos % kBlock == 0) {
          ++need;
        } else if (t == 0) {
          const int32_t b = A.table[s][pos / kBlock];
          if (b < 0) return fail(PKV_ERR_INVALID_ARG, "sequence %d: last block was evicted", s);
          if (A.refcount[b] - A.dropped(b) > 1) {
            ++need;
            ++A.dropped(b);
          }
        }
      }
    }
    if (need > (int64_t)A.free_blocks.size())
      return fail(PKV_ERR_OUT_OF_BLOCKS, "append needs %lld blocks, %zu free", (long long)need, A.free_blocks.size());
    int32_t ncow = 0;
    for (int32_t i = 0; i < n; ++i) {
      const int32_t s = ids[i];
      for (int32_t t = 0; t < T; ++t) {
        const int32_t pos = A.len[s];
        const int32_t lb = pos / kBlock;
        if (pos % kBlock == 0) {
          A.set_entry(s, lb, A.take());
        } else if (A.refcount[A.table[s][lb]] > 1) {
          const int32_t old = A.table[s][lb];
          const int32_t fresh = A.take();
          A.release(old);  // still held by another sequence
          A.set_entry(s, lb, fresh);
          if (A.queue) {
            A.pending_cow.push_back(old);
            A.pending_cow.push_back(fresh);
          }
          if (cow_out && ncow < cow_cap) {
            cow_out[2 * ncow] = old;
            cow_out[2 * ncow + 1] = fresh;
          }
          ++ncow;
          ++A.cow_count;
        }
        if (slots_out) slots_out[(size_t)i * T + t] = (int64_t)A.table[s][lb] * kBlock + pos % kBlock;
        A.len[s] = pos + 1;
      }
    }
    if (n_cow_out) *n_cow_out = ncow;
    return PKV_OK;
  });
}

pkv_status pkv_append(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, int32_t T, const void* k_new,
                      const void* v_new) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
    if ((int64_t)n * T > 0 && (!k_new || !v_new)) return fail(PKV_ERR_INVALID_ARG, "k_new / v_new is NULL");
    const size_t ntok = (size_t)n * (size_t)std::max(T, 0);
    std::vector<int64_t> slots(ntok);
    if (pkv_status r = pkv_reserve_slots(p, n, ids, T, slots.data(), nullptr, 0, nullptr)) return r;
    cudaStream_t st = (cudaStream_t)stream;
    // copies first: the new rows of a copied block land in the copy
    if (pkv_status r = flush_pending(p, st, /*with_patches=*/false)) return r;
    std::vector<TablePatch> patches = dedup_patches(p->alloc, p->alloc.pending_patch);
    p->alloc.pending_patch.clear();
    if (ntok == 0 && patches.empty()) return PKV_OK;
    const auto& c = p->cfg;
    const size_t row_bytes = (size_t)c.n_kv_heads * c.head_dim * (c.kv_dtype == PKV_KV_FP32 ? 4 : 2);
    AppendArgs a;
    a.kv_dtype = c.kv_dtype;
    a.Hk = c.n_kv_heads;
    a.D = c.head_dim;
    a.k_pool = p->buf.k_pool;
    a.v_pool = p->buf.v_pool;
    a.k_scale = p->buf.k_scale;
    a.v_scale = p->buf.v_scale;
    a.k_channel = p->k_channel;
    a.v_channel = p->v_channel;
    a.tables = p->buf.block_tables;
    if (ntok <= (size_t)kInlineAppend && patches.size() <= (size_t)kInlineAppend) {
      // small (decode-step) append: slots and patches ride in the parameters
      a.n_tokens = (int)ntok;
      a.n_patches = (int)patches.size();
      a.slots = nullptr;
      a.patches = nullptr;
      for (size_t i = 0; i < ntok; ++i) a.inline_slots[i] = slots[i];
      for (size_t i = 0; i < patches.size(); ++i) {
        a.inline_patches[2 * i] = patches[i].index;
        a.inline_patches[2 * i + 1] = patches[i].value;
      }
      a.k_new = k_new;
      a.v_new = v_new;
      return launch(p, PKV_KERNEL_APPEND, st, [&] { return launch_append(a, st); });
    }
    // large appends go through the staging ring in chunks of tokens; the first
    // chunk carries the patches
    const size_t chunk = size_t(1) << 20;
    size_t t0 = 0;
    do {
      const size_t nt = std::min(chunk, ntok - t0);
      const size_t np = t0 == 0 ? patches.size() : 0;
      const size_t slot_off = (np * sizeof(TablePatch) + 255) & ~size_t(255);
      StagingSlot* s;
      if (pkv_status r = p->staging.acquire(slot_off + nt * sizeof(int64_t), &s)) return r;
      if (np) memcpy(s->host, patches.data(), np * sizeof(TablePatch));
      if (nt) memcpy(s->host + slot_off, slots.data() + t0, nt * sizeof(int64_t));
      if (pkv_status r = Staging::upload(s, slot_off + nt * sizeof(int64_t), st)) return r;
      a.n_tokens = (int)nt;
      a.n_patches = (int)np;
      a.patches = (const int32_t*)s->dev;
      a.slots = (const int64_t*)(s->dev + slot_off);
      a.k_new = (const char*)k_new + t0 * row_bytes;
      a.v_new = (const char*)v_new + t0 * row_bytes;
      if (pkv_status r = launch(p, PKV_KERNEL_APPEND, st, [&] { return launch_append(a, st); })) return r;
      if (pkv_status r = Staging::release(s, st)) return r;
      t0 += nt;
    } while (t0 < ntok);
    return PKV_OK;
  });
}

pkv_status pkv_seq_compact(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const int32_t* keep_idx,
                           int64_t keep_stride, const int32_t* counts, float* acc, int64_t acc_stride) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (pkv_status r = check_seq_list(p, n, ids)) return r;
    if (n > 0 && !counts) return fail(PKV_ERR_INVALID_ARG, "counts is NULL");
    auto& A = p->alloc;
    int64_t need = 0;
    int32_t max_count = 0, max_len = 0;
    if (const int32_t d = A.first_repeat(n, ids); d >= 0)
      return fail(PKV_ERR_INVALID_ARG, "sequence %d listed twice", d);
    for (int32_t i = 0; i < n; ++i) {
      if (counts[i] < 0 || counts[i] > A.len[ids[i]])
        return fail(PKV_ERR_INVALID_ARG, "count %d outside [0, %d]", counts[i], A.len[ids[i]]);
      need += ceil_div(counts[i], kBlock);
      max_count = std::max(max_count, counts[i]);
      max_len = std::max(max_len, A.len[ids[i]]);
    }
    if (p->device) {
      if (max_count > 0 && (!keep_idx || keep_stride < max_count))
        return fail(PKV_ERR_INVALID_ARG, "keep_idx is NULL or keep_stride < largest count");
      if (acc && acc_stride < max_len) return fail(PKV_ERR_INVALID_ARG, "acc_stride < length");
    }
    if (need > (int64_t)A.free_blocks.size())
      return fail(PKV_ERR_OUT_OF_BLOCKS, "compaction needs %lld fresh blocks, %zu free", (long long)need,
                  A.free_blocks.size());
    cudaStream_t st = (cudaStream_t)stream;
    if (p->device)
      if (pkv_status r = flush_pending(p, st)) return r;  // the gather reads the current device table
    // fresh blocks for every sequence first, then release the old ones
    std::vector<CompactSeq> seqs(n);
    std::vector<int32_t> fresh;
    fresh.reserve(need);
    for (int32_t i = 0; i < n; ++i) {
      seqs[i] = {ids[i], i, counts[i], (int32_t)fresh.size(), A.len[ids[i]], 0, 0, 0};
      for (int32_t k = 0; k < ceil_div(counts[i], kBlock); ++k) fresh.push_back(A.take());
    }
    // a failure before the gather is queued gives the fresh blocks back
    auto undo = [&](pkv_status r) {
      for (size_t k = fresh.size(); k-- > 0;) A.untake(fresh[k]);
      return r;
    };
    StagingSlot* s = nullptr;
    if (p->device && n > 0) {
      const size_t seq_bytes = n * sizeof(CompactSeq), off = (seq_bytes + 255) & ~size_t(255);
      if (pkv_status r = p->staging.acquire(off + fresh.size() * sizeof(int32_t) + 4, &s)) return undo(r);
      memcpy(s->host, seqs.data(), seq_bytes);
      if (!fresh.empty()) memcpy(s->host + off, fresh.data(), fresh.size() * sizeof(int32_t));
      if (pkv_status r = Staging::upload(s, off + fresh.size() * sizeof(int32_t), st)) return undo(r);
      const auto& c = p->cfg;
      const int row_bytes = c.head_dim * elem_bytes(c.kv_dtype);
      const bool fp8 = has_scales(c.kv_dtype);
      if (pkv_status r = launch(p, PKV_KERNEL_COMPACT, st, [&] {
            return launch_compact_gather((const CompactSeq*)s->dev, n, max_count, (const int32_t*)(s->dev + off),
                                         p->buf.block_tables, c.max_blocks_per_seq, c.num_blocks, keep_idx, keep_stride,
                                         c.n_kv_heads, row_bytes, p->buf.k_pool, p->buf.v_pool,
                                         fp8 ? p->buf.k_scale : nullptr, fp8 ? p->buf.v_scale : nullptr, p->buf.status,
                                         st);
          }))
        return undo(r);
    }
    size_t pos = 0;
    // old blocks, ascending, sequence by sequence; each entry gets one patch
    // (its fresh block below the new length, -1 past it)
    for (int32_t i = 0; i < n; ++i) A.drop_from(ids[i], 0, ceil_div(counts[i], kBlock));
    for (int32_t i = 0; i < n; ++i) {
      for (int32_t k = 0; k < ceil_div(counts[i], kBlock); ++k) A.set_entry(ids[i], k, fresh[pos++]);
      A.len[ids[i]] = counts[i];
      A.holes[ids[i]] = 0;
    }
    if (!p->device) return PKV_OK;
    // new tables, after the gather (the queue holds this call's patches only:
    // the flush before the gather emptied it)
    if (pkv_status r = flush_pending(p, st, true, true)) return r;
    if (acc && n > 0)
      if (pkv_status r = launch(p, PKV_KERNEL_COMPACT, st, [&] {
            return launch_compact_scores((const CompactSeq*)s->dev, n, keep_idx, keep_stride, acc, acc_stride, st);
          }))
        return r;
    return s ? Staging::release(s, st) : PKV_OK;
  });
}

pkv_status pkv_swap_space_create(pkv_pool* p, int64_t nh, void* hk, void* hv, float* hks, float* hvs) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    auto& A = p->alloc;
    if (nh < 0 || nh > INT32_MAX) return fail(PKV_ERR_INVALID_ARG, "num_host_blocks %lld out of range", (long long)nh);
    for (int32_t s = 0; s < A.max_seqs; ++s)
      if (A.swapped[s]) return fail(PKV_ERR_INVALID_ARG, "sequence %d is swapped out", s);
    const bool scaled = has_scales(p->cfg.kv_dtype);
    void *kd = nullptr, *vd = nullptr, *ksd = nullptr, *vsd = nullptr;
    if (p->device) {
      if (nh > 0 && (!hk || !hv || (scaled && (!hks || !hvs))))
        return fail(PKV_ERR_INVALID_ARG, "a host buffer of the swap space is NULL");
      if (pkv_status r = map_host(hk, &kd, "host_k")) return r;
      if (pkv_status r = map_host(hv, &vd, "host_v")) return r;
      if (scaled) {
        if (pkv_status r = map_host(hks, &ksd, "host_k_scale")) return r;
        if (pkv_status r = map_host(hvs, &vsd, "host_v_scale")) return r;
      }
    } else if (hk || hv || hks || hvs) {
      return fail(PKV_ERR_INVALID_ARG, "a host-only pool takes no swap buffers");
    }
    p->host_k = hk;
    p->host_v = hv;
    p->host_ks = scaled ? hks : nullptr;
    p->host_vs = scaled ? hvs : nullptr;
    p->host_k_dev = kd;
    p->host_v_dev = vd;
    p->host_ks_dev = (float*)ksd;
    p->host_vs_dev = (float*)vsd;
    A.set_swap_space((int32_t)nh);
    p->swap_space = true;
    return PKV_OK;
  });
}

pkv_status pkv_swap_out(pkv_pool* p, void* stream, int32_t n, const int32_t* ids) {
  return guarded([&]() -> pkv_status {
    return swap_move(p, stream, n, ids, true);
  });
}

pkv_status pkv_swap_in(pkv_pool* p, void* stream, int32_t n, const int32_t* ids) {
  return guarded([&]() -> pkv_status {
    return swap_move(p, stream, n, ids, false);
  });
}

pkv_status pkv_seq_swapped(const pkv_pool* p, int32_t s, int32_t* swapped_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !swapped_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (!p->alloc.valid_seq(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live", s);
    *swapped_out = p->alloc.swapped[s];
    return PKV_OK;
  });
}

pkv_status pkv_get_host_block_table(const pkv_pool* p, int32_t s, int32_t* host_out, int32_t cap, int32_t* n_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !n_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    const auto& A = p->alloc;
    if (!A.valid_seq(s)) return fail(PKV_ERR_INVALID_ARG, "sequence %d is not live", s);
    const int32_t n = A.swapped[s] ? ceil_div(A.len[s], kBlock) : 0;
    *n_out = n;
    if (n > cap || (n > 0 && !host_out)) return fail(PKV_ERR_INVALID_ARG, "capacity %d < %d entries", cap, n);
    for (int32_t i = 0; i < n; ++i) host_out[i] = A.host_table[s][i];
    return PKV_OK;
  });
}

pkv_status pkv_host_free_blocks(const pkv_pool* p, int64_t* n_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !n_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    *n_out = (int64_t)p->alloc.host_free.size();
    return PKV_OK;
  });
}

pkv_status pkv_decode_workspace_size(const pkv_pool* p, int32_t n, int32_t num_splits, size_t* bytes_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !bytes_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (n < 0 || num_splits < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
    if (p->cfg.kv_dtype == PKV_KV_FP32) {
      *bytes_out = 0;
      return PKV_OK;
    }
    *bytes_out = max_pieces(p, n, num_splits) * partial_floats(p->G * p->HG, p->cfg.head_dim) * sizeof(float);
    return PKV_OK;
  });
}

pkv_status pkv_decode_attn(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const void* q, float scale,
                           int32_t mode, int32_t S, int32_t W, int32_t num_splits, void* out, float* lse,
                           float* logits, int64_t logits_stride, void* workspace, size_t workspace_bytes) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
    if (pkv_status r = check_seq_list(p, n, ids)) return r;
    if (!valid_mask(mode, S, W)) return fail(PKV_ERR_INVALID_ARG, "invalid mask %d (%d, %d)", mode, S, W);
    if (num_splits < 0) return fail(PKV_ERR_INVALID_ARG, "num_splits < 0");
    if (n > 0 && (!q || !out)) return fail(PKV_ERR_INVALID_ARG, "q / out is NULL");
    const auto& A = p->alloc;
    int32_t maxlen = 0;
    for (int32_t i = 0; i < n; ++i) maxlen = std::max(maxlen, A.len[ids[i]]);
    if (logits && logits_stride < maxlen) return fail(PKV_ERR_INVALID_ARG, "logits_stride < max length");
    if (pkv_status r = check_keep_blocks_present(p, n, ids, mode, S, W)) return r;
    cudaStream_t st = (cudaStream_t)stream;
    if (pkv_status r = flush_pending(p, st)) return r;
    if (n == 0) return PKV_OK;
    const auto& c = p->cfg;

    if (c.kv_dtype == PKV_KV_FP32) {
      StagingSlot* s;
      if (pkv_status r = p->staging.acquire(n * sizeof(SeqRow), &s)) return r;
      SeqRow* rows = (SeqRow*)s->host;
      for (int32_t i = 0; i < n; ++i) rows[i] = {ids[i], i, A.len[ids[i]], 0};
      if (pkv_status r = Staging::upload(s, n * sizeof(SeqRow), st)) return r;
      DecodeF32Params prm;
      prm.k_pool = (const float*)p->buf.k_pool;
      prm.v_pool = (const float*)p->buf.v_pool;
      prm.tables = p->buf.block_tables;
      prm.max_blocks = c.max_blocks_per_seq;
      prm.num_blocks = c.num_blocks;
      prm.n_heads = c.n_heads;
      prm.n_kv_heads = c.n_kv_heads;
      prm.head_dim = c.head_dim;
      prm.rows = (const SeqRow*)s->dev;
      prm.n_seqs = n;
      prm.q = (const float*)q;
      prm.out = (float*)out;
      prm.lse = lse;
      prm.logits = logits;
      prm.logits_stride = logits_stride;
      prm.scale = scale;
      prm.mask_mode = mode;
      prm.num_sinks = S;
      prm.window = W;
      prm.status = p->buf.status;
      if (pkv_status r = launch(p, PKV_KERNEL_DECODE, st, [&] { return launch_decode_f32(prm, st); })) return r;
      return Staging::release(s, st);
    }

    size_t need = 0;
    pkv_decode_workspace_size(p, n, num_splits, &need);
    Plan& plan = build_plan(p, n, ids, mode, S, W, num_splits);
    const size_t pf = (size_t)partial_floats(p->G * p->HG, c.head_dim) * sizeof(float);
    if (plan.n_partials > 0 && (!workspace || workspace_bytes < plan.n_partials * pf))
      return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
    if (plan.n_partials > 0 && ((uintptr_t)workspace & 15))
      return fail(PKV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const PlanLayout L = plan_layout(plan, warps_per_cta(p, plan.nq), 0);
    StagingSlot* s;
    if (pkv_status r = p->staging.acquire(L.bytes, &s)) return r;
    plan_write(plan, L, s->host);
    if (pkv_status r = p->staging.upload_overlapped(s, L.bytes, st)) return r;
    if (pkv_status r = launch_tc_plan(p, st, plan, L, s->dev, q, scale, mode, S, W, out, lse, logits, logits_stride,
                                      workspace))
      return r;
    return Staging::release(s, st);
  });
}

pkv_status pkv_h2o_scores(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const float* logits,
                          int64_t logits_stride, const float* lse, int32_t mode, int32_t S, int32_t W, float* acc,
                          int64_t acc_stride) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
    if (pkv_status r = check_seq_list(p, n, ids)) return r;
    if (!valid_mask(mode, S, W)) return fail(PKV_ERR_INVALID_ARG, "invalid mask");
    if (n > 0 && (!logits || !lse || !acc)) return fail(PKV_ERR_INVALID_ARG, "NULL device array");
    if (n > 65535) return fail(PKV_ERR_UNSUPPORTED, "%d sequences in one score update (at most 65535)", n);
    const auto& A = p->alloc;
    int32_t maxlen = 0, max_keep = 0;
    for (int32_t i = 0; i < n; ++i) {
      const int32_t L = A.len[ids[i]];
      maxlen = std::max(maxlen, L);
      int32_t k = L;
      if (mode == PKV_MASK_SLIDING) k = std::min(L, W + 1);
      if (mode == PKV_MASK_SINK_WINDOW && (int64_t)L > (int64_t)S + W) k = S + W;
      max_keep = std::max(max_keep, k);
    }
    if (logits_stride < maxlen || acc_stride < maxlen) return fail(PKV_ERR_INVALID_ARG, "stride < max length");
    cudaStream_t st = (cudaStream_t)stream;
    if (pkv_status r = flush_pending(p, st)) return r;
    if (n == 0 || max_keep == 0) return PKV_OK;
    StagingSlot* s;
    if (pkv_status r = p->staging.acquire(n * sizeof(SeqRow), &s)) return r;
    SeqRow* rows = (SeqRow*)s->host;
    for (int32_t i = 0; i < n; ++i) rows[i] = {ids[i], i, A.len[ids[i]], 0};
    if (pkv_status r = p->staging.upload_overlapped(s, n * sizeof(SeqRow), st)) return r;
    const auto& c = p->cfg;
    if (pkv_status r = launch(p, PKV_KERNEL_H2O_SCORE, st, [&] {
          return launch_h2o_score((const SeqRow*)s->dev, n, c.n_heads, c.n_kv_heads, logits, logits_stride, lse, mode,
                                  S, W, acc, acc_stride, max_keep, st);
        }))
      return r;
    return Staging::release(s, st);
  });
}

namespace {

pkv_status select_keep(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const float* acc,
                       int64_t acc_stride, const SelPolicy& pol, int64_t max_keep, int32_t* keep_idx,
                       int64_t keep_stride, int32_t* keep_count) {
  if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
  if (pkv_status r = check_seq_list(p, n, ids)) return r;
  if (n > 0 && (!acc || !keep_idx || !keep_count)) return fail(PKV_ERR_INVALID_ARG, "NULL device array");
  const auto& A = p->alloc;
  int32_t max_len = 0;
  for (int32_t i = 0; i < n; ++i) max_len = std::max(max_len, A.len[ids[i]]);
  if (max_len > acc_stride) return fail(PKV_ERR_INVALID_ARG, "acc_stride %lld below the longest sequence (%d)",
                                        (long long)acc_stride, max_len);
  if (keep_stride < std::min<int64_t>(max_keep, max_len))
    return fail(PKV_ERR_INVALID_ARG, "keep_stride %lld below the largest keep-set", (long long)keep_stride);
  cudaStream_t st = (cudaStream_t)stream;
  if (pkv_status r = flush_pending(p, st)) return r;
  if (n == 0) return PKV_OK;
  StagingSlot* s;
  if (pkv_status r = p->staging.acquire(n * sizeof(SeqRow), &s)) return r;
  SeqRow* rows = (SeqRow*)s->host;
  for (int32_t i = 0; i < n; ++i) rows[i] = {ids[i], i, A.len[ids[i]], 0};
  if (pkv_status r = p->staging.upload_overlapped(s, n * sizeof(SeqRow), st)) return r;
  const bool starve = p->starve_select;
  p->starve_select = false;
  if (pkv_status r = launch(p, PKV_KERNEL_H2O_SELECT, st, [&] {
        return launch_h2o_select((const SeqRow*)s->dev, n, acc, acc_stride, pol, keep_idx, keep_stride, keep_count,
                                 p->buf.status, p->wait_limit_ns, starve, st);
      }))
    return r;
  return Staging::release(s, st);
}

}  // namespace

pkv_status pkv_h2o_select(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const float* acc,
                          int64_t acc_stride, int32_t budget, int32_t recent, int32_t* keep_idx, int64_t keep_stride,
                          int32_t* keep_count) {
  return guarded([&]() -> pkv_status {
    if (recent < 0 || budget < recent || budget < 1) return fail(PKV_ERR_INVALID_ARG, "need 0 <= recent <= budget, budget >= 1");
    if (keep_stride < budget) return fail(PKV_ERR_INVALID_ARG, "keep_stride < budget");
    return select_keep(p, stream, n, ids, acc, acc_stride, SelPolicy{0, recent, budget - recent, 0}, budget, keep_idx,
                       keep_stride, keep_count);
  });
}

pkv_status pkv_policy_select(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const float* acc,
                             int64_t acc_stride, int32_t sink_size, int32_t window_size, int32_t h2o_size,
                             int32_t* keep_idx, int64_t keep_stride, int32_t* keep_count) {
  return guarded([&]() -> pkv_status {
    if (sink_size < 0 || window_size < 0 || h2o_size < 0)
      return fail(PKV_ERR_INVALID_ARG, "sink_size, window_size and h2o_size must be >= 0");
    return select_keep(p, stream, n, ids, acc, acc_stride, SelPolicy{sink_size, window_size, h2o_size, 1},
                       (int64_t)sink_size + window_size + h2o_size, keep_idx, keep_stride, keep_count);
  });
}

pkv_status pkv_sync_status(pkv_pool* p, void* stream) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
    cudaStream_t st = (cudaStream_t)stream;
    PKV_CUDA(cudaStreamSynchronize(st));
    int32_t w[4] = {0, 0, 0, 0};
    PKV_CUDA(cudaMemcpy(w, p->buf.status, sizeof w, cudaMemcpyDeviceToHost));
    if (w[0]) {
      PKV_CUDA(cudaMemset(p->buf.status, 0, sizeof w));
      PKV_CUDA(cudaDeviceSynchronize());
      if (w[0] & kStatusUndrained)
        return fail(PKV_ERR_UNDRAINED,
                    "a device wait timed out (info %d) and copies it had issued were still in flight when the "
                    "kernel gave up on them; later results on this CUDA context are not reliable",
                    w[1]);
      if (w[0] & kStatusTimeout) return fail(PKV_ERR_TIMEOUT, "a device wait timed out (info %d)", w[1]);
      return fail(PKV_ERR_DEVICE_ASSERT, "device range check failed (info %d, %d)", w[1], w[2]);
    }
    return PKV_OK;
  });
}

pkv_status pkv_timing_enable(pkv_pool* p, int32_t kernel_mask) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    p->timing.mask = p->device ? kernel_mask : 0;
    return PKV_OK;
  });
}

pkv_status pkv_timing_read(pkv_pool* p, double* total_ms, int64_t* launches) {
  return guarded([&]() -> pkv_status {
    if (!p || !total_ms || !launches) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    for (int k = 0; k < PKV_KERNEL_COUNT; ++k) {
      double sum = 0;
      for (auto& pr : p->timing.marks[k]) {
        PKV_CUDA(cudaEventSynchronize(pr.second));
        float ms = 0;
        PKV_CUDA(cudaEventElapsedTime(&ms, pr.first, pr.second));
        sum += ms;
        p->timing.spare.push_back(pr.first);
        p->timing.spare.push_back(pr.second);
      }
      total_ms[k] = sum;
      launches[k] = (int64_t)p->timing.marks[k].size();
      p->timing.marks[k].clear();
    }
    return PKV_OK;
  });
}

pkv_status pkv_set_wait_limit(pkv_pool* p, int64_t wait_limit_ns) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (wait_limit_ns < 1000000 || wait_limit_ns > 60000000000LL)
      return fail(PKV_ERR_INVALID_ARG, "wait limit must lie in [1 ms, 60 s]");
    p->wait_limit_ns = (uint64_t)wait_limit_ns;
    return PKV_OK;
  });
}

pkv_status pkv_set_channel_scales(pkv_pool* p, const float* k_channel, const float* v_channel) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (!p->device) return fail(PKV_ERR_NO_DEVICE, "host-only pool");
    if (!has_scales(p->cfg.kv_dtype)) return fail(PKV_ERR_UNSUPPORTED, "channel scales need an FP8 or INT8 pool");
    if ((k_channel == nullptr) != (v_channel == nullptr))
      return fail(PKV_ERR_INVALID_ARG, "give both channel scale arrays or neither");
    const auto& A = p->alloc;
    for (int32_t s = 0; s < A.max_seqs; ++s)
      if (A.live[s] && A.len[s] > 0)
        return fail(PKV_ERR_INVALID_ARG, "channel scales change only while the pool holds no token (sequence %d)", s);
    if (k_channel) {
      const size_t n = (size_t)p->cfg.n_kv_heads * p->cfg.head_dim;
      std::vector<float> h(2 * n);
      PKV_CUDA(cudaMemcpy(h.data(), k_channel, n * sizeof(float), cudaMemcpyDeviceToHost));
      PKV_CUDA(cudaMemcpy(h.data() + n, v_channel, n * sizeof(float), cudaMemcpyDeviceToHost));
      for (size_t i = 0; i < 2 * n; ++i) {
        uint32_t bits;
        memcpy(&bits, &h[i], sizeof bits);
        const uint32_t ex = (bits >> 23) & 0xFF;
        // a power of two, 2^-126 .. 2^127: sign 0, mantissa 0, a normal exponent
        if ((bits & 0x807FFFFFu) != 0 || ex == 0 || ex == 0xFF)
          return fail(PKV_ERR_INVALID_ARG, "channel scale %zu of %s (%g) is not a positive power of two", i % n,
                      i < n ? "K" : "V", (double)h[i]);
      }
    }
    p->k_channel = k_channel;
    p->v_channel = v_channel;
    return PKV_OK;
  });
}

pkv_status pkv_set_cascade(pkv_pool* p, int32_t mode) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (mode < 0 || mode > 2) return fail(PKV_ERR_INVALID_ARG, "cascade mode %d not in {0, 1, 2}", mode);
    p->cascade = mode;
    return PKV_OK;
  });
}

pkv_status pkv_test_starve_next_decode(pkv_pool* p, int32_t warp) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (warp < 0) return fail(PKV_ERR_INVALID_ARG, "warp < 0");
    p->starve_warp = warp;
    return PKV_OK;
  });
}

pkv_status pkv_test_starve_next_select(pkv_pool* p) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    p->starve_select = true;
    return PKV_OK;
  });
}

pkv_status pkv_test_set_geometry(pkv_pool* p, int32_t num_sms, int32_t wpc, int32_t wpc2, int32_t group) {
  return guarded([&]() -> pkv_status {
    if (!p) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (p->device) return fail(PKV_ERR_INVALID_ARG, "the geometry of a device pool is its GPU's");
    if (num_sms < 1 || wpc < 1 || wpc2 < 1 || group < 1) return fail(PKV_ERR_INVALID_ARG, "geometry must be positive");
    p->num_sms = num_sms;
    p->tc_warps_per_cta = wpc;
    p->tc2_warps_per_cta = wpc2;
    p->tc_ctas_per_sm = p->tc2_ctas_per_sm = 1;
    p->G = group;
    p->HG = unit_heads(p->cfg, group);
    return PKV_OK;
  });
}

pkv_status pkv_test_plan_bytes(pkv_pool* p, int32_t n, const int32_t* ids, int32_t mode, int32_t S, int32_t W,
                               int32_t num_splits, int32_t general, void* out, size_t cap, size_t* size,
                               int32_t* info) {
  return guarded([&]() -> pkv_status {
    if (!p || !size || !info) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (pkv_status r = check_seq_list(p, n, ids)) return r;
    if (n < 1) return fail(PKV_ERR_INVALID_ARG, "no sequences");
    if (!valid_mask(mode, S, W)) return fail(PKV_ERR_INVALID_ARG, "invalid mask %d (%d, %d)", mode, S, W);
    if (num_splits < 0) return fail(PKV_ERR_INVALID_ARG, "num_splits < 0");
    p->general_plan = general != 0;
    Plan& plan = build_plan(p, n, ids, mode, S, W, num_splits);
    p->general_plan = false;
    const PlanLayout L = plan_layout(plan, warps_per_cta(p, plan.nq), 0);
    *size = L.bytes;
    info[0] = plan.total_warps;
    info[1] = plan.ctas;
    info[2] = plan.n_partials;
    info[3] = plan.nq;
    info[4] = (int32_t)plan.pieces.size();
    info[5] = (int32_t)plan.combine.size();
    info[6] = (int32_t)plan.empty.size();
    info[7] = (int32_t)plan.prefix_items.size();
    info[8] = (int32_t)plan.prefix_members.size();
    if (cap < L.bytes || !out) return fail(PKV_ERR_INVALID_ARG, "plan of %zu bytes > cap %zu", L.bytes, cap);
    plan_write(plan, L, (char*)out);
    return PKV_OK;
  });
}

pkv_status pkv_test_cow_waves(pkv_pool* p, int32_t n_pairs, const int32_t* pairs, int32_t* starts_out, int32_t cap,
                              int32_t* n_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !n_out || n_pairs < 0 || (n_pairs > 0 && !pairs)) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
    auto& A = p->alloc;
    for (int64_t i = 0; i < 2 * (int64_t)n_pairs; ++i)
      if (pairs[i] < 0 || pairs[i] >= A.NB) return fail(PKV_ERR_INVALID_ARG, "block %d out of range", pairs[i]);
    std::vector<int32_t> queued;
    queued.swap(A.pending_cow);
    A.pending_cow.assign(pairs, pairs + 2 * (size_t)n_pairs);
    const std::vector<size_t> w = cow_waves(A);
    A.pending_cow.swap(queued);
    *n_out = (int32_t)w.size();
    if ((int32_t)w.size() > cap || !starts_out) return fail(PKV_ERR_INVALID_ARG, "capacity %d < %zu", cap, w.size());
    for (size_t i = 0; i < w.size(); ++i) starts_out[i] = (int32_t)w[i];
    return PKV_OK;
  });
}

pkv_status pkv_test_take_patches(pkv_pool* p, int32_t queue_patches, int32_t* out, int32_t cap, int32_t* n_out) {
  return guarded([&]() -> pkv_status {
    if (!p || !n_out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (p->device) return fail(PKV_ERR_INVALID_ARG, "a device pool flushes its own queue");
    auto& A = p->alloc;
    A.queue = queue_patches != 0;
    *n_out = (int32_t)A.pending_patch.size();
    if (*n_out > cap || (*n_out > 0 && !out)) return fail(PKV_ERR_INVALID_ARG, "capacity %d < %d patches", cap, *n_out);
    for (size_t i = 0; i < A.pending_patch.size(); ++i) {
      out[2 * i] = A.pending_patch[i].index;
      out[2 * i + 1] = A.pending_patch[i].value;
    }
    A.pending_patch.clear();
    A.pending_cow.clear();
    return PKV_OK;
  });
}

pkv_status pkv_launch_count(const pkv_pool* p, int64_t* out) {
  return guarded([&]() -> pkv_status {
    if (!p || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    *out = p->launches;
    return PKV_OK;
  });
}

}  // extern "C"
