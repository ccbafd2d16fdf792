/*
 * pkv.h -- C ABI of libpkv: decode attention over a paged KV cache on GB300.
 *
 * The cache keeps every sequence's keys and values in fixed 16-token
 * physical blocks drawn from one shared pool; a per-sequence block table maps
 * logical block i (tokens 16i .. 16i+15) to a physical block.  Blocks can be
 * shared between sequences with reference counts and are copied on the first
 * write to a shared block.  Decode attends one query token per sequence over
 * its cached tokens, with grouped-query heads, optional FP8-E4M3 or INT8
 * storage with per-token scales (and optional per-channel scales), optional
 * sliding-window or sink + window
 * keep-sets, and
 * optional H2O accumulated-score output and keep-set selection.
 *
 * Sources (page title, section):
 *   [LC] "长上下文优化：注意力稀疏化与 KV Cache 管理": KV bytes per token;
 *        sliding-window mask; StreamingKVCache; H2OEviction; block-table
 *        sketch; GQA head counts.
 *   [PA] "KV Cache 与 PagedAttention：显存复用与长上下文推理": sections
 *        PagedAttention 的设计, 物理布局示意, 三大运行时组件 (block allocator,
 *        block table, reference count + copy-on-write), the Block/copy_on_write
 *        sketch, 量化原理 (FP16 -> INT8 / FP8 E4M3, per-token scaling), and the monitoring
 *        note (free/used blocks).
 *   [SO] "系统优化": 滑动窗口注意力 / StreamingLLM 详解 (sinks + window), KV
 *        Cache 淘汰 (H2O), Flash Attention (tiled online softmax).
 *
 * Conventions
 *   - Every call returns a pkv_status; nothing throws across the ABI (a
 *     failed host allocation inside the library returns PKV_ERR_HOST_MEMORY).
 *     pkv_last_error() gives a message for the calling thread's last failure.
 *   - "device" pointers are CUDA device memory owned by the caller; the
 *     library never frees them.  "host" pointers are ordinary host memory.
 *     The library owns only its host-side allocator state and pinned staging
 *     buffers.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued asynchronously on it; host arrays
 *     passed in are fully consumed before the call returns.
 *   - A pool is used from one host thread at a time, and its device work
 *     must run in call order: pass one stream to every call, or order the
 *     streams yourself.  (Blocks that one call frees on the host can be the
 *     ones the next call's kernels write, while the first call's kernels may
 *     still read them.)
 *   - Layouts (row-major, innermost last):
 *       k_pool, v_pool  [num_blocks][n_kv_heads][16][head_dim]  kv dtype
 *       k_scale,v_scale [num_blocks][n_kv_heads][16]            fp32 (FP8 / INT8 only)
 *       block_tables    [max_seqs][max_blocks_per_seq]          int32, -1 = none
 *       q, out          [n_seqs][n_heads][head_dim]   fp32 (fp32 KV) else bf16
 *       lse             [n_seqs][n_heads]                        fp32, natural log
 *       logits          [n_seqs][n_kv_heads][logits_stride][G]   fp32
 *     with G = n_heads / n_kv_heads; query head h reads kv head h / G.
 *   - Device-side failures (a bounded wait that ran out, a table entry out of
 *     range) set the pool's device status word; pkv_sync_status() reports
 *     and clears them.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_BLOCK_SIZE 16

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* bad argument; state unchanged */
  PKV_ERR_UNSUPPORTED = 2,   /* valid but unsupported shape or dtype */
  PKV_ERR_OUT_OF_BLOCKS = 3, /* the free pool cannot cover the request; state unchanged */
  PKV_ERR_OUT_OF_SEQS = 4,   /* every sequence id is in use */
  PKV_ERR_CUDA = 5,          /* a CUDA runtime call failed (message in pkv_last_error) */
  PKV_ERR_TIMEOUT = 6,       /* a device-side bounded wait ran out */
  PKV_ERR_DEVICE_ASSERT = 7, /* a device-side range check failed */
  PKV_ERR_NO_DEVICE = 8,     /* device work requested on a host-only pool */
  PKV_ERR_WORKSPACE = 9,     /* workspace too small (see pkv_decode_workspace_size) */
  PKV_ERR_HOST_MEMORY = 10,  /* a host allocation failed; the pool may be part-way
                                through the call and should be destroyed */
  PKV_ERR_UNDRAINED = 11     /* a device-side bounded wait ran out, and so did the
                                wait for the copies the kernel had already issued:
                                they may still land in shared memory after the
                                kernel exits, so later work on this CUDA context
                                is not reliable (recreate the context) */
} pkv_status;

typedef enum { PKV_KV_FP32 = 0, PKV_KV_BF16 = 1, PKV_KV_FP8_E4M3 = 2, PKV_KV_INT8 = 3 } pkv_kv_dtype;

/* Keep-sets for decode query position i = L - 1 over keys j in [0, L):
 *   FULL         every key.
 *   SLIDING      |i - j| <= window ([LC] sliding-window mask), i.e. the
 *                window + 1 keys j >= L - 1 - window.
 *   SINK_WINDOW  [LC] StreamingKVCache / [SO] StreamingLLM: when L exceeds
 *                num_sinks + window, keys j < num_sinks and j >= L - window;
 *                otherwise every key. */
typedef enum { PKV_MASK_FULL = 0, PKV_MASK_SLIDING = 1, PKV_MASK_SINK_WINDOW = 2 } pkv_mask_mode;

/* [PA] PagedAttention 的设计 / 三大运行时组件.  Shapes supported: block_size
 * 16; head_dim 64 or 128 (every kv dtype); G in {1, 2, 4, 8} ([LC] MHA / GQA /
 * MQA head counts).  Anything else: PKV_ERR_UNSUPPORTED. */
typedef struct {
  int32_t num_blocks;         /* physical blocks in the pool */
  int32_t block_size;         /* must be 16 */
  int32_t n_heads;            /* query heads */
  int32_t n_kv_heads;         /* KV heads (GQA: n_heads % n_kv_heads == 0) */
  int32_t head_dim;
  int32_t max_seqs;           /* rows of the block table */
  int32_t max_blocks_per_seq; /* columns of the block table */
  int32_t kv_dtype;           /* pkv_kv_dtype */
  uint64_t alloc_seed;        /* initial free-pool order: Fisher-Yates shuffle of
                                 [0, num_blocks) driven by splitmix64(alloc_seed);
                                 0 = ascending order */
  const int32_t* free_order;  /* host, optional: explicit initial free-pool order
                                 (num_blocks distinct ids, front first); overrides
                                 alloc_seed; copied during create */
} pkv_pool_config;

/* Device buffers of a pool, all allocated and owned by the caller. */
typedef struct {
  void* k_pool;          /* device, [num_blocks][n_kv_heads][16][head_dim] */
  void* v_pool;          /* device, same shape */
  float* k_scale;        /* device, [num_blocks][n_kv_heads][16] (FP8 / INT8 only, else NULL) */
  float* v_scale;        /* device, same (FP8 / INT8 only, else NULL) */
  int32_t* block_tables; /* device, [max_seqs][max_blocks_per_seq]; the library
                            initialises it to -1 during create and keeps it in
                            step with the host tables */
  int32_t* status;       /* device, 4 int32: device error word, zeroed by create */
} pkv_pool_buffers;

typedef struct {
  size_t k_pool, v_pool, k_scale, v_scale, block_tables, status; /* bytes */
} pkv_buffer_sizes;

typedef struct {
  int64_t num_blocks, free_blocks, used_blocks;
  int64_t shared_blocks; /* blocks with refcount > 1 */
  int64_t active_seqs;
  int64_t cow_copies;    /* copy-on-write block copies so far */
  int64_t blocks_allocated, blocks_freed;
} pkv_stats;

typedef struct pkv_pool pkv_pool;

/* ---- pool lifetime ------------------------------------------------------ */

/* Bytes each device buffer of a pool with this config needs. */
pkv_status pkv_pool_required_bytes(const pkv_pool_config* cfg, pkv_buffer_sizes* out);

/* Creates a pool.  `buffers` NULL gives a host-only pool: the allocator calls
 * work, device calls return PKV_ERR_NO_DEVICE.  With buffers, the current CUDA
 * device must be the one that holds them; the block tables are set to -1 and
 * the status word to 0 (synchronously). */
pkv_status pkv_pool_create(const pkv_pool_config* cfg, const pkv_pool_buffers* buffers,
                           pkv_pool** out);
void pkv_pool_destroy(pkv_pool* pool);

/* ---- sequences (host allocator, [PA] 三大运行时组件) ---------------------- */

/* New empty sequence; the id is the smallest one not in use. */
pkv_status pkv_seq_add(pkv_pool* pool, int32_t* seq_out);
/* New sequence sharing every block of `src` (refcount + 1 each): parallel
 * sampling / beam fork ([PA] 共享场景的价值). */
pkv_status pkv_seq_fork(pkv_pool* pool, int32_t src, int32_t* dst_out);
/* Drops every block reference (blocks reaching 0 return to the front of the
 * free pool, in ascending logical order) and releases the id. */
pkv_status pkv_seq_free(pkv_pool* pool, int32_t seq);
/* Shortens a sequence to new_len tokens, dropping blocks past it (ascending).
 * Refused if the new last block is partial and was evicted. */
pkv_status pkv_seq_truncate(pkv_pool* pool, int32_t seq, int32_t new_len);
/* pkv_seq_truncate for n distinct sequences (host arrays ids[n], new_lens[n]),
 * in the order given; every argument is checked before anything changes. */
pkv_status pkv_seq_truncate_many(pkv_pool* pool, int32_t n, const int32_t* seq_ids, const int32_t* new_lens);
/* StreamingLLM eviction ([LC] StreamingKVCache, [SO] StreamingLLM 详解): drops
 * every block lying wholly outside [0, num_sinks) U [L - window, L); those
 * table entries become -1.  No-op when L <= num_sinks + window.  window >= 1. */
pkv_status pkv_seq_evict(pkv_pool* pool, int32_t seq, int32_t num_sinks, int32_t window);
pkv_status pkv_seq_len(const pkv_pool* pool, int32_t seq, int32_t* len_out);
/* Copies ceil(len/16) table entries of `seq` into host_out (capacity cap). */
pkv_status pkv_get_block_table(const pkv_pool* pool, int32_t seq, int32_t* host_out, int32_t cap,
                               int32_t* n_out);
pkv_status pkv_pool_stats(const pkv_pool* pool, pkv_stats* out);

/* Allocator step of an append ([PA] copy_on_write sketch), host side only.
 * For each listed sequence in order, for each of T new tokens at position p:
 * p % 16 == 0 takes the front block of the free pool; otherwise a shared last
 * block (refcount > 1) is first copied to a fresh block (copy-on-write).
 * Writes slots[i*T + t] = block * 16 + p % 16 (host, may be NULL) and the COW
 * (src, dst) pairs (host [cow_cap][2], may be NULL).  All or nothing:
 * PKV_ERR_OUT_OF_BLOCKS leaves the state unchanged.  On a device pool the
 * block copies and table updates are queued and run at the start of the next
 * call that takes a stream, with the result of running them one by one in
 * queue order (a block freed after it was queued as a copy's source may be
 * the destination of a later copy). */
pkv_status pkv_reserve_slots(pkv_pool* pool, int32_t n_seqs, const int32_t* seq_ids, int32_t T,
                             int64_t* slots_out, int32_t* cow_pairs_out, int32_t cow_cap,
                             int32_t* n_cow_out);

/* ---- device work -------------------------------------------------------- */

/* Appends T tokens per sequence: pkv_reserve_slots, then on `stream` the
 * queued COW block copies (whole blocks: K, V and scales of every kv head),
 * the table updates and the scatter of the new rows into their slots.
 * k_new, v_new: device [n_seqs][T][n_kv_heads][head_dim], fp32 for an FP32
 * pool, bf16 otherwise.  FP8 pools quantise each (token, kv head) row:
 * s = absmax / 448 in fp32 (1 when absmax is 0), code = E4M3(x / s) with
 * round-to-nearest-even and saturation to +-448 ([PA] 量化原理).  INT8 pools
 * alike with s = absmax / 127 and code = x / s rounded to the nearest
 * integer (ties to even), clamped to +-127. */
pkv_status pkv_append(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                      int32_t T, const void* k_new, const void* v_new);

/* Workspace bytes pkv_decode_attn needs for n_seqs sequences and the given
 * num_splits (0 = automatic). */
pkv_status pkv_decode_workspace_size(const pkv_pool* pool, int32_t n_seqs, int32_t num_splits,
                                     size_t* bytes_out);

/* Decode attention ([PA] decode loads KV block by block through the table;
 * [SO] Flash Attention's tiled online softmax).  For each listed sequence b
 * (context length L_b, the current token included) and query head h:
 *   s_j = scale * q[b][h] . K_j   for kept keys j (FP8 / INT8: K_j = code_j * s_j)
 *   out[b][h] = sum_j softmax(s)_j V_j,   lse[b][h] = ln sum_j exp(s_j)
 * Empty keep-set: out = 0, lse = -inf.  Accumulation is fp32.  FP8 / INT8
 * pools: the codes enter the tensor-core products exactly; q is rounded to
 * fp16 after scaling each head by a power of two (so no element overflows),
 * and the softmax weights, normalised by the largest weight times V scale,
 * are rounded to fp16 -- valid for any magnitudes of q, K and V, with V
 * scales above 2^-100.
 *   q, out      device [n_seqs][n_heads][head_dim] (fp32 for FP32 pools, else bf16)
 *   lse         device [n_seqs][n_heads] fp32, or NULL
 *   logits      device [n_seqs][n_kv_heads][logits_stride][G] fp32, or NULL:
 *               receives s_j of every kept key (for pkv_h2o_scores); other
 *               positions are left untouched.  logits_stride >= max L_b.
 *   num_splits  0: the keys of all sequences are split evenly over the GPU's
 *               warps; n > 0: each (sequence, kv head) range is cut into n
 *               equal parts.  Partial results are merged by log-sum-exp.
 *   workspace   device scratch of at least pkv_decode_workspace_size bytes;
 *               it must not be in use by other work on the GPU meanwhile.
 * Every block of the keep-set must be present (not evicted): else
 * PKV_ERR_INVALID_ARG. */
pkv_status pkv_decode_attn(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                           const void* q, float scale, int32_t mask_mode, int32_t num_sinks,
                           int32_t window, int32_t num_splits, void* out, float* lse,
                           float* logits, int64_t logits_stride, void* workspace,
                           size_t workspace_bytes);

/* Same computation and arguments as pkv_decode_attn, minus the workspace: the
 * split-KV scratch lives in a fixed 32 MiB array compiled into the library
 * (2 MiB for the per-call plan and queued block-table / copy-on-write updates,
 * 30 MiB for partial records).  The pages describe nothing like it; it exists
 * for callers that cannot allocate device memory on their own -- code running
 * under a framework allocator that owns the whole device budget, or inside a
 * latency-critical loop where cudaMalloc / cudaFree would synchronise the
 * device.  It allocates no device or pinned memory (host-side planning uses
 * ordinary heap memory) and copies its plan from pageable memory.
 *   - bf16, FP8 and INT8 pools (PKV_ERR_UNSUPPORTED for fp32); the pool's
 *     device must be the current device.
 *   - A call that needs more than the array holds fails with
 *     PKV_ERR_WORKSPACE and a message giving both sizes; nothing is launched.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current) and keeps it for the life of the
 *     process.  After the device's primary context is reset, the kept
 *     address is stale: do not call this entry point again in that process.
 *   - Every device that runs this entry point keeps the 32 MiB until the
 *     process exits.  All calls share the array: calls whose work overlaps on
 *     the GPU (other streams, other pools on the same device) race on it. */
pkv_status pkv_decode_attn_static(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                                  const void* q, float scale, int32_t mask_mode, int32_t num_sinks,
                                  int32_t window, int32_t num_splits, void* out, float* lse, float* logits,
                                  int64_t logits_stride);

/* H2O score update ([LC] H2OEviction.update_scores): for each listed sequence
 * and each kept key j, acc[b][j] += (1/n_heads) * sum_h exp(s_hj - lse_h),
 * the attention weight summed over the single decode query and averaged over
 * all query heads.  logits/lse as written by pkv_decode_attn with the same
 * sequences and keep-set.  acc: device [n_seqs][acc_stride] fp32.  At most
 * 65535 sequences per call (PKV_ERR_UNSUPPORTED above that). */
pkv_status pkv_h2o_scores(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                          const float* logits, int64_t logits_stride, const float* lse,
                          int32_t mask_mode, int32_t num_sinks, int32_t window, float* acc,
                          int64_t acc_stride);

/* H2O keep-set ([LC] H2OEviction.select, [SO] evict_tokens with recent = 0):
 * for each listed sequence (length L, the pool's own), with keep = budget -
 * recent, the positions [L - recent, L) plus the keep highest acc values among
 * [0, L - recent) (ties to the lower position), in ascending order; all of
 * [0, L) when L <= budget.  seq_ids: host [n_seqs], live sequences on the
 * device.  acc: device [n_seqs][acc_stride] fp32 (>= 0; row i belongs to
 * seq_ids[i]; acc_stride >= every listed length).  keep_idx: device
 * [n_seqs][keep_stride] int32 (keep_stride >= budget); keep_count: device
 * [n_seqs] int32.  0 <= recent <= budget. */
pkv_status pkv_h2o_select(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                          const float* acc, int64_t acc_stride, int32_t budget, int32_t recent,
                          int32_t* keep_idx, int64_t keep_stride, int32_t* keep_count);

/* The combined keep rule ([PA] KV compression: initial tokens + recent window
 * + high-attention tokens, printed with sink 4, window 256 and 512 - 4 - 256
 * heavy hitters): position p of a length-L sequence is kept when
 * p < sink_size, when p >= L - window_size, or when acc[b][p] is among the
 * h2o_size highest of all L positions (ties to the lower position).  The
 * ranking spans every position, so a heavy hitter that is also a sink or
 * recent is kept once and the set may be smaller than the three sizes'
 * sum.  Output ascending in keep_idx (device [n_seqs][keep_stride], with
 * keep_stride >= min(sink_size + window_size + h2o_size, largest length)),
 * its size in keep_count (device [n_seqs]).  seq_ids: host [n_seqs], live
 * sequences on the device (L is each one's length in the pool); acc: device
 * [n_seqs][acc_stride] fp32 (>= 0; acc_stride >= every listed length). */
pkv_status pkv_policy_select(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                             const float* acc, int64_t acc_stride, int32_t sink_size, int32_t window_size,
                             int32_t h2o_size, int32_t* keep_idx, int64_t keep_stride, int32_t* keep_count);

/* H2O compaction ([LC] H2OEviction keeps only the selected positions; [PA]
 * 剪枝/淘汰: memory goes from O(seq) to O(budget)).  For each listed sequence,
 * the counts[i] tokens at positions keep_idx[i][0 .. counts[i]) (ascending,
 * e.g. the output of pkv_h2o_select) become its whole contents, in that
 * order, in freshly allocated blocks; the sequence's length becomes counts[i]
 * and its old blocks are released.  Order: every sequence's fresh blocks are
 * taken first (list order), then the old blocks are released (list order,
 * ascending logical order).  acc (device [n_seqs][acc_stride] fp32, or NULL)
 * is compacted alike: acc[i][j] = acc[i][keep_idx[i][j]] for j < counts[i],
 * 0 from counts[i] up to the old length.
 *   keep_idx  device [n_seqs][keep_stride] int32 (keep_stride >= max count)
 *   counts    host [n_seqs]
 * keep_idx must be ascending for acc's in-place compaction to be correct.
 * A position outside [0, old length) or in an evicted block is not copied
 * and sets the device status word (PKV_ERR_DEVICE_ASSERT at the next
 * pkv_sync_status).  On a host-only pool only the allocator changes
 * (keep_idx and acc unused).  PKV_ERR_INVALID_ARG (a sequence listed twice,
 * a count above the length) or PKV_ERR_OUT_OF_BLOCKS (the fresh blocks do
 * not fit) leave every state unchanged. */
pkv_status pkv_seq_compact(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                           const int32_t* keep_idx, int64_t keep_stride, const int32_t* counts, float* acc,
                           int64_t acc_stride);

/* ---- CPU swap space ------------------------------------------------------ */

/* CPU swap ([PA] three runtime components: the block allocator manages the
 * pool in blocks and can swap them out to CPU RAM; [LC] CPU offloading keeps
 * inactive requests' KV in host memory and loads it back when needed).
 *
 * pkv_swap_space_create gives the pool a host pool of num_host_blocks
 * blocks with the device pool's layout:
 *   host_k, host_v            [num_host_blocks][n_kv_heads][16][head_dim]
 *   host_k_scale, host_v_scale [num_host_blocks][n_kv_heads][16] fp32
 *                              (FP8 / INT8 pools only, else NULL)
 * On a device pool they must be page-locked host memory the device can
 * address (cudaHostAlloc, or cudaHostRegister with mapping); the copies run
 * as one kernel per call that reads or writes them directly.  On a host-only
 * pool they must be NULL (the allocator alone is tracked).  The host pool
 * starts in ascending order; allocation takes its front and a released host
 * block goes back to the front.  Refused while a sequence is swapped out.
 *
 * pkv_swap_out: every listed sequence's blocks, in list order and ascending
 * logical order, get host blocks (a device block shared by several listed
 * sequences is copied once and its host block shared as many times); the
 * copies are enqueued on `stream`; then every device block is released (same
 * order) and the device table rows become -1.  A swapped-out sequence keeps
 * its length; append, fork, truncate, evict, compaction and decode refuse it;
 * pkv_seq_free releases its host blocks.
 * pkv_swap_in mirrors it: device blocks from the front of the device pool (a
 * host block shared by several listed sequences becomes one shared device
 * block), copies on `stream`, then the host blocks are released.
 * Both: PKV_ERR_OUT_OF_BLOCKS when the destination pool is short (state
 * unchanged); PKV_ERR_INVALID_ARG for a sequence that is not live, already in
 * the requested place, or listed twice.  Host memory the copies touch may be
 * read by the caller only after `stream` has passed them. */
pkv_status pkv_swap_space_create(pkv_pool* pool, int64_t num_host_blocks, void* host_k, void* host_v,
                                 float* host_k_scale, float* host_v_scale);
pkv_status pkv_swap_out(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids);
pkv_status pkv_swap_in(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids);
/* 1 if the sequence is swapped out, else 0. */
pkv_status pkv_seq_swapped(const pkv_pool* pool, int32_t seq, int32_t* swapped_out);
/* Host block table of a swapped-out sequence (ceil(len / 16) entries, -1 for
 * blocks it did not hold); like pkv_get_block_table. */
pkv_status pkv_get_host_block_table(const pkv_pool* pool, int32_t seq, int32_t* host_out, int32_t cap,
                                    int32_t* n_out);
/* Free blocks of the host pool. */
pkv_status pkv_host_free_blocks(const pkv_pool* pool, int64_t* n_out);

/* Synchronises `stream`, then reports and clears the device status word:
 * PKV_ERR_UNDRAINED, PKV_ERR_TIMEOUT, PKV_ERR_DEVICE_ASSERT or PKV_OK. */
pkv_status pkv_sync_status(pkv_pool* pool, void* stream);

/* ---- measurement -------------------------------------------------------- */

typedef enum {
  PKV_KERNEL_COW_COPY = 0,
  PKV_KERNEL_APPEND = 1,
  PKV_KERNEL_DECODE = 2,
  PKV_KERNEL_COMBINE = 3, /* the split-KV merge runs inside the decode kernel: no launches */
  PKV_KERNEL_H2O_SCORE = 4,
  PKV_KERNEL_H2O_SELECT = 5,
  PKV_KERNEL_TABLE_PATCH = 6,
  PKV_KERNEL_SWAP_COPY = 7, /* CPU swap-out / swap-in block copies */
  PKV_KERNEL_COMPACT = 8,   /* H2O compaction: row gather and score compaction */
  PKV_KERNEL_PREFIX = 9,    /* shared-prefix multi-query decode */
  PKV_KERNEL_COUNT = 10
} pkv_kernel_id;

/* Bit k of kernel_mask (k a pkv_kernel_id) brackets every launch of kernel k
 * with CUDA events on its stream; 0 turns timing off, -1 times every kernel.
 * Events between launches can add small gaps: time only what you read. */
pkv_status pkv_timing_enable(pkv_pool* pool, int32_t kernel_mask);
/* Synchronises on the recorded events and returns, per kernel id, the summed
 * device time (ms) and launch count since the last reset; then resets. */
pkv_status pkv_timing_read(pkv_pool* pool, double* total_ms_out /* [PKV_KERNEL_COUNT] */,
                           int64_t* launches_out /* [PKV_KERNEL_COUNT] */);
/* Bound (ns, within [1 ms, 60 s]; default 4 s) of every wait of the decode
 * kernel on its shared-memory stages, and of the keep-set selection's waits
 * on the score rows it streams into shared memory.  A wait that runs out sets
 * PKV_ERR_TIMEOUT in the status word; the warp (decode) or block (selection;
 * its keep_count is then 0) waits for its own copies in flight (bounded
 * again: 50 ms) and returns.  When those copies landed, the context stays
 * usable; when that second wait runs out too, the status word reports
 * PKV_ERR_UNDRAINED instead, and the context is not to be trusted. */
pkv_status pkv_set_wait_limit(pkv_pool* pool, int64_t wait_limit_ns);
/* Shared-prefix (cascade) decode ([PA] prefix sharing: a system prompt
 * reused by many requests, parallel sampling).  In decode over whole
 * keep-sets (PKV_MASK_FULL, num_splits = 0):
 *   - mode 1 (default): the planner pairs sequences that share leading full
 *     blocks; a pair's shared blocks are read once, by one warp attending
 *     for both (skipped when it would save under an eighth of the batch's
 *     block reads); each sequence's remaining blocks are read alone;
 *   - mode 2 (BF16 pools): sequences whose first block is the same physical
 *     block form groups (at least 4 sequences sharing at least 8 full
 *     blocks); a group's common prefix is read once per CTA of a multi-query
 *     kernel that attends for up to 128 query rows at once, and the rest of
 *     every sequence is read alone (no pairs); without groups, mode 2 pairs
 *     like mode 1;
 *   - mode 0: every sequence reads its own blocks.
 * All parts are merged by log-sum-exp like any split. */
pkv_status pkv_set_cascade(pkv_pool* pool, int32_t mode);
/* Per-channel scales ([PA] 量化原理 names per-channel and per-token scaling;
 * FP8 / INT8 pools).  Each (kv head, channel d) gets a fixed scale c_d, a
 * power of two (one exponent per channel, as in the OCP microscaling
 * formats), set by the caller -- from calibration data rounded to powers of
 * two, for instance -- while the pool holds no token; the per-token scales
 * stay on top of them.  An appended row x is divided by its channel scales
 * first, y_d = x_d / c_d (exact), and y is quantised per token as pkv_append
 * describes; the value stored is code_d * s * c_d.  Decode folds the K
 * scales into q once per (sequence, kv head) and the V scales into the
 * output, so it reads no extra bytes; with powers of two both products are
 * exact, and the numerics are those of plain per-token scaling.
 * Compaction, copy-on-write and CPU swap move codes and per-token scales as
 * before.
 *   k_channel, v_channel  device [n_kv_heads][head_dim] fp32, borrowed: they
 *                         must stay valid and unchanged while the pool is
 *                         used; both NULL returns to plain per-token scales.
 * Errors: PKV_ERR_UNSUPPORTED (a BF16 / FP32 pool); PKV_ERR_INVALID_ARG (a
 * sequence holds tokens, only one array given, or a scale that is not a
 * power of two in [2^-126, 2^127] -- checked with a synchronous copy to the
 * host); PKV_ERR_NO_DEVICE (a host-only pool). */
pkv_status pkv_set_channel_scales(pkv_pool* pool, const float* k_channel, const float* v_channel);
/* Test hook for the bound above: in the next decode on this pool, warp `warp`
 * of the grid arms its first stage without issuing the copies, so that wait
 * can only run out.  Outputs of that call are undefined; the status word
 * reports PKV_ERR_TIMEOUT. */
pkv_status pkv_test_starve_next_decode(pkv_pool* pool, int32_t warp);
/* Test hook for the same bound in the keep-set selection: in the next
 * pkv_h2o_select / pkv_policy_select on this pool, the block of the first
 * listed sequence never issues the first copy of its score row, so its wait
 * can only run out (when that row is streamed at all: budget < length).
 * That sequence's keep-set is undefined; the status word reports
 * PKV_ERR_TIMEOUT. */
pkv_status pkv_test_starve_next_select(pkv_pool* pool);
/* Test hooks for the decode planner (host only, no device work).
 * pkv_test_set_geometry: the launch geometry a host-only pool plans for --
 * SMs, warps per CTA of the one-sequence and of the two-sequence kernel (one
 * CTA per SM each) -- and the GQA group size.  pkv_test_plan_bytes: builds
 * the plan of a decode call (the same arguments) and copies its uploaded
 * bytes into `out` (cap bytes; *size gets the length) and into info[9] the
 * physical warps, CTAs, partial records, sequences per warp, and the counts
 * of pieces, merge items, empty items, group-prefix items and group-prefix
 * members (the sections of the uploaded plan, in that order, each starting
 * on a 32-byte boundary after the warp_begin array of warps + 1 entries);
 * general != 0 forces the general planner instead of the one-pass paths,
 * which must give the same bytes. */
pkv_status pkv_test_set_geometry(pkv_pool* pool, int32_t num_sms, int32_t warps_per_cta, int32_t pair_warps_per_cta,
                                 int32_t group);
pkv_status pkv_test_plan_bytes(pkv_pool* pool, int32_t n_seqs, const int32_t* seq_ids, int32_t mask_mode,
                               int32_t num_sinks, int32_t window, int32_t num_splits, int32_t general, void* out,
                               size_t cap, size_t* size, int32_t* info);

/* Test hook (host only): how the library would cut this list of queued
 * block copies (src, dst pairs, host) into waves that run one after another
 * (the copies inside a wave run in parallel).  starts_out (host, cap
 * entries) receives the index of each wave's first copy and, last, n_pairs;
 * *n_out gets the count (waves + 1; an empty list gives {0, 0}).  The
 * pool's own queue is untouched. */
pkv_status pkv_test_cow_waves(pkv_pool* pool, int32_t n_pairs, const int32_t* pairs, int32_t* starts_out,
                              int32_t cap, int32_t* n_out);

/* Test hook (host-only pools): queue_patches != 0 makes the pool queue the
 * block-table patches a device pool would send to its device table.  Each
 * call moves the patches queued so far into out (host, (flat index, value)
 * pairs in queue order, cap pairs), clears the queue (and the queued copies)
 * and gives their count in *n_out. */
pkv_status pkv_test_take_patches(pkv_pool* pool, int32_t queue_patches, int32_t* out, int32_t cap, int32_t* n_out);

/* Total kernel launches issued by this pool so far (all kernels). */
pkv_status pkv_launch_count(const pkv_pool* pool, int64_t* out);

const char* pkv_last_error(void);
const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
