// pkv_internal.h -- structures shared by the host planner and the kernels of
// libpkv.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

constexpr int kBlock = 16;   // tokens per physical block

// Device status word bits (pool status buffer, element 0).  kStatusUndrained:
// after a wait ran out, copies the waiting warp or block had issued were
// still in flight when it gave up waiting for them too.
enum : int32_t { kStatusTimeout = 1, kStatusBadBlock = 2, kStatusUndrained = 4 };

// Kv heads per unit of the tensor-core decode kernel (kv dtype 1 bf16, 2 FP8,
// 3 INT8; group size G; head_dim D).  A unit is one 16-token block of HG
// adjacent kv heads, which lie next to each other in the pool: HG is chosen
// so that a unit's K (and V) is one contiguous piece of at least 4 KB (DRAM
// serves small scattered pieces markedly slower), while its query heads, HG x
// G, still fit the 8 columns of one MMA tile.  The planner then sees n_kv_heads
// / HG kv heads of HG x G query heads each (the query heads of adjacent kv
// heads are adjacent too).  Pools whose n_kv_heads HG does not divide use 1.
#ifndef PKV_MAX_HEAD_GROUP
#define PKV_MAX_HEAD_GROUP 1
#endif
constexpr int tc_head_group(int kv, int G, int D) {
  const int chunk = kBlock * D * (kv == 1 ? 2 : 1);  // bytes of one head's K in a block
  int hg = chunk >= 4096 ? 1 : 4096 / chunk;
  while (hg > 1 && (hg * G > 8 || hg > PKV_MAX_HEAD_GROUP)) hg >>= 1;
  return hg;
}

// Geometry of the tensor-core decode kernel for a kv dtype, sequences per
// warp (nq), head_dim D and kv heads per unit (hg): warps per CTA (one CTA per
// SM), teams (hg warps sharing a ring of stages; the plan's "warps"), stages
// of each ring and dynamic shared memory.  One-head units keep a ring per
// warp (7 warps x 2 stages of 8 KB for bf16 head_dim 128: fewer, longer
// runs per SM stream faster than 12 x 2; 16 warps for one-byte codes, which
// the 64-split batch needs; 12 for bf16 at head_dim 64, 12 or 16
// otherwise); units of several heads fill about 200 KB with stages.
// Bytes of one unit in a stage: K then V of hg heads (+ their scales).
constexpr int tc_unit_bytes(int kv, int D, int hg) {
  return 2 * hg * kBlock * D * (kv == 1 ? 2 : 1) + (kv == 1 ? 0 : hg * 128);
}
#ifndef PKV_TEAM_WARPS
#define PKV_TEAM_WARPS 16  // warps per CTA of several-head units, one sequence per warp
#endif
#ifndef PKV_OB_WARPS  // one-head units of one-byte codes at head_dim 128, one sequence per warp
#define PKV_OB_WARPS 16
#endif
#ifndef PKV_OB_STAGES
#define PKV_OB_STAGES 2
#endif
#ifndef PKV_OB_UPS  // units per stage
#define PKV_OB_UPS 1
#endif
#ifndef PKV_BF_WARPS  // one-head units of bf16 at head_dim 128, one sequence per warp
#define PKV_BF_WARPS 7
#endif
#ifndef PKV_BF_STAGES
#define PKV_BF_STAGES 2
#endif
#ifndef PKV_BF_UPS
#define PKV_BF_UPS 1
#endif
#ifndef PKV_D64_BF_WARPS  // one-head units at head_dim 64, one sequence per warp: bf16
#define PKV_D64_BF_WARPS 12
#endif
#ifndef PKV_D64_OB_WARPS  // ... and one-byte codes
#define PKV_D64_OB_WARPS 16
#endif
#ifndef PKV_D64_STAGES
#define PKV_D64_STAGES 0  // 0: 2 for bf16, 3 for one-byte codes
#endif
#ifndef PKV_D64_UPS
#define PKV_D64_UPS 1
#endif
#ifndef PKV_KV_EVICT_FIRST  // allows the L2 evict-first policy on K / V copies read once per call
#define PKV_KV_EVICT_FIRST 1
#endif
#ifndef PKV_PAIR_WARPS  // two sequences per warp (shared-prefix pairs)
#define PKV_PAIR_WARPS 12
#endif
#ifndef PKV_PAIR_STAGES
#define PKV_PAIR_STAGES 0  // 0: 2 for bf16, 3 for one-byte codes
#endif
constexpr int tc_warps(int kv, int nq, int D, int hg) {
  return hg > 1                               ? (nq == 2 ? 12 : PKV_TEAM_WARPS / hg * hg)
         : nq == 2 && (D == 128 || kv != 1)   ? PKV_PAIR_WARPS
         : nq == 1 && D == 128 && kv != 1     ? PKV_OB_WARPS
         : nq == 1 && D == 128 && kv == 1     ? PKV_BF_WARPS
         : nq == 1                            ? (kv == 1 ? PKV_D64_BF_WARPS : PKV_D64_OB_WARPS)
         : D == 128 && kv == 1                ? 12
                                              : 16;
}
// Units per stage: a stage holds that many consecutive units of its ring's
// stream under one barrier (one-sequence rings only).
constexpr int tc_ups(int kv, int nq, int D, int hg) {
  return hg > 1 || nq == 2 ? 1 : D == 64 ? PKV_D64_UPS : kv != 1 ? PKV_OB_UPS : PKV_BF_UPS;
}
constexpr int tc_stage_bytes(int kv, int nq, int D, int hg) { return tc_ups(kv, nq, D, hg) * tc_unit_bytes(kv, D, hg); }
constexpr int tc_teams(int kv, int nq, int D, int hg) { return tc_warps(kv, nq, D, hg) / hg; }
#ifndef PKV_TEAM_STAGES
#define PKV_TEAM_STAGES 0  // 0: fill about 200 KB
#endif
constexpr int tc_stages(int kv, int nq, int D, int hg) {
  return hg == 1 ? (nq == 1 && D == 128 ? (kv != 1 ? PKV_OB_STAGES : PKV_BF_STAGES)
                  : nq == 1 && PKV_D64_STAGES > 0 ? PKV_D64_STAGES
                  : nq == 2 && PKV_PAIR_STAGES > 0 ? PKV_PAIR_STAGES
                  : kv != 1 && (nq == 2 || D == 64) ? 3 : 2)
         : PKV_TEAM_STAGES > 0 ? PKV_TEAM_STAGES
         : 204800 / (tc_teams(kv, nq, D, hg) * (tc_stage_bytes(kv, nq, D, hg) + 16)) < 2 ? 2
         : 204800 / (tc_teams(kv, nq, D, hg) * (tc_stage_bytes(kv, nq, D, hg) + 16)) > 6
             ? 6
             : 204800 / (tc_teams(kv, nq, D, hg) * (tc_stage_bytes(kv, nq, D, hg) + 16));
}
constexpr size_t tc_smem_bytes(int kv, int nq, int D, int hg) {
  return 1024 + (size_t)tc_teams(kv, nq, D, hg) * tc_stages(kv, nq, D, hg) * (size_t)(tc_stage_bytes(kv, nq, D, hg) + 16);
}

// One contiguous range of logical blocks of one (sequence, kv head), handled
// by one warp of the decode kernel.  Consecutive pieces of the same
// (sequence, kv head) inside one warp form a "run"; the run is finalised
// after the piece whose flags carry kPieceLastOfRun.  A run that does not
// cover its whole (sequence, kv head) writes a partial record; flags >> 1 is
// then the index of the merge item that owns the record.
enum : int32_t { kPieceLastOfRun = 1 };
struct Piece {
  int32_t seq_slot;    // block-table row
  int32_t q_row;       // batch index into q / out / lse / logits
  int32_t kv_head;
  int32_t lblk_begin;  // logical block range [begin, end)
  int32_t lblk_end;
  int32_t ctx_len;     // L: context length, current token included
  int32_t out_index;   // >= 0: partial record index; -1: write the final output
  int32_t flags;       // bit 0: last piece of its run; bits 31..1: merge item
  // A second sequence whose blocks [lblk_begin, lblk_end) are the same
  // physical blocks (shared-prefix decode); q_row1 = -1: none.  Its run
  // always ends in a partial record out_index1 of merge item item1.
  int32_t q_row1;
  int32_t out_index1;
  int32_t item1;
  // Logical blocks from this one on are read once by this call (no other
  // sequence holds them, or only the pair itself): their copies may leave L2
  // first.  lblk_end or more: none.  Read by the two-sequence rings; the
  // one-sequence rings take DecodeTCParams::kv_evict_first.
  int32_t stream_from;
};
static_assert(sizeof(Piece) == 48, "Piece layout");

// A (sequence, kv head) whose n_partials (>= 2) partial records, stored
// consecutively from first_partial, are merged by log-sum-exp.  The warp that
// writes the last of them (counted with an atomic per item) does the merge.
struct CombineItem {
  int32_t q_row, kv_head, first_partial, n_partials;
};

// Shared-prefix group work for the multi-query kernel: the logical blocks
// [lblk_begin, lblk_end) of kv head kv_head, which every member sequence
// holds as the same physical blocks (read through table_seq's table row),
// attended by all members' query heads at once.  Each member writes one
// partial record per item.
struct PrefixItem {
  int32_t kv_head, table_seq, lblk_begin, lblk_end, member_begin, n_members, pad0, pad1;
};
struct PrefixMember {
  int32_t q_row, out_index, item, pad;  // item: the merge item of (q_row, kv_head)
};

// A (sequence, kv head) with an empty keep-set: out = 0, lse = -inf.
struct EmptyItem {
  int32_t q_row, kv_head;
};

// One sequence of an H2O compaction: its count kept tokens move, in order,
// into the fresh blocks new_blocks[new_off ...].
struct CompactSeq {
  int32_t seq_slot, q_row, count, new_off, old_len, pad0, pad1, pad2;
};

// A keep-set rule: the first `sinks` positions, the last `window` positions,
// and the `heavy` highest scores among all positions (rank_all) or among the
// positions before the window.
struct SelPolicy {
  int32_t sinks, window, heavy, rank_all;
};

// Per-sequence row for kernels that walk one sequence at a time.
struct SeqRow {
  int32_t seq_slot, q_row, ctx_len, pad;
};

// Floats per partial record: O[G][D] (unnormalised), M[G] (log2 units),
// l[G], padded so that every record starts on a 16-byte boundary.
inline __host__ __device__ int partial_floats(int G, int D) { return G * D + ((2 * G + 3) & ~3); }

struct DecodeTCParams {
  CUtensorMap tmap_k;  // 2-D view of the K pool in 128-byte rows, 128B swizzle (see make_tensor_map)
  CUtensorMap tmap_v;
  const float* k_scale;  // FP8 only
  const float* v_scale;
  const int32_t* tables;
  int32_t max_blocks, num_blocks;
  int32_t n_heads, n_kv_heads;
  const void* q;
  void* out;
  float* lse;
  float* logits;
  int64_t logits_stride;
  const Piece* pieces;
  const int32_t* warp_begin;  // [total_warps + 1]
  int32_t total_warps;
  float* partials;
  const CombineItem* combine;  // merge items, with one arrival counter each
  int32_t* counters;           // zero at launch
  const EmptyItem* empty;
  int32_t n_empty;
  float scale;       // natural-unit softmax scale
  int32_t mask_mode, num_sinks, window;
  int32_t* status;
  uint64_t wait_limit_ns;  // bound of every mbarrier wait
  int32_t starve_warp;     // >= 0: that warp arms its first stage but issues no copy (wait-expiry test)
  const PrefixItem* prefix_items;  // the multi-query kernel's work (one CTA each)
  const PrefixMember* prefix_members;
  int32_t n_prefix_items;
  const float* k_channel;  // per-channel scales [Hk][D] of an FP8 / INT8 pool, or nullptr
  const float* v_channel;
  int32_t kv_evict_first;  // one-sequence rings: launch the variant whose K / V copies are evict-first in L2
};

struct DecodeF32Params {
  const float* k_pool;
  const float* v_pool;
  const int32_t* tables;
  int32_t max_blocks, num_blocks;
  int32_t n_heads, n_kv_heads, head_dim;
  const SeqRow* rows;
  int32_t n_seqs;
  const float* q;
  float* out;
  float* lse;
  float* logits;
  int64_t logits_stride;
  float scale;
  int32_t mask_mode, num_sinks, window;
  int32_t* status;
};

// ---- kernel launchers (defined in the .cu files) -------------------------

// Tensor-core decode: kv_dtype 1 = bf16, 2 = FP8, 3 = INT8; nq = 1, or 2 for
// the variant whose pieces may carry a second sequence over shared blocks;
// one set per head_dim (64, 128).  Return the launch / attribute error.
// G is the kv head's group size; hg (1 or tc_head_group) the kv heads per unit.
cudaError_t launch_decode_tc_d64(int kv_dtype, int G, int hg, int nq, const DecodeTCParams& p, int grid_ctas,
                                 cudaStream_t stream);
cudaError_t launch_decode_tc_d128(int kv_dtype, int G, int hg, int nq, const DecodeTCParams& p, int grid_ctas,
                                  cudaStream_t stream);
cudaError_t decode_tc_prepare_d64(int kv_dtype, int G, int hg, int nq);
cudaError_t decode_tc_prepare_d128(int kv_dtype, int G, int hg, int nq);
cudaError_t decode_tc_occupancy_d64(int kv_dtype, int G, int hg, int nq, int* ctas_per_sm);
cudaError_t decode_tc_occupancy_d128(int kv_dtype, int G, int hg, int nq, int* ctas_per_sm);
inline cudaError_t launch_decode_tc(int kv_dtype, int G, int hg, int nq, int D, const DecodeTCParams& p,
                                    int grid_ctas, cudaStream_t stream) {
  return D == 64 ? launch_decode_tc_d64(kv_dtype, G, hg, nq, p, grid_ctas, stream)
                 : launch_decode_tc_d128(kv_dtype, G, hg, nq, p, grid_ctas, stream);
}
// sets the dynamic shared-memory attribute
inline cudaError_t decode_tc_prepare(int kv_dtype, int G, int hg, int nq, int D) {
  return D == 64 ? decode_tc_prepare_d64(kv_dtype, G, hg, nq) : decode_tc_prepare_d128(kv_dtype, G, hg, nq);
}
inline cudaError_t decode_tc_occupancy(int kv_dtype, int G, int hg, int nq, int D, int* ctas_per_sm) {
  return D == 64 ? decode_tc_occupancy_d64(kv_dtype, G, hg, nq, ctas_per_sm)
                 : decode_tc_occupancy_d128(kv_dtype, G, hg, nq, ctas_per_sm);
}
// Shared-prefix multi-query kernel (bf16 KV, head_dim 128): one CTA per PrefixItem.
cudaError_t launch_prefix_decode(int G, const DecodeTCParams& p, cudaStream_t stream);
cudaError_t prefix_decode_prepare(int G);
constexpr int kPrefixRowsPerCta = 128;  // 8 warps x 16 query rows


cudaError_t launch_decode_f32(const DecodeF32Params& p, cudaStream_t stream);

cudaError_t launch_block_copy(const int32_t* pairs, int n_pairs, const void* src_k, const void* src_v,
                              const float* src_ks, const float* src_vs, void* dst_k, void* dst_v, float* dst_ks,
                              float* dst_vs, size_t block_bytes, size_t scale_floats, cudaStream_t stream);
cudaError_t launch_cow_copy(const int32_t* pairs, int n_pairs, void* k_pool, void* v_pool,
                            float* k_scale, float* v_scale, size_t block_bytes,
                            size_t scale_floats_per_block, cudaStream_t stream);

cudaError_t launch_table_patch(const int32_t* patches, int n_patches, int32_t* tables,
                               cudaStream_t stream);

// Append (scatter / FP8 quantise) of new rows, plus the block-table patches
// queued with it.  Up to kInlineAppend slots and patches travel inside the
// kernel parameters; larger lists come from device memory.
constexpr int kInlineAppend = 256;
struct AppendArgs {
  int kv_dtype, n_tokens, n_patches, Hk, D;
  const int64_t* slots;     // device, or nullptr: inline_slots
  const int32_t* patches;   // device (index, value) pairs, or nullptr: inline_patches
  const void* k_new;
  const void* v_new;
  void* k_pool;
  void* v_pool;
  float* k_scale;
  float* v_scale;
  const float* k_channel;  // per-channel scales [Hk][D] (FP8 / INT8), or nullptr
  const float* v_channel;
  int32_t* tables;
  int64_t inline_slots[kInlineAppend];
  int32_t inline_patches[2 * kInlineAppend];
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

cudaError_t launch_h2o_score(const SeqRow* rows, int n_seqs, int n_heads, int n_kv_heads,
                             const float* logits, int64_t logits_stride, const float* lse,
                             int mask_mode, int num_sinks, int window, float* acc,
                             int64_t acc_stride, int max_keep, cudaStream_t stream);

cudaError_t launch_compact_gather(const CompactSeq* seqs, int n, int max_count, const int32_t* new_blocks,
                                  const int32_t* tables, int max_blocks, int num_blocks, const int32_t* keep_idx,
                                  int64_t keep_stride, int Hk, int row_bytes, void* k_pool, void* v_pool, float* k_scale,
                                  float* v_scale, int32_t* status, cudaStream_t stream);
cudaError_t launch_compact_scores(const CompactSeq* seqs, int n, const int32_t* keep_idx, int64_t keep_stride,
                                  float* acc, int64_t acc_stride, cudaStream_t stream);

cudaError_t launch_h2o_select(const SeqRow* rows, int n_seqs, const float* acc, int64_t acc_stride,
                              const SelPolicy& pol, int32_t* keep_idx, int64_t keep_stride, int32_t* keep_count,
                              int32_t* status, uint64_t wait_limit_ns, bool starve_first, cudaStream_t stream);

}  // namespace pkv

// ---- decode with caller-supplied device regions (no library allocation) ----
struct pkv_pool;
namespace pkv {
// Sets the message pkv_last_error() returns on this thread.
void set_error(const char* msg);
// Runs the bf16 / FP8 decode of pkv_decode_attn, staging every host-built
// array (queued copy-on-write pairs and table patches, the work plan) with
// one pageable copy into `plan_dev` and keeping the split-KV partial records
// in `partials_dev`.  Allocates no device or pinned memory.
int decode_attn_into(pkv_pool* p, void* stream, int32_t n, const int32_t* ids, const void* q, float scale,
                     int32_t mode, int32_t S, int32_t W, int32_t num_splits, void* out, float* lse, float* logits,
                     int64_t logits_stride, void* plan_dev, size_t plan_cap, void* partials_dev, size_t partials_cap);
}  // namespace pkv
