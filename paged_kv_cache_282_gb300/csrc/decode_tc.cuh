// decode_tc.cuh -- decode attention over the paged KV cache, BF16, FP8-E4M3
// and INT8 KV, head_dim D in {64, 128}, GQA group G in {1, 2, 4, 8}; sm_103a.
// Included by one translation unit per head_dim, which instantiates the
// kernel for it.
//
// What it computes (pages: "KV Cache 与 PagedAttention：显存复用与长上下文推理",
// PagedAttention 的设计 -- decode loads KV block by block through the block
// table; "系统优化", Flash Attention -- tiled online softmax; "长上下文优化：
// 注意力稀疏化与 KV Cache 管理", GQA): for each (sequence, kv head) and the G
// query heads that share it, softmax(scale * q K^T) V over the kept keys.
//
// GB300 design:
//  - Work unit = one 16-token block of one kv head: a 16 x D chunk of K plus
//    the same for V, each contiguous in HBM.  The host cuts the concatenated
//    units of all (sequence, kv head) pairs into equal contiguous runs, one
//    per warp of a persistent grid (one CTA per SM), so ragged lengths balance
//    exactly.  A run that covers only part of its (sequence, kv head) writes a
//    partial record; the warp that writes the last record of a (sequence, kv
//    head) -- counted with one atomic per item -- merges them by
//    log-sum-exp, so no separate combine launch is needed.
//  - Every warp owns a private ring of shared-memory stages filled by TMA
//    (cp.async.bulk.tensor, 2-D tiles with rows of 128 bytes and the 128-byte
//    swizzle, so the fragment loads below are bank-conflict free) and
//    completed through mbarrier transaction counts.  Lane 0 refills a stage as
//    soon as the warp has consumed it; physical block ids for the next 32
//    units are fetched one batch ahead.  K / V that the call reads only once
//    are copied with an L2 evict-first policy, so they do not push the block
//    tables, plans, records and shared prefixes out of L2 (one-sequence rings:
//    a launch variant chosen per call; pair rings: per piece).
//  - Every K/V byte is read once per GQA group: the G query heads are the N
//    dimension of m16n8k16 tensor-core MMAs (S = K Q^T, then O^T = V^T P),
//    with fp32 accumulation.  The path is HBM-bound (4 flop/byte for BF16,
//    G = 4); the MMAs only keep instruction issue far below the memory time.
//  - FP8 / INT8: codes widen to fp16 in registers, exactly.  q is scaled by a
//    power of two per (sequence, head) so that its largest element lies in
//    [2^14, 2^15) before it is rounded to fp16 (no element can overflow, and
//    an element loses bits only when it is below 2^-24 of the largest); the
//    factor leaves the logit after the product, together with the token's K
//    scale.  The V scale enters the softmax weight through its log2: the
//    running maximum m is taken over logit + log2(v_scale), the weight
//    2^(logit + log2 v_scale - m) <= 1 is what the fp16 MMA multiplies the V
//    codes by, and l sums 2^(logit - m).  So the fp16 weights never overflow,
//    and a weight flushes to zero only when its V-scaled value is below 2^-24
//    of the largest one, whatever the magnitudes of q, K and V.
//  - Per-channel scales (FP8 / INT8 pools that have them; powers of two, so
//    the products are exact): the K channel scales multiply q once per run,
//    the V channel scales multiply the output; neither touches the per-unit
//    work.
//  - Every wait is bounded: after the limit the warp sets the status word,
//    drains its own copies in flight (bounded again; a drain that also runs
//    out sets a second bit) and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainTimeoutNs = 50000000ull;

// Geometry of a unit: one 16-token block of HG adjacent kv heads.
template <int KV, int NQ, int D, int HG>
struct TC {
  static constexpr int kEs = KV == 1 ? 2 : 1;          // bytes per element
  static constexpr int kRowBytes = D * kEs;            // one token of one kv head
  static constexpr int kHeadChunk = 16 * kRowBytes;    // K (or V) of one kv head of a block
  static constexpr int kChunkBytes = HG * kHeadChunk;  // K (or V) of one unit, contiguous in HBM
  static constexpr int kUPS = tc_ups(KV, NQ, D, HG);             // units per stage
  static constexpr int kUnitBytes = 2 * kChunkBytes;              // K then V of one unit
  static constexpr int kStageBytes = kUPS * kUnitBytes;
  static constexpr int kUnitScaleBytes = KV == 1 ? 0 : HG * 128;  // 16 K scales per head, then the V scales
  static constexpr int kScaleBytes = kUPS * kUnitScaleBytes;      // per stage
  static constexpr uint32_t kUnitTxBytes = kUnitBytes + kUnitScaleBytes;
  static constexpr int kWarps = tc_warps(KV, NQ, D, HG);
  static constexpr int kTeams = kWarps / HG;  // each team shares one ring of stages
  static constexpr int kStages = tc_stages(KV, NQ, D, HG);
  // TMA boxes per chunk, each 128 bytes wide: two for bf16 rows of 256 bytes
  // (HG = 1), one otherwise; one-byte codes with D = 64 are viewed as rows of
  // two tokens
  static constexpr int kBoxes = kRowBytes > 128 ? kRowBytes / 128 : 1;
  static constexpr int kBoxBytes = kChunkBytes / kBoxes;
  static constexpr bool kPairRows = kRowBytes < 128;
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------

// Release / acquire fence at GPU scope: orders a warp's partial-record stores
// before the arrival count that publishes them, and the count before the
// merging warp's loads of the other warps' records.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// NW consecutive 32-bit words (16 or 8 bytes) from shared memory
template <int NW>
__device__ __forceinline__ void load_words(uint32_t addr, uint32_t (&w)[NW]) {
  static_assert(NW == 4 || NW == 2, "16 or 8 bytes");
  if constexpr (NW == 4) {
    const uint4 v = lds128(addr);
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  } else {
    const uint2 v = lds64(addr);
    w[0] = v.x, w[1] = v.y;
  }
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// four E4M3 codes (byte 0 first) -> two f16x2 registers: lo = (byte 0, byte 1),
// hi = (byte 2, byte 3), lower half first.  Exact: E4M3 is a subset of fp16.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 c0, c1;\n\t"
      "mov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
}

// four INT8 codes (byte 0 first) -> two f16x2 registers, same layout as
// above.  Exact: with u = c + 128 in [1, 255], the fp16 bit pattern
// 0x6400 | u is 1024 + u (fp16 spacing is 1 on [1024, 2048)), and
// subtracting 1152 leaves c.
__device__ __forceinline__ void i8x4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = codes ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140), b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&x);
  hi = *reinterpret_cast<const uint32_t*>(&y);
}

// one-byte codes of the pool's type -> fp16 pairs
template <int KV>
__device__ __forceinline__ void codes4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  if (KV == 3)
    i8x4_to_f16x2x2(codes, lo, hi);
  else
    e4m3x4_to_f16x2x2(codes, lo, hi);
}

// 2^x and log2(x) with the hardware approximations (relative error ~2^-22;
// subnormal inputs and results flush to zero), used for the softmax weights.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory byte offset of byte x of token t inside a one-byte chunk of
// D codes per token, as TMA wrote it with the 128-byte swizzle (16-byte piece
// k of 128-byte row y sits at piece k ^ (y % 8)).  D = 128: one token a row.
// D = 64: two tokens a row (token t is the (t % 2)-th half of row t / 2).
template <int D>
__device__ __forceinline__ uint32_t ob_off(int t, int x) {
  if (D == 128) return (uint32_t)(t * 128 + ((((x >> 4) ^ t) & 7) << 4) + (x & 15));
  const int y = t >> 1, k = ((t & 1) << 2) | (x >> 4);
  return (uint32_t)(y * 128 + (((k ^ y) & 7) << 4) + (x & 15));
}

__device__ __forceinline__ bool kept(int j, int L, int mode, int S, int W) {
  if (j >= L) return false;
  if (mode == 0) return true;
  if (mode == 1) return (L - 1 - j) <= W;
  if ((long long)L <= (long long)S + W) return true;
  return j < S || j >= L - W;
}

// Walk a unit cursor (piece index, logical block) forward by n units.
__device__ __forceinline__ void advance(const Piece* __restrict__ P, int pe, int& ip, int& il, int n) {
  while (ip < pe) {
    const int end = P[ip].lblk_end;
    if (il + n < end) {
      il += n;
      return;
    }
    n -= end - il;
    ++ip;
    if (ip < pe) il = P[ip].lblk_begin;
  }
}

// Row coordinate r = (block * Hk + first kv head) * 16 of the unit `lane`
// positions past the cursor (a piece's kv_head names its unit's group of HG
// kv heads), or -1 past the end.  Two-sequence rings (PER_UNIT) return r when
// the unit is read once (Piece::stream_from) and -r - 2 otherwise.
template <int HG, bool PER_UNIT>
__device__ __forceinline__ int unit_row(const DecodeTCParams& p, int pe, int ip, int il, int lane) {
  advance(p.pieces, pe, ip, il, lane);
  if (ip >= pe) return -1;
  const Piece pc = p.pieces[ip];
  int blk = p.tables[(size_t)pc.seq_slot * p.max_blocks + il];
  if (blk < 0 || blk >= p.num_blocks) {
    atomicOr(p.status, kStatusBadBlock);
    p.status[1] = pc.seq_slot;
    p.status[2] = il;
    blk = 0;  // keep the copy in bounds; the status word reports the fault
  }
  const int row = (blk * p.n_kv_heads + pc.kv_head * HG) * kBlock;
  if (!PER_UNIT) return row;
  return il >= pc.stream_from ? row : -row - 2;
}

// Log-sum-exp merge of the partial records of one (sequence, kv head) by one
// warp (the last writer): M = max_p M_p, w_p = 2^(M_p - M),
// out = sum_p w_p O_p / sum_p w_p l_p, lse = (M + log2 sum_p w_p l_p) ln 2.
// Records are taken 32/G at a time: lane (j, h) = (lane / G, lane % G) owns
// the scalars of record j, head h, so every head is merged at once and all
// loads of a chunk are independent.  Each lane owns D/32 consecutive output
// columns.  Records written by other SMs are read through L2 (ld.global.cg).
// HG: kv heads of the item's unit (its row h belongs to kv head
// kv_head * HG + h / (G / HG)), for the per-channel V scales.
template <int G, int D, int HG = 1>
__device__ void merge_partials(const DecodeTCParams& p, const CombineItem it, int lane) {
  constexpr int PF = G * D + ((2 * G + 3) & ~3);
  constexpr int RPC = 32 / G;  // records per chunk
  constexpr int NV = D / 32;   // columns per lane
  const float* base = p.partials + (size_t)it.first_partial * PF;
  const int hl = lane % G, jl = lane / G;
  const int n = it.n_partials;
  float M = -INFINITY;
  for (int k0 = 0; k0 < n; k0 += RPC)
    if (k0 + jl < n) M = fmaxf(M, __ldcg(base + (size_t)(k0 + jl) * PF + G * D + hl));
#pragma unroll
  for (int off = 16; off >= G; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  float acc[G][NV];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < NV; ++e) acc[h][e] = 0.f;
  float lsum = 0.f;
  for (int k0 = 0; k0 < n; k0 += RPC) {
    float w = 0.f;
    if (k0 + jl < n) {
      const float* rec = base + (size_t)(k0 + jl) * PF;
      const float Mk = __ldcg(rec + G * D + hl);
      w = Mk == -INFINITY ? 0.f : exp2f(Mk - M);
      lsum += w * __ldcg(rec + G * D + G + hl);
    }
#pragma unroll
    for (int j = 0; j < RPC; ++j) {
      if (k0 + j >= n) break;
      const float* rec = base + (size_t)(k0 + j) * PF;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float wj = __shfl_sync(kFull, w, j * G + h);
        if (NV == 4) {
          const float4 o = __ldcg(reinterpret_cast<const float4*>(rec + h * D) + lane);
          acc[h][0] += wj * o.x;
          acc[h][1] += wj * o.y;
          acc[h][2] += wj * o.z;
          acc[h][3] += wj * o.w;
        } else {
          const float2 o = __ldcg(reinterpret_cast<const float2*>(rec + h * D) + lane);
          acc[h][0] += wj * o.x;
          acc[h][1] += wj * o.y;
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= G; off >>= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float l = __shfl_sync(kFull, lsum, h);  // lane h holds head h's total
    const float Mh = __shfl_sync(kFull, M, h);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const size_t row = (size_t)it.q_row * p.n_heads + it.kv_head * G + h;
    float cv[NV];  // per-channel V scales of this lane's columns (1 without them)
#pragma unroll
    for (int e = 0; e < NV; ++e)
      cv[e] = p.v_channel != nullptr ? p.v_channel[(size_t)(it.kv_head * HG + h / (G / HG)) * D + lane * NV + e] : 1.f;
    if (NV == 4) {
      uint2 packed;
      packed.x = pack_bf16(acc[h][0] * inv * cv[0], acc[h][1] * inv * cv[1]);
      packed.y = pack_bf16(acc[h][2] * inv * cv[2], acc[h][3] * inv * cv[3]);
      *reinterpret_cast<uint2*>(out + row * D + lane * 4) = packed;
    } else {
      *reinterpret_cast<uint32_t*>(out + row * D + lane * 2) =
          pack_bf16(acc[h][0] * inv * cv[0], acc[h][1] * inv * cv[1]);
    }
    if (lane == 0 && p.lse != nullptr) p.lse[row] = l > 0.f ? (Mh + log2f(l)) * kLn2 : -INFINITY;
  }
}

// Reports a wait that ran out (the team's leader also waits, bounded again,
// for the copies it has in flight into its team's stages -- the stages from
// `from` to `issued` in ring order -- and flags a drain that ran out too).
template <int S>
__device__ void fail_and_drain(const DecodeTCParams& p, uint32_t full, int from, int issued, bool leader, int gw,
                               int lane) {
  if (lane == 0) {
    atomicOr(p.status, kStatusTimeout);
    p.status[1] = gw;
  }
  if (!leader) return;
  bool drained = true;
  for (int v = from; v < issued; ++v)
    drained &= mbar_wait(full + 8 * (v % S), (uint32_t)((v / S) & 1), kDrainTimeoutNs);
  if (!drained && lane == 0) atomicOr(p.status, kStatusUndrained);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// GP: query heads per kv head.  HG: kv heads per unit = warps of a team.  A
// team shares one ring of stages, each holding a unit (one block of HG
// adjacent kv heads); its warp jh attends with kv head jh of every unit for
// that head's GP query heads, so a unit's K and V arrive as two contiguous
// pieces of HG chunks while every warp runs the one-head computation.  The
// plan names teams ("warps" of the plan) and units of HG heads, whose records
// hold GV = GP HG query heads.
// EF: one-sequence rings whose K / V copies all take the L2 evict-first
// policy (chosen per call on the host, DecodeTCParams::kv_evict_first).
template <int KV, int GP, int HG, int NQ, int D, bool EF = false>
__global__ void __launch_bounds__(TC<KV, NQ, D, HG>::kWarps * 32, 1)
    decode_tc_kernel(const __grid_constant__ DecodeTCParams p) {
  using C = TC<KV, NQ, D, HG>;
  constexpr int S = C::kStages;
  constexpr int KT = D / 16;  // k16 steps of QK, m16 tiles of PV
  constexpr int GV = GP * HG;
  constexpr int T = C::kTeams;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int team = wl / HG, jh = wl % HG;
  const bool leader = jh == 0;  // issues the team's copies
  const int gw = blockIdx.x * T + team;

  const uint32_t data = smem_addr(base) + (uint32_t)(team * S * C::kStageBytes);
  const uint32_t scl = smem_addr(base) + (uint32_t)(T * S * C::kStageBytes + team * S * C::kScaleBytes);
  const uint32_t full = smem_addr(base) + (uint32_t)(T * S * (C::kStageBytes + C::kScaleBytes) + team * S * 16);
  const uint32_t empty = full + 8 * S;  // HG arrivals: every warp of the team is done with the stage
  if (threadIdx.x == 0) {
    for (int s = 0; s < T * S; ++s) {
      const uint32_t f = smem_addr(base) + (uint32_t)(T * S * (C::kStageBytes + C::kScaleBytes) + (s / S) * S * 16 +
                                                     (s % S) * 8);
      mbar_init(f, 1);
      mbar_init(f + 8 * S, HG);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (gw >= p.total_warps) return;
  // (sequence, unit head group) pairs with an empty keep-set: zeros and -inf
  for (int e = gw; e < p.n_empty; e += p.total_warps) {
    const EmptyItem it = p.empty[e];
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    for (int h = 0; h < GP; ++h) {
      const size_t row = ((size_t)it.q_row * p.n_heads + it.kv_head * GV + jh * GP + h);
      if (D == 128)
        *reinterpret_cast<uint2*>(out + row * D + lane * 4) = make_uint2(0u, 0u);
      else
        *reinterpret_cast<uint32_t*>(out + row * D + lane * 2) = 0u;
      if (lane == 0 && p.lse != nullptr) p.lse[row] = -INFINITY;
    }
  }
  const int pb = p.warp_begin[gw], pe = p.warp_begin[gw + 1];
  if (pb >= pe) return;

  const int r = lane >> 2, c = lane & 3;
  const int Hk = p.n_kv_heads, H = p.n_heads;
  const float sl2 = p.scale * kLog2e;

  // total units of this team
  int n_units = 0;
  for (int k = pb; k < pe; ++k) n_units += p.pieces[k].lblk_end - p.pieces[k].lblk_begin;

  // issue side (the leader warp): rows of the current and the next batch of 32 units
  int bip = pb, bil = p.pieces[pb].lblk_begin;  // cursor at the current batch start
  int cur_rows = -1, next_rows = -1, nip = bip, nil = bil;
  if (leader) {
    cur_rows = unit_row<HG, NQ == 2>(p, pe, bip, bil, lane);
    advance(p.pieces, pe, nip, nil, 32);
    next_rows = unit_row<HG, NQ == 2>(p, pe, nip, nil, lane);
  }
  int batch_base = 0;
  int issued = 0, ist = 0;  // units issued; the stage the next stage of units goes to
  // parity of that stage's empty barrier to wait for: refill v (teams: one
  // unit per stage) waits for the consumption of unit v - S, phase (v / S - 1)
  // of the barrier; the S first issues wait for nothing and wrap the stage
  // index once, so start at 1
  uint32_t iph = 1;

  const uint64_t kv_policy = l2_evict_first_policy();
  // TMA y coordinate of a unit's chunk: token rows, or pairs of tokens
  auto ycoord = [](int row) { return C::kPairRows ? row >> 1 : row; };
  // leader warp, all lanes: fills the next stage with the next (up to) kUPS
  // units of the stream; lane 0 issues the copies.  Returns the units issued
  // (0 past the end of the stream) or -1 when the wait for the team to
  // release the stage ran out.
  auto issue = [&]() -> int {
    const int v0 = issued;
    if (v0 >= n_units) return 0;
    const int nu = min(C::kUPS, n_units - v0);
    const int st = ist;
    bool ok = true;
    if (HG > 1 && v0 >= S) ok = mbar_wait(empty + 8 * st, iph, p.wait_limit_ns);  // lanes agree
    if (++ist == S) {
      ist = 0;
      iph ^= 1u;
    }
    if (!ok) return -1;
    int rows[C::kUPS];
#pragma unroll
    for (int j = 0; j < C::kUPS; ++j) {
      rows[j] = -1;
      if (j < nu) {
        const int v = v0 + j;
        if (v - batch_base >= 32) {
          batch_base += 32;
          cur_rows = next_rows;
          advance(p.pieces, pe, nip, nil, 32);
          next_rows = unit_row<HG, NQ == 2>(p, pe, nip, nil, lane);
        }
        rows[j] = __shfl_sync(kFull, cur_rows, v - batch_base);  // encoded as unit_row returns it
      }
    }
    issued = v0 + nu;
    if (lane == 0) {
      const uint32_t bar = full + 8 * st;
      mbar_expect_tx(bar, (uint32_t)nu * C::kUnitTxBytes);
      if (v0 == 0 && gw == p.starve_warp) return nu;  // test hook: this stage never completes
#pragma unroll
      for (int j = 0; j < C::kUPS; ++j) {
        if (j >= nu) break;
        // read once by this call: the copies may leave L2 first (the pair
        // rings decide per unit, the one-sequence rings per call, as EF)
        const bool once = NQ == 2 ? rows[j] >= 0 : EF;
        const int row = NQ == 2 && rows[j] < 0 ? -rows[j] - 2 : rows[j];
        const uint32_t dst = data + (uint32_t)(st * C::kStageBytes + j * C::kUnitBytes);
        const int y = ycoord(row);
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b) {
          if (once) {
            tma_load_2d_hint(dst + C::kBoxBytes * b, &p.tmap_k, 64 * b, y, bar, kv_policy);
            tma_load_2d_hint(dst + C::kChunkBytes + C::kBoxBytes * b, &p.tmap_v, 64 * b, y, bar, kv_policy);
          } else {
            tma_load_2d(dst + C::kBoxBytes * b, &p.tmap_k, 64 * b, y, bar);
            tma_load_2d(dst + C::kChunkBytes + C::kBoxBytes * b, &p.tmap_v, 64 * b, y, bar);
          }
        }
        if (KV != 1) {
          const uint32_t sd = scl + (uint32_t)(st * C::kScaleBytes + j * C::kUnitScaleBytes);
          bulk_load(sd, p.k_scale + row, HG * 64, bar);
          bulk_load(sd + HG * 64, p.v_scale + row, HG * 64, bar);
        }
      }
    }
    return nu;
  };

  if (leader)
    for (int s0 = 0; s0 < S; ++s0)
      if (issue() <= 0) break;

  // per-lane fragment address pieces
  const int mi = lane >> 3, rr = lane & 7;
  // bf16 K (ldmatrix, non-transposed): matrices (tok 0-7|8-15) x (d lo|hi 8)
  const uint32_t k_row_off = (uint32_t)((rr + ((mi & 1) << 3)) * 128);
  const int k_hi = mi >> 1;
  // bf16 V (ldmatrix, transposed): matrices (d lo|hi 8) x (tok 0-7|8-15)
  const uint32_t v_row_off = (uint32_t)((rr + ((mi >> 1) << 3)) * 128);
  const int v_hi = mi & 1;
  // this warp's kv head within each unit: its K / V chunks and scales
  const uint32_t head_off = (uint32_t)(jh * C::kHeadChunk), head_scl = (uint32_t)(jh * 64);

  // Per sequence t of the piece (t = 1 only in the two-sequence variant):
  // Q^T fragments, O^T accumulators, the softmax state of columns 2c, 2c+1,
  // and (one-byte codes) the per-column factors that undo q's scaling.
  uint32_t qf[NQ][KT][2];
  float o[NQ][KT][4];
  float m0[NQ], m1[NQ], l0[NQ], l1[NQ];
  float sl2c[NQ][2], lgc[NQ][2];
  bool run_open = false, two = false;
  int u = 0, cst = 0;  // units consumed; the stage of the next one
  uint32_t cph = 0;    // the phase that stage completes next

  for (int pi = pb; pi < pe; ++pi) {
    const Piece pc = p.pieces[pi];
    const int g = pc.kv_head * HG + jh, L = pc.ctx_len;  // this warp's kv head
    // blocks whose every token is kept: [wb0, wb1) (the tail of the keep-set)
    // and [0, wsb) (blocks wholly inside the sinks); all other blocks test
    // their tokens one by one
    int wb0 = 0, wsb = 0;
    const int wb1 = L / kBlock;
    if (p.mask_mode == 1) {
      wb0 = max(0, (L - 1 - p.window + kBlock - 1) / kBlock);
    } else if (p.mask_mode == 2 && (long long)L > (long long)p.num_sinks + p.window) {
      wb0 = (L - p.window + kBlock - 1) / kBlock;
      wsb = p.num_sinks / kBlock;
    }
    if (!run_open) {
      two = NQ == 2 && pc.q_row1 >= 0;
      // Q^T fragments (B operand): rows k = head-dim slots, column n = query head r
      const int h = g * GP + r;
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        const int qr = t == 0 ? pc.q_row : pc.q_row1;
        const bool valid = r < GP && qr >= 0;
        const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)(valid ? qr : 0) * H + (valid ? h : 0)) * D;
        if (KV == 1) {
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            qf[t][kk][0] = valid ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * c) : 0u;
            qf[t][kk][1] = valid ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * c) : 0u;
          }
          sl2c[t][0] = sl2c[t][1] = sl2;
          lgc[t][0] = lgc[t][1] = p.scale;
        } else {
          // one-byte codes: k-slot 2c+e <-> d = (D/4)c + 4kk + e, slot 2c+8+e <-> d + 2;
          // q scaled by 2^eq so that max |q| lies in [2^14, 2^15), then rounded to fp16
          // (per-channel K scales c: the code products need q * c, formed in fp32)
          uint2 raw[KT];
          const float* kch = p.k_channel != nullptr ? p.k_channel + (size_t)g * D + (D / 4) * c : nullptr;
          auto qval = [&](int kk, int e) {  // element (D/4)c + 4kk + e of q (times c)
            const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(e < 2 ? &raw[kk].x : &raw[kk].y);
            const float v = (e & 1) ? __high2float(x) : __low2float(x);
            return kch != nullptr ? v * __ldg(kch + 4 * kk + e) : v;
          };
          float mx = 0.f;
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            raw[kk] = valid ? *reinterpret_cast<const uint2*>(qrow + (D / 4) * c + 4 * kk) : make_uint2(0u, 0u);
#pragma unroll
            for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(qval(kk, e)));
          }
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
          // floor(log2(mx)) from the exponent field (-127 for 0 or subnormal)
          const int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
          const int eq = min(126, 14 - e);  // >= -113: bf16 magnitudes stay below 2^128
          const float qs = __uint_as_float((uint32_t)(eq + 127) << 23);
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            qf[t][kk][0] = pack_f16(qval(kk, 0) * qs, qval(kk, 1) * qs);
            qf[t][kk][1] = pack_f16(qval(kk, 2) * qs, qval(kk, 3) * qs);
          }
          // columns 2c, 2c+1 are the heads of lanes 8c and 8c + 4
          const int eq0 = __shfl_sync(kFull, eq, 8 * c), eq1 = __shfl_sync(kFull, eq, 8 * c + 4);
          const float iq0 = __uint_as_float((uint32_t)(127 - eq0) << 23);
          const float iq1 = __uint_as_float((uint32_t)(127 - eq1) << 23);
          sl2c[t][0] = sl2 * iq0;
          sl2c[t][1] = sl2 * iq1;
          lgc[t][0] = p.scale * iq0;
          lgc[t][1] = p.scale * iq1;
        }
#pragma unroll
        for (int i = 0; i < KT; ++i) o[t][i][0] = o[t][i][1] = o[t][i][2] = o[t][i][3] = 0.f;
        m0[t] = m1[t] = -INFINITY;
        l0[t] = l1[t] = 0.f;
      }
      run_open = true;
    }

    for (int lb = pc.lblk_begin; lb < pc.lblk_end; ++lb, ++u) {
      const int st = cst;
      const int slot = C::kUPS == 1 ? 0 : u % C::kUPS;  // the unit's place in its stage
      if (slot == 0 && !mbar_wait(full + 8 * st, cph, p.wait_limit_ns)) {
        fail_and_drain<S>(p, full, u / C::kUPS + 1, (issued + C::kUPS - 1) / C::kUPS, leader, gw, lane);
        return;
      }
      const uint32_t kb = data + (uint32_t)(st * C::kStageBytes + slot * C::kUnitBytes) + head_off;
      const uint32_t vb = data + (uint32_t)(st * C::kStageBytes + slot * C::kUnitBytes + C::kChunkBytes) + head_off;

      // ---- S = K Q^T : rows = tokens, columns = query heads of the group
      float sa[NQ][4], sb[NQ][4];
#pragma unroll
      for (int t = 0; t < NQ; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[t][e] = sb[t][e] = 0.f;
      float ks_r = 1.f, ks_r8 = 1.f, lv_r = 0.f, lv_r8 = 0.f;
      if (KV == 1) {
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          const int c16 = 2 * kk + k_hi;  // 16-byte chunk index across the row
          uint32_t a[4];
          ldsm_x4(kb + (uint32_t)((c16 >> 3) * C::kBoxBytes) + k_row_off + (uint32_t)((((c16 & 7) ^ rr)) << 4), a);
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (t == 1 && !two) break;
            if (kk & 1)
              mma_bf16(sb[t], a, qf[t][kk][0], qf[t][kk][1]);
            else
              mma_bf16(sa[t], a, qf[t][kk][0], qf[t][kk][1]);
          }
        }
      } else {
        // tokens r and r + 8, codes d in [(D/4)c, (D/4)(c + 1))
        uint32_t tA[KT], tB[KT];
#pragma unroll
        for (int h16 = 0; h16 < KT / 4; ++h16) {
          const uint4 x = lds128(kb + ob_off<D>(r, (D / 4) * c + 16 * h16));
          const uint4 y = lds128(kb + ob_off<D>(r + 8, (D / 4) * c + 16 * h16));
          tA[4 * h16 + 0] = x.x, tA[4 * h16 + 1] = x.y, tA[4 * h16 + 2] = x.z, tA[4 * h16 + 3] = x.w;
          tB[4 * h16 + 0] = y.x, tB[4 * h16 + 1] = y.y, tB[4 * h16 + 2] = y.z, tB[4 * h16 + 3] = y.w;
        }
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          uint32_t a[4];
          codes4_to_f16x2x2<KV>(tA[kk], a[0], a[2]);
          codes4_to_f16x2x2<KV>(tB[kk], a[1], a[3]);
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (t == 1 && !two) break;
            if (kk & 1)
              mma_f16(sb[t], a, qf[t][kk][0], qf[t][kk][1]);
            else
              mma_f16(sa[t], a, qf[t][kk][0], qf[t][kk][1]);
          }
        }
        const uint32_t sc = scl + (uint32_t)(st * C::kScaleBytes + slot * C::kUnitScaleBytes) + head_scl;
        ks_r = lds_f32(sc + 4 * r);
        ks_r8 = lds_f32(sc + 4 * (r + 8));
        lv_r = lds_f32(sc + HG * 64 + 4 * r);
        lv_r8 = lds_f32(sc + HG * 64 + 4 * (r + 8));
      }

      // ---- mask (per token: the same for both sequences, whose shared
      // blocks are whole), logits out, online softmax (log2 units)
      const int tok0 = lb * kBlock + r, tok1 = tok0 + 8;
      // most units lie wholly inside the keep-set: their first and last
      // token decide it, and the per-token test is skipped
      const bool whole = (lb >= wb0 && lb < wb1) || lb < wsb;
      const bool k0 = whole || kept(tok0, L, p.mask_mode, p.num_sinks, p.window);
      const bool k1 = whole || kept(tok1, L, p.mask_mode, p.num_sinks, p.window);
      const bool h0v = 2 * c < GP, h1v = 2 * c + 1 < GP;
      if (KV != 1) {
        // log2 of the V scales of tokens r, r + 8; a masked slot may hold
        // unwritten memory, so its scale never reaches the arithmetic
        lv_r = k0 ? fast_log2(lv_r) : 0.f;
        lv_r8 = k1 ? fast_log2(lv_r8) : 0.f;
      }
      if (!whole && __ballot_sync(kFull, !(k0 && k1))) {
        // zero this head's V rows of masked tokens in the stage (0 * NaN = NaN)
        constexpr int kPieces = C::kRowBytes / 16;  // 16-byte pieces per token row
        constexpr int kRowsPerPass = 32 / kPieces;
        const int k = lane % kPieces;
#pragma unroll
        for (int t0 = 0; t0 < 16; t0 += kRowsPerPass) {
          const int t = t0 + lane / kPieces;
          if (!kept(lb * kBlock + t, L, p.mask_mode, p.num_sinks, p.window)) {
            uint32_t addr;
            if (KV == 1)
              addr = vb + (uint32_t)((k >> 3) * C::kBoxBytes + t * 128 + (((k & 7) ^ (t & 7)) << 4));
            else
              addr = vb + ob_off<D>(t, 16 * k);
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
          }
        }
        // order these generic-proxy writes before the TMA refill of this stage
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      uint32_t pb0[NQ], pb1[NQ];
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        if (t == 1 && !two) break;
        const float s0 = (sa[t][0] + sb[t][0]) * ks_r, s1 = (sa[t][1] + sb[t][1]) * ks_r;
        const float s2 = (sa[t][2] + sb[t][2]) * ks_r8, s3 = (sa[t][3] + sb[t][3]) * ks_r8;
        if (p.logits != nullptr) {
          const int qr = t == 0 ? pc.q_row : pc.q_row1;
          float* lg = p.logits + ((size_t)qr * Hk + g) * p.logits_stride * GP;
          if (k0 && h0v) lg[(size_t)tok0 * GP + 2 * c] = s0 * lgc[t][0];
          if (k0 && h1v) lg[(size_t)tok0 * GP + 2 * c + 1] = s1 * lgc[t][1];
          if (k1 && h0v) lg[(size_t)tok1 * GP + 2 * c] = s2 * lgc[t][0];
          if (k1 && h1v) lg[(size_t)tok1 * GP + 2 * c + 1] = s3 * lgc[t][1];
        }
        const float a0 = k0 ? s0 * sl2c[t][0] : -INFINITY, a1 = k0 ? s1 * sl2c[t][1] : -INFINITY;
        const float a2 = k1 ? s2 * sl2c[t][0] : -INFINITY, a3 = k1 ? s3 * sl2c[t][1] : -INFINITY;
        // one-byte codes: the maximum runs over logit + log2(v scale)
        const float b0 = KV == 1 ? a0 : a0 + lv_r, b1 = KV == 1 ? a1 : a1 + lv_r;
        const float b2 = KV == 1 ? a2 : a2 + lv_r8, b3 = KV == 1 ? a3 : a3 + lv_r8;
        float bm0 = fmaxf(b0, b2), bm1 = fmaxf(b1, b3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
          bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
        }
        const float mn0 = fmaxf(m0[t], bm0), mn1 = fmaxf(m1[t], bm1);
        const float z0 = mn0 == -INFINITY ? 0.f : mn0, z1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0[t] - z0), al1 = fast_exp2(m1[t] - z1);
        const float p0 = fast_exp2(b0 - z0), p1 = fast_exp2(b1 - z1), p2 = fast_exp2(b2 - z0),
                    p3 = fast_exp2(b3 - z1);
        if (KV == 1) {
          l0[t] = l0[t] * al0 + (p0 + p2);
          l1[t] = l1[t] * al1 + (p1 + p3);
        } else {
          // l sums the unscaled weights 2^(a - m) (capped at 2^126: only V
          // scales below 2^-100 could reach it)
          const float e0 = fast_exp2(fminf(a0 - z0, 126.f)), e1 = fast_exp2(fminf(a1 - z1, 126.f));
          const float e2 = fast_exp2(fminf(a2 - z0, 126.f)), e3 = fast_exp2(fminf(a3 - z1, 126.f));
          l0[t] = l0[t] * al0 + (e0 + e2);
          l1[t] = l1[t] * al1 + (e1 + e3);
        }
        m0[t] = mn0;
        m1[t] = mn1;
        if (__any_sync(kFull, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
          for (int i = 0; i < KT; ++i) {
            o[t][i][0] *= al0;
            o[t][i][1] *= al1;
            o[t][i][2] *= al0;
            o[t][i][3] *= al1;
          }
        }
        if (KV == 1) {
          pb0[t] = movmatrix_t(pack_bf16(p0, p1));
          pb1[t] = movmatrix_t(pack_bf16(p2, p3));
        } else {
          pb0[t] = movmatrix_t(pack_f16(p0, p1));
          pb1[t] = movmatrix_t(pack_f16(p2, p3));
        }
      }

      // ---- O^T += V^T P : rows = head-dim, columns = query heads
      if (KV == 1) {
#pragma unroll
        for (int i = 0; i < KT; ++i) {
          const int c16 = 2 * i + v_hi;
          uint32_t a[4];
          ldsm_x4_t(vb + (uint32_t)((c16 >> 3) * C::kBoxBytes) + v_row_off + (uint32_t)((((c16 & 7) ^ rr)) << 4), a);
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (t == 1 && !two) break;
            mma_bf16(o[t][i], a, pb0[t], pb1[t]);
          }
        }
      } else {
        // tokens 2c, 2c+1, 2c+8, 2c+9; codes d in [(D/8)r, (D/8)(r + 1))
        constexpr int NW = D / 32;  // code words per token
        uint32_t A4[NW], B4[NW], C4[NW], D4[NW];
        const int x = (D / 8) * r;
        load_words<NW>(vb + ob_off<D>(2 * c, x), A4);
        load_words<NW>(vb + ob_off<D>(2 * c + 1, x), B4);
        load_words<NW>(vb + ob_off<D>(2 * c + 8, x), C4);
        load_words<NW>(vb + ob_off<D>(2 * c + 9, x), D4);
        uint32_t pab[D / 8], pcd[D / 8];  // (token pair) values at d = (D/8)r + e
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const uint32_t lo = __byte_perm(A4[w], B4[w], 0x5140), hi = __byte_perm(A4[w], B4[w], 0x7362);
          codes4_to_f16x2x2<KV>(lo, pab[4 * w + 0], pab[4 * w + 1]);
          codes4_to_f16x2x2<KV>(hi, pab[4 * w + 2], pab[4 * w + 3]);
          const uint32_t lo2 = __byte_perm(C4[w], D4[w], 0x5140), hi2 = __byte_perm(C4[w], D4[w], 0x7362);
          codes4_to_f16x2x2<KV>(lo2, pcd[4 * w + 0], pcd[4 * w + 1]);
          codes4_to_f16x2x2<KV>(hi2, pcd[4 * w + 2], pcd[4 * w + 3]);
        }
#pragma unroll
        for (int i = 0; i < KT; ++i) {
          const uint32_t a[4] = {pab[i], pab[KT + i], pcd[i], pcd[KT + i]};
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (t == 1 && !two) break;
            mma_f16(o[t][i], a, pb0[t], pb1[t]);
          }
        }
      }
      if (slot == C::kUPS - 1 || u + 1 == n_units) {  // the stage is consumed
        __syncwarp();
        if (HG > 1 && lane == 0) mbar_arrive(empty + 8 * st);  // this warp is done with the stage
        if (++cst == S) {
          cst = 0;
          cph ^= 1u;
        }
        if (leader && issue() < 0) {
          fail_and_drain<S>(p, full, u / C::kUPS + 1, (issued + C::kUPS - 1) / C::kUPS, true, gw, lane);
          return;
        }
      }
    }

    if (pc.flags & kPieceLastOfRun) {
      // ---- finalise the run: this warp's GP rows of the output or of the
      // unit's partial record, per sequence
      int rec_items[NQ];  // merge item of each record written, or -1
#pragma unroll
      for (int t = 0; t < NQ; ++t) rec_items[t] = -1;
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        if (t == 1 && !two) break;
        float L0 = l0[t], L1 = l1[t];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          L0 += __shfl_xor_sync(kFull, L0, off);
          L1 += __shfl_xor_sync(kFull, L1, off);
        }
        const int qr = t == 0 ? pc.q_row : pc.q_row1;
        const int oi = t == 0 ? pc.out_index : pc.out_index1;
        const int ci = t == 0 ? pc.flags >> 1 : pc.item1;
        const int h0 = 2 * c, h1 = 2 * c + 1;
        auto dpos = [&](int i, int half) {
          return KV == 1 ? 16 * i + 8 * half + r : (D / 8) * r + (D / 16) * half + i;
        };
        if (oi < 0) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
          const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
          const size_t row0 = ((size_t)qr * H + g * GP + h0) * D;
          const size_t row1 = row0 + D;
          const float* vch = p.v_channel != nullptr ? p.v_channel + (size_t)g * D : nullptr;
#pragma unroll
          for (int i = 0; i < KT; ++i)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int d = dpos(i, half);
              const float cv = vch != nullptr ? __ldg(vch + d) : 1.f;  // per-channel V scale
              if (h0 < GP) out[row0 + d] = __float2bfloat16(o[t][i][2 * half] * inv0 * cv);
              if (h1 < GP) out[row1 + d] = __float2bfloat16(o[t][i][2 * half + 1] * inv1 * cv);
            }
          if (r == 0 && p.lse != nullptr) {
            const size_t li = (size_t)qr * H + g * GP;
            if (h0 < GP) p.lse[li + h0] = L0 > 0.f ? (m0[t] + log2f(L0)) * kLn2 : -INFINITY;
            if (h1 < GP) p.lse[li + h1] = L1 > 0.f ? (m1[t] + log2f(L1)) * kLn2 : -INFINITY;
          }
        } else {
          // record rows of this warp's heads: jh GP + h of the unit's GV
          float* rec = p.partials + (size_t)oi * partial_floats(GV, D);
          const int rh0 = jh * GP + h0, rh1 = jh * GP + h1;
#pragma unroll
          for (int i = 0; i < KT; ++i)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int d = dpos(i, half);
              if (h0 < GP) rec[rh0 * D + d] = o[t][i][2 * half];
              if (h1 < GP) rec[rh1 * D + d] = o[t][i][2 * half + 1];
            }
          if (r == 0) {
            if (h0 < GP) {
              rec[GV * D + rh0] = m0[t];
              rec[GV * D + GV + rh0] = L0;
            }
            if (h1 < GP) {
              rec[GV * D + rh1] = m1[t];
              rec[GV * D + GV + rh1] = L1;
            }
          }
          rec_items[t] = ci;
        }
      }
      // publish the run's records (one release fence for both sequences of a
      // pair) and count them -- every warp of the team counts its part, so an
      // item is complete after n_partials x HG arrivals; the warp that brings
      // the last one merges the (sequence, unit) (acquire before reading)
      if (rec_items[0] >= 0 || (NQ == 2 && rec_items[NQ - 1] >= 0)) {
        fence_acq_rel_gpu();
        __syncwarp();
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          const int ci = rec_items[t];
          if (ci < 0) continue;
          int last = 0;
          if (lane == 0) last = atomicAdd(p.counters + ci, 1) == p.combine[ci].n_partials * HG - 1;
          last = __shfl_sync(kFull, last, 0);
          if (last) {
            fence_acq_rel_gpu();
            merge_partials<GV, D, HG>(p, p.combine[ci], lane);
          }
        }
      }
      run_open = false;
    }
  }
}

// GP: query heads per kv head; HG: kv heads per unit (warps per team).
template <int KV, int GP, int HG, int NQ, int D>
cudaError_t launch_t(const DecodeTCParams& p, int ctas, cudaStream_t st) {
  constexpr int threads = TC<KV, NQ, D, HG>::kWarps * 32;
  constexpr size_t smem = tc_smem_bytes(KV, NQ, D, HG);
  if constexpr (NQ == 1 && HG == 1) {
    if (p.kv_evict_first) {
      decode_tc_kernel<KV, GP, HG, NQ, D, true><<<ctas, threads, smem, st>>>(p);
      return cudaGetLastError();
    }
  }
  decode_tc_kernel<KV, GP, HG, NQ, D><<<ctas, threads, smem, st>>>(p);
  return cudaGetLastError();
}

template <int KV, int GP, int HG, int NQ, int D>
cudaError_t prepare_t() {
  const int smem = (int)tc_smem_bytes(KV, NQ, D, HG);
  if constexpr (NQ == 1 && HG == 1) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_tc_kernel<KV, GP, HG, NQ, D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(decode_tc_kernel<KV, GP, HG, NQ, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int KV, int GP, int HG, int NQ, int D>
cudaError_t occupancy_t(int* n) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, decode_tc_kernel<KV, GP, HG, NQ, D>,
                                                       TC<KV, NQ, D, HG>::kWarps * 32, tc_smem_bytes(KV, NQ, D, HG));
}

// Expands X(KV, G, NQ) for every compiled (dtype, group, sequences per warp);
// each is built with units of one kv head and of tc_head_group heads.
#define PKV_FOR_VARIANTS(X)                                                                 \
  X(1, 1, 1) X(1, 2, 1) X(1, 4, 1) X(1, 8, 1) X(2, 1, 1) X(2, 2, 1) X(2, 4, 1) X(2, 8, 1)          \
  X(3, 1, 1) X(3, 2, 1) X(3, 4, 1) X(3, 8, 1) X(1, 1, 2) X(1, 2, 2) X(1, 4, 2) X(1, 8, 2)          \
  X(2, 1, 2) X(2, 2, 2) X(2, 4, 2) X(2, 8, 2) X(3, 1, 2) X(3, 2, 2) X(3, 4, 2) X(3, 8, 2)

}  // namespace

}  // namespace pkv
