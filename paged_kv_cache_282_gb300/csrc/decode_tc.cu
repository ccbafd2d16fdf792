// decode_tc.cu -- decode attention over the paged KV cache, BF16, FP8-E4M3
// and INT8 KV, head_dim 128, GQA group G in {1, 2, 4, 8}; sm_103a.
//
// What it computes (pages: "KV Cache 与 PagedAttention：显存复用与长上下文推理",
// PagedAttention 的设计 -- decode loads KV block by block through the block
// table; "系统优化", Flash Attention -- tiled online softmax; "长上下文优化：
// 注意力稀疏化与 KV Cache 管理", GQA): for each (sequence, kv head) and the G
// query heads that share it, softmax(scale * q K^T) V over the kept keys.
//
// GB300 design:
//  - Work unit = one 16-token block of one kv head: a 4 KB (BF16) or 2 KB
//    (FP8) K chunk plus the same for V, each contiguous in HBM.  The host cuts
//    the concatenated units of all (sequence, kv head) pairs into equal
//    contiguous runs, one per warp of a persistent grid (one CTA per SM), so
//    ragged lengths balance exactly.  A run that covers only part of its
//    (sequence, kv head) writes a partial record; the warp that writes the
//    last record of a (sequence, kv head) -- counted with one atomic per item
//    -- merges them by log-sum-exp, so no separate combine launch is needed.
//  - Every warp owns a private ring of shared-memory stages filled by TMA
//    (cp.async.bulk.tensor, 2-D tiles of 16 rows x 128 bytes with the 128-byte
//    swizzle, so the fragment loads below are bank-conflict free) and
//    completed through mbarrier transaction counts.  Lane 0 refills a stage as
//    soon as the warp has consumed it; physical block ids for the next 32
//    units are fetched one batch ahead.
//  - Every K/V byte is read once per GQA group: the G query heads are the N
//    dimension of m16n8k16 tensor-core MMAs (S = K Q^T, then O^T = V^T P),
//    with fp32 accumulation.  The path is HBM-bound (4 flop/byte for BF16,
//    G = 4); the MMAs only keep instruction issue far below the memory time.
//  - FP8 / INT8: codes are widened to fp16 in registers (exact); the per-token K
//    scale multiplies the logit, and the per-token V scale multiplies the
//    softmax weight before it is rounded to fp16 (the running max and the sum
//    l are those of the unscaled weights).
//  - Every wait is bounded: after about 4 s the warp sets the status word,
//    drains its own copies in flight (bounded again) and returns.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainTimeoutNs = 50000000ull;

template <int KV, int NQ>
struct TC;
template <>
struct TC<1, 1> {  // BF16
  static constexpr int kWarps = 12, kStages = 2;
  static constexpr int kStageBytes = 8192;  // K: 2 swizzled boxes of 2 KB, V: same
  static constexpr int kScaleBytes = 0;
  static constexpr uint32_t kTxBytes = 8192;
};
template <>
struct TC<2, 1> {  // FP8 E4M3: half-size units, so twice the warps to keep enough in flight
  static constexpr int kWarps = 16, kStages = 2;
  static constexpr int kStageBytes = 4096;  // K: one swizzled box of 2 KB, V: same
  static constexpr int kScaleBytes = 128;   // 16 K scales + 16 V scales
  static constexpr uint32_t kTxBytes = 4096 + 128;
};
// Two sequences per warp: twice the accumulators.  12 warps at 168 registers
// (a little spilled) beat 8 warps at 243 with deeper rings: the pairs are
// latency-bound, and more warps hide more of it.
template <>
struct TC<1, 2> {
  static constexpr int kWarps = 12, kStages = 2;
  static constexpr int kStageBytes = 8192;
  static constexpr int kScaleBytes = 0;
  static constexpr uint32_t kTxBytes = 8192;
};
template <>
struct TC<2, 2> {
  static constexpr int kWarps = 12, kStages = 3;
  static constexpr int kStageBytes = 4096;
  static constexpr int kScaleBytes = 128;
  static constexpr uint32_t kTxBytes = 4096 + 128;
};

// INT8 codes: the same geometry as FP8
template <int NQ>
struct TC<3, NQ> : TC<2, NQ> {};

template <int KV, int NQ>
constexpr size_t smem_bytes() {
  using C = TC<KV, NQ>;
  return 1024 + (size_t)C::kWarps * C::kStages * (C::kStageBytes + C::kScaleBytes) + (size_t)C::kWarps * C::kStages * 8;
}

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

// 2^x with the hardware approximation (relative error ~2^-22; subnormal
// results flush to zero), used for the softmax weights.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// Row coordinate (block * Hk + kv_head) * 16 of the unit `lane` positions past
// the cursor, or -1 past the end.
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
  return (blk * p.n_kv_heads + pc.kv_head) * kBlock;
}

// Log-sum-exp merge of the partial records of one (sequence, kv head) by one
// warp (the last writer): M = max_p M_p, w_p = 2^(M_p - M),
// out = sum_p w_p O_p / sum_p w_p l_p, lse = (M + log2 sum_p w_p l_p) ln 2.
// Records are taken 32/G at a time: lane (j, h) = (lane / G, lane % G) owns
// the scalars of record j, head h, so every head is merged at once and all
// loads of a chunk are independent.  Records written by other SMs are read
// through L2 (ld.global.cg).
template <int G>
__device__ void merge_partials(const DecodeTCParams& p, const CombineItem it, int lane) {
  constexpr int PF = G * 128 + ((2 * G + 3) & ~3);
  constexpr int RPC = 32 / G;  // records per chunk
  const float* base = p.partials + (size_t)it.first_partial * PF;
  const int hl = lane % G, jl = lane / G;
  const int n = it.n_partials;
  float M = -INFINITY;
  for (int k0 = 0; k0 < n; k0 += RPC)
    if (k0 + jl < n) M = fmaxf(M, __ldcg(base + (size_t)(k0 + jl) * PF + G * 128 + hl));
#pragma unroll
  for (int off = 16; off >= G; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  float4 acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
  for (int k0 = 0; k0 < n; k0 += RPC) {
    float w = 0.f;
    if (k0 + jl < n) {
      const float* rec = base + (size_t)(k0 + jl) * PF;
      const float Mk = __ldcg(rec + G * 128 + hl);
      w = Mk == -INFINITY ? 0.f : exp2f(Mk - M);
      lsum += w * __ldcg(rec + G * 128 + G + hl);
    }
#pragma unroll
    for (int j = 0; j < RPC; ++j) {
      if (k0 + j >= n) break;
      const float* rec = base + (size_t)(k0 + j) * PF;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float wj = __shfl_sync(kFull, w, j * G + h);
        const float4 o = __ldcg(reinterpret_cast<const float4*>(rec + h * 128) + lane);
        acc[h].x += wj * o.x;
        acc[h].y += wj * o.y;
        acc[h].z += wj * o.z;
        acc[h].w += wj * o.w;
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
    uint2 packed;
    packed.x = pack_bf16(acc[h].x * inv, acc[h].y * inv);
    packed.y = pack_bf16(acc[h].z * inv, acc[h].w * inv);
    *reinterpret_cast<uint2*>(out + row * 128 + lane * 4) = packed;
    if (lane == 0 && p.lse != nullptr) p.lse[row] = l > 0.f ? (Mh + log2f(l)) * kLn2 : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int KV, int G, int NQ>
__global__ void __launch_bounds__(TC<KV, NQ>::kWarps * 32, 1)
    decode_tc_kernel(const __grid_constant__ DecodeTCParams p) {
  using C = TC<KV, NQ>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int gw = blockIdx.x * C::kWarps + wl;
  if (gw >= p.total_warps) return;
  // (sequence, kv head) pairs with an empty keep-set: zeros and -inf
  for (int e = gw; e < p.n_empty; e += p.total_warps) {
    const EmptyItem it = p.empty[e];
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    for (int h = 0; h < G; ++h) {
      const size_t row = ((size_t)it.q_row * p.n_heads + it.kv_head * G + h);
      *reinterpret_cast<uint2*>(out + row * 128 + lane * 4) = make_uint2(0u, 0u);
      if (lane == 0 && p.lse != nullptr) p.lse[row] = -INFINITY;
    }
  }
  const int pb = p.warp_begin[gw], pe = p.warp_begin[gw + 1];
  if (pb >= pe) return;

  const uint32_t data = smem_addr(base) + (uint32_t)(wl * S * C::kStageBytes);
  const uint32_t scl = smem_addr(base) + (uint32_t)(C::kWarps * S * C::kStageBytes + wl * S * C::kScaleBytes);
  const uint32_t bars =
      smem_addr(base) + (uint32_t)(C::kWarps * S * (C::kStageBytes + C::kScaleBytes) + wl * S * 8);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();

  const int r = lane >> 2, c = lane & 3;
  const int Hk = p.n_kv_heads, H = p.n_heads;
  const float sl2 = p.scale * kLog2e;

  // total units of this warp
  int n_units = 0;
  for (int k = pb; k < pe; ++k) n_units += p.pieces[k].lblk_end - p.pieces[k].lblk_begin;

  // issue side: rows of the current and the next batch of 32 units
  int bip = pb, bil = p.pieces[pb].lblk_begin;  // cursor at the current batch start
  int cur_rows = unit_row(p, pe, bip, bil, lane);
  int nip = bip, nil = bil;
  advance(p.pieces, pe, nip, nil, 32);
  int next_rows = unit_row(p, pe, nip, nil, lane);
  int batch_base = 0;
  int issued = 0;

  auto issue = [&](int v) {  // all lanes; lane 0 issues the copies of unit v
    if (v - batch_base >= 32) {
      batch_base += 32;
      cur_rows = next_rows;
      advance(p.pieces, pe, nip, nil, 32);
      next_rows = unit_row(p, pe, nip, nil, lane);
    }
    const int row = __shfl_sync(kFull, cur_rows, v - batch_base);
    if (lane == 0) {
      const int st = v % S;
      const uint32_t bar = bars + 8 * st;
      const uint32_t dst = data + (uint32_t)(st * C::kStageBytes);
      mbar_expect_tx(bar, C::kTxBytes);
      if (v == 0 && gw == p.starve_warp) return;  // test hook: this stage never completes
      if (KV == 1) {
        tma_load_2d(dst, &p.tmap_k, 0, row, bar);
        tma_load_2d(dst + 2048, &p.tmap_k, 64, row, bar);
        tma_load_2d(dst + 4096, &p.tmap_v, 0, row, bar);
        tma_load_2d(dst + 6144, &p.tmap_v, 64, row, bar);
      } else {
        tma_load_2d(dst, &p.tmap_k, 0, row, bar);
        tma_load_2d(dst + 2048, &p.tmap_v, 0, row, bar);
        const uint32_t sd = scl + (uint32_t)(st * C::kScaleBytes);
        bulk_load(sd, p.k_scale + row, 64, bar);
        bulk_load(sd + 64, p.v_scale + row, 64, bar);
      }
    }
  };

  for (; issued < n_units && issued < S; ++issued) issue(issued);

  // per-lane fragment address pieces
  const int mi = lane >> 3, rr = lane & 7;
  // bf16 K (ldmatrix, non-transposed): matrices (tok 0-7|8-15) x (d lo|hi 8)
  const uint32_t k_row_off = (uint32_t)((rr + ((mi & 1) << 3)) * 128);
  const int k_hi = mi >> 1;
  // bf16 V (ldmatrix, transposed): matrices (d lo|hi 8) x (tok 0-7|8-15)
  const uint32_t v_row_off = (uint32_t)((rr + ((mi >> 1) << 3)) * 128);
  const int v_hi = mi & 1;

  // Per sequence t of the piece (t = 1 only in the two-sequence variant):
  // Q^T fragments, O^T accumulators and the softmax state of columns 2c, 2c+1.
  uint32_t qf[NQ][8][2];
  float o[NQ][8][4];
  float m0[NQ], m1[NQ], l0[NQ], l1[NQ];
  bool run_open = false, two = false;
  int u = 0;

  for (int pi = pb; pi < pe; ++pi) {
    const Piece pc = p.pieces[pi];
    const int g = pc.kv_head, L = pc.ctx_len;
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
      const int h = g * G + r;
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        const int qr = t == 0 ? pc.q_row : pc.q_row1;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t b0 = 0, b1 = 0;
          if (r < G && qr >= 0) {
            const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)qr * H + h) * 128;
            if (KV == 1) {
              b0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * c);
              b1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * c);
            } else {
              // FP8 path: k-slot 2c+e <-> d = 32c + 4kk + e, slot 2c+8+e <-> d + 2
              const uint2 raw = *reinterpret_cast<const uint2*>(qrow + 32 * c + 4 * kk);
              const __nv_bfloat162 x01 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
              const __nv_bfloat162 x23 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
              b0 = pack_f16(__low2float(x01), __high2float(x01));
              b1 = pack_f16(__low2float(x23), __high2float(x23));
            }
          }
          qf[t][kk][0] = b0;
          qf[t][kk][1] = b1;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) o[t][i][0] = o[t][i][1] = o[t][i][2] = o[t][i][3] = 0.f;
        m0[t] = m1[t] = -INFINITY;
        l0[t] = l1[t] = 0.f;
      }
      run_open = true;
    }

    for (int lb = pc.lblk_begin; lb < pc.lblk_end; ++lb, ++u) {
      const int st = u % S;
      if (!mbar_wait(bars + 8 * st, (uint32_t)((u / S) & 1), p.wait_limit_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeout);
          p.status[1] = gw;
        }
        for (int v = u + 1; v < issued; ++v) mbar_wait(bars + 8 * (v % S), (uint32_t)((v / S) & 1), kDrainTimeoutNs);
        return;
      }
      const uint32_t kb = data + (uint32_t)(st * C::kStageBytes);
      const uint32_t vb = kb + (KV == 1 ? 4096u : 2048u);

      // ---- S = K Q^T : rows = tokens, columns = query heads of the group
      float sa[NQ][4], sb[NQ][4];
#pragma unroll
      for (int t = 0; t < NQ; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[t][e] = sb[t][e] = 0.f;
      float ks_r = 1.f, ks_r8 = 1.f, vs_r = 1.f, vs_r8 = 1.f;
      if (KV == 1) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int c16 = 2 * kk + k_hi;  // 16-byte chunk index across the 256-byte row
          uint32_t a[4];
          ldsm_x4(kb + (uint32_t)((c16 >> 3) * 2048) + k_row_off + (uint32_t)((((c16 & 7) ^ rr)) << 4), a);
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
        // tokens r and r + 8, codes d in [32c, 32c + 32)
        const uint4 x0 = lds128(kb + (uint32_t)(r * 128) + (uint32_t)(((2 * c) ^ r) << 4));
        const uint4 x1 = lds128(kb + (uint32_t)(r * 128) + (uint32_t)(((2 * c + 1) ^ r) << 4));
        const uint4 y0 = lds128(kb + (uint32_t)((r + 8) * 128) + (uint32_t)(((2 * c) ^ r) << 4));
        const uint4 y1 = lds128(kb + (uint32_t)((r + 8) * 128) + (uint32_t)(((2 * c + 1) ^ r) << 4));
        const uint32_t tA[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t tB[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
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
        const uint32_t sc = scl + (uint32_t)(st * C::kScaleBytes);
        ks_r = lds_f32(sc + 4 * r);
        ks_r8 = lds_f32(sc + 4 * (r + 8));
        vs_r = lds_f32(sc + 64 + 4 * r);
        vs_r8 = lds_f32(sc + 64 + 4 * (r + 8));
      }

      // ---- mask (per token: the same for both sequences, whose shared
      // blocks are whole), logits out, online softmax (log2 units)
      const int tok0 = lb * kBlock + r, tok1 = tok0 + 8;
      // most units lie wholly inside the keep-set: their first and last
      // token decide it, and the per-token test is skipped
      const bool whole = (lb >= wb0 && lb < wb1) || lb < wsb;
      const bool k0 = whole || kept(tok0, L, p.mask_mode, p.num_sinks, p.window);
      const bool k1 = whole || kept(tok1, L, p.mask_mode, p.num_sinks, p.window);
      const bool h0v = 2 * c < G, h1v = 2 * c + 1 < G;
      if (!whole && __ballot_sync(kFull, !(k0 && k1))) {
        // zero the V rows of masked tokens in this warp's stage (0 * NaN = NaN)
        constexpr int kRowBytes = KV == 1 ? 256 : 128;
        constexpr int kChunksPerRow = kRowBytes / 16;
        constexpr int kRowsPerPass = 32 / kChunksPerRow;
        const int ch = lane % kChunksPerRow;
#pragma unroll
        for (int t0 = 0; t0 < 16; t0 += kRowsPerPass) {
          const int t = t0 + lane / kChunksPerRow;
          if (!kept(lb * kBlock + t, L, p.mask_mode, p.num_sinks, p.window)) {
            const uint32_t addr = vb + (uint32_t)((ch >> 3) * 2048 + t * 128 + (ch & 7) * 16);
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
          float* lg = p.logits + ((size_t)qr * Hk + g) * p.logits_stride * G;
          if (k0 && h0v) lg[(size_t)tok0 * G + 2 * c] = s0 * p.scale;
          if (k0 && h1v) lg[(size_t)tok0 * G + 2 * c + 1] = s1 * p.scale;
          if (k1 && h0v) lg[(size_t)tok1 * G + 2 * c] = s2 * p.scale;
          if (k1 && h1v) lg[(size_t)tok1 * G + 2 * c + 1] = s3 * p.scale;
        }
        const float a0 = k0 ? s0 * sl2 : -INFINITY, a1 = k0 ? s1 * sl2 : -INFINITY;
        const float a2 = k1 ? s2 * sl2 : -INFINITY, a3 = k1 ? s3 * sl2 : -INFINITY;
        float bm0 = fmaxf(a0, a2), bm1 = fmaxf(a1, a3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
          bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
        }
        const float mn0 = fmaxf(m0[t], bm0), mn1 = fmaxf(m1[t], bm1);
        const float z0 = mn0 == -INFINITY ? 0.f : mn0, z1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0[t] - z0), al1 = fast_exp2(m1[t] - z1);
        const float p0 = fast_exp2(a0 - z0), p1 = fast_exp2(a1 - z1), p2 = fast_exp2(a2 - z0),
                    p3 = fast_exp2(a3 - z1);
        l0[t] = l0[t] * al0 + (p0 + p2);
        l1[t] = l1[t] * al1 + (p1 + p3);
        m0[t] = mn0;
        m1[t] = mn1;
        if (__any_sync(kFull, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[t][i][0] *= al0;
            o[t][i][1] *= al1;
            o[t][i][2] *= al0;
            o[t][i][3] *= al1;
          }
        }
        // FP8 / INT8: the weight multiplies the V code times the token's V
        // scale.  Slots of masked tokens may hold anything (unwritten memory),
        // so their scale must not reach the arithmetic (0 * NaN is NaN).
        if (KV == 1) {
          pb0[t] = movmatrix_t(pack_bf16(p0, p1));
          pb1[t] = movmatrix_t(pack_bf16(p2, p3));
        } else {
          const float w0 = k0 ? vs_r : 0.f, w1 = k1 ? vs_r8 : 0.f;
          pb0[t] = movmatrix_t(pack_f16(p0 * w0, p1 * w0));
          pb1[t] = movmatrix_t(pack_f16(p2 * w1, p3 * w1));
        }
      }

      // ---- O^T += V^T P : rows = head-dim, columns = query heads
      if (KV == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c16 = 2 * i + v_hi;
          uint32_t a[4];
          ldsm_x4_t(vb + (uint32_t)((c16 >> 3) * 2048) + v_row_off + (uint32_t)((((c16 & 7) ^ rr)) << 4), a);
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (t == 1 && !two) break;
            mma_bf16(o[t][i], a, pb0[t], pb1[t]);
          }
        }
      } else {
        // tokens 2c, 2c+1, 2c+8, 2c+9; codes d in [16r, 16r + 16)
        const uint4 va = lds128(vb + (uint32_t)((2 * c) * 128) + (uint32_t)((r ^ (2 * c)) << 4));
        const uint4 vbb = lds128(vb + (uint32_t)((2 * c + 1) * 128) + (uint32_t)((r ^ (2 * c + 1)) << 4));
        const uint4 vc = lds128(vb + (uint32_t)((2 * c + 8) * 128) + (uint32_t)((r ^ (2 * c)) << 4));
        const uint4 vd = lds128(vb + (uint32_t)((2 * c + 9) * 128) + (uint32_t)((r ^ (2 * c + 1)) << 4));
        const uint32_t A4[4] = {va.x, va.y, va.z, va.w}, B4[4] = {vbb.x, vbb.y, vbb.z, vbb.w};
        const uint32_t C4[4] = {vc.x, vc.y, vc.z, vc.w}, D4[4] = {vd.x, vd.y, vd.z, vd.w};
        uint32_t pab[16], pcd[16];  // (token pair) values at d = 16r + e
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t lo = __byte_perm(A4[w], B4[w], 0x5140), hi = __byte_perm(A4[w], B4[w], 0x7362);
          codes4_to_f16x2x2<KV>(lo, pab[4 * w + 0], pab[4 * w + 1]);
          codes4_to_f16x2x2<KV>(hi, pab[4 * w + 2], pab[4 * w + 3]);
          const uint32_t lo2 = __byte_perm(C4[w], D4[w], 0x5140), hi2 = __byte_perm(C4[w], D4[w], 0x7362);
          codes4_to_f16x2x2<KV>(lo2, pcd[4 * w + 0], pcd[4 * w + 1]);
          codes4_to_f16x2x2<KV>(hi2, pcd[4 * w + 2], pcd[4 * w + 3]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t a[4] = {pab[i], pab[8 + i], pcd[i], pcd[8 + i]};
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (t == 1 && !two) break;
            mma_f16(o[t][i], a, pb0[t], pb1[t]);
          }
        }
      }
      __syncwarp();
      if (issued < n_units) {
        issue(issued);
        ++issued;
      }
    }

    if (pc.flags & kPieceLastOfRun) {
      // ---- finalise the run: one output or partial record per sequence
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
        auto dpos = [&](int i, int half) { return KV == 1 ? 16 * i + 8 * half + r : 16 * r + 8 * half + i; };
        if (oi < 0) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
          const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
          const size_t row0 = ((size_t)qr * H + g * G + h0) * 128;
          const size_t row1 = row0 + 128;
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int d = dpos(i, half);
              if (h0 < G) out[row0 + d] = __float2bfloat16(o[t][i][2 * half] * inv0);
              if (h1 < G) out[row1 + d] = __float2bfloat16(o[t][i][2 * half + 1] * inv1);
            }
          if (r == 0 && p.lse != nullptr) {
            const size_t li = (size_t)qr * H + g * G;
            if (h0 < G) p.lse[li + h0] = L0 > 0.f ? (m0[t] + log2f(L0)) * kLn2 : -INFINITY;
            if (h1 < G) p.lse[li + h1] = L1 > 0.f ? (m1[t] + log2f(L1)) * kLn2 : -INFINITY;
          }
        } else {
          float* rec = p.partials + (size_t)oi * partial_floats(G, 128);
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int d = dpos(i, half);
              if (h0 < G) rec[h0 * 128 + d] = o[t][i][2 * half];
              if (h1 < G) rec[h1 * 128 + d] = o[t][i][2 * half + 1];
            }
          if (r == 0) {
            if (h0 < G) {
              rec[G * 128 + h0] = m0[t];
              rec[G * 128 + G + h0] = L0;
            }
            if (h1 < G) {
              rec[G * 128 + h1] = m1[t];
              rec[G * 128 + G + h1] = L1;
            }
          }
          rec_items[t] = ci;
        }
      }
      // publish the run's records (one release fence for both sequences of a
      // pair), count them, and merge any (sequence, kv head) whose last
      // record this was (acquire before reading the others' records)
      if (rec_items[0] >= 0 || (NQ == 2 && rec_items[NQ - 1] >= 0)) {
        fence_acq_rel_gpu();
        __syncwarp();
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          const int ci = rec_items[t];
          if (ci < 0) continue;
          int last = 0;
          if (lane == 0) last = atomicAdd(p.counters + ci, 1) == p.combine[ci].n_partials - 1;
          last = __shfl_sync(kFull, last, 0);
          if (last) {
            fence_acq_rel_gpu();
            merge_partials<G>(p, p.combine[ci], lane);
          }
        }
      }
      run_open = false;
    }
  }
}

// ---------------------------------------------------------------------------
// Shared-prefix multi-query kernel (bf16 KV).  One CTA per PrefixItem: the
// item's blocks are loaded once per CTA by TMA into a 3-stage ring of 64-token
// chunks and consumed by all 8 warps; each warp owns 16 query rows (16 / G
// member sequences x G heads) and runs FlashAttention-2 style: S = Q K^T with
// the query rows as M (m16n8k16, K fragments by ldmatrix), the online softmax
// on the rows in registers (a row lives in one quad), the probabilities reused
// in registers as the A operand of O = P V (V fragments by ldmatrix.trans).
// Every block of an item is a full block of every member, so no token mask
// applies.  Each member's rows end in one partial record, merged like any
// split by the warp that writes the last record of a (sequence, kv head).
// ---------------------------------------------------------------------------

constexpr int kPWarps = 8, kPStages = 3, kPChunkBlocks = 4;
constexpr int kPStageBytes = kPChunkBlocks * 8192;

constexpr size_t prefix_smem_bytes() { return 1024 + (size_t)kPStages * kPStageBytes + 2 * kPStages * 8; }

template <int G>
__global__ void __launch_bounds__(kPWarps * 32, 1) prefix_decode_kernel(const __grid_constant__ DecodeTCParams p) {
  constexpr int MPW = 16 / G;  // member sequences per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const PrefixItem it = p.prefix_items[blockIdx.x];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int r = lane >> 2, c = lane & 3, mi = lane >> 3, rr = lane & 7;
  const int g = it.kv_head, Hk = p.n_kv_heads, H = p.n_heads;
  const uint32_t data = smem_addr(base);
  const uint32_t full = data + (uint32_t)(kPStages * kPStageBytes), empty = full + 8 * kPStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, kPWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  const int nblk = it.lblk_end - it.lblk_begin;
  const int nchunks = (nblk + kPChunkBlocks - 1) / kPChunkBlocks;
  auto issue = [&](int ch) {  // thread 0 only
    const int st = ch % kPStages, nb = min(kPChunkBlocks, nblk - ch * kPChunkBlocks);
    const uint32_t bar = full + 8 * st, dst = data + (uint32_t)(st * kPStageBytes);
    mbar_expect_tx(bar, (uint32_t)nb * 8192u);
    for (int j = 0; j < nb; ++j) {
      const int lb = it.lblk_begin + ch * kPChunkBlocks + j;
      int blk = p.tables[(size_t)it.table_seq * p.max_blocks + lb];
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.status, kStatusBadBlock);
        p.status[1] = it.table_seq;
        p.status[2] = lb;
        blk = 0;  // keep the copy in bounds; the status word reports the fault
      }
      const int row = (blk * Hk + g) * kBlock;
      const uint32_t d0 = dst + (uint32_t)(j * 8192);
      tma_load_2d(d0, &p.tmap_k, 0, row, bar);
      tma_load_2d(d0 + 2048, &p.tmap_k, 64, row, bar);
      tma_load_2d(d0 + 4096, &p.tmap_v, 0, row, bar);
      tma_load_2d(d0 + 6144, &p.tmap_v, 64, row, bar);
    }
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < nchunks && issued < kPStages; ++issued) issue(issued);

  // Q fragments (A operand): rows r and r + 8 of this warp, k = d
  const int mbase = wl * MPW;  // first member of this warp within the item
  auto row_valid = [&](int row) { return mbase + row / G < it.n_members; };
  auto row_qrow = [&](int row) { return p.prefix_members[it.member_begin + mbase + row / G].q_row; };
  uint32_t qa[8][4];
  {
    const bool v0 = row_valid(r), v1 = row_valid(r + 8);
    const __nv_bfloat16* q0 = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                              ((size_t)(v0 ? row_qrow(r) : 0) * H + g * G + r % G) * 128;
    const __nv_bfloat16* q1 = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                              ((size_t)(v1 ? row_qrow(r + 8) : 0) * H + g * G + (r + 8) % G) * 128;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + 16 * kk + 2 * c) : 0u;
      qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + 16 * kk + 2 * c) : 0u;
      qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + 16 * kk + 8 + 2 * c) : 0u;
      qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + 16 * kk + 8 + 2 * c) : 0u;
    }
  }
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r = -INFINITY, m_r8 = -INFINITY, l_r = 0.f, l_r8 = 0.f;
  const float sl2 = p.scale * kLog2e;
  bool failed = false;
  int ch = 0;  // chunks this warp has consumed

  for (; ch < nchunks; ++ch) {
    const int st = ch % kPStages, nb = min(kPChunkBlocks, nblk - ch * kPChunkBlocks);
    if (!mbar_wait(full + 8 * st, (uint32_t)((ch / kPStages) & 1), p.wait_limit_ns)) {
      if (lane == 0) {
        atomicOr(p.status, kStatusTimeout);
        p.status[1] = -1 - (int)blockIdx.x;
      }
      failed = true;
      break;
    }
    const uint32_t cb = data + (uint32_t)(st * kPStageBytes);

    // ---- S = Q K^T: rows = query rows, columns = the chunk's tokens
    float sacc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int j = 0; j < kPChunkBlocks; ++j) {
      if (j >= nb) break;
      const uint32_t kb = cb + (uint32_t)(j * 8192);
      const int tok = rr + ((mi >> 1) << 3);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ch16 = 2 * kk + (mi & 1);
        uint32_t b[4];
        ldsm_x4(kb + (uint32_t)((ch16 >> 3) * 2048 + tok * 128 + (((ch16 & 7) ^ rr) << 4)), b);
        mma_bf16(sacc[2 * j], qa[kk], b[0], b[1]);
        mma_bf16(sacc[2 * j + 1], qa[kk], b[2], b[3]);
      }
    }
    if (p.logits != nullptr) {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        if (n >= 2 * nb) break;
        const int tok0 = (it.lblk_begin + ch * kPChunkBlocks) * kBlock + 8 * n + 2 * c;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int row = r + 8 * half;
          if (!row_valid(row)) continue;
          float* lg = p.logits + ((size_t)row_qrow(row) * Hk + g) * p.logits_stride * G;
          lg[(size_t)tok0 * G + row % G] = sacc[n][2 * half] * p.scale;
          lg[(size_t)(tok0 + 1) * G + row % G] = sacc[n][2 * half + 1] * p.scale;
        }
      }
    }
    // ---- online softmax on rows r and r + 8 (log2 units)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      if (n >= 2 * nb) break;
      mx0 = fmaxf(mx0, fmaxf(sacc[n][0], sacc[n][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[n][2], sacc[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    const float mn0 = fmaxf(m_r, mx0 * sl2), mn1 = fmaxf(m_r8, mx1 * sl2);
    const float al0 = fast_exp2(m_r - mn0), al1 = fast_exp2(m_r8 - mn1);
    float ps0 = 0.f, ps1 = 0.f;
    uint32_t pa[4][4];  // P as the A operand of each block's k16 step
#pragma unroll
    for (int j = 0; j < kPChunkBlocks; ++j) {
      if (j >= nb) break;
      float e[2][4];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float* sv = sacc[2 * j + h2];
        e[h2][0] = fast_exp2(fmaf(sv[0], sl2, -mn0));
        e[h2][1] = fast_exp2(fmaf(sv[1], sl2, -mn0));
        e[h2][2] = fast_exp2(fmaf(sv[2], sl2, -mn1));
        e[h2][3] = fast_exp2(fmaf(sv[3], sl2, -mn1));
        ps0 += e[h2][0] + e[h2][1];
        ps1 += e[h2][2] + e[h2][3];
      }
      pa[j][0] = pack_bf16(e[0][0], e[0][1]);
      pa[j][1] = pack_bf16(e[0][2], e[0][3]);
      pa[j][2] = pack_bf16(e[1][0], e[1][1]);
      pa[j][3] = pack_bf16(e[1][2], e[1][3]);
    }
    l_r = l_r * al0 + ps0;
    l_r8 = l_r8 * al1 + ps1;
    m_r = mn0;
    m_r8 = mn1;
    if (__any_sync(kFull, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
    }
    // ---- O += P V: k = the block's 16 tokens, n = 8-wide d tiles
#pragma unroll
    for (int j = 0; j < kPChunkBlocks; ++j) {
      if (j >= nb) break;
      const uint32_t vb = cb + (uint32_t)(j * 8192 + 4096);
      const int tok = rr + ((mi & 1) << 3);
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const int ch16 = i + (mi >> 1);
        uint32_t b[4];
        ldsm_x4_t(vb + (uint32_t)((ch16 >> 3) * 2048 + tok * 128 + (((ch16 & 7) ^ rr) << 4)), b);
        mma_bf16(o[i], pa[j], b[0], b[1]);
        mma_bf16(o[i + 1], pa[j], b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty + 8 * st) : "memory");
    if (threadIdx.x == 0 && issued < nchunks) {
      // the stage is free once all warps have consumed this chunk
      if (!mbar_wait(empty + 8 * st, (uint32_t)((ch / kPStages) & 1), p.wait_limit_ns)) {
        atomicOr(p.status, kStatusTimeout);
        failed = true;
        ++ch;  // this chunk was consumed
        break;
      }
      issue(issued);
      ++issued;
    }
  }
  if (threadIdx.x == 0 && failed) {
    // copies still in flight (chunks issued but not consumed) target this
    // CTA's shared memory: wait them out, bounded
    for (int v = ch; v < issued; ++v)
      mbar_wait(full + 8 * (v % kPStages), (uint32_t)((v / kPStages) & 1), kDrainTimeoutNs);
  }
  if (failed) return;

  // ---- records: O (unnormalised), M (log2 units) and l of every row
  l_r += __shfl_xor_sync(kFull, l_r, 1);
  l_r += __shfl_xor_sync(kFull, l_r, 2);
  l_r8 += __shfl_xor_sync(kFull, l_r8, 1);
  l_r8 += __shfl_xor_sync(kFull, l_r8, 2);
  constexpr int PF = G * 128 + ((2 * G + 3) & ~3);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = r + 8 * half;
    if (!row_valid(row)) continue;
    const PrefixMember mb = p.prefix_members[it.member_begin + mbase + row / G];
    float* rec = p.partials + (size_t)mb.out_index * PF;
    const int h = row % G;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      *reinterpret_cast<float2*>(rec + h * 128 + 8 * i + 2 * c) = make_float2(o[i][2 * half], o[i][2 * half + 1]);
    if (c == 0) {
      rec[G * 128 + h] = half ? m_r8 : m_r;
      rec[G * 128 + G + h] = half ? l_r8 : l_r;
    }
  }
  fence_acq_rel_gpu();
  __syncwarp();
  for (int k = 0; k < MPW; ++k) {
    if (mbase + k >= it.n_members) break;
    const PrefixMember mb = p.prefix_members[it.member_begin + mbase + k];
    int last = 0;
    if (lane == 0) last = atomicAdd(p.counters + mb.item, 1) == p.combine[mb.item].n_partials - 1;
    last = __shfl_sync(kFull, last, 0);
    if (last) {
      fence_acq_rel_gpu();
      merge_partials<G>(p, p.combine[mb.item], lane);
    }
  }
}

template <int KV, int G, int NQ>
cudaError_t launch_t(const DecodeTCParams& p, int ctas, cudaStream_t st) {
  decode_tc_kernel<KV, G, NQ><<<ctas, TC<KV, NQ>::kWarps * 32, smem_bytes<KV, NQ>(), st>>>(p);
  return cudaGetLastError();
}

template <int KV, int G, int NQ>
cudaError_t prepare_t() {
  return cudaFuncSetAttribute(decode_tc_kernel<KV, G, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<KV, NQ>());
}

template <int KV, int G, int NQ>
cudaError_t occupancy_t(int* n) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, decode_tc_kernel<KV, G, NQ>, TC<KV, NQ>::kWarps * 32,
                                                       smem_bytes<KV, NQ>());
}

// Expands X(KV, G, NQ) for every compiled variant, returning its result when
// it matches the runtime (kv_dtype, G, nq).
#define PKV_FOR_VARIANTS(X)                                                                 \
  X(1, 1, 1) X(1, 2, 1) X(1, 4, 1) X(1, 8, 1) X(2, 1, 1) X(2, 2, 1) X(2, 4, 1) X(2, 8, 1)          \
  X(3, 1, 1) X(3, 2, 1) X(3, 4, 1) X(3, 8, 1) X(1, 1, 2) X(1, 2, 2) X(1, 4, 2) X(1, 8, 2)          \
  X(2, 1, 2) X(2, 2, 2) X(2, 4, 2) X(2, 8, 2) X(3, 1, 2) X(3, 2, 2) X(3, 4, 2) X(3, 8, 2)

}  // namespace

cudaError_t launch_decode_tc(int kv_dtype, int G, int nq, const DecodeTCParams& p, int ctas, cudaStream_t st) {
  if (ctas <= 0) return cudaSuccess;
#define X(KV, GG, NQ) \
  if (kv_dtype == KV && G == GG && nq == NQ) return launch_t<KV, GG, NQ>(p, ctas, st);
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

int decode_tc_warps_per_cta(int kv_dtype, int nq) {
  if (kv_dtype == 2 || kv_dtype == 3) return nq == 2 ? TC<2, 2>::kWarps : TC<2, 1>::kWarps;
  return nq == 2 ? TC<1, 2>::kWarps : TC<1, 1>::kWarps;
}

size_t decode_tc_smem_bytes(int kv_dtype, int nq) {
  if (kv_dtype == 2 || kv_dtype == 3) return nq == 2 ? smem_bytes<2, 2>() : smem_bytes<2, 1>();
  return nq == 2 ? smem_bytes<1, 2>() : smem_bytes<1, 1>();
}

cudaError_t decode_tc_prepare(int kv_dtype, int G, int nq) {
#define X(KV, GG, NQ) \
  if (kv_dtype == KV && G == GG && nq == NQ) return prepare_t<KV, GG, NQ>();
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t decode_tc_occupancy(int kv_dtype, int G, int nq, int* n) {
#define X(KV, GG, NQ) \
  if (kv_dtype == KV && G == GG && nq == NQ) return occupancy_t<KV, GG, NQ>(n);
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

#undef PKV_FOR_VARIANTS

cudaError_t launch_prefix_decode(int G, const DecodeTCParams& p, cudaStream_t st) {
  if (p.n_prefix_items <= 0) return cudaSuccess;
  const size_t smem = prefix_smem_bytes();
  switch (G) {
    case 1: prefix_decode_kernel<1><<<p.n_prefix_items, kPWarps * 32, smem, st>>>(p); break;
    case 2: prefix_decode_kernel<2><<<p.n_prefix_items, kPWarps * 32, smem, st>>>(p); break;
    case 4: prefix_decode_kernel<4><<<p.n_prefix_items, kPWarps * 32, smem, st>>>(p); break;
    case 8: prefix_decode_kernel<8><<<p.n_prefix_items, kPWarps * 32, smem, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t prefix_decode_prepare(int G) {
  const int smem = (int)prefix_smem_bytes();
  switch (G) {
    case 1: return cudaFuncSetAttribute(prefix_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 2: return cudaFuncSetAttribute(prefix_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 4: return cudaFuncSetAttribute(prefix_decode_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 8: return cudaFuncSetAttribute(prefix_decode_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pkv
