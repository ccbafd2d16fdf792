// kernels.cu -- the HBM-bound helper kernels of libpkv (sm_103a):
//   append / reshape_and_cache (+ FP8 E4M3 per-token quantisation),
//   copy-on-write block copy, block-table patch,
//   H2O score accumulation, H2O top-k keep-set selection, and the fp32
//   CUDA-core decode used for fp32 pools.
//
// Pages (title, section): "KV Cache 与 PagedAttention：显存复用与长上下文推理"
// (三大运行时组件, copy_on_write sketch, 量化原理); "长上下文优化：注意力稀疏化与
// KV Cache 管理" (H2OEviction, StreamingKVCache, sliding-window mask);
// "系统优化" (Flash Attention's online softmax; KV Cache 淘汰).

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <float.h>

#include <algorithm>
#include <atomic>

#include "async_copy.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// number of kept keys and the k-th kept position, in ascending order
__device__ __forceinline__ int keep_count_of(int L, int mode, int S, int W) {
  if (L <= 0) return 0;
  if (mode == 0) return L;
  if (mode == 1) return min(L, W + 1);
  if ((long long)L <= (long long)S + W) return L;
  return S + W;
}
__device__ __forceinline__ int keep_pos(int k, int L, int mode, int S, int W) {
  if (mode == 0) return k;
  if (mode == 1) return max(0, L - 1 - W) + k;
  if ((long long)L <= (long long)S + W) return k;
  return k < S ? k : L - W + (k - S);
}

// ---------------------------------------------------------------------------
// append: scatter new rows into their slots (bf16 / fp32 copy, or FP8
// quantisation), and apply the block-table patches queued with them
// ---------------------------------------------------------------------------

__device__ __forceinline__ int64_t slot_of(const AppendArgs& a, int64_t t) {
  return a.slots ? a.slots[t] : a.inline_slots[t];
}

__device__ __forceinline__ void apply_patches(const AppendArgs& a) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_patches; i += gridDim.x * blockDim.x) {
    const int32_t idx = a.patches ? a.patches[2 * i] : a.inline_patches[2 * i];
    const int32_t val = a.patches ? a.patches[2 * i + 1] : a.inline_patches[2 * i + 1];
    a.tables[idx] = val;
  }
}

__global__ void append_copy_kernel(const __grid_constant__ AppendArgs a, int row_chunks) {
  apply_patches(a);
  const uint4* k_new = static_cast<const uint4*>(a.k_new);
  const uint4* v_new = static_cast<const uint4*>(a.v_new);
  uint4* k_pool = static_cast<uint4*>(a.k_pool);
  uint4* v_pool = static_cast<uint4*>(a.v_pool);
  const int64_t per_tok = (int64_t)a.Hk * row_chunks;
  const int64_t total = (int64_t)a.n_tokens * per_tok;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < 2 * total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= total;
    const int64_t e = is_v ? i - total : i;
    const int64_t t = e / per_tok;
    const int64_t rem = e - t * per_tok;  // = g * row_chunks + chunk
    const int64_t slot = slot_of(a, t);
    const int64_t blk = slot >> 4, off = slot & 15;
    const int64_t g = rem / row_chunks, ch = rem - g * row_chunks;
    const int64_t dst = ((blk * a.Hk + g) * kBlock + off) * row_chunks + ch;
    if (is_v)
      v_pool[dst] = v_new[e];
    else
      k_pool[dst] = k_new[e];
  }
}

// FP8 / INT8: one warp per (token, kv head, K|V) row of D values (D / 32 per
// lane).  With per-channel scales c the row is divided by them first
// (y = x / c), and y is what is quantised per token.
//   FP8:  s = absmax / 448, code = E4M3(x / s), round to nearest even,
//         saturate to +-448
//   INT8: s = absmax / 127, code = x / s rounded to the nearest integer
//         (ties to even), clamped to +-127
// (fp32, IEEE division; s = 1 when absmax is 0)
template <int KV, int D>
__global__ void append_quant_kernel(const __grid_constant__ AppendArgs a) {
  constexpr float kMaxCode = KV == 3 ? 127.0f : 448.0f;
  constexpr int E = D / 32;  // values per lane: 4 or 2
  apply_patches(a);
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.n_tokens * a.Hk;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t w = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5); w < 2 * rows; w += warps) {
    const bool is_v = w >= rows;
    const int64_t row = is_v ? w - rows : w;  // = t * Hk + g
    const int64_t t = row / a.Hk, g = row - t * a.Hk;
    const __nv_bfloat16* src =
        static_cast<const __nv_bfloat16*>(is_v ? a.v_new : a.k_new) + row * D + lane * E;
    float x[E];
    if constexpr (E == 4) {
      const uint2 raw = *reinterpret_cast<const uint2*>(src);
      const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      x[0] = __low2float(lo), x[1] = __high2float(lo), x[2] = __low2float(hi), x[3] = __high2float(hi);
    } else {
      const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(src);
      x[0] = __low2float(v), x[1] = __high2float(v);
    }
    if (a.k_channel != nullptr) {  // per-channel scales: y = x / c first (IEEE division)
      const float* ch = (is_v ? a.v_channel : a.k_channel) + g * D + lane * E;
#pragma unroll
      for (int k = 0; k < E; ++k) x[k] = __fdiv_rn(x[k], ch[k]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kMaxCode);
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < E; ++k) {
      uint32_t code;
      if (KV == 3) {
        const int n = __float2int_rn(__fdiv_rn(x[k], s));
        code = (uint32_t)(uint8_t)(int8_t)max(-127, min(127, n));
      } else {
        code = __nv_cvt_float_to_fp8(__fdiv_rn(x[k], s), __NV_SATFINITE, __NV_E4M3);
      }
      packed |= code << (8 * k);
    }
    const int64_t slot = slot_of(a, t);
    const int64_t blk = slot >> 4, off = slot & 15;
    const int64_t srow = (blk * a.Hk + g) * kBlock + off;
    uint8_t* dst = static_cast<uint8_t*>(is_v ? a.v_pool : a.k_pool) + srow * D + lane * E;
    if constexpr (E == 4)
      *reinterpret_cast<uint32_t*>(dst) = packed;
    else
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    if (lane == 0) (is_v ? a.v_scale : a.k_scale)[srow] = s;
  }
}

// ---------------------------------------------------------------------------
// copy-on-write and CPU swap: copy whole physical blocks (K, V, and FP8 /
// INT8 scales)
// ---------------------------------------------------------------------------

// Whole-block copies pairs[2i] -> pairs[2i+1] from one pool to another (the
// same pool for copy-on-write; device <-> pinned host pool for CPU swap, the
// host side reached through its device-mapped address).
__global__ void block_copy_kernel(const int32_t* __restrict__ pairs, const uint4* src_k, const uint4* src_v,
                                  uint4* dst_k, uint4* dst_v, int64_t chunks, const float* src_ks,
                                  const float* src_vs, float* dst_ks, float* dst_vs, int64_t sfloats) {
  const int64_t src = pairs[2 * blockIdx.y], dst = pairs[2 * blockIdx.y + 1];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < chunks; i += (int64_t)gridDim.x * blockDim.x) {
    dst_k[dst * chunks + i] = src_k[src * chunks + i];
    dst_v[dst * chunks + i] = src_v[src * chunks + i];
  }
  if (src_ks && blockIdx.x == 0)
    for (int64_t i = threadIdx.x; i < sfloats; i += blockDim.x) {
      dst_ks[dst * sfloats + i] = src_ks[src * sfloats + i];
      dst_vs[dst * sfloats + i] = src_vs[src * sfloats + i];
    }
}

__global__ void table_patch_kernel(const int32_t* __restrict__ patches, int n, int32_t* __restrict__ tables) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    tables[patches[2 * i]] = patches[2 * i + 1];
}

// ---------------------------------------------------------------------------
// H2O score: acc[b][j] += mean over query heads of exp(s_hj - lse_h)
// ---------------------------------------------------------------------------

// Each term is 2^(s log2(e) - lse log2(e)) on the hardware ex2: the exponent
// comes from one fused multiply-add of the fp32 logit against lse log2(e)
// staged in shared memory, so its absolute error is about |s - lse| 2^-24
// plus half an ulp of lse log2(e); with the instruction's own relative error
// (about 2^-22) a term is within 2e-6 of exp(s - lse) for |s - lse| < 20,
// and terms below that weigh nothing at the scores' 1e-5 relative bound.
// The accurate expf spent most of this kernel's time in instructions.
__device__ __forceinline__ float h2o_term(float s, float lse2) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(fmaf(s, 1.4426950408889634f, -lse2)));
  return y;
}

__global__ void h2o_score_kernel(const SeqRow* __restrict__ rows, int n_heads, int n_kv_heads,
                                 const float* __restrict__ logits, int64_t stride, const float* __restrict__ lse,
                                 int mode, int S, int W, float* __restrict__ acc, int64_t acc_stride) {
  extern __shared__ float s_lse[];  // lse log2(e) per query head
  const SeqRow row = rows[blockIdx.y];
  const int b = row.q_row, L = row.ctx_len;
  for (int h = threadIdx.x; h < n_heads; h += blockDim.x) s_lse[h] = lse[(size_t)b * n_heads + h] * 1.4426950408889634f;
  __syncthreads();
  const int nk = keep_count_of(L, mode, S, W);
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= nk) return;
  const int j = keep_pos(k, L, mode, S, W);
  const int G = n_heads / n_kv_heads;
  float* accj = acc + (size_t)b * acc_stride + j;
  const float prev = *accj;  // in flight with the logit loads
  float sum = 0.0f;
  if ((G & 3) == 0 && ((reinterpret_cast<uintptr_t>(logits) | (uintptr_t)(stride * G * 4)) & 15) == 0) {
    // heads in groups of four (one float4 each), visited in head order; a
    // batch of 8 float4 loads is issued before any of them is used
    const int q4 = G >> 2, nf = n_heads >> 2;
    for (int f0 = 0; f0 < nf; f0 += 8) {
      int g = f0 / q4, i = f0 - g * q4;
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (f0 + u < nf)
          x[u] = *reinterpret_cast<const float4*>(logits + (((size_t)b * n_kv_heads + g) * stride + j) * G + 4 * i);
        if (++i == q4) {
          i = 0;
          ++g;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (f0 + u < nf) {
          const float* ls = s_lse + 4 * (f0 + u);
          sum += h2o_term(x[u].x, ls[0]) + h2o_term(x[u].y, ls[1]) + h2o_term(x[u].z, ls[2]) +
                 h2o_term(x[u].w, ls[3]);
        }
      }
    }
  } else {
#pragma unroll 8
    for (int g = 0; g < n_kv_heads; ++g) {
      const float* lg = logits + (((size_t)b * n_kv_heads + g) * stride + j) * G;
      for (int i = 0; i < G; ++i) sum += h2o_term(lg[i], s_lse[g * G + i]);
    }
  }
  *accj = prev + sum / (float)n_heads;
}

// ---------------------------------------------------------------------------
// H2O select: exact top-k by radix select on order-preserving keys, ties to
// the lower position, output in ascending position order.
// ---------------------------------------------------------------------------

constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0;  // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// exclusive block scan of v (blockDim.x == kSelThreads); returns the total
__device__ int block_excl_scan(int v, int* excl, int* s_warp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, t, o);
      if (lane >= o) t += y;
    }
    s_warp[lane] = t;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int before = w ? s_warp[w - 1] : 0;
  const int total = s_warp[31];
  *excl = before + x - v;
  __syncthreads();
  return total;
}

constexpr int kSelUnroll = 16;     // keys per thread per sweep (independent loads)
constexpr int kSelCap = 8192;       // candidates held in shared memory
constexpr int kSelSample = 2048;    // keys sampled to pick the one-pass threshold (<= kSelCap)
constexpr int kSelSampleMinRow = 16384;  // rows longer than this take the sampled one-pass path
// The gather streams a row through a ring of bulk copies: kSelRing stages of
// kSelChunk scores, one chunk per sweep (kSelChunk / kSelThreads per thread).
#ifndef PKV_SEL_CHUNK
#define PKV_SEL_CHUNK 8192
#endif
#ifndef PKV_SEL_RING
#define PKV_SEL_RING 4
#endif
constexpr int kSelChunk = PKV_SEL_CHUNK;
constexpr int kSelRing = PKV_SEL_RING;
constexpr size_t kSelSmem = (size_t)kSelCap * 8 + (size_t)kSelRing * kSelChunk * 4;
static_assert(kSelSample % kSelThreads == 0 && kSelChunk % (4 * kSelThreads) == 0, "select geometry");

template <int N>
struct IntTag {
  static constexpr int value = N;
};

struct SelShared {
  unsigned long long bar[kSelRing];  // ring stage mbarriers (one arrival + the copy's bytes)
  uint32_t hist[256];
  uint32_t hist2[2][256];  // radix passes: one filled while the other is cleared
  int warp[32];
  int tot[32];     // per-warp candidate counts of a sweep
  uint32_t prefix, mask;
  int k, n_cand, top, n_head;
  int starve;     // test hook: the first chunk of this block's row is never issued
  int undrained;  // a copy into the ring was still in flight when the drain gave up
};
static_assert(kSelSmem + sizeof(SelShared) <= 227 * 1024, "select shared memory");

// Slot of candidate i in the shared candidate arrays: the word index with its
// low 3 bits XORed by bits 5-7.  A row of 32 consecutive candidates stays one
// row (conflict-free linear reads), and a warp whose lanes write 8 consecutive
// candidates each (stride 8) spreads over all 32 banks.
__device__ __forceinline__ int cand_slot(int i) { return i ^ ((i >> 5) & 7); }

// Histogram of digit (key >> shift) & 255 over the keys i < m whose bits under
// `mask` equal `prefix`.  Scores are often equal (zero outside the keep-set,
// or of one magnitude), so lanes of a warp holding the same digit are
// grouped (match.any) and their leader adds the group's count: one shared
// atomic per distinct digit per warp step instead of one per key.
// U keys per thread per sweep: few for the short candidate lists in shared
// memory (every thread runs every slot of the sweep), kSelUnroll for rows
// read from global memory.
template <int U, class KeyAt>
__device__ void accumulate_digits(KeyAt key_at, int m, uint32_t prefix, uint32_t mask, int shift, uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < m; base += U * kSelThreads) {
    uint32_t key[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kSelThreads + threadIdx.x;
      key[u] = i < m ? key_at(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kSelThreads + threadIdx.x;
      const bool in = i < m && (key[u] & mask) == prefix;
      if (!__any_sync(0xffffffffu, in)) continue;
      const uint32_t digit = in ? (key[u] >> shift) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
    }
  }
}
template <int U, class KeyAt>
__device__ void digit_histogram(KeyAt key_at, int m, uint32_t prefix, uint32_t mask, int shift, SelShared& sh) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist[i] = 0;
  __syncthreads();
  accumulate_digits<U>(key_at, m, prefix, mask, shift, sh.hist);
  __syncthreads();
}

// Warp 0 alone: the digit d of a 256-bin histogram whose bin holds the k-th
// largest key, (keys in bins above d) < k <= (keys in bins d and above).  Lane
// l scans bins 255 - 8l down to 248 - 8l.  The one lane that holds d returns
// true with d, k minus the keys above d, and the keys in bins d and above.
__device__ __forceinline__ bool find_digit_warp(const uint32_t* hist, int k, int* digit, int* k_rem, int* count) {
  const int lane = threadIdx.x & 31;
  int c[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = (int)hist[255 - 8 * lane - j];
    sum += c[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  int above = incl - sum;
  if (!(above < k && k <= incl)) return false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (above < k && k <= above + c[j]) {
      *digit = 255 - 8 * lane - j;
      *k_rem = k - above;
      *count = above + c[j];
      return true;
    }
    above += c[j];
  }
  return false;
}

// Finds, in parallel over the 256 bins, the digit d whose bin holds the k-th
// largest key: (keys in bins above d) < k <= (keys in bins d and above).
// Writes d to *digit_out and k minus the keys above it to *k_out, and the
// keys in bins d and above to *count_out (when not NULL).  Called by the
// whole block; ends with a barrier.
__device__ void find_digit(SelShared& sh, int k, int* digit_out, int* k_out, int* count_out) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  // bins in descending digit order: position j holds digit 255 - j
  int c = t < 256 ? (int)sh.hist[255 - t] : 0;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (t < 256 && lane == 31) sh.warp[w] = incl;
  __syncthreads();
  if (t < 256) {
    int before = 0;
    for (int i = 0; i < w; ++i) before += sh.warp[i];
    const int above = before + incl - c, upto = before + incl;
    if (above < k && k <= upto) {
      *digit_out = 255 - t;
      *k_out = k - above;
      if (count_out) *count_out = upto;
    }
  }
  __syncthreads();
}

// Exact keep-th largest key among keys i < m (radix select, 8 bits a pass):
// on return sh.prefix is that key and sh.k the number of keys equal to it
// that belong to the selection (the lowest positions among them).
// With last_shift > 0 the passes stop after that digit: sh.prefix then holds
// the keep-th largest key's top bits with the rest zero, a lower bound of it.
template <int U, class KeyAt>
__device__ void radix_select(KeyAt key_at, int m, int keep, SelShared& sh, int last_shift = 0) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist2[0][i] = 0;
  if (threadIdx.x == 0) {
    sh.prefix = 0;
    sh.mask = 0;
    sh.k = keep;
  }
  __syncthreads();
  int pass = 0;
  for (int shift = 24; shift >= last_shift; shift -= 8, ++pass) {
    const uint32_t prefix = sh.prefix, mask = sh.mask;
    const int k = sh.k;
    // the other buffer was last read before the previous pass's final barrier
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist2[(pass + 1) & 1][i] = 0;
    accumulate_digits<U>(key_at, m, prefix, mask, shift, sh.hist2[pass & 1]);
    __syncthreads();
    if (threadIdx.x < 32) {
      int d, kr, cnt;
      if (find_digit_warp(sh.hist2[pass & 1], k, &d, &kr, &cnt)) {
        sh.prefix = prefix | ((uint32_t)d << shift);
        sh.mask = mask | (255u << shift);
        sh.k = kr;
      }
    }
    __syncthreads();
  }
}

// Writes, in ascending order, the positions in [emit_lo, emit_hi) of the
// selected keys among i < m: those above T, plus the first need_eq keys equal
// to T (counted over all i, in or out of the range); keys are visited in the
// order of i, which must be the order of positions.  Returns the number
// written.
template <int U, class KeyAt, class PosAt>
__device__ int ordered_emit(KeyAt key_at, PosAt pos_at, int m, uint32_t T, int need_eq, int emit_lo, int emit_hi,
                            int32_t* out, SelShared& sh) {
  int taken = 0, eq_seen = 0;
  for (int base = 0; base < m; base += U * kSelThreads) {
    const int i0 = base + U * threadIdx.x;
    uint32_t key[U];
    int n_eq = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      key[u] = i0 + u < m ? key_at(i0 + u) : 0u;
      n_eq += (i0 + u < m && key[u] == T);
    }
    int eq_excl;
    const int eq_tot = block_excl_scan(n_eq, &eq_excl, sh.warp);
    int rank = eq_seen + eq_excl, n_sel = 0;
    uint32_t take = 0;  // bit u: key u is selected and inside the range
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + u >= m) continue;
      const bool sel = key[u] > T || (key[u] == T && rank++ < need_eq);
      const int p = pos_at(i0 + u);
      if (sel && p >= emit_lo && p < emit_hi) {
        take |= 1u << u;
        ++n_sel;
      }
    }
    int sel_excl;
    const int sel_tot = block_excl_scan(n_sel, &sel_excl, sh.warp);
    int pos = taken + sel_excl;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (take >> u & 1u) out[pos++] = pos_at(i0 + u);
    taken += sel_tot;
    eq_seen += eq_tot;
  }
  return taken;
}

// The ring's geometry for a row: the head (positions before the row's first
// 128-byte boundary, fewer than 32, read directly) and the chunks after it.
__device__ __forceinline__ int ring_head(const float* a, int n) {
  return min(n, (int)(((128u - (uint32_t)(reinterpret_cast<uintptr_t>(a) & 127u)) & 127u) >> 2));
}
// Thread 0: chunk c of the row into stage c % kSelRing, one bulk copy from a
// 128-byte aligned address (the ragged end, under 16 bytes, is read directly).
__device__ __forceinline__ void ring_issue(const float* a, int n, int head, int c, float* ring, SelShared& sh) {
  const int st = c % kSelRing, k0 = head + c * kSelChunk;
  const int bulk = min(kSelChunk, n - k0) & ~3;
  const uint32_t bar = smem_addr(&sh.bar[st]);
  if (c == 0 && sh.starve) return;  // test hook: this stage never completes
  if (bulk > 0) {
    mbar_expect_tx(bar, (uint32_t)bulk * 4u);
    bulk_load(smem_addr(ring + (size_t)st * kSelChunk), a + k0, (uint32_t)bulk * 4u, bar);
  } else {
    mbar_arrive(bar);
  }
}
// Thread 0: initialises the ring's barriers and issues its first chunks.  A
// barrier of the whole block must separate this from the first wait.
__device__ void ring_prime(const float* a, int n, float* ring, SelShared& sh) {
  const int head = ring_head(a, n), nch = (n - head + kSelChunk - 1) / kSelChunk;
  for (int i = 0; i < kSelRing; ++i) mbar_init(smem_addr(&sh.bar[i]), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  for (int c = 0; c < min(nch, kSelRing); ++c) ring_issue(a, n, head, c, ring, sh);
}

// Streams the scores a[0, n) through the shared-memory ring and gathers, in
// position order, the keys at or above thr into c_key / c_pos (at most
// kSelCap stored).  The head is read directly by warp 0; the chunks arrive
// kSelRing - 1 ahead of the sweep (primed: ring_prime already ran for this
// row).  A sweep whose chunk holds no candidate costs one barrier (which also
// hands its stage back to the copies); a sweep with candidates adds one more
// to exchange the warps' counts.  Returns the number of qualifying keys, or
// -1 when a copy did not complete within limit_ns (the copies still in flight
// are waited for, within a bound, first).  Called by the whole block.
__device__ int gather_ring(const float* __restrict__ a, int n, uint32_t thr, bool primed, float* ring,
                           uint32_t* c_key, int32_t* c_pos, SelShared& sh, uint64_t limit_ns) {
  constexpr int P = kSelChunk / kSelThreads;  // keys per thread per sweep
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const uint32_t lt = (1u << lane) - 1u;  // lanes below this one
  // the float whose order key is thr: keys >= thr are exactly the non-NaN
  // floats >= thr_f (-0 and +0 share one key)
  const float thr_f = __uint_as_float((thr & 0x80000000u) ? (thr & 0x7fffffffu) : ~thr);
  const int head = ring_head(a, n);
  const int nch = (n - head + kSelChunk - 1) / kSelChunk;
  if (t < 32) {
    const uint32_t key = t < head ? order_key(a[t]) : 0u;
    const uint32_t hb = __ballot_sync(kFull, t < head && key >= thr);
    if ((hb >> lane) & 1u) {
      c_key[cand_slot(__popc(hb & lt))] = key;
      c_pos[cand_slot(__popc(hb & lt))] = t;
    }
    if (t == 0) sh.n_head = __popc(hb);
  }
  // Thread 0 alone waits on the ring's barriers: for chunk c + 1 before the
  // barrier that ends sweep c (chunk 0 before the first), so each sweep's
  // chunk is resident once the previous barrier is passed.
  bool ok = true;
  if (t == 0) {
    if (!primed) ring_prime(a, n, ring, sh);
    if (nch > 0) ok = mbar_wait(smem_addr(&sh.bar[0]), 0u, limit_ns);
  }
  auto drain = [&](int first, int end) {  // thread 0: chunks [first, end) were issued, not consumed
    if (t == 0)
      for (int v = first; v < end; ++v)
        if (!(v == 0 && sh.starve) &&  // the test hook's stage has no copy to wait for
            !mbar_wait(smem_addr(&sh.bar[v % kSelRing]), (uint32_t)((v / kSelRing) & 1), limit_ns))
          sh.undrained = 1;
    __syncthreads();
  };
  if (__syncthreads_or(ok ? 0 : 1)) {
    drain(0, min(nch, kSelRing));
    return -1;
  }
  int filled = sh.n_head;
  for (int c = 0; c < nch; ++c) {
    const int st = c % kSelRing, k0 = head + c * kSelChunk;
    const int cnt = min(kSelChunk, n - k0), bulk = cnt & ~3;
    const int i0 = P * t;
    const float* src = ring + (size_t)st * kSelChunk;
    float x[P];
    if (i0 + P <= bulk) {
#pragma unroll
      for (int v = 0; v < P / 4; ++v) {
        const float4 y = reinterpret_cast<const float4*>(src + i0)[v];
        x[4 * v] = y.x;
        x[4 * v + 1] = y.y;
        x[4 * v + 2] = y.z;
        x[4 * v + 3] = y.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < P; ++u) {
        const int i = i0 + u;
        x[u] = i >= cnt ? -INFINITY : (i < bulk ? src[i] : a[k0 + i]);
      }
    }
    // Prefilter in float: !(x < thr_f) holds for every key at or above thr
    // (and for NaN); the exact key test runs only in sweeps where it fires.
    bool maybe = false;
#pragma unroll
    for (int u = 0; u < P; ++u) maybe |= !(x[u] < thr_f);
    if (t == 0 && c + 1 < nch)
      ok = mbar_wait(smem_addr(&sh.bar[(c + 1) % kSelRing]), (uint32_t)(((c + 1) / kSelRing) & 1), limit_ns);
    // every thread has read stage st; any candidate, or a copy that timed out?
    const int flags = __syncthreads_or((maybe ? 1 : 0) | (ok ? 0 : 0x10000));
    if (flags & 0x10000) {
      drain(c + 1, min(nch, c + kSelRing));
      return -1;
    }
    if (t == 0 && c + kSelRing < nch) ring_issue(a, n, head, c + kSelRing, ring, sh);
    if (flags == 0) continue;
    uint32_t sel = 0;  // bit u: key u qualifies
    int below = 0, wcount = 0;  // candidates before this thread's within its warp, and the warp's count
    if (__any_sync(kFull, maybe)) {
#pragma unroll
      for (int u = 0; u < P; ++u) sel |= (uint32_t)(i0 + u < cnt && order_key(x[u]) >= thr) << u;
#pragma unroll
      for (int u = 0; u < P; ++u) {
        const uint32_t bu = __ballot_sync(kFull, (sel >> u) & 1u);
        below += __popc(bu & lt);
        wcount += __popc(bu);
      }
    }
    if (lane == 0) sh.tot[w] = wcount;
    __syncthreads();
    const int tw = sh.tot[lane];
    const int before = (int)__reduce_add_sync(kFull, (uint32_t)(lane < w ? tw : 0));
    const int total = (int)__reduce_add_sync(kFull, (uint32_t)tw);
    int pos = filled + before + below;
#pragma unroll
    for (int u = 0; u < P; ++u)
      if ((sel >> u) & 1u) {
        if (pos < kSelCap) {
          c_key[cand_slot(pos)] = order_key(x[u]);
          c_pos[cand_slot(pos)] = k0 + i0 + u;
        }
        ++pos;
      }
    filled += total;
  }
  __syncthreads();
  if (t == 0)
    for (int i = 0; i < kSelRing; ++i) mbar_inval(smem_addr(&sh.bar[i]));
  __syncthreads();
  return filled;
}

// One CTA per sequence.  The kept set is [0, lo) (sinks), the selected
// positions inside [lo, hi), and [hi, L) (the recent window), where the
// selection is the `heavy` highest scores among the ranked positions [0, n).
// Two passes over the scores in global memory: a histogram of the top byte
// finds the smallest top-byte bucket that, with the buckets above it, holds
// at least `keep` keys; those candidates are gathered, in position order,
// into shared memory, where the exact radix select and the ordered output
// run.  If the candidates do not fit, the select and the output run over
// global memory instead.
__global__ void __launch_bounds__(kSelThreads) h2o_select_kernel(const SeqRow* __restrict__ rows,
                                                                 const float* __restrict__ acc, int64_t acc_stride,
                                                                 SelPolicy pol, int32_t* __restrict__ keep_idx,
                                                                 int64_t keep_stride, int32_t* __restrict__ keep_count,
                                                                 int32_t* __restrict__ status, uint64_t wait_limit_ns,
                                                                 int starve_first) {
  __shared__ SelShared sh;
  if (threadIdx.x == 0) {
    sh.starve = starve_first && blockIdx.x == 0;
    sh.undrained = 0;
  }
  extern __shared__ uint32_t cand[];  // kSelCap keys, kSelCap positions, then the ring
  uint32_t* c_key = cand;
  int32_t* c_pos = reinterpret_cast<int32_t*>(cand + kSelCap);
  float* ring = reinterpret_cast<float*>(cand + 2 * kSelCap);
  const SeqRow row = rows[blockIdx.x];
  const int b = row.q_row, L = row.ctx_len;
  const float* a = acc + (size_t)b * acc_stride;
  int32_t* out = keep_idx + (size_t)b * keep_stride;
  const int hi = max(L - pol.window, 0), lo = min(pol.sinks, hi);
  const int n = pol.rank_all ? L : hi, keep = pol.heavy;
  if (hi <= lo || n <= keep) {  // every position is kept
    for (int j = threadIdx.x; j < L; j += blockDim.x) out[j] = j;
    if (threadIdx.x == 0) keep_count[b] = L;
    return;
  }
  for (int j = threadIdx.x; j < lo; j += blockDim.x) out[j] = j;
  int n_heavy = 0;
  // Gathers, in position order, the keys of [0, n) at or above thr into the
  // shared candidate arrays (at most kSelCap written); returns how many keys
  // qualified, or -1 when a copy timed out.
  auto gather = [&](uint32_t thr, bool primed) {
    return gather_ring(a, n, thr, primed, ring, c_key, c_pos, sh, wait_limit_ns);
  };
  auto timed_out = [&]() {
    if (threadIdx.x == 0) {
      atomicOr(status, sh.undrained ? kStatusTimeout | kStatusUndrained : kStatusTimeout);
      keep_count[b] = 0;
    }
  };
  auto smem_key = [c_key](int i) { return c_key[cand_slot(i)]; };
  auto smem_pos = [c_pos](int i) { return c_pos[cand_slot(i)]; };
  // exact select and ordered output over the m (<= kSelCap) candidates in
  // shared memory, with as few keys per thread as cover m in one sweep
  auto select_candidates = [&](int m) {
    auto run = [&](auto tag) {
      constexpr int U = decltype(tag)::value;
      radix_select<U>(smem_key, m, keep, sh);
      const uint32_t T = sh.prefix;
      const int need_eq = sh.k;
      return ordered_emit<U>(smem_key, smem_pos, m, T, need_eq, lo, hi, out + lo, sh);
    };
    if (m <= 2 * kSelThreads) return run(IntTag<2>{});
    if (m <= 4 * kSelThreads) return run(IntTag<4>{});
    return run(IntTag<kSelCap / kSelThreads>{});
  };
  bool done = false;
  if (keep > 0 && n > kSelSampleMinRow) {
    // Long rows: a strided sample of kSelSample keys gives a threshold a bit
    // below the expected keep-th largest; one pass gathers every key at or
    // above it.  When at least keep (and at most kSelCap) keys qualify, the
    // keep-th largest is among them and the exact select runs on them alone;
    // otherwise the two-pass path below runs.  The row's first chunks stream
    // into the ring while the sample is read and ranked.
    if (threadIdx.x == 0) ring_prime(a, n, ring, sh);
    {
      constexpr int U = kSelSample / kSelThreads;  // every load issued before the first store
      uint32_t sk[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        sk[u] = order_key(a[(int)((int64_t)(threadIdx.x + u * kSelThreads) * n / kSelSample)]);
#pragma unroll
      for (int u = 0; u < U; ++u) c_key[cand_slot(threadIdx.x + u * kSelThreads)] = sk[u];
    }
    __syncthreads();
    const int64_t want = ((int64_t)keep * kSelSample + n - 1) / n * 5 / 4 + 8;
    const int r = want < kSelSample ? (int)want : kSelSample;
    // the r-th largest sample's top 16 bits: a threshold at or below it
    radix_select<kSelSample / kSelThreads>(smem_key, kSelSample, r, sh, 16);
    const uint32_t thr = sh.prefix;
    __syncthreads();
    const int m = gather(thr, true);
    if (m < 0) return timed_out();
    if (m >= keep && m <= kSelCap) {
      n_heavy = select_candidates(m);
      done = true;
    }
  }
  if (keep > 0 && !done) {
    auto global_key = [a](int i) { return order_key(a[i]); };
    auto global_pos = [](int i) { return i; };
    // pass 1: top-byte histogram and the candidate bucket
    digit_histogram<kSelUnroll>(global_key, n, 0u, 0u, 24, sh);
    {
      __shared__ int s_top, s_rest, s_cnt;
      find_digit(sh, keep, &s_top, &s_rest, &s_cnt);
      if (threadIdx.x == 0) {
        sh.top = s_top;
        sh.n_cand = s_cnt;
      }
      __syncthreads();
    }
    const uint32_t lo_key = (uint32_t)sh.top << 24;
    const int m = sh.n_cand;
    if (m <= kSelCap) {
      // pass 2: gather the candidates in position order
      if (gather(lo_key, false) < 0) return timed_out();
      n_heavy = select_candidates(m);
    } else {
      radix_select<kSelUnroll>(global_key, n, keep, sh);
      const uint32_t T = sh.prefix;
      const int need_eq = sh.k;
      n_heavy = ordered_emit<kSelUnroll>(global_key, global_pos, n, T, need_eq, lo, hi, out + lo, sh);
    }
  }
  for (int i = threadIdx.x; i < L - hi; i += blockDim.x) out[lo + n_heavy + i] = hi + i;
  if (threadIdx.x == 0) keep_count[b] = lo + n_heavy + (L - hi);
}

// ---------------------------------------------------------------------------
// H2O compaction: kept tokens move, in order, into fresh blocks (one warp per
// (token, kv head) row: K, V and the FP8 / INT8 scales); the score array follows.
// ---------------------------------------------------------------------------

// Moves each kept (token, kv head) row -- its K and V row and, for one-byte
// codes, the two scales -- from the sequence's current block to its fresh
// block.  A task of 2 x row_bytes / 16 lanes (at most a warp) moves one row
// pair in 16-byte chunks, K in the task's first half and V in its second;
// tasks run head-major (consecutive tasks: consecutive kept tokens of one
// kv head), so neighbouring lanes and warps read and write neighbouring rows.
// Each lane serves kCompactTasks tasks, spaced a grid's worth of tasks
// apart, and issues all their loads before its stores.
constexpr int kCompactTasks = 2;
__global__ void compact_gather_kernel(const CompactSeq* __restrict__ seqs, const int32_t* __restrict__ new_blocks,
                                      const int32_t* __restrict__ tables, int max_blocks, int num_blocks,
                                      const int32_t* __restrict__ keep_idx, int64_t keep_stride, int Hk, int row_bytes,
                                      char* __restrict__ k_pool, char* __restrict__ v_pool,
                                      float* __restrict__ k_scale, float* __restrict__ v_scale,
                                      int32_t* __restrict__ status) {
  const CompactSeq sq = seqs[blockIdx.y];
  const int C = row_bytes / 16;          // chunks per row
  const int per = min(32, 2 * C);        // lanes per task
  const int lane = threadIdx.x & 31, sub = lane % per;
  const int64_t tasks = (int64_t)sq.count * Hk;
  const int64_t slot = ((int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * (32 / per) + lane / per;
  const int64_t span = (int64_t)gridDim.x * (blockDim.x / 32) * (32 / per);  // tasks one round of the grid covers
  size_t srow[kCompactTasks], drow[kCompactTasks];
  bool live[kCompactTasks];
#pragma unroll
  for (int u = 0; u < kCompactTasks; ++u) {
    const int64_t t = slot + u * span;
    live[u] = false;
    if (t >= tasks) continue;
    const int g = (int)(t / sq.count), i = (int)(t - (int64_t)g * sq.count);
    const int src = keep_idx[(size_t)sq.q_row * keep_stride + i];
    const int sb = (src >= 0 && src < sq.old_len) ? tables[(size_t)sq.seq_slot * max_blocks + src / kBlock] : -1;
    if (sb < 0 || sb >= num_blocks) {
      if (sub == 0) atomicOr(status, kStatusBadBlock);
      continue;
    }
    const int db = new_blocks[sq.new_off + i / kBlock];
    srow[u] = ((size_t)sb * Hk + g) * kBlock + (src & 15);
    drow[u] = ((size_t)db * Hk + g) * kBlock + (i & 15);
    live[u] = true;
  }
  for (int q = sub; q < 2 * C; q += per) {
    char* pool = q < C ? k_pool : v_pool;
    const int ch = q < C ? q : q - C;
    uint4 x[kCompactTasks];
#pragma unroll
    for (int u = 0; u < kCompactTasks; ++u)
      if (live[u]) x[u] = reinterpret_cast<const uint4*>(pool + srow[u] * row_bytes)[ch];
#pragma unroll
    for (int u = 0; u < kCompactTasks; ++u)
      if (live[u]) reinterpret_cast<uint4*>(pool + drow[u] * row_bytes)[ch] = x[u];
  }
#pragma unroll
  for (int u = 0; u < kCompactTasks; ++u) {
    if (!live[u]) continue;
    if (k_scale && sub == 0) k_scale[drow[u]] = k_scale[srow[u]];
    if (v_scale && sub == per - 1) v_scale[drow[u]] = v_scale[srow[u]];
  }
}

// acc[b][i] = acc[b][keep_idx[i]] for i < count, zero for count <= i < old_len.
// Kept positions are ascending, so keep_idx[i] >= i: a chunk reads only
// positions no earlier chunk has written, and reads before it writes.
__global__ void __launch_bounds__(1024) compact_scores_kernel(const CompactSeq* __restrict__ seqs,
                                                              const int32_t* __restrict__ keep_idx, int64_t keep_stride,
                                                              float* __restrict__ acc, int64_t acc_stride) {
  constexpr int kChunk = 4096;
  const CompactSeq sq = seqs[blockIdx.x];
  float* a = acc + (size_t)sq.q_row * acc_stride;
  const int32_t* k = keep_idx + (size_t)sq.q_row * keep_stride;
  for (int base = 0; base < sq.count; base += kChunk) {
    float v[kChunk / 1024];
#pragma unroll
    for (int u = 0; u < kChunk / 1024; ++u) {
      const int i = base + u * 1024 + threadIdx.x;
      v[u] = i < sq.count ? a[k[i]] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kChunk / 1024; ++u) {
      const int i = base + u * 1024 + threadIdx.x;
      if (i < sq.count) a[i] = v[u];
    }
    __syncthreads();
  }
  for (int i = sq.count + threadIdx.x; i < sq.old_len; i += blockDim.x) a[i] = 0.0f;
}

// ---------------------------------------------------------------------------
// fp32 decode on CUDA cores: one warp per query head, one CTA per
// (sequence, kv head); online softmax over the kept keys in order.
// ---------------------------------------------------------------------------

template <int D>
__global__ void decode_f32_kernel(const DecodeF32Params p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31, i = threadIdx.x >> 5;
  const SeqRow row = p.rows[blockIdx.x];
  const int g = blockIdx.y, Hk = p.n_kv_heads, G = p.n_heads / Hk, h = g * G + i;
  const int b = row.q_row, L = row.ctx_len;
  float q[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = p.q[((size_t)b * p.n_heads + h) * D + lane + 32 * e];
    o[e] = 0.0f;
  }
  float m = -INFINITY, l = 0.0f;
  const int nk = keep_count_of(L, p.mask_mode, p.num_sinks, p.window);
  for (int k = 0; k < nk; ++k) {
    const int j = keep_pos(k, L, p.mask_mode, p.num_sinks, p.window);
    const int blk = p.tables[(size_t)row.seq_slot * p.max_blocks + j / kBlock];
    if (blk < 0 || blk >= p.num_blocks) {
      if (lane == 0) atomicOr(p.status, kStatusBadBlock);
      continue;
    }
    const size_t r = ((size_t)blk * Hk + g) * kBlock + (j & 15);
    const float* kr = p.k_pool + r * D;
    const float* vr = p.v_pool + r * D;
    float dot = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot += q[e] * kr[lane + 32 * e];
#pragma unroll
    for (int off = 16; off; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
    const float s = dot * p.scale;
    if (p.logits && lane == 0) p.logits[(((size_t)b * Hk + g) * p.logits_stride + j) * G + i] = s;
    const float mn = fmaxf(m, s);
    const float alpha = expf(m - mn);
    const float pj = expf(s - mn);
    l = l * alpha + pj;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = o[e] * alpha + pj * vr[lane + 32 * e];
    m = mn;
  }
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) p.out[((size_t)b * p.n_heads + h) * D + lane + 32 * e] = o[e] * inv;
  if (p.lse && lane == 0) p.lse[(size_t)b * p.n_heads + h] = l > 0.0f ? m + logf(l) : -INFINITY;
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  if (g > 65535LL * 32) g = 65535LL * 32;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  if (a.n_tokens <= 0 && a.n_patches <= 0) return cudaSuccess;
  if (a.kv_dtype == 2 || a.kv_dtype == 3) {
    const int64_t warps = 2LL * a.n_tokens * a.Hk;
    const int grid = grid_for(std::max<int64_t>(warps * 32, a.n_patches), 256);
    if (a.D != 64 && a.D != 128) return cudaErrorInvalidValue;
    if (a.kv_dtype == 3) {
      if (a.D == 64)
        append_quant_kernel<3, 64><<<grid, 256, 0, st>>>(a);
      else
        append_quant_kernel<3, 128><<<grid, 256, 0, st>>>(a);
    } else {
      if (a.D == 64)
        append_quant_kernel<2, 64><<<grid, 256, 0, st>>>(a);
      else
        append_quant_kernel<2, 128><<<grid, 256, 0, st>>>(a);
    }
  } else {
    const int row_chunks = a.D * (a.kv_dtype == 0 ? 4 : 2) / 16;
    const int64_t work = 2LL * a.n_tokens * a.Hk * row_chunks;
    append_copy_kernel<<<grid_for(std::max<int64_t>(work, a.n_patches), 256), 256, 0, st>>>(a, row_chunks);
  }
  return cudaGetLastError();
}

cudaError_t launch_block_copy(const int32_t* pairs, int n_pairs, const void* src_k, const void* src_v,
                              const float* src_ks, const float* src_vs, void* dst_k, void* dst_v, float* dst_ks,
                              float* dst_vs, size_t block_bytes, size_t scale_floats, cudaStream_t st) {
  if (n_pairs <= 0) return cudaSuccess;
  const int64_t chunks = (int64_t)(block_bytes / 16);
  for (int first = 0; first < n_pairs; first += 65535) {
    const int n = std::min(65535, n_pairs - first);
    dim3 grid((unsigned)std::min<int64_t>((chunks + 255) / 256, 64), (unsigned)n);
    block_copy_kernel<<<grid, 256, 0, st>>>(pairs + 2 * first, (const uint4*)src_k, (const uint4*)src_v,
                                            (uint4*)dst_k, (uint4*)dst_v, chunks, scale_floats ? src_ks : nullptr,
                                            scale_floats ? src_vs : nullptr, dst_ks, dst_vs, (int64_t)scale_floats);
    if (cudaError_t e = cudaGetLastError()) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_cow_copy(const int32_t* pairs, int n_pairs, void* k_pool, void* v_pool, float* k_scale,
                            float* v_scale, size_t block_bytes, size_t scale_floats, cudaStream_t st) {
  return launch_block_copy(pairs, n_pairs, k_pool, v_pool, k_scale, v_scale, k_pool, v_pool, k_scale, v_scale,
                           block_bytes, scale_floats, st);
}

cudaError_t launch_table_patch(const int32_t* patches, int n, int32_t* tables, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  table_patch_kernel<<<std::min((n + 255) / 256, 1024), 256, 0, st>>>(patches, n, tables);
  return cudaGetLastError();
}

cudaError_t launch_h2o_score(const SeqRow* rows, int n_seqs, int n_heads, int n_kv_heads, const float* logits,
                             int64_t stride, const float* lse, int mode, int S, int W, float* acc, int64_t acc_stride,
                             int max_keep, cudaStream_t st) {
  if (n_seqs <= 0 || max_keep <= 0) return cudaSuccess;
  dim3 grid((unsigned)((max_keep + 255) / 256), (unsigned)n_seqs);
  h2o_score_kernel<<<grid, 256, n_heads * sizeof(float), st>>>(rows, n_heads, n_kv_heads, logits, stride, lse, mode,
                                                                S, W, acc, acc_stride);
  return cudaGetLastError();
}

cudaError_t launch_compact_gather(const CompactSeq* seqs, int n, int max_count, const int32_t* new_blocks,
                                  const int32_t* tables, int max_blocks, int num_blocks, const int32_t* keep_idx,
                                  int64_t keep_stride, int Hk, int row_bytes, void* k_pool, void* v_pool, float* k_scale,
                                  float* v_scale, int32_t* status, cudaStream_t st) {
  if (n <= 0 || max_count <= 0) return cudaSuccess;
  const int tasks_per_warp = 32 / std::min(32, 2 * (row_bytes / 16)) * kCompactTasks;
  const int64_t warps = ((int64_t)max_count * Hk + tasks_per_warp - 1) / tasks_per_warp;
  for (int first = 0; first < n; first += 65535) {  // grid.y limit
    dim3 grid((unsigned)((warps + 7) / 8), (unsigned)std::min(65535, n - first));
    compact_gather_kernel<<<grid, 256, 0, st>>>(seqs + first, new_blocks, tables, max_blocks, num_blocks, keep_idx,
                                                keep_stride, Hk, row_bytes, (char*)k_pool, (char*)v_pool, k_scale,
                                                v_scale, status);
    if (cudaError_t e = cudaGetLastError()) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_compact_scores(const CompactSeq* seqs, int n, const int32_t* keep_idx, int64_t keep_stride,
                                  float* acc, int64_t acc_stride, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  compact_scores_kernel<<<n, 1024, 0, st>>>(seqs, keep_idx, keep_stride, acc, acc_stride);
  return cudaGetLastError();
}

cudaError_t launch_h2o_select(const SeqRow* rows, int n_seqs, const float* acc, int64_t acc_stride,
                              const SelPolicy& pol, int32_t* keep_idx, int64_t keep_stride, int32_t* keep_count,
                              int32_t* status, uint64_t wait_limit_ns, bool starve_first, cudaStream_t st) {
  if (n_seqs <= 0) return cudaSuccess;
  static std::atomic<uint64_t> attr_set{0};  // one bit per device
  const int smem = (int)kSelSmem;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const uint64_t bit = dev < 64 ? uint64_t(1) << dev : 0;
  if (!(attr_set.load() & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(h2o_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  h2o_select_kernel<<<n_seqs, kSelThreads, smem, st>>>(rows, acc, acc_stride, pol, keep_idx, keep_stride, keep_count,
                                                       status, wait_limit_ns, starve_first ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_decode_f32(const DecodeF32Params& p, cudaStream_t st) {
  if (p.n_seqs <= 0) return cudaSuccess;
  dim3 grid((unsigned)p.n_seqs, (unsigned)p.n_kv_heads);
  const int threads = 32 * (p.n_heads / p.n_kv_heads);
  if (p.head_dim == 64)
    decode_f32_kernel<64><<<grid, threads, 0, st>>>(p);
  else
    decode_f32_kernel<128><<<grid, threads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
