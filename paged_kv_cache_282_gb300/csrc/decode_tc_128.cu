// decode_tc_128.cu -- the decode kernel of decode_tc.cuh instantiated for
// head_dim 128 (BF16, FP8-E4M3 and INT8 KV; G in {1, 2, 4, 8}; one or two
// sequences per warp), with its launch, shared-memory and occupancy dispatch,
// and the shared-prefix multi-query kernel (BF16, head_dim 128).

#include "decode_tc.cuh"

namespace pkv {

// hg: 1, or tc_head_group(kv_dtype, G, 128) kv heads per unit.
cudaError_t launch_decode_tc_d128(int kv_dtype, int G, int hg, int nq, const DecodeTCParams& p, int ctas,
                                 cudaStream_t st) {
  if (ctas <= 0) return cudaSuccess;
#define X(KV, GG, NQ)                                                           \
  if (kv_dtype == KV && G == GG && nq == NQ) {                                  \
    constexpr int H = tc_head_group(KV, GG, 128);                                 \
    if (hg == 1) return launch_t<KV, GG, 1, NQ, 128>(p, ctas, st);                \
    if (hg == H) return launch_t<KV, GG, H, NQ, 128>(p, ctas, st);                \
    return cudaErrorInvalidValue;                                               \
  }
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t decode_tc_prepare_d128(int kv_dtype, int G, int hg, int nq) {
#define X(KV, GG, NQ)                                                           \
  if (kv_dtype == KV && G == GG && nq == NQ) {                                  \
    constexpr int H = tc_head_group(KV, GG, 128);                                 \
    if (hg == 1) return prepare_t<KV, GG, 1, NQ, 128>();                          \
    if (hg == H) return prepare_t<KV, GG, H, NQ, 128>();                          \
    return cudaErrorInvalidValue;                                               \
  }
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t decode_tc_occupancy_d128(int kv_dtype, int G, int hg, int nq, int* n) {
#define X(KV, GG, NQ)                                                           \
  if (kv_dtype == KV && G == GG && nq == NQ) {                                  \
    constexpr int H = tc_head_group(KV, GG, 128);                                 \
    if (hg == 1) return occupancy_t<KV, GG, 1, NQ, 128>(n);                       \
    if (hg == H) return occupancy_t<KV, GG, H, NQ, 128>(n);                       \
    return cudaErrorInvalidValue;                                               \
  }
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

namespace {

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
    bool drained = true;
    for (int v = ch; v < issued; ++v)
      drained &= mbar_wait(full + 8 * (v % kPStages), (uint32_t)((v / kPStages) & 1), kDrainTimeoutNs);
    if (!drained) atomicOr(p.status, kStatusUndrained);
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
      merge_partials<G, 128>(p, p.combine[mb.item], lane);
    }
  }
}

}  // namespace

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
