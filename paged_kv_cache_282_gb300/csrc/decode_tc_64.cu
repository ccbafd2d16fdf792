// decode_tc_64.cu -- the decode kernel of decode_tc.cuh instantiated for
// head_dim 64 (BF16, FP8-E4M3 and INT8 KV; G in {1, 2, 4, 8}; one or two
// sequences per warp), with its launch, shared-memory and occupancy dispatch.

#include "decode_tc.cuh"

namespace pkv {

// hg: 1, or tc_head_group(kv_dtype, G, 64) kv heads per unit.
cudaError_t launch_decode_tc_d64(int kv_dtype, int G, int hg, int nq, const DecodeTCParams& p, int ctas,
                                 cudaStream_t st) {
  if (ctas <= 0) return cudaSuccess;
#define X(KV, GG, NQ)                                                           \
  if (kv_dtype == KV && G == GG && nq == NQ) {                                  \
    constexpr int H = tc_head_group(KV, GG, 64);                                 \
    if (hg == 1) return launch_t<KV, GG, 1, NQ, 64>(p, ctas, st);                \
    if (hg == H) return launch_t<KV, GG, H, NQ, 64>(p, ctas, st);                \
    return cudaErrorInvalidValue;                                               \
  }
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t decode_tc_prepare_d64(int kv_dtype, int G, int hg, int nq) {
#define X(KV, GG, NQ)                                                           \
  if (kv_dtype == KV && G == GG && nq == NQ) {                                  \
    constexpr int H = tc_head_group(KV, GG, 64);                                 \
    if (hg == 1) return prepare_t<KV, GG, 1, NQ, 64>();                          \
    if (hg == H) return prepare_t<KV, GG, H, NQ, 64>();                          \
    return cudaErrorInvalidValue;                                               \
  }
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t decode_tc_occupancy_d64(int kv_dtype, int G, int hg, int nq, int* n) {
#define X(KV, GG, NQ)                                                           \
  if (kv_dtype == KV && G == GG && nq == NQ) {                                  \
    constexpr int H = tc_head_group(KV, GG, 64);                                 \
    if (hg == 1) return occupancy_t<KV, GG, 1, NQ, 64>(n);                       \
    if (hg == H) return occupancy_t<KV, GG, H, NQ, 64>(n);                       \
    return cudaErrorInvalidValue;                                               \
  }
  PKV_FOR_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace pkv
