// decode_static.cu -- decode attention whose scratch memory is a fixed array
// compiled into the library, for callers that cannot allocate device memory
// themselves (see pkv_decode_attn_static in include/pkv.h).
//
// The scratch holds the per-call work plan (and any queued copy-on-write pairs
// and block-table updates) in its first kPlanBytes and the split-KV partial
// records in the rest.  Every device that runs this entry point keeps the
// array until the process exits.  All calls share it: two calls whose work
// overlaps on the GPU (different streams, or different pools on one device
// used concurrently) race on it.  Nothing in it needs to start at zero -- each
// call writes every plan byte and every partial record it later reads.

#include <mutex>

#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr size_t kPlanBytes = size_t(2) << 20;      // first 2 MiB: plan and queued updates
constexpr int kMaxDevices = 64;

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device

}  // namespace

static __device__ __align__(256) unsigned char g_pkv_static_scratch[kScratchBytes];

extern "C" pkv_status pkv_decode_attn_static(pkv_pool* pool, void* stream, int32_t n_seqs, const int32_t* seq_ids,
                                             const void* q, float scale, int32_t mask_mode, int32_t num_sinks,
                                             int32_t window, int32_t num_splits, void* out, float* lse,
                                             float* logits, int64_t logits_stride) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    pkv::set_error("pkv_decode_attn_static: no usable current CUDA device");
    return PKV_ERR_CUDA;
  }
  void* base = nullptr;
  {
    // Set-up, once per device, with that device current: in host code the
    // array's name is only a stand-in; its address on this device comes from
    // the runtime.
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_pkv_static_scratch);
      if (e != cudaSuccess || !ptr) {
        pkv::set_error(cudaGetErrorString(e));
        return PKV_ERR_CUDA;
      }
      g_scratch_addr[dev] = ptr;
    }
    base = g_scratch_addr[dev];
  }
  return (pkv_status)pkv::decode_attn_into(pool, stream, n_seqs, seq_ids, q, scale, mask_mode, num_sinks, window,
                                           num_splits, out, lse, logits, logits_stride, base, kPlanBytes,
                                           static_cast<char*>(base) + kPlanBytes, kScratchBytes - kPlanBytes);
}
