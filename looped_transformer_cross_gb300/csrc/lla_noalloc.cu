// lla_noalloc.cu — lla_decode_attn_noalloc: the decode entry point for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where a device allocation is not allowed or not
// wanted — a plugin inside a host framework whose memory pool owns the whole
// GPU, or a latency-critical serving path that must never call cudaMalloc
// (which can synchronise the device and can fail at run time).  Such callers
// still own their inputs and outputs; only the decode scratch (split-KV
// records, the query-operand images and the status word) moves into a fixed array that
// this library defines.
//
// The array is a file-scope __device__ variable of LLA_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (that device
// current) and caches it.  Every call shares the array and it keeps the last
// call's contents; the status word is cleared on the caller's stream once the
// host checks have passed, before the first launch, and lla_device_status with
// no workspace reads it back.  Calls that overlap on the GPU (different streams,
// or several host threads) race on the array and must be serialised by the caller.
#include <mutex>

#include "lla_kernels.h"

namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[LLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

namespace lla {

// Device address of g_noalloc_scratch on the current device (looked up once).
lla_status noalloc_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LLA_OK;
}

}  // namespace lla

extern "C" lla_status lla_decode_attn_noalloc(const lla_dims* dims, int loop_t, const void* q,
                                              lla_cache cache, const int32_t* seq_lens,
                                              const int32_t* q_pos, const void* w_up_k,
                                              const void* w_up_v, const float* mu_k,
                                              const float* mu_v, const float* rope_cos,
                                              const float* rope_sin, int64_t rope_len, float* out,
                                              float* lse, void* stream) {
  const size_t need = lla_workspace_size(dims, cache.B, cache.L_max, 0);
  if (need == 0)  // invalid dims: let the workspace entry point report which error
    return lla_decode_attn(dims, loop_t, q, cache, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v,
                           rope_cos, rope_sin, rope_len, out, lse, nullptr, 0, stream);
  if (need > LLA_NOALLOC_SCRATCH_BYTES) return LLA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const lla_status st = lla::noalloc_scratch_address(&scratch);
  if (st != LLA_OK) return st;
  // the status word is zeroed on `stream` only once every host check has passed
  return lla::decode_attn_status_cleared(dims, loop_t, q, cache, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v,
                                         rope_cos, rope_sin, rope_len, out, lse, scratch,
                                         LLA_NOALLOC_SCRATCH_BYTES, stream);
}
