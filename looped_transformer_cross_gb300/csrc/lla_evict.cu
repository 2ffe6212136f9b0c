// lla_evict.cu — token eviction composed with LLA ("Looped Latent Attention:
// Cross-Loop KV Compression for Looped Transformers", arXiv 2607.15456v2, Appendix D
// "Token-eviction composition table", Table 9, and Appendix J "Eviction and
// long-context prefill").
//
// A StreamingLLM/H2O-style budget keeps the first `sink` tokens and the `window`
// newest; with LLA only the kept tokens' latents are stored, so the two savings
// multiply.  For every sequence with L > sink + window the window's latent rows
// L-window .. L-1 move in order to slots sink .. sink+window-1 (in place, every head,
// both axes), then the sequence's length becomes sink + window.  A later decode
// rotates slot j at position j (positions within the kept cache).
//
// evict_move_kernel: block = (sequence, head or LLA-2D latent, axis).  The window
// moves D = L - window - sink rows towards the front; it is copied in chunks of at
// most D rows, each staged in shared memory between two block barriers, so a chunk
// writes only rows an earlier chunk has already read (or evicted rows).
// evict_lens_kernel (after it, same stream): the new lengths.
#include "lla_kernels.h"

namespace lla {

namespace {

constexpr int kEvictThreads = 256;
constexpr int kStageBytes = 32768;            // one chunk in shared memory

__device__ __forceinline__ bool over_budget(const EvictArgs& a, int b, int& L) {
  L = __ldg(a.seq_lens + b);
  if (L < 0 || L > a.L_max) return false;
  return L > a.sink + a.window;
}

__global__ void __launch_bounds__(kEvictThreads) evict_move_kernel(const __grid_constant__ EvictArgs a) {
  __shared__ uint4 stage[kStageBytes / 16];
  const int unit = blockIdx.x, axis = blockIdx.y, tid = threadIdx.x;
  const int b = unit / a.units_per_seq;
  int L;
  if (!over_budget(a, b, L)) return;
  const int r = axis == 0 ? a.r_k : a.r_v;
  const int64_t rb = static_cast<int64_t>(r) * a.esize;             // row bytes, a multiple of 32
  uint8_t* rows = static_cast<uint8_t*>(axis == 0 ? a.cache_k : a.cache_v) + static_cast<int64_t>(unit) * a.L_max * rb;
  const uint8_t* src = rows + static_cast<int64_t>(L - a.window) * rb;
  uint8_t* dst = rows + static_cast<int64_t>(a.sink) * rb;
  const int D = L - a.window - a.sink;                              // shift, >= 1
  const int C = min(D, static_cast<int>(kStageBytes / rb));         // rows per chunk
  for (int c0 = 0; c0 < a.window; c0 += C) {
    const int n16 = static_cast<int>(min(C, a.window - c0) * rb / 16);
    const uint4* s4 = reinterpret_cast<const uint4*>(src + c0 * rb);
    for (int i = tid; i < n16; i += kEvictThreads) stage[i] = s4[i];
    __syncthreads();
    uint4* d4 = reinterpret_cast<uint4*>(dst + c0 * rb);
    for (int i = tid; i < n16; i += kEvictThreads) d4[i] = stage[i];
    __syncthreads();
  }
}

__global__ void evict_lens_kernel(const __grid_constant__ EvictArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.B) return;
  const int L = a.seq_lens[b];
  if (L < 0 || L > a.L_max) {
    record_status(a.status, LLA_ERR_DEVICE_ARG);
    return;
  }
  if (L > a.sink + a.window) a.seq_lens[b] = a.sink + a.window;
}

}  // namespace

cudaError_t launch_evict_window(const EvictArgs& a, cudaStream_t s) {
  if (a.window > 0) {
    evict_move_kernel<<<dim3(static_cast<unsigned>(a.B) * a.units_per_seq, 2), kEvictThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  evict_lens_kernel<<<(a.B + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lla
