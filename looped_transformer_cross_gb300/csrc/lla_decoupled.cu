// lla_decoupled.cu — absorbed decoupled-RoPE decode, fp32 mode ("Looped Latent
// Attention: Cross-Loop KV Compression for Looped Transformers", arXiv 2607.15456v2,
// Appendix J "Absorbed attention", Tables 13-14).
//
// Appendix J moves the K up-projection to the query side, q^T (W_up c) =
// (W_up^T q)^T c, and, since RoPE blocks that for the rotary part, keeps an
// MLA-style NoPE content path on the latents plus a small explicit rotary branch
// (d_rope = 64) stored once per token for all loops.  Per (sequence, head) at loop t:
//   w  = W_up,k,t^T q_c,  b0 = q_c . mu_k,t              (absorbed content query)
//   s_j = (w . c_k,j + b0 + RoPE(q_r, q_pos) . RoPE(r_j, j)) / sqrt(d + d_rope)
//   out = (sum_j p_j c_v,j) W_up,v,t^T + mu_v,t           (absorbed values)
// with the rotary branch's frequencies base^(-2f/d_rope).  Nothing of width d is
// ever formed per token: the content score is an r_k-long dot product on the latent.
//
// This file holds the fp32 mode: one block per (unit, 128-token tile) writes the
// scores, then the shared fp32 softmax / V kernel finishes.  The bf16 storage runs on
// the tensor-core kernels of lla_decoupled_tc.cu.
#include "lla_kernels.h"

#include <cmath>

namespace lla {

namespace {

constexpr int kRope = 64;   // rotary branch width supported

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

// Rotary pair (i0, i1) of frequency f within the d_rope branch.
__host__ __device__ __forceinline__ void rope_pair(int style, int f, int& i0, int& i1) {
  i0 = style == 0 ? f : 2 * f;
  i1 = style == 0 ? f + kRope / 2 : 2 * f + 1;
}

// fp32 mode: block = (unit, 128-token tile), thread = token; scores in natural units.
__global__ void __launch_bounds__(128) decoupled_f32_scores_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float w[256], qr[kRope], red[4];
  const int u = blockIdx.x, tid = threadIdx.x;
  const int b = u / a.H, h = u % a.H;
  const int L = clamp_len(__ldg(a.seq_lens + b), a.L_max);
  const int j0 = blockIdx.y * kTile;
  if (j0 >= L) return;
  int qp = __ldg(a.q_pos + b);
  if (qp < 0 || qp >= a.rope_len) {
    if (tid == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
  }
  const float* qv = static_cast<const float*>(a.q) + static_cast<int64_t>(u) * (kHeadDim + kRope);
  const float* W = static_cast<const float*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * a.r_k;
  for (int k = tid; k < a.r_k; k += 128) {
    float s = 0.f;
    for (int e = 0; e < kHeadDim; ++e) s = fmaf(qv[e], W[e * a.r_k + k], s);
    w[k] = s;
  }
  {
    float part = qv[tid] * a.mu_k[static_cast<int64_t>(h) * a.mu_hstride + tid];
    part = warp_sum(part);
    if ((tid & 31) == 0) red[tid >> 5] = part;
  }
  if (tid < kRope / 2) {
    int i0, i1;
    rope_pair(a.rope_style, tid, i0, i1);
    const float c = a.rope_cos[static_cast<int64_t>(qp) * (kRope / 2) + tid];
    const float s = a.rope_sin[static_cast<int64_t>(qp) * (kRope / 2) + tid];
    const float x0 = qv[kHeadDim + i0], x1 = qv[kHeadDim + i1];
    qr[i0] = x0 * c - x1 * s;
    qr[i1] = x0 * s + x1 * c;
  }
  __syncthreads();
  const int j = j0 + tid;
  if (j >= L) return;
  const float* ck = static_cast<const float*>(a.cache_k) + (static_cast<int64_t>(u) * a.L_max + j) * a.r_k;
  const float* rk = static_cast<const float*>(a.k_rope) + (static_cast<int64_t>(u) * a.L_max + j) * kRope;
  float s = red[0] + red[1] + red[2] + red[3];
  for (int k = 0; k < a.r_k; ++k) s = fmaf(w[k], ck[k], s);
  for (int f = 0; f < kRope / 2; ++f) {
    int i0, i1;
    rope_pair(a.rope_style, f, i0, i1);
    const float c = a.rope_cos[static_cast<int64_t>(j) * (kRope / 2) + f];
    const float sn = a.rope_sin[static_cast<int64_t>(j) * (kRope / 2) + f];
    const float k0 = rk[i0] * c - rk[i1] * sn, k1 = rk[i0] * sn + rk[i1] * c;
    s = fmaf(qr[i0], k0, fmaf(qr[i1], k1, s));
  }
  a.scores[static_cast<int64_t>(u) * a.L_max + j] = s * rsqrtf(static_cast<float>(kHeadDim + kRope));
}

}  // namespace

cudaError_t launch_decoupled_f32(const DecodeArgs& a, cudaStream_t s) {
  const dim3 g1(a.B * a.H, static_cast<unsigned>((a.L_max + kTile - 1) / kTile));
  decoupled_f32_scores_kernel<<<g1, 128, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_decode_f32_values(a, s);
}

}  // namespace lla
