// lla_paged_generic.cu — bf16 decode over a paged latent cache whose page size the
// tile kernel's copy path does not take ("Enabling dynamic computation in Looped
// LMs", §"Ragged KV" and App. A.1: a page table per sequence; its vLLM setting is
// one-token pages).  The tile kernel copies a 128-token tile as whole pages or as
// 128/P pieces of P tokens (P a multiple of 8 dividing 128); every other page size
// comes here.
//
// One CTA per (sequence, head), 128 threads, one token per thread per 128-token
// tile, token rows gathered one by one through the block table.  The score is that
// of the LLA paper's Eq. (3) with RoPE after reconstruction, regrouped per frequency
// pair f = (i0, i1):
//     s_j = sum_f cos(j th_f) (Zc_f . c_j + bc_f) + sin(j th_f) (Zs_f . c_j + bs_f),
// with Zc_f = q'_i0 W_i0 + q'_i1 W_i1, Zs_f = q'_i1 W_i0 - q'_i0 W_i1 (q' = RoPE(q,
// q_pos), W = W_up,k,t rows) and bc, bs the same forms over mu_k,t: an exact
// reassociation of q'.RoPE(W c_j + mu, j).  Zc, Zs are rounded once to bf16, as the
// tile kernel's query operand is.  Online softmax in fp32 over the tiles; the value
// path accumulates sum_j p_j c_v,j and applies W_up,v,t once at the end (Appendix J
// "Absorbed attention").  Slow next to the tile kernel (the gather is per row and the
// 128 x r_k contraction per token runs on the CUDA cores), but any page size >= 1
// works.
#include "lla_kernels.h"

namespace lla {

namespace {

constexpr int kGenThreads = 128;
constexpr float kGenInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)

__device__ __forceinline__ int gen_clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

// Dynamic shared memory: Z pairs [r_k][64] (bf16 Zc_f, Zs_f per 32-bit word), then the
// tile's K rows [128][r_k] and V rows [128][r_v] (rows padded by 16 bytes, so the
// 16-byte row reads of consecutive threads fall in distinct banks).
__global__ void __launch_bounds__(kGenThreads)
decode_paged_generic_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float bc[64], bs[64], qr[kHeadDim], pw[kGenThreads], red[4], acc[256];
  const int rk = a.r_k, rv = a.r_v;
  const int ckst = rk * 2 + 16, cvst = rv * 2 + 16;
  uint32_t* zw = reinterpret_cast<uint32_t*>(smem);                   // [rk][64]
  uint8_t* ck = smem + static_cast<size_t>(rk) * 64 * 4;             // [128][ckst]
  uint8_t* cv = ck + static_cast<size_t>(kGenThreads) * ckst;         // [128][cvst]
  const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int b = u / a.H, h = u % a.H;
  const int L0 = __ldg(a.seq_lens + b);
  if ((L0 < 0 || L0 > a.L_max) && tid == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
  const int L = gen_clamp_len(L0, a.L_max);
  float* out = a.out + static_cast<int64_t>(u) * kHeadDim;
  if (L == 0) {
    out[tid] = 0.f;
    if (tid == 0) a.lse[u] = -INFINITY;
    return;
  }
  int qp = __ldg(a.q_pos + b);
  if (qp < 0 || qp >= a.rope_len) {
    if (tid == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
  }
  auto pair_of = [&](int f, int& i0, int& i1) {
    i0 = a.rope_style == 0 ? f : 2 * f;
    i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
  };
  // ---- rotated query, folded query operand (Zc, Zs) and its bias terms
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + static_cast<int64_t>(u) * kHeadDim;
  if (tid < 64) {
    int i0, i1;
    pair_of(tid, i0, i1);
    const float c = __ldg(a.rope_cos + static_cast<int64_t>(qp) * 64 + tid);
    const float sn = __ldg(a.rope_sin + static_cast<int64_t>(qp) * 64 + tid);
    const float x0 = __bfloat162float(q[i0]), x1 = __bfloat162float(q[i1]);
    qr[i0] = x0 * c - x1 * sn;
    qr[i1] = x0 * sn + x1 * c;
  }
  __syncthreads();
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * rk;
  const float* mk = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
  for (int idx = tid; idx < 64 * rk; idx += kGenThreads) {
    const int f = idx % 64, k = idx / 64;
    int i0, i1;
    pair_of(f, i0, i1);
    const float w0 = __bfloat162float(W[static_cast<int64_t>(i0) * rk + k]);
    const float w1 = __bfloat162float(W[static_cast<int64_t>(i1) * rk + k]);
    const __nv_bfloat162 z = __floats2bfloat162_rn(qr[i0] * w0 + qr[i1] * w1, qr[i1] * w0 - qr[i0] * w1);
    zw[k * 64 + f] = *reinterpret_cast<const uint32_t*>(&z);
  }
  if (tid < 64) {
    int i0, i1;
    pair_of(tid, i0, i1);
    bc[tid] = qr[i0] * mk[i0] + qr[i1] * mk[i1];
    bs[tid] = qr[i1] * mk[i0] - qr[i0] * mk[i1];
  }
  for (int k = tid; k < rv; k += kGenThreads) acc[k] = 0.f;
  __syncthreads();

  const __nv_bfloat16* CK = static_cast<const __nv_bfloat16*>(a.cache_k);
  const __nv_bfloat16* CV = static_cast<const __nv_bfloat16*>(a.cache_v);
  float m_run = -INFINITY, l_run = 0.f;
  for (int j0 = 0; j0 < L; j0 += kGenThreads) {
    const int j = j0 + tid;
    const bool valid = j < L;
    // ---- gather this thread's token rows (its page through the block table)
    if (valid) {
      const int64_t row = latent_row(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max, a.H, b, h, j,
                                     a.status);
      const uint4* sk = reinterpret_cast<const uint4*>(CK + row * rk);
      const uint4* sv = reinterpret_cast<const uint4*>(CV + row * rv);
      uint4* dk = reinterpret_cast<uint4*>(ck + static_cast<size_t>(tid) * ckst);
      uint4* dv = reinterpret_cast<uint4*>(cv + static_cast<size_t>(tid) * cvst);
      for (int i = 0; i < rk / 8; ++i) dk[i] = __ldg(sk + i);
      for (int i = 0; i < rv / 8; ++i) dv[i] = __ldg(sv + i);
    }
    __syncthreads();
    // ---- score of this thread's token
    float s = -INFINITY;
    if (valid) {
      float A[64], Bs[64];
#pragma unroll
      for (int f = 0; f < 64; ++f) { A[f] = 0.f; Bs[f] = 0.f; }
      const uint4* crow = reinterpret_cast<const uint4*>(ck + static_cast<size_t>(tid) * ckst);
      for (int k0 = 0; k0 < rk; k0 += 8) {
        float c8[8];
        unpack_bf16x8(crow[k0 / 8], c8);
#pragma unroll 2
        for (int kk = 0; kk < 8; ++kk) {
          const uint4* zr = reinterpret_cast<const uint4*>(zw + (k0 + kk) * 64);
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            const uint4 z4 = zr[g];
            const uint32_t zz[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 z2 = *reinterpret_cast<const __nv_bfloat162*>(&zz[e]);
              A[4 * g + e] = fmaf(c8[kk], __low2float(z2), A[4 * g + e]);
              Bs[4 * g + e] = fmaf(c8[kk], __high2float(z2), Bs[4 * g + e]);
            }
          }
        }
      }
      const float* cr = a.rope_cos + static_cast<int64_t>(j) * 64;
      const float* sr = a.rope_sin + static_cast<int64_t>(j) * 64;
      s = 0.f;
#pragma unroll
      for (int f = 0; f < 64; f += 4) {
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(cr + f));
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(sr + f));
        s = fmaf(c4.x, A[f] + bc[f], fmaf(s4.x, Bs[f] + bs[f], s));
        s = fmaf(c4.y, A[f + 1] + bc[f + 1], fmaf(s4.y, Bs[f + 1] + bs[f + 1], s));
        s = fmaf(c4.z, A[f + 2] + bc[f + 2], fmaf(s4.z, Bs[f + 2] + bs[f + 2], s));
        s = fmaf(c4.w, A[f + 3] + bc[f + 3], fmaf(s4.w, Bs[f + 3] + bs[f + 3], s));
      }
      s *= kGenInvSqrtD;
    }
    // ---- online softmax over the tile
    float mt = warp_max(s);
    if (lane == 0) red[wid] = mt;
    __syncthreads();
    mt = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float m_new = fmaxf(m_run, mt);
    const float scale = expf(m_run - m_new);   // m_run = -inf on the first tile: 0
    const float p = valid ? expf(s - m_new) : 0.f;
    pw[tid] = p;
    __syncthreads();   // pw complete; red free again
    float ps = warp_sum(p);
    if (lane == 0) red[wid] = ps;
    const int nt = min(kGenThreads, L - j0);
    for (int k = tid; k < rv; k += kGenThreads) {
      float v = acc[k] * scale;
      for (int i = 0; i < nt; ++i)
        v = fmaf(pw[i], __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(cv + static_cast<size_t>(i) * cvst)[k]),
                 v);
      acc[k] = v;
    }
    __syncthreads();   // red sums complete; rows free for the next tile
    l_run = l_run * scale + (red[0] + red[1] + red[2] + red[3]);
    m_run = m_new;
    __syncthreads();   // everyone read red before the next tile writes it
  }
  // ---- out = (acc W_up,v,t^T) / l + mu_v,t ; lse = m + ln l
  const __nv_bfloat16* Wv = static_cast<const __nv_bfloat16*>(a.w_up_v) + (static_cast<int64_t>(h) * kHeadDim + tid) * rv;
  float o = 0.f;
  for (int k = 0; k < rv; ++k) o = fmaf(acc[k], __bfloat162float(Wv[k]), o);
  out[tid] = o / l_run + a.mu_v[static_cast<int64_t>(h) * a.mu_hstride + tid];
  if (tid == 0) a.lse[u] = m_run + logf(l_run);
}

}  // namespace

size_t decode_paged_generic_smem(int r_k, int r_v) {
  return static_cast<size_t>(r_k) * 64 * 4 + static_cast<size_t>(kGenThreads) * (r_k * 2 + 16) +
         static_cast<size_t>(kGenThreads) * (r_v * 2 + 16);
}

cudaError_t launch_decode_paged_generic(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = decode_paged_generic_smem(a.r_k, a.r_v);
  static size_t configured = 0;
  if (configured < smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_paged_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  decode_paged_generic_kernel<<<a.B * a.H, kGenThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lla
