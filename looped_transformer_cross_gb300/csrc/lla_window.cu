// lla_window.cu — exact attention over each sequence's window of recent tokens,
// merged into the latent-store result by log-sum-exp ("Hybrid Latent Attention for
// Looped Language Models", §3.4 "Exact sliding window", Eq. (4); Appendix I
// "Serving Implementation", one decoding step).
//
// Eq. (4) puts the latent tokens' scores and the window tokens' exact scores into
// one softmax.  lla_decode_attn returns the latent part normalised on its own with
// its log-sum-exp; this kernel forms the window part the same way and merges the
// two, which equals the single softmax.  Block = one (sequence, head): the window's
// keys and values arrive in shared memory as plain bulk copies of 32-token chunks,
// double-buffered, each warp runs an online softmax over every fourth token of a
// chunk, eight per step, the warps are merged in shared memory, and the result is
// merged into out / lse in place.  Lane l owns the frequencies 2l and 2l + 1 and
// both dimensions of each of their pairs, so rotating the keys needs no exchange;
// the eight scores of a step come out of one shuffle reduce-scatter.
#include "lla_kernels.h"

#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr int kWinThreads = 128;
constexpr int kWinWarps = kWinThreads / 32;
constexpr int kUnroll = 8;                          // window tokens per warp step
constexpr int kChunkBytes = 8192;                   // staged keys (and values) per chunk, two chunks in flight

// Two consecutive elements as floats.
__device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
  const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float2 ld2(const float* p) { return __ldg(reinterpret_cast<const float2*>(p)); }

// The lane's four dimensions of a d = 128 row, ordered (i0(f0), i1(f0), i0(f1), i1(f1))
// for its frequencies f0 = 2 lane, f1 = 2 lane + 1: rotate-half pairs (f, f + 64)
// or interleaved pairs (2f, 2f + 1).
template <typename T>
__device__ __forceinline__ float4 load_pairs(const T* row, int lane, int style) {
  if (style == 0) {
    const float2 a = ld2(row + 2 * lane), b = ld2(row + 64 + 2 * lane);
    return make_float4(a.x, b.x, a.y, b.y);
  }
  const float2 a = ld2(row + 4 * lane), b = ld2(row + 4 * lane + 2);
  return make_float4(a.x, a.y, b.x, b.y);
}

// The same from a row staged in shared memory (plain loads, not the read-only path).
__device__ __forceinline__ float2 ls2(const __nv_bfloat16* p) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float2 ls2(const float* p) { return *reinterpret_cast<const float2*>(p); }

template <typename T>
__device__ __forceinline__ float4 lds_pairs(const T* row, int lane, int style) {
  if (style == 0) {
    const float2 a = ls2(row + 2 * lane), b = ls2(row + 64 + 2 * lane);
    return make_float4(a.x, b.x, a.y, b.y);
  }
  const float2 a = ls2(row + 4 * lane), b = ls2(row + 4 * lane + 2);
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__global__ void __launch_bounds__(kWinThreads) window_attn_kernel(const __grid_constant__ WindowArgs a) {
  constexpr int CW = kChunkBytes / (kHeadDim * static_cast<int>(sizeof(T)));   // tokens per staged chunk
  extern __shared__ __align__(128) uint8_t wsm[];   // 2 x ([CW][128] keys, [CW][128] values)
  __shared__ float sm_m[kWinWarps], sm_l[kWinWarps];
  __shared__ float4 sm_acc[kWinWarps][32];
  __shared__ uint64_t full[2];
  __shared__ volatile int abort_flag;
  const int u = blockIdx.x, b = u / a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto kbuf = [&](int i) { return reinterpret_cast<T*>(wsm) + i * 2 * CW * kHeadDim; };

  // ---- device-side range checks: a bad window is skipped, a bad query position clamped
  int n = __ldg(a.win_len + b);
  const int p0 = __ldg(a.win_pos + b);
  if (n < 0 || n > a.W) {
    if (tid == 0 && u % a.H == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    n = 0;
  }
  if (n > 0 && (p0 < 0 || static_cast<int64_t>(p0) + n > a.rope_len)) {
    if (tid == 0 && u % a.H == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    n = 0;
  }
  int qp = __ldg(a.q_pos + b);
  if (qp < 0 || qp >= a.rope_len) {
    if (tid == 0 && u % a.H == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
  }
  const T* kb = static_cast<const T*>(a.k_win) + static_cast<int64_t>(u) * a.W * kHeadDim;
  const T* vb = static_cast<const T*>(a.v_win) + static_cast<int64_t>(u) * a.W * kHeadDim;
  // the window's keys and values arrive as plain bulk copies, chunk ci into buffer
  // ci & 1, the next chunk's copy in flight while this one is used
  auto issue = [&](int ci) {
    const int c0 = ci * CW;
    const uint32_t cn = static_cast<uint32_t>(min(CW, n - c0));
    const uint32_t fb = smem_u32(&full[ci & 1]);
    T* kd = kbuf(ci & 1);
    mbar_arrive_expect_tx(fb, 2 * cn * kHeadDim * static_cast<uint32_t>(sizeof(T)));
    bulk_load(smem_u32(kd), kb + static_cast<int64_t>(c0) * kHeadDim, cn * kHeadDim * sizeof(T), fb);
    bulk_load(smem_u32(kd + CW * kHeadDim), vb + static_cast<int64_t>(c0) * kHeadDim, cn * kHeadDim * sizeof(T), fb);
  };
  const int nch = (n + CW - 1) / CW;
  if (tid == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    abort_flag = 0;
    fence_mbar_init();
    if (nch > 0) issue(0);
    if (nch > 1) issue(1);
  }
  __syncthreads();

  // ---- q' = RoPE(q, q_pos), scaled so that scores are in log2 units
  const T* qv = static_cast<const T*>(a.q) + static_cast<int64_t>(u) * kHeadDim;
  float4 qr;
  {
    const float4 x = load_pairs(qv, lane, a.rope_style);
    const float2 c = __ldg(reinterpret_cast<const float2*>(a.rope_cos + static_cast<int64_t>(qp) * 64 + 2 * lane));
    const float2 s = __ldg(reinterpret_cast<const float2*>(a.rope_sin + static_cast<int64_t>(qp) * 64 + 2 * lane));
    const float sc = kLog2e * kInvSqrtD;
    qr = make_float4((x.x * c.x - x.y * s.x) * sc, (x.x * s.x + x.y * c.x) * sc,
                     (x.z * c.y - x.w * s.y) * sc, (x.z * s.y + x.w * c.y) * sc);
  }

  // cos / sin of kWinWarps theta_f for the lane's frequencies (table row kWinWarps)
  const float2 cs = __ldg(reinterpret_cast<const float2*>(a.rope_cos + kWinWarps * 64 + 2 * lane));
  const float2 sn = __ldg(reinterpret_cast<const float2*>(a.rope_sin + kWinWarps * 64 + 2 * lane));

  // ---- online softmax of this warp's window tokens (every kWinWarps-th of a chunk),
  // kUnroll per step: the step's scores come out of one shuffle reduce-scatter
  // (lanes 4i .. 4i + 3 end with token i's sum), then one broadcast per weight
  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int ci = 0; ci < nch; ++ci) {
    const int c0 = ci * CW, cn = min(CW, n - c0);
    const T* ks = kbuf(ci & 1);
    const T* vs = ks + CW * kHeadDim;
    // (bounded; on expiry the status word records it and the block leaves the loop
    // together, after the barrier below)
    const bool got = warp_wait(smem_u32(&full[ci & 1]), (ci >> 1) & 1, &abort_flag, a.status);
    for (int w0 = warp; got && w0 < cn; w0 += kWinWarps * kUnroll) {
      // the step's tokens sit kWinWarps positions apart: one table row for its first
      // token, the others by rotating with R(kWinWarps) (angle sum; positions of
      // masked tokens may run past the table, their weights are 0)
      float2 cc[kUnroll], ss[kUnroll];
      {
        const int64_t p = static_cast<int64_t>(p0) + c0 + w0;
        cc[0] = __ldg(reinterpret_cast<const float2*>(a.rope_cos + p * 64 + 2 * lane));
        ss[0] = __ldg(reinterpret_cast<const float2*>(a.rope_sin + p * 64 + 2 * lane));
      }
#pragma unroll
      for (int i = 1; i < kUnroll; ++i) {
        cc[i] = make_float2(fmaf(cc[i - 1].x, cs.x, -ss[i - 1].x * sn.x), fmaf(cc[i - 1].y, cs.y, -ss[i - 1].y * sn.y));
        ss[i] = make_float2(fmaf(ss[i - 1].x, cs.x, cc[i - 1].x * sn.x), fmaf(ss[i - 1].y, cs.y, cc[i - 1].y * sn.y));
      }
      float part[kUnroll];
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const int w = min(w0 + i * kWinWarps, cn - 1);
        const float4 k = lds_pairs(ks + w * kHeadDim, lane, a.rope_style);
        const float k0 = k.x * cc[i].x - k.y * ss[i].x, k1 = k.x * ss[i].x + k.y * cc[i].x;
        const float k2 = k.z * cc[i].y - k.w * ss[i].y, k3 = k.z * ss[i].y + k.w * cc[i].y;
        part[i] = fmaf(qr.x, k0, fmaf(qr.y, k1, fmaf(qr.z, k2, qr.w * k3)));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool up = lane & 16;
        const float send = up ? part[i] : part[i + 4], keep = up ? part[i + 4] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool up = lane & 8;
        const float send = up ? part[i] : part[i + 2], keep = up ? part[i + 2] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      {
        const bool up = lane & 4;
        const float send = up ? part[0] : part[1], keep = up ? part[1] : part[0];
        part[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      part[0] += __shfl_xor_sync(0xffffffffu, part[0], 2);
      part[0] += __shfl_xor_sync(0xffffffffu, part[0], 1);
      const bool live = w0 + (lane >> 2) * kWinWarps < cn;
      const float sv = live ? part[0] : -INFINITY;
      const float mt = warp_max_redux(sv);   // token 0 of the step is always live
      if (mt > m) {
        const float alpha = m == -INFINITY ? 0.f : exp2f(m - mt);
        l *= alpha;
        acc.x *= alpha; acc.y *= alpha; acc.z *= alpha; acc.w *= alpha;
        m = mt;
      }
      const float pv = live ? exp2f(sv - m) : 0.f;
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const float p = __shfl_sync(0xffffffffu, pv, 4 * i);
        const float4 v = lds_pairs(vs + min(w0 + i * kWinWarps, cn - 1) * kHeadDim, lane, a.rope_style);
        l += p;
        acc.x = fmaf(p, v.x, acc.x);
        acc.y = fmaf(p, v.y, acc.y);
        acc.z = fmaf(p, v.z, acc.z);
        acc.w = fmaf(p, v.w, acc.w);
      }
    }
    __syncthreads();   // every warp is done with the buffer before chunk ci + 2 lands in it
    if (abort_flag) break;   // read by all threads after the barrier: a uniform exit
    if (tid == 0 && ci + 2 < nch) issue(ci + 2);
  }
  if (abort_flag) { m = -INFINITY; l = 0.f; }   // timed out (status recorded): keep the latent result
  sm_acc[warp][lane] = acc;
  if (lane == 0) { sm_m[warp] = m; sm_l[warp] = l; }
  __syncthreads();

  // ---- merge the warps, then the latent part (out, lse) of the same row
  if (warp == 0) {
    float M = sm_m[0];
#pragma unroll
    for (int i = 1; i < kWinWarps; ++i) M = fmaxf(M, sm_m[i]);
    if (M == -INFINITY) return;   // no window token: the latent result stands
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kWinWarps; ++i) {
      const float f = sm_m[i] == -INFINITY ? 0.f : exp2f(sm_m[i] - M);
      const float4 ai = sm_acc[i][lane];
      L = fmaf(f, sm_l[i], L);
      o.x = fmaf(f, ai.x, o.x); o.y = fmaf(f, ai.y, o.y); o.z = fmaf(f, ai.z, o.z); o.w = fmaf(f, ai.w, o.w);
    }
    const float lw = M + log2f(L);                       // window log-sum-exp (log2 units)
    const float ll = __ldg(a.lse + u) * kLog2e;          // latent log-sum-exp (log2 units)
    const float MM = fmaxf(lw, ll);
    const float wa = ll == -INFINITY ? 0.f : exp2f(ll - MM), wb = exp2f(lw - MM);
    const float inv = 1.f / (wa + wb), fb = wb * inv / L;
    float* orow = a.out + static_cast<int64_t>(u) * kHeadDim;
    const int e0 = a.rope_style == 0 ? 2 * lane : 4 * lane;
    const int e1 = a.rope_style == 0 ? 64 + 2 * lane : 4 * lane + 1;
    const int e2 = a.rope_style == 0 ? 2 * lane + 1 : 4 * lane + 2;
    const int e3 = a.rope_style == 0 ? 64 + 2 * lane + 1 : 4 * lane + 3;
    const float fa = wa * inv;
    // a latent row with lse = -inf holds zeros (no latent token): weight 0 above
    orow[e0] = fmaf(fa, orow[e0], fb * o.x);
    orow[e1] = fmaf(fa, orow[e1], fb * o.y);
    orow[e2] = fmaf(fa, orow[e2], fb * o.z);
    orow[e3] = fmaf(fa, orow[e3], fb * o.w);
    __syncwarp();
    if (lane == 0) a.lse[u] = (MM + log2f(wa + wb)) * kLn2;
  }
}

}  // namespace

cudaError_t launch_window_attn(const WindowArgs& a, bool bf16, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(a.B) * a.H;
  static bool configured[2] = {false, false};
  if (!configured[bf16]) {
    cudaError_t e = bf16 ? cudaFuncSetAttribute(window_attn_kernel<__nv_bfloat16>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * kChunkBytes)
                         : cudaFuncSetAttribute(window_attn_kernel<float>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * kChunkBytes);
    if (e != cudaSuccess) return e;
    configured[bf16] = true;
  }
  if (bf16) window_attn_kernel<__nv_bfloat16><<<grid, kWinThreads, 4 * kChunkBytes, s>>>(a);
  else window_attn_kernel<float><<<grid, kWinThreads, 4 * kChunkBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lla
