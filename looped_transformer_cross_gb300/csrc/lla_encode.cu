// lla_encode.cu — the cross-loop encode of Looped Latent Attention on sm_103a
// ("Looped Latent Attention: Cross-Loop KV Compression for Looped
// Transformers", arXiv 2607.15456v2, §3 Eq. (1)-(2)):
//     c = (x - mu) W_down ,  x = [x_1; ...; x_T] in R^{T d}
// for every token and head, written into the token's cache slot.
//
// bf16 path: one CTA per (128-token tile, head, axis K/V).  TMA streams
// 64-wide K-slices of x (K-major) and W_down (MN-major) through a ring; warp 1
// issues tcgen05 MMAs accumulating x W_down in TMEM; four epilogue warps (one
// token per TMEM lane) subtract mu W_down (computed once per call by a small
// kernel), round to bf16 and store the latent row.  Computing x W - mu W
// instead of (x - mu) W is exact in real arithmetic.
//
// fp32 path: one block per (token, head, axis), the literal sum in fp32.
#include "lla_kernels.h"

namespace lla {

namespace {

struct alignas(16) EncodeMisc {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t dfull;
  uint32_t tmem_base;
  int abort;
};

// bias[axis][h][k] = sum_u mu[h][u] * W_down[h][u][k]  (fp32).  Block = (head,
// axis): warp w sums rows u = w, w + 8, ...; lane l covers columns 8l..8l+7 with
// 16-byte loads, sixteen rows in flight; the eight warps' partial sums are added
// in shared memory.
__global__ void __launch_bounds__(256) encode_bias_kernel(const __grid_constant__ EncodeArgs a) {
  __shared__ float part[8][256];
  const int h = blockIdx.x, axis = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = axis == 0 ? a.r_k : a.r_v;
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(axis == 0 ? a.w_down_k : a.w_down_v) +
                           static_cast<int64_t>(h) * a.Td * r;
  const float* mu = (axis == 0 ? a.mu_k : a.mu_v) + static_cast<int64_t>(h) * a.Td;
  const int k = 8 * lane;
  constexpr int kRows = 16;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (k < r) {
    for (int u0 = warp; u0 < a.Td; u0 += 8 * kRows) {
      uint4 wv[kRows];
      float m[kRows];
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        const int u = u0 + 8 * j;
        const bool in = u < a.Td;
        wv[j] = in ? __ldg(reinterpret_cast<const uint4*>(W + static_cast<int64_t>(u) * r + k)) : make_uint4(0, 0, 0, 0);
        m[j] = in ? __ldg(mu + u) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        float w8[8];
        unpack_bf16x8(wv[j], w8);
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] = fmaf(m[j], w8[t], acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) part[warp][k + t] = acc[t];
  }
  __syncthreads();
  const int t = threadIdx.x;
  if (t < r) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][t];
    a.bias[(static_cast<int64_t>(axis) * a.H + h) * 256 + t] = s;
  }
}

__device__ __forceinline__ bool slot_ok(const EncodeArgs& a, int sid, int p) {
  return sid >= 0 && sid < a.B && p >= 0 && p < a.L_max;
}

__global__ void __launch_bounds__(kEncodeThreads, 1)
encode_bf16_kernel(const __grid_constant__ EncodeArgs a, const __grid_constant__ EncodePlan P,
                   const __grid_constant__ EncodeMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  EncodeMisc* misc = reinterpret_cast<EncodeMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, h = blockIdx.y, axis = blockIdx.z;
  const int r = axis == 0 ? a.r_k : a.r_v;
  const ChunkPlan& bp = axis == 0 ? P.bk : P.bv;
  const CUtensorMap* xmap = axis == 0 ? &maps.xk : &maps.xv;
  const CUtensorMap* wmaps = axis == 0 ? maps.wk : maps.wv;
  const int KB = a.Td / 64;
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };

  if (tid == 0) {
    for (int s = 0; s < P.S; ++s) { mbar_init(bar(misc->full[s]), 1); mbar_init(bar(misc->empty[s]), 1); }
    mbar_init(bar(misc->dfull), 1);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&misc->tmem_base), P.tmem_cols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t bytes = 128 * 64 * 2 + bp.bytes;
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % P.S;
        if (!mbar_wait(bar(misc->empty[s]), ((kb / P.S) & 1) ^ 1, abort, a.status)) break;
        const uint32_t fb = bar(misc->full[s]);
        mbar_arrive_expect_tx(fb, bytes);
        const uint32_t st = sbase + P.ring + s * P.stage;
        tma_load_3d(st + P.a_off, xmap, fb, kb * 64, h, tile * 128);
        for (int c = 0; c < bp.n; ++c)
          tma_load_3d(st + P.b_off + bp.off[c], &wmaps[chunk_map_index(bp.width[c])], fb, bp.start[c],
                      kb * 64, h);
        issued = kb + 1;
      }
      for (int kb = max(0, issued - P.S); kb < issued; ++kb) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->full[kb % P.S]), (kb / P.S) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < KB && ok; ++kb) {
        const int s = kb % P.S;
        if (!(ok = mbar_wait(bar(misc->full[s]), (kb / P.S) & 1, abort, a.status))) break;
        tc_fence_after();
        const uint32_t st = sbase + P.ring + s * P.stage;
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = umma_desc(st + P.a_off + k * 32, 16, 1024, kSw128);
          // N-runs: up to four 64-wide chunks per MMA, narrower chunks alone
          for (int c = 0; c < bp.n;) {
            const int w = bp.width[c];
            int nch = 1;
            if (w == 64) while (c + nch < bp.n && bp.width[c + nch] == 64 && nch < 4) ++nch;
            const int rb = w * 2;
            const uint64_t bd = umma_desc(st + P.b_off + bp.off[c] + k * 16 * rb, 64 * rb, 8 * rb,
                                          sw_mode_for_row_bytes(rb));
            umma_bf16(tmem + bp.start[c], ad, bd, umma_idesc_bf16(128, w * nch, false, true),
                      (kb > 0 || k > 0) ? 1u : 0u);
            c += nch;
          }
        }
        umma_commit(bar(misc->empty[s]));
      }
      umma_commit(bar(misc->dfull));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->dfull), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    if (warp_wait(bar(misc->dfull), 0, abort, a.status)) {
      tc_fence_after();
      const int n = tile * 128 + row;
      int sid = -1, p = -1;
      if (n < a.N) {
        sid = __ldg(a.seq_idx + n);
        p = __ldg(a.pos + n);
        if (!slot_ok(a, sid, p)) record_status(a.status, LLA_ERR_DEVICE_ARG);
      }
      const int64_t drow = n < a.N && slot_ok(a, sid, p)
                               ? latent_row_for_write(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max,
                                                      a.H, sid, h, p, a.status)
                               : -1;
      const bool write = drow >= 0;
      const float* bias = a.bias + (static_cast<int64_t>(axis) * a.H + h) * 256;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(axis == 0 ? a.cache_k : a.cache_v) + (write ? drow : 0) * r;
      for (int c0 = 0; c0 < r; c0 += 16) {
        float v[16];
        tmem_ld_x16(tmem + lane_base + c0, v);   // every lane of the warp takes part
        tmem_wait_ld();
        if (write) {
          uint32_t wds[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i] - bias[c0 + 2 * i],
                                                            v[2 * i + 1] - bias[c0 + 2 * i + 1]);
            wds[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
          d4[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
          d4[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, P.tmem_cols);
  }
}

// fp32: literal c[k] = sum_u (x[u] - mu[u]) W[u][k]; block = (token, head, axis).
__global__ void __launch_bounds__(256) encode_f32_kernel(const __grid_constant__ EncodeArgs a) {
  const int n = blockIdx.x, h = blockIdx.y, axis = blockIdx.z, k = threadIdx.x;
  const int r = axis == 0 ? a.r_k : a.r_v;
  const int sid = __ldg(a.seq_idx + n), p = __ldg(a.pos + n);
  if (!slot_ok(a, sid, p)) {
    if (k == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    return;
  }
  if (k >= r) return;
  const float* x = static_cast<const float*>(axis == 0 ? a.x_k : a.x_v) + (static_cast<int64_t>(n) * a.H + h) * a.Td;
  const float* mu = (axis == 0 ? a.mu_k : a.mu_v) + static_cast<int64_t>(h) * a.Td;
  const float* W = static_cast<const float*>(axis == 0 ? a.w_down_k : a.w_down_v) + static_cast<int64_t>(h) * a.Td * r;
  float s = 0.f;
  for (int u = 0; u < a.Td; ++u) s = fmaf(x[u] - mu[u], W[static_cast<int64_t>(u) * r + k], s);
  const int64_t row =
      latent_row_for_write(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max, a.H, sid, h, p, a.status);
  if (row < 0) return;
  float* dst = static_cast<float*>(axis == 0 ? a.cache_k : a.cache_v);
  dst[row * r + k] = s;
}

}  // namespace

bool make_encode_plan(int r_k, int r_v, int Td, EncodePlan* p) {
  *p = EncodePlan{};
  if (Td % 64 != 0) return false;
  p->bk = make_chunk_plan(r_k, 64);
  p->bv = make_chunk_plan(r_v, 64);
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  const int bmax = p->bk.bytes > p->bv.bytes ? p->bk.bytes : p->bv.bytes;
  p->a_off = 0;
  p->b_off = 128 * 64 * 2;
  p->stage = al(p->b_off + bmax, 1024);
  const int fixed = 1024 + 1024;   // misc + alignment slack
  int S = kMaxStages;
  while (S > 2 && fixed + S * p->stage > kSmemLimit) --S;
  if (fixed + S * p->stage > kSmemLimit) return false;
  p->S = S;
  p->ring = 0;
  p->misc = S * p->stage;
  p->bytes = p->misc + 1024 + 1024;
  const int rmax = r_k > r_v ? r_k : r_v;
  int cols = 32;
  while (cols < rmax) cols <<= 1;
  p->tmem_cols = cols;
  return true;
}

cudaError_t launch_encode_bf16(const EncodeArgs& a, const EncodePlan& plan, const EncodeMaps& m,
                               cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  encode_bias_kernel<<<dim3(a.H, 2), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static int configured = 0;
  if (configured < plan.bytes) {
    e = cudaFuncSetAttribute(encode_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.bytes);
    if (e != cudaSuccess) return e;
    configured = plan.bytes;
  }
  const dim3 grid((a.N + 127) / 128, a.H, 2);
  encode_bf16_kernel<<<grid, kEncodeThreads, plan.bytes, s>>>(a, plan, m);
  return cudaGetLastError();
}

cudaError_t launch_encode_f32(const EncodeArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  encode_f32_kernel<<<dim3(a.N, a.H, 2), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lla
