// lla_decode2d.cu — LLA-2D latent-store decode attention on sm_103a ("Looped
// Latent Attention: Cross-Loop KV Compression for Looped Transformers", arXiv
// 2607.15456v2: §3 "The LLA-2D variant", Eq. (3), "RoPE and reconstruction",
// Appendix J "Absorbed attention").
//
// LLA-2D keeps ONE K latent (r_k) and ONE V latent (r_v) per token and layer,
// shared by all H heads, and loop t rebuilds every head's key from it:
// k_{t,h} = c_k W_up,k,t,h^T + mu_k,t,h.  One call (one layer, one loop, all heads
// and sequences) therefore contracts [tokens x r_k] with [r_k x H*128]: at H = 16,
// r_k = 128 that is about 0.5 MFLOP per cached token and ~700 flop per latent
// byte, so the score pass is bound by the tensor pipe, not by HBM.
//
// Four launches:
//  1. decode2d_z_kernel: the query operand Z of every (sequence, head) (the
//     RoPE-rotated, scaled query folded into W_up,k,t,h) and an f16 RoPE table.
//  2. decode2d_score_kernel (CTA pairs, tcgen05 cta_group::2): blocks of 256 tokens
//     of one sequence; CTA `rank` holds the block's K latent tile at rows
//     256 kb + 128 rank.  Each stage is one pair MMA U = C_k [Z_2p; Z_2p+1]^T over
//     a pair of heads (M = 256 tokens, N = 256, K = r_k), the even CTA supplying
//     head 2p's 128 operand rows and the odd CTA head 2p+1's.  A pair MMA issues
//     at most about one per 70 cycles, so N = 256 (128 cycles of tensor work per
//     MMA) keeps the pipe fed where N = 128 could not.  Both CTAs' copies of an
//     operand complete on one barrier of the even CTA (cta_group::2 copies).  The
//     two 256-column score buffers fill TMEM.  Epilogue warps (one token per
//     thread, warp group g takes head 2p + g) form the rotary score
//     s = sum_f cos(j th_f) U_f + sin(j th_f) U_64+f from the token's cos/sin row
//     held in registers and write, per 32-token group (one warp), the weights
//     p = 2^(s - m) (bf16) with m = ceil(max s), an integer, and m.
//  3. decode2d_value_kernel (one CTA per SM): D_v = sum_j p_j c_v,j for every head
//     over contiguous runs of 128-token tiles, on the tensor cores (M = 128 r_v
//     rows, N = 16 heads, K = tokens; Appendix J), the weights of each group first
//     scaled by 2^(m_group - M_run) (exact: both are integers) and summed into
//     l_run, one record (M_run, l_run, D_v) per run.
//  4. decode2d_combine_kernel: merges the records of a sequence (log-sum-exp
//     merge) and applies the V up-projection once.
//
#include "lla_kernels.h"

#include <algorithm>
#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr int kSNK = 3;        // latent tile slots of the score kernel (one tile per block)
constexpr int kSNZ = 3;        // query-operand windows in flight (one head per CTA each)
constexpr int kZRowBytes = 128;    // one 64-wide bf16 chunk row
constexpr int kVTile = 128;        // tokens of a value tile (= score tile)
constexpr int kVS = 3;             // value ring stages

struct alignas(16) MiscScore {
  // full barriers (used in the even CTA): the copies of both CTAs complete on them
  uint64_t kfull[kSNK], kempty[kSNK];
  uint64_t zfull[kSNZ], zempty[kSNZ];
  // score buffers: ufull takes the MMA commit; uempty (used in the even CTA) the
  // 8 epilogue warps of both CTAs
  uint64_t ufull[2], uempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int start_b, start_kb, count, total_blocks;
  float xch[2][2][kTile];   // [stage parity][head of the pair][token]: the other group's half score
  int scan[kScore2dThreads];
};
static_assert(sizeof(MiscScore) <= 4096, "misc region");

struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) { slot = 0; phase ^= 1u; }
  }
};

// Block of one sequence: tokens [256 kb, 256 kb + 256).
struct Walker2d {
  int b, kb, nb, L;
};

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

__device__ __forceinline__ int nblocks(int L) { return (L + kBlock2dTokens - 1) / kBlock2dTokens; }
__device__ __forceinline__ int ntiles_of(int L) { return (L + kVTile - 1) / kVTile; }

__device__ __forceinline__ void walk_advance(Walker2d& w, const Decode2dArgs& a) {
  if (++w.kb < w.nb) return;
  w.kb = 0;
  while (true) {
    if (++w.b >= a.B) { w.nb = 0; return; }
    w.L = clamp_len(__ldg(a.seq_lens + w.b), a.L_max);
    w.nb = nblocks(w.L);
    if (w.nb > 0) return;
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}

// Query operand of every (sequence, head) for the LLA-2D kernel: the rows of
// the per-head construction, stacked per sequence.  With q' = RoPE(q, q_pos),
// sc = log2(e)/sqrt(d) and the frequency pair (i0, i1) of f < 64, head h gives
//   row h*128 + f      : sc (q'_i0 W_i0 + q'_i1 W_i1),  bias sc (q'_i0 mu_i0 + q'_i1 mu_i1)
//   row h*128 + 64 + f : sc (q'_i1 W_i0 - q'_i0 W_i1),  bias sc (q'_i1 mu_i0 - q'_i0 mu_i1)
// with W = W_up,k,t,h (rows h*128 + e of the loop-t slice) and mu = mu_k,t,h, so
// that sum_f cos(j th_f) U_f + sin(j th_f) U_64+f with U = c_j Z^T + bias is
// log2(e) RoPE(q, q_pos).RoPE(k_j, j) / sqrt(d) for the key of Eq. (3).  Layout
// per sequence: nkc chunks of [H*128 rows][64 bf16] in the 128-byte swizzle of a
// K-major operand (row n swizzled by n mod 8), then the bias operand [H*128
// rows][16 bf16] (32-byte swizzle): column 0 = bias rounded to bf16, column 1 =
// the rounding remainder, so a 16-wide MMA against ones in columns 0 and 1 adds
// the bias in ~16-bit precision.  Blocks = (sequence, head); the blocks after
// them write the RoPE table transposed, trigT[c][j] = cos(j th_c) (c < 64) or
// sin(j th_c-64), so that the epilogue's loads of 32 consecutive tokens coalesce
// (32 tokens per block).
constexpr int kZThreads = 256;
constexpr int kTrigTokensPerBlock = 32;
__global__ void __launch_bounds__(kZThreads) decode2d_z_kernel(const __grid_constant__ Decode2dArgs a) {
  // the decode grid may start its set-up now; it waits for this grid before it
  // copies an image
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float qs[2][64];
  const int u = blockIdx.x, tid = threadIdx.x;
  if (u >= a.B * a.H) {
    __shared__ float tr[128][kTrigTokensPerBlock + 1];
    const int64_t j0 = static_cast<int64_t>(u - a.B * a.H) * kTrigTokensPerBlock;
    for (int i = tid; i < kTrigTokensPerBlock * 128; i += kZThreads) {
      const int jj = i / 128, c = i % 128;
      int64_t j = j0 + jj;
      if (j >= a.rope_len) j = a.rope_len - 1;   // rows past the table: masked tokens
      tr[c][jj] = __ldg((c < 64 ? a.rope_cos : a.rope_sin) + j * 64 + (c & 63));
    }
    __syncthreads();
    for (int i = tid; i < kTrigTokensPerBlock * 128; i += kZThreads) {
      const int c = i / kTrigTokensPerBlock, jj = i % kTrigTokensPerBlock;
      a.trigT[c * a.trig_rows + j0 + jj] = tr[c][jj];
    }
    return;
  }
  const int b = u / a.H, h = u - (u / a.H) * a.H;
  if (clamp_len(__ldg(a.seq_lens + b), a.L_max) == 0) return;
  uint8_t* img = a.zimg + static_cast<int64_t>(b) * a.zimg_stride;
  const __nv_bfloat16* W =
      static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * a.r_k;
  const int ng = a.r_k / 8;
  constexpr int kItems = 64 * 16 / kZThreads;   // items per thread at r_k = 128
  uint4 ra[kItems], rb[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int it = tid + j * kZThreads;
    if (it < 64 * ng) {
      const int f = it / ng, k = 8 * (it - (it / ng) * ng);
      const int i0 = a.rope_style == 0 ? f : 2 * f;
      const int i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
      ra[j] = __ldg(reinterpret_cast<const uint4*>(W + static_cast<int64_t>(i0) * a.r_k + k));
      rb[j] = __ldg(reinterpret_cast<const uint4*>(W + static_cast<int64_t>(i1) * a.r_k + k));
    }
  }
  if (tid < 64) {
    const int f = tid;
    int qp = __ldg(a.q_pos + b);
    if (qp < 0 || qp >= a.rope_len) {
      if (f == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
      qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
    }
    const int i0 = a.rope_style == 0 ? f : 2 * f;
    const int i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
    const __nv_bfloat16* qv =
        static_cast<const __nv_bfloat16*>(a.q) + (static_cast<int64_t>(b) * a.H + h) * kHeadDim;
    const float* mu = a.mu_k + static_cast<int64_t>(h) * kHeadDim;
    const float cq = __ldg(a.rope_cos + static_cast<int64_t>(qp) * 64 + f);
    const float sq = __ldg(a.rope_sin + static_cast<int64_t>(qp) * 64 + f);
    const float x0 = __bfloat162float(qv[i0]), x1 = __bfloat162float(qv[i1]);
    const float m0 = __ldg(mu + i0), m1 = __ldg(mu + i1);
    const float scale = kLog2e * kInvSqrtD;
    const float q0 = (x0 * cq - x1 * sq) * scale;   // sc * q'_i0
    const float q1 = (x0 * sq + x1 * cq) * scale;   // sc * q'_i1
    qs[0][f] = q0;
    qs[1][f] = q1;
    const float bias[2] = {q0 * m0 + q1 * m1, q1 * m0 - q0 * m1};
    uint8_t* ab = img + a.plan.nkc * a.zchunk_bytes;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int n = h * kHeadDim + f + 64 * half;
      const __nv_bfloat16 zh = __float2bfloat16_rn(bias[half]);
      const __nv_bfloat16 zl = __float2bfloat16_rn(bias[half] - __bfloat162float(zh));
      const uint32_t pair = bf16x2_bits(__halves2bfloat162(zh, zl));
      *reinterpret_cast<uint4*>(ab + swizzle_offset(n * 32, 32)) = make_uint4(pair, 0, 0, 0);
      *reinterpret_cast<uint4*>(ab + swizzle_offset(n * 32 + 16, 32)) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int it = tid + j * kZThreads;
    if (it >= 64 * ng) break;
    const int f = it / ng, k = 8 * (it - f * ng);
    float wa[8], wb[8];
    unpack_bf16x8(ra[j], wa);
    unpack_bf16x8(rb[j], wb);
    const float q0 = qs[0][f], q1 = qs[1][f];
    uint32_t z0[4], z1[4];   // rows f and 64 + f of head h
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      z0[t] = bf16x2_bits(__floats2bfloat162_rn(q0 * wa[2 * t] + q1 * wb[2 * t],
                                                q0 * wa[2 * t + 1] + q1 * wb[2 * t + 1]));
      z1[t] = bf16x2_bits(__floats2bfloat162_rn(q1 * wa[2 * t] - q0 * wb[2 * t],
                                                q1 * wa[2 * t + 1] - q0 * wb[2 * t + 1]));
    }
    uint8_t* zc = img + static_cast<int64_t>(k >> 6) * a.zchunk_bytes;
    const int col = (k & 63) * 2;
    const int n0 = h * kHeadDim + f, n1 = n0 + 64;
    *reinterpret_cast<uint4*>(zc + swizzle_offset(n0 * kZRowBytes + col, kZRowBytes)) =
        make_uint4(z0[0], z0[1], z0[2], z0[3]);
    *reinterpret_cast<uint4*>(zc + swizzle_offset(n1 * kZRowBytes + col, kZRowBytes)) =
        make_uint4(z1[0], z1[1], z1[2], z1[3]);
  }
}


// d = a * b + d on a pair of f32 lanes (one packed instruction)
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mov.b64 pd, {%0, %1};\n\tfma.rn.f32x2 pd, pa, pb, pd;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Contiguous share `part` of `parts` of the work units (blocks or tiles) of all
// sequences, in sequence order: its first (sequence, unit) and its length.  Every
// thread of the CTA calls it (it synchronises); scan holds kThreads ints.
template <int kThreads, typename CountOf>
__device__ void share_of(const Decode2dArgs& a, CountOf count_of, long long part, long long parts, int* scan,
                         int* start_b, int* start_k, int* count, int* total) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_thr = (a.B + kThreads - 1) / kThreads;
  const int b0 = min(a.B, tid * per_thr), b1 = min(a.B, b0 + per_thr);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += count_of(b);
  scan[tid] = local;
  __syncthreads();
  if (warp == 0) {
    constexpr int kPer = kThreads / 32;
    int v[kPer];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) { v[i] = scan[lane * kPer + i]; s += v[i]; }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int excl = incl - s;
#pragma unroll
    for (int i = 0; i < kPer; ++i) { scan[lane * kPer + i] = excl; excl += v[i]; }
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  const long long NB = *total;
  const long long lo = part * NB / parts, hi = (part + 1) * NB / parts;
  long long P0 = scan[tid];
  for (int b = b0; b < b1; ++b) {
    const int nb = count_of(b);
    if (nb > 0 && lo < hi && P0 <= lo && lo < P0 + nb) {
      *start_b = b;
      *start_k = static_cast<int>(lo - P0);
    }
    P0 += nb;
  }
  if (tid == 0) *count = static_cast<int>(hi - lo);
  __syncthreads();
}

// Warp-collective wait in which every lane polls (no suspend hint, no broadcast
// from one lane afterwards): the epilogue's per-stage wait is on its critical path.
// Bounded like mbar_wait.
__device__ __forceinline__ bool warp_poll(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (__all_sync(0xffffffffu, done != 0)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        record_status(status, LLA_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// Spinning form of the bounded wait (no suspend hint): for the issuer, whose every
// wait is on the critical path of the tensor pipe.  Its barriers are its own CTA's:
// the copies of both CTAs complete on them, and the score-buffer releases carry no
// data (the TMEM reads they announce were waited for and fenced).
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        record_status(status, LLA_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kScore2dThreads, 1)
decode2d_score_kernel(const __grid_constant__ Decode2dArgs a, const __grid_constant__ Decode2dMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Decode2dPlan& P = a.plan;
  const uint32_t sbase = smem_u32(sm);
  MiscScore* misc = reinterpret_cast<MiscScore*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_cta_rank();
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int HP = a.H / 2;   // stages (head pairs) of a block

  // ---------------------------------------------------------- work range (same in both CTAs)
  if (tid == 0) misc->abort = 0;
  if (blockIdx.x == 0 && tid < a.B) {
    for (int b = tid; b < a.B; b += kScore2dThreads) {
      const int L0 = __ldg(a.seq_lens + b);
      if (L0 < 0 || L0 > a.L_max) record_status(a.status, LLA_ERR_DEVICE_ARG);
    }
  }
  share_of<kScore2dThreads>(
      a, [&](int b) { return nblocks(clamp_len(__ldg(a.seq_lens + b), a.L_max)); }, pair, a.pairs, misc->scan,
      &misc->start_b, &misc->start_kb, &misc->count, &misc->total_blocks);
  const int count = misc->count;
  if (count == 0) return;   // both CTAs of the pair leave here together

  Walker2d start;
  start.b = misc->start_b;
  start.kb = misc->start_kb;
  start.L = clamp_len(__ldg(a.seq_lens + start.b), a.L_max);
  start.nb = nblocks(start.L);

  // ---------------------------------------------------------- set-up
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    for (int s = 0; s < kSNK; ++s) {
      mbar_init(bar(misc->kfull[s]), 1);        // the even producer's expect_tx (both CTAs' bytes)
      mbar_init(bar(misc->kempty[s]), 1);       // MMA commit after the block's last stage
    }
    for (int s = 0; s < kSNZ; ++s) {
      mbar_init(bar(misc->zfull[s]), 1);
      mbar_init(bar(misc->zempty[s]), 1);       // MMA commit of the window's stage
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(misc->ufull[s]), 1);
      mbar_init(bar(misc->uempty[s]), 16);      // 8 epilogue warps of each CTA
    }
    mbar_init(bar(misc->mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.z);
    prefetch_tmap(&maps.zb);
  }
  // bias operand A: columns 0 and 1 of every token row are 1 (they meet bias hi / lo)
  if (tid < kTile) {
    const uint32_t ones = bf16x2_bits(__floats2bfloat162_rn(1.f, 1.f));
    *reinterpret_cast<uint4*>(sm + P.aug_a + swizzle_offset(tid * 32, 32)) = make_uint4(ones, 0, 0, 0);
    *reinterpret_cast<uint4*>(sm + P.aug_a + swizzle_offset(tid * 32 + 16, 32)) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any remote arrive
  if (warp == 1) {
    __syncwarp();
    tmem_alloc_pair(smem_u32(&misc->tmem_base), 512);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the value grid may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    // ======================================================== TMA producer (each CTA)
    // Per block: the latent tile, then per head pair this CTA's head of the pair
    // (2p + rank): its 128 query-operand rows and their bias rows.  The copies of
    // both CTAs complete on the even CTA's full barrier, which the even producer
    // arms with the bytes of both.
    if (lane == 0) {
      Walker2d w = start;
      RingPos kr, zr;
      int issued_k = 0, issued_z = 0;
      bool ok = true, images_ready = false;
      // latents stream through once; a sequence's query operand is read by every block
      const uint64_t pol_stream = l2_policy_evict_first(), pol_keep = l2_policy_evict_last();
      for (int n = 0; n < count && ok; ++n) {
        {
          const int sk = kr.slot;
          if (!(ok = mbar_wait(bar(misc->kempty[sk]), kr.phase ^ 1u, abort, a.status))) break;
          const uint32_t fb = bar(misc->kfull[sk]);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * P.nkc * 16384);
          const uint32_t fbe = map_to_rank(fb, 0);
          const int y = w.kb * kBlock2dTokens + static_cast<int>(rank) * kTile;
          for (int c = 0; c < P.nkc; ++c)
            tma_load_3d_pair(sbase + P.k_ring + sk * P.k_stage + c * 16384, &maps.k, fbe, 64 * c, y, w.b, pol_stream);
          ++issued_k;
          kr.next(kSNK);
        }
        for (int p = 0; p < HP && ok; ++p) {
          const int sz = zr.slot;
          if (!(ok = mbar_wait(bar(misc->zempty[sz]), zr.phase ^ 1u, abort, a.status))) break;
          if (!images_ready) {
            asm volatile("griddepcontrol.wait;" ::: "memory");   // images written
            images_ready = true;
          }
          const uint32_t fb = bar(misc->zfull[sz]);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (P.nkc * 16384 + 4096));
          const uint32_t fbe = map_to_rank(fb, 0);
          const uint32_t dst = sbase + P.z_ring + sz * P.z_stage;
          const int row0 = (2 * p + static_cast<int>(rank)) * kHeadDim;
          for (int c = 0; c < P.nkc; ++c)
            tma_load_3d_pair(dst + c * 16384, &maps.z, fbe, 0, c * a.H * kHeadDim + row0, w.b, pol_keep);
          tma_load_3d_pair(dst + P.nkc * 16384, &maps.zb, fbe, 0, row0, w.b, pol_keep);
          ++issued_z;
          zr.next(kSNZ);
        }
        walk_advance(w, a);
      }
      // every copy of the pair lands before the CTAs can exit (the odd CTA's copies
      // count on the even CTA's barriers; the final cluster barrier holds it)
      if (rank == 0) {
        auto drain = [&](uint64_t* full, int n, int issued) {
          for (int i = max(0, issued - n); i < issued; ++i) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(full[i % n]), (i / n) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
          }
        };
        drain(misc->kfull, kSNK, issued_k);
        drain(misc->zfull, kSNZ, issued_z);
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ======================================================== pair MMA issuer (even CTA)
    // The whole warp runs the loop (warp-uniform descriptors) and one elected lane
    // issues.  Stage G (block n, head pair p) uses score buffer G & 1, latent slot
    // n mod 3 and query window G mod 3; it releases the window and, after the
    // block's last stage, the latent slot by MMA commit.
    const uint32_t idesc = umma_idesc_bf16(256, 256, false, false);
    const int ksteps = a.r_k / 16;
    const uint64_t dA0 = umma_desc(sbase + P.k_ring, 16, 1024, kSw128);
    const uint64_t dZ0 = umma_desc(sbase + P.z_ring, 16, 1024, kSw128);
    const uint64_t dZb0 = umma_desc(sbase + P.z_ring + P.nkc * 16384, 16, 256, kSw32);
    const uint64_t daug = umma_desc(sbase + P.aug_a, 16, 256, kSw32);
    const uint32_t kst = static_cast<uint32_t>(P.k_stage) >> 4, zst = static_cast<uint32_t>(P.z_stage) >> 4;
    // every lane polls each barrier; the vote keeps the warp's decision uniform (a
    // wait that gave up in any lane ends the loop in all of them)
    auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
    bool ok = true;
    uint32_t G = 0;
    for (uint32_t n = 0; n < static_cast<uint32_t>(count) && ok; ++n) {
      const uint32_t ts = n % kSNK;
      if (!(ok = agree(mbar_spin(bar(misc->kfull[ts]), (n / kSNK) & 1u, abort, a.status)))) break;
      const uint64_t a0 = dA0 + ts * kst;
      for (int p = 0; p < HP && ok; ++p, ++G) {
        const uint32_t zs = G % kSNZ, buf = G & 1u;
        if (!(ok = agree(mbar_spin(bar(misc->zfull[zs]), (G / kSNZ) & 1u, abort, a.status)))) break;
        if (!(ok = agree(mbar_spin(bar(misc->uempty[buf]), ((G >> 1) & 1u) ^ 1u, abort, a.status)))) break;
        tc_fence_after();
        const uint64_t b0 = dZ0 + zs * zst, bb = dZb0 + zs * zst;
        const uint32_t d = tmem + 256 * buf;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          // 64-wide K chunks 16 KB apart in both operands; 32 B per K step
          if (k < ksteps)
            umma_bf16_pair_warp(d, a0 + (k >> 2) * (16384 >> 4) + (k & 3) * 2, b0 + (k >> 2) * (16384 >> 4) + (k & 3) * 2,
                                idesc, k > 0 ? 1u : 0u);
        }
        umma_bf16_pair_warp(d, daug, bb, idesc, 1u);   // + bias
        umma_commit_pair_warp(bar(misc->ufull[buf]));
        umma_commit_pair_warp(bar(misc->zempty[zs]));
        if (p == HP - 1) umma_commit_pair_warp(bar(misc->kempty[ts]));
      }
    }
    // this warp's MMAs complete before TMEM is released
    umma_commit_pair_warp(bar(misc->mma_done));
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar(misc->mma_done), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
  } else if (warp >= 2 && warp < 10) {
    // ======================================================== epilogue (warps 2-9)
    // One token per thread (TMEM lane); warp group g holds the frequencies
    // f in [32 g, 32 g + 32) of the rotary score of both heads of a stage:
    //   s_h = sum_f cos(j th_f) U_h,f + sin(j th_f) U_h,64+f,
    // adds the other group's half through shared memory and takes head 2p + g's
    // softmax weights.
    const int we = warp - 2, g = we >> 2, q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int H = a.H;
    const int64_t prow = a.ntiles * kVTile;   // weights per (sequence, head)
    const int64_t ngroups = a.ntiles * 4;     // 32-token groups per (sequence, head)

    // cos / sin(j th_f) of this thread's token j for its 32 frequencies, from the
    // transposed table (a warp's 32 tokens are one 128-byte line per frequency)
    float cs[32], sn[32];
    auto load_trig = [&](const Walker2d& wb) {
      const int64_t j = static_cast<int64_t>(wb.kb) * kBlock2dTokens + rank * kTile + row;
      const float* tc = a.trigT + static_cast<int64_t>(32 * g) * a.trig_rows + j;
      const float* ts = tc + 64 * a.trig_rows;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        cs[i] = tc[i * a.trig_rows];
        sn[i] = ts[i * a.trig_rows];
      }
    };
    auto epi_sync = []() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    // score-buffer release: this thread's TMEM reads completed (tcgen05.wait::ld) and
    // were fenced before the arrive, so the pair's later MMA into the buffer cannot
    // overtake them; nothing else needs to be made visible, so no cluster release
    auto release_u = [&](uint32_t b) {
      if (rank == 0) {
        mbar_arrive(b);
      } else {
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(map_to_rank(b, 0))
                     : "memory");
      }
    };
    // sum over this group's frequencies of one head: cos part u_c, sin part u_s
    auto half_score = [&](const float (&u_c)[32], const float (&u_s)[32]) {
      float x0 = 0.f, x1 = 0.f, y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        ffma2(x0, x1, u_c[2 * i], u_c[2 * i + 1], cs[2 * i], cs[2 * i + 1]);
        ffma2(y0, y1, u_s[2 * i], u_s[2 * i + 1], sn[2 * i], sn[2 * i + 1]);
      }
      return (x0 + x1) + (y0 + y1);
    };

    Walker2d w = start;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the transposed RoPE table is written
    load_trig(w);
    bool ok = true;
    uint32_t G = 0;
    for (int n = 0; n < count; ++n) {
      const int tile_tok = w.kb * kBlock2dTokens + static_cast<int>(rank) * kTile;
      const int j = tile_tok + row;
      const bool valid = j < w.L;
      const bool tvalid = tile_tok < w.L;     // the tile holds a token of the sequence
      const int64_t grp = tile_tok / 32 + q;  // this warp's 32 tokens
#pragma unroll 1
      for (int p = 0; p < HP; ++p, ++G) {
        const uint32_t buf = G & 1u;
        if (ok) ok = warp_poll(bar(misc->ufull[buf]), (G >> 1) & 1u, abort, a.status);
        bool released = false;
        float part[2] = {0.f, 0.f};   // this group's half of head 2p, 2p + 1
        if (ok) {
          tc_fence_after();
          const uint32_t tU = tmem + lane_base + 256 * buf + 32 * g;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float u_c[32], u_s[32];
            tmem_ld_x32(tU + 128 * hh, u_c);
            tmem_ld_x32(tU + 128 * hh + 64, u_s);
            tmem_wait_ld();
            if (hh == 1) {
              // every read of the buffer has completed: hand it back before the sums
              tc_fence_before();
              __syncwarp();
              if (lane == 0) release_u(bar(misc->uempty[buf]));
              released = true;
            }
            part[hh] = half_score(u_c, u_s);
          }
        }
        if (!released) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_u(bar(misc->uempty[buf]));
        }
        // exchange halves: this group keeps head 2p + g
        const float mine = g ? part[1] : part[0], other = g ? part[0] : part[1];
        misc->xch[buf][1 - g][row] = other;
        epi_sync();
        const float s = valid ? mine + misc->xch[buf][g][row] : -INFINITY;
        // the group's weights 2^(s - m), m = ceil(max s) over its 32 tokens (-inf
        // when none of them is in the sequence)
        const float m = ceilf(warp_max_redux(s));
        const __nv_bfloat16 pb = __float2bfloat16_rn(valid ? exp2f(s - m) : 0.f);
        const int h = 2 * p + g;
        if (tvalid) {
          a.pw[(static_cast<int64_t>(w.b) * H + h) * prow + j] = __bfloat16_as_ushort(pb);
          if (lane == 0) a.grp_m[(static_cast<int64_t>(w.b) * H + h) * ngroups + grp] = m;
        }
      }
      walk_advance(w, a);
      // this thread's token row is no longer needed: fetch the next block's now
      if (n + 1 < count) load_trig(w);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's MMAs and remote arrives are done with this CTA's memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

struct alignas(16) MiscValue {
  uint64_t full[kVS], fixed[kVS], empty[kVS];
  uint64_t dfull[2], dempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int start_b, start_t, count, total_tiles;
  float mrun[2][kMax2dHeads];    // per run parity: M of each head
  float pm[8][kMax2dHeads];      // partial maxima of 8 group subsets
  int scan[kValue2dThreads];
};
static_assert(sizeof(MiscValue) <= 4096, "value misc region");

// Tile of one sequence: tokens [128 t, 128 t + 128).
struct TileWalker {
  int b, t, nt, L;
  __device__ __forceinline__ void advance(const Decode2dArgs& a) {
    if (++t < nt) return;
    t = 0;
    while (true) {
      if (++b >= a.B) { nt = 0; return; }
      L = clamp_len(__ldg(a.seq_lens + b), a.L_max);
      nt = ntiles_of(L);
      if (nt > 0) return;
    }
  }
};

// D_v of every head over runs of 128-token tiles (Appendix J):
//   D[r][h] = sum_j w_j,h c_v,j[r],   l[h] = sum_j w_j,h,   w_j,h = 2^(m_g(j) - M) p_j,h,
// over the 32-token groups g of the run, with M the largest m_g (all of them
// integers, so each scale is an exact power of two and w is the bf16 weight the
// MMA reads).  One record (M, l, D) per (sequence, CTA).  Roles: warp 0
// copies (V tile + weight tile per ring stage), warp 1 issues the MMAs (M = 128
// rows of r_v, N = 16 heads, K = 16 tokens), warps 2-5 scale each weight tile,
// zero V rows past the sequence end, and write the records.
__global__ void __launch_bounds__(kValue2dThreads, 1)
decode2d_value_kernel(const __grid_constant__ Decode2dArgs a, const __grid_constant__ Decode2dMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Decode2dPlan& P = a.plan;
  const uint32_t sbase = smem_u32(sm);
  MiscValue* misc = reinterpret_cast<MiscValue*>(sm + P.v_misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) misc->abort = 0;
  share_of<kValue2dThreads>(
      a, [&](int b) { return ntiles_of(clamp_len(__ldg(a.seq_lens + b), a.L_max)); }, blockIdx.x, gridDim.x,
      misc->scan, &misc->start_b, &misc->start_t, &misc->count, &misc->total_tiles);
  const int count = misc->count;
  if (count == 0) return;
  TileWalker start;
  start.b = misc->start_b;
  start.t = misc->start_t;
  start.L = clamp_len(__ldg(a.seq_lens + start.b), a.L_max);
  start.nt = ntiles_of(start.L);

  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    for (int s = 0; s < kVS; ++s) {
      mbar_init(bar(misc->full[s]), 1);
      mbar_init(bar(misc->fixed[s]), 4);   // the 4 scaling warps
      mbar_init(bar(misc->empty[s]), 1);   // MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(misc->dfull[i]), 1);   // MMA commit after a run's last tile
      mbar_init(bar(misc->dempty[i]), 4);  // the 4 record warps
    }
    mbar_init(bar(misc->mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.v);
    prefetch_tmap(&maps.p);
  }
  // weight rows of heads >= H stay zero (the copies write H rows of each box)
  for (int s = 0; s < kVS; ++s)
    for (int i = tid; i < 4096 / 16; i += kValue2dThreads)
      reinterpret_cast<uint4*>(sm + P.v_ring + s * P.v_stage + P.nvb * 16384)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&misc->tmem_base), 64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  // the combine grid may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the weights and tile maxima are written by the score grid
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ======================================================== TMA producer
    if (lane == 0) {
      TileWalker w = start;
      RingPos r;
      int issued = 0;
      bool ok = true;
      const uint64_t pol_stream = l2_policy_evict_first();
      for (int i = 0; i < count && ok; ++i) {
        const int s = r.slot;
        if (!(ok = mbar_wait(bar(misc->empty[s]), r.phase ^ 1u, abort, a.status))) break;
        const uint32_t fb = bar(misc->full[s]);
        mbar_arrive_expect_tx(fb, P.nvb * 16384 + 2 * 64 * 2 * a.H);
        const uint32_t dst = sbase + P.v_ring + s * P.v_stage;
        const int y = w.t * kVTile;
        for (int bx = 0; bx < P.nvb; ++bx) tma_load_3d_hint(dst + bx * 16384, &maps.v, fb, 64 * bx, y, w.b, pol_stream);
        for (int kb = 0; kb < 2; ++kb) tma_load_3d(dst + P.nvb * 16384 + kb * 2048, &maps.p, fb, y + 64 * kb, 0, w.b);
        ++issued;
        r.next(kVS);
        w.advance(a);
      }
      for (int i = max(0, issued - kVS); i < issued; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->full[i % kVS]), (i / kVS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    // ======================================================== MMA issuer (whole warp)
    const uint32_t idesc = umma_idesc_bf16(128, 16, true, false);
    // MN-major V: 64-row r_v boxes 16 KB apart (LBO), 8 token rows 1 KB apart (SBO);
    // K-major weights: 16 head rows, 64-token boxes 2 KB apart
    const uint64_t dV0 = umma_desc(sbase + P.v_ring, 16384, 1024, kSw128);
    const uint64_t dP0 = umma_desc(sbase + P.v_ring + P.nvb * 16384, 16, 1024, kSw128);
    const uint32_t vst = static_cast<uint32_t>(P.v_stage) >> 4;
    auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
    TileWalker w = start;
    RingPos r;
    bool ok = true;
    uint32_t run = 0;
    for (int i = 0; i < count && ok; ++i) {
      const int s = r.slot;
      const bool run_start = i == 0 || w.t == 0;
      const bool run_end = i == count - 1 || w.t == w.nt - 1;
      const uint32_t db = run & 1u;
      if (!(ok = agree(mbar_wait(bar(misc->fixed[s]), r.phase, abort, a.status)))) break;
      if (run_start && !(ok = agree(mbar_wait(bar(misc->dempty[db]), ((run >> 1) & 1u) ^ 1u, abort, a.status)))) break;
      tc_fence_after();
      const uint64_t av = dV0 + s * vst, bp = dP0 + s * vst;
      const int valid = w.L - w.t * kVTile;
#pragma unroll
      for (int k = 0; k < 8; ++k) {   // 16-token K steps: +2 KB in each V box, +32 B in the weight rows
        if (16 * k >= valid) break;
#pragma unroll
        for (int ci = 0; ci < 2; ++ci)
          if (ci < P.nvc)
            umma_bf16_warp(tmem + 32 * db + 16 * ci, av + ci * ((2 * 16384) >> 4) + k * (2048 >> 4),
                           bp + (k >> 2) * (2048 >> 4) + (k & 3) * 2, idesc, (!run_start || k > 0) ? 1u : 0u);
      }
      umma_commit_warp(bar(misc->empty[s]));
      if (run_end) {
        umma_commit_warp(bar(misc->dfull[db]));
        ++run;
      }
      r.next(kVS);
      w.advance(a);
    }
    umma_commit_warp(bar(misc->mma_done));
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar(misc->mma_done), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
  } else {
    // ======================================================== scaling and records (warps 2-5)
    const int ft = tid - 64, q = warp & 3;
    const int row = 32 * q + lane;                     // r_v row in a 128-row chunk (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int H = a.H;
    auto grp_sync = []() { asm volatile("bar.sync 2, 128;" ::: "memory"); };
    // weight row (head) this thread scales, and the 8-token piece of it: the 16-byte
    // chunk ft & 7 as stored holds logical chunk (ft & 7) ^ (row & 7) (128-byte swizzle)
    const int hs = ft >> 3, piece = (ft & 7) ^ (hs & 7);
    const int64_t ngroups = a.ntiles * 4;
    float lsum = 0.f;   // this thread's share of the run's l of head hs
    TileWalker w = start;
    RingPos r;
    bool ok = true;
    uint32_t run = 0;
    for (int i = 0; i < count; ++i) {
      const bool run_start = i == 0 || w.t == 0;
      const bool run_end = i == count - 1 || w.t == w.nt - 1;
      const int par = run & 1;
      if (run_start) {
        // the run: tiles [w.t, te) of sequence w.b; its M per head, the largest m of
        // its groups (groups past the sequence end hold -inf)
        const int te = min(w.nt, w.t + (count - i));
        const int h = ft & 15, sub = ft >> 4;
        float M = -INFINITY;
        if (h < H) {
          const float* gm = a.grp_m + (static_cast<int64_t>(w.b) * H + h) * ngroups;
          for (int gi = 4 * w.t + sub; gi < 4 * te; gi += 8) M = fmaxf(M, gm[gi]);
        }
        misc->pm[sub][h] = M;
        grp_sync();
        if (ft < H) {
          float Mr = misc->pm[0][ft];
#pragma unroll
          for (int u = 1; u < 8; ++u) Mr = fmaxf(Mr, misc->pm[u][ft]);
          misc->mrun[par][ft] = Mr;
        }
        grp_sync();
        lsum = 0.f;
      }
      // 2^(m_g - M_run), an exact power of two, for the group of each of this
      // thread's two pieces (tokens 64 kb + 8 piece ...)
      float sc[2] = {0.f, 0.f};
      if (hs < H) {
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const int64_t gi = 4 * static_cast<int64_t>(w.t) + 2 * kb + (piece >> 2);
          const float m = a.grp_m[(static_cast<int64_t>(w.b) * H + hs) * ngroups + gi];
          const float Mr = misc->mrun[par][hs];
          if (m != -INFINITY && Mr != -INFINITY) {
            const int e = static_cast<int>(m - Mr);
            sc[kb] = e < -126 ? 0.f : __int_as_float((127 + e) << 23);
          }
        }
      }
      const int s = r.slot;
      if (ok) ok = warp_wait(bar(misc->full[s]), r.phase, abort, a.status);
      uint8_t* st = sm + P.v_ring + s * P.v_stage;
      if (ok) {
        // weights: 16 rows of 128 B in each of the two 64-token boxes; thread ft takes
        // 16 bytes of row hs in both (the swizzle moves chunks within a row only)
        if (hs < H) {
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            uint4* pp = reinterpret_cast<uint4*>(st + P.nvb * 16384 + kb * 2048) + ft;
            uint4 v = *pp;
            uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[c]));
              const __nv_bfloat162 wv = __floats2bfloat162_rn(f.x * sc[kb], f.y * sc[kb]);
              const float2 wf = __bfloat1622float2(wv);
              lsum += wf.x + wf.y;
              u[c] = bf16x2_bits(wv);
            }
            *pp = v;
          }
        }
        // V rows past the sequence end may hold anything: zero them (0 * x stays 0)
        const int valid = w.L - w.t * kVTile;
        if (valid < kVTile) {
          const int per_box = (kVTile - valid) * 8;
          for (int x = ft; x < P.nvb * per_box; x += 128) {
            const int bx = x / per_box, rr = valid + (x - bx * per_box) / 8, c16 = x & 7;
            *reinterpret_cast<uint4*>(st + bx * 16384 + rr * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(misc->fixed[s]));
      r.next(kVS);
      if (run_end) {
        // the run's record, once its last MMAs are complete
        const uint32_t db = run & 1u;
        if (ok) ok = warp_wait(bar(misc->dfull[db]), (run >> 1) & 1u, abort, a.status);
        tc_fence_after();
        const int64_t rec = static_cast<int64_t>(w.b) + blockIdx.x;
        if (ok) {
#pragma unroll
          for (int ci = 0; ci < 2; ++ci) {
            if (ci < P.nvc) {
              float v[16];
              tmem_ld_x16(tmem + lane_base + 32 * db + 16 * ci, v);
              tmem_wait_ld();
              const int rr = 128 * ci + row;
              if (rr < a.r_v) {
#pragma unroll
                for (int h = 0; h < kMax2dHeads; ++h)
                  if (h < H) a.rec_acc[(rec * H + h) * a.r_v + rr] = v[h];
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->dempty[db]));
        // l: the sum over the 8 threads (lanes) of each head row
        float l = lsum;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        if ((ft & 7) == 0 && hs < H) {
          a.rec_ml[(rec * H + hs) * 2] = misc->mrun[par][hs];
          a.rec_ml[(rec * H + hs) * 2 + 1] = l;
        }
        ++run;
      }
      w.advance(a);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// Merge the run records of each (sequence, head) by log-sum-exp, apply the V
// up-projection once (Appendix J identity) and normalise:
//   out = (sum_c 2^(m_c - M) acc_c) W_up,v,t,h^T / (sum_c 2^(m_c - M) l_c) + mu_v,t,h.
// A sequence's records come from the value CTAs whose tile ranges overlap it.  Block = (head h, two consecutive sequences); W_up,v,t,h is
// staged in shared memory (rows padded by one word) before the wait for the
// decode grid.
constexpr int kCombineUnits = 16;   // sequences per block (W_up,v,t,h staged once for all)
constexpr int kCombineThreads = 128;

size_t combine_smem_bytes(int r_v) {
  return (static_cast<size_t>(128) * (r_v / 2 + 1) + kCombineUnits * 256 + 3 * kCombineUnits) * 4;
}

__global__ void __launch_bounds__(kCombineThreads) decode2d_combine_kernel(const __grid_constant__ Decode2dArgs a) {
  extern __shared__ float csm[];
  __shared__ int red[kCombineThreads / 32];
  const int h = blockIdx.x, b0 = blockIdx.y * kCombineUnits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rw = a.r_v / 2, wpr = rw + 1;
  uint32_t* Ws = reinterpret_cast<uint32_t*>(csm);
  float* accs = csm + 128 * wpr;   // [kCombineUnits][256]
  float* Ms = accs + kCombineUnits * 256;
  float* Ls = Ms + kCombineUnits;
  int* Tp = reinterpret_cast<int*>(Ls + kCombineUnits);   // tiles of the block's sequences before each
  {
    const uint4* Wg = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w_up_v) +
                                                     static_cast<int64_t>(h) * kHeadDim * a.r_v);
    const int n16 = 128 * rw / 4;
    constexpr int kMax = 128 * 128 / 4 / kCombineThreads;
    uint4 v[kMax];
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
      const int i = tid + j * kCombineThreads;
      v[j] = i < n16 ? __ldg(Wg + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
      const int i = tid + j * kCombineThreads;
      if (i < n16) {
        const int e = i / (rw / 4), k = 4 * (i - e * (rw / 4));
        uint32_t* d = Ws + e * wpr + k;
        d[0] = v[j].x; d[1] = v[j].y; d[2] = v[j].z; d[3] = v[j].w;
      }
    }
  }
  int before = 0, all = 0;   // tiles of sequences [0, b0) and [0, B)
  for (int bb = tid; bb < a.B; bb += kCombineThreads) {
    const int n = ntiles_of(clamp_len(__ldg(a.seq_lens + bb), a.L_max));
    all += n;
    if (bb < b0) before += n;
  }
  before = __reduce_add_sync(0xffffffffu, before);
  all = __reduce_add_sync(0xffffffffu, all);
  if (lane == 0) red[warp] = before;
  __syncthreads();
  int pre = 0;
#pragma unroll
  for (int w = 0; w < kCombineThreads / 32; ++w) pre += red[w];
  __syncthreads();
  if (lane == 0) red[warp] = all;
  __syncthreads();
  int tot = 0;
#pragma unroll
  for (int w = 0; w < kCombineThreads / 32; ++w) tot += red[w];

  if (tid == 0) {
    int t = 0;
    for (int u = 0; u < kCombineUnits; ++u) {
      Tp[u] = t;
      if (b0 + u < a.B) t += ntiles_of(clamp_len(__ldg(a.seq_lens + b0 + u), a.L_max));
    }
  }
  __syncthreads();

  asm volatile("griddepcontrol.wait;" ::: "memory");   // records written

  // warp w merges the records of sequences b0 + w, b0 + w + 4, ...
  for (int u = warp; u < kCombineUnits; u += kCombineThreads / 32) {
    const int b = b0 + u;
    float M = -INFINITY, Lt = 0.f;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    const int nb = b < a.B ? ntiles_of(clamp_len(__ldg(a.seq_lens + b), a.L_max)) : 0;
    if (nb > 0) {
      const long long B0 = pre + Tp[u];
      const long long NB = tot, NP = a.units;
      const long long p0 = ((B0 + 1) * NP - 1) / NB, p1 = ((B0 + nb) * NP - 1) / NB;
      for (long long p = p0; p <= p1; ++p) {
        const long long lo = p * NB / NP, hi = (p + 1) * NB / NP;
        if (max(lo, B0) >= min(hi, B0 + nb)) continue;   // the value CTA saw no tile of b
        const long long rec = b + p;
        const float mr = a.rec_ml[(rec * a.H + h) * 2], lr = a.rec_ml[(rec * a.H + h) * 2 + 1];
        const float* ar = a.rec_acc + (rec * a.H + h) * a.r_v;
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = lane + 32 * j < a.r_v ? ar[lane + 32 * j] : 0.f;
        if (mr == -INFINITY) continue;
        const float Mn = fmaxf(M, mr);
        const float alpha = M == -INFINITY ? 0.f : exp2f(M - Mn), wr = exp2f(mr - Mn);
        Lt = fmaf(lr, wr, Lt * alpha);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(x[j], wr, acc[j] * alpha);
        M = Mn;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < a.r_v) accs[u * 256 + lane + 32 * j] = acc[j];
    if (lane == 0) { Ms[u] = M; Ls[u] = Lt; }
  }
  __syncthreads();

  const int e = tid;
  float o[kCombineUnits];
#pragma unroll
  for (int j = 0; j < kCombineUnits; ++j) o[j] = 0.f;
  const uint32_t* wr = Ws + e * wpr;
#pragma unroll 4
  for (int k = 0; k < rw; ++k) {
    const uint32_t w2 = wr[k];
    const float wlo = __uint_as_float(w2 << 16), whi = __uint_as_float(w2 & 0xFFFF0000u);
#pragma unroll
    for (int j = 0; j < kCombineUnits; ++j) {
      const float2 av = *reinterpret_cast<const float2*>(accs + j * 256 + 2 * k);
      o[j] = fmaf(av.x, wlo, fmaf(av.y, whi, o[j]));
    }
  }
  const float mu = __ldg(a.mu_v + static_cast<int64_t>(h) * kHeadDim + e);
#pragma unroll
  for (int j = 0; j < kCombineUnits; ++j) {
    const int bb = b0 + j;
    if (bb >= a.B) continue;
    const int64_t uu = static_cast<int64_t>(bb) * a.H + h;
    const bool empty = Ms[j] == -INFINITY;
    a.out[uu * kHeadDim + e] = empty ? 0.f : o[j] / Ls[j] + mu;
    if (e == 0) a.lse[uu] = empty ? -INFINITY : (Ms[j] + log2f(Ls[j])) * kLn2;
  }
}

}  // namespace

bool make_decode2d_plan(int H, int r_k, int r_v, Decode2dPlan* p) {
  *p = Decode2dPlan{};
  if (H < 2 || H > kMax2dHeads || H % 2 || r_k < 16 || r_k > 128 || r_v < 16 || r_v > 256 || r_k % 16 ||
      r_v % 16)
    return false;
  // score kernel
  p->nkc = (r_k + 63) / 64;
  p->k_stage = p->nkc * 16384;
  p->z_stage = p->nkc * 16384 + 4096;   // one head's 128 operand rows, then their bias operand
  int off = 0;
  p->k_ring = off; off += kSNK * p->k_stage;
  p->z_ring = off; off += kSNZ * p->z_stage;
  p->aug_a = off;  off += 4096;
  p->misc = off;   off += 4096;
  p->bytes = off + 1024;
  // value kernel: per stage the V tile (64-wide r_v boxes of 128 tokens), then the
  // weight tile (two 64-token boxes of 16 head rows)
  p->nvb = (r_v + 63) / 64;
  p->nvc = (r_v + 127) / 128;
  p->v_stage = p->nvb * 16384 + 4096;
  p->v_ring = 0;
  p->v_misc = kVS * p->v_stage;
  p->v_bytes = p->v_misc + 4096 + 1024;
  return p->bytes <= kSmemLimit && p->v_bytes <= kSmemLimit;
}

size_t decode2d_zimg_stride(int H, int r_k) {
  const size_t nkc = (r_k + 63) / 64;
  const size_t b = nkc * H * kHeadDim * kZRowBytes + static_cast<size_t>(H) * kHeadDim * 32;
  return (b + 1023) / 1024 * 1024;
}

int64_t decode2d_trig_rows(int64_t L_max) {
  return (L_max + kBlock2dTokens - 1) / kBlock2dTokens * kBlock2dTokens;
}

cudaError_t launch_decode2d_bf16(Decode2dArgs& a, const Decode2dMaps& maps, cudaStream_t s) {
  static int configured = 0, vconfigured = 0;
  if (configured < a.plan.bytes) {
    cudaError_t e = cudaFuncSetAttribute(decode2d_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         a.plan.bytes);
    if (e != cudaSuccess) return e;
    configured = a.plan.bytes;
  }
  if (vconfigured < a.plan.v_bytes) {
    cudaError_t e = cudaFuncSetAttribute(decode2d_value_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         a.plan.v_bytes);
    if (e != cudaSuccess) return e;
    vconfigured = a.plan.v_bytes;
  }
  // pairs that can be resident at once (each CTA needs a whole SM)
  static int pairs_for = -1, max_pairs = 0;
  if (pairs_for != a.plan.bytes) {
    cudaLaunchConfig_t occ = {};
    occ.gridDim = dim3(2);
    occ.blockDim = dim3(kScore2dThreads);
    occ.dynamicSmemBytes = a.plan.bytes;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, decode2d_score_kernel, &occ);
    if (e != cudaSuccess) return e;
    max_pairs = n;
    pairs_for = a.plan.bytes;
  }
  if (max_pairs < 1) return cudaErrorLaunchOutOfResources;
  a.pairs = std::min(a.pairs, std::min(max_pairs, kMaxPairs));
  if (a.pairs < 1) a.pairs = 1;
  if (a.units < 1) a.units = 1;

  decode2d_z_kernel<<<a.B * a.H + static_cast<int>(a.trig_rows / kTrigTokensPerBlock), kZThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.pairs);
  cfg.blockDim = dim3(kScore2dThreads);
  cfg.dynamicSmemBytes = a.plan.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode2d_score_kernel, a, maps);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(a.units);
  cfg.blockDim = dim3(kValue2dThreads);
  cfg.dynamicSmemBytes = a.plan.v_bytes;
  e = cudaLaunchKernelEx(&cfg, decode2d_value_kernel, a, maps);
  if (e != cudaSuccess) return e;
  const size_t csmem = combine_smem_bytes(a.r_v);
  static size_t cconfigured = 0;
  if (cconfigured < csmem) {
    e = cudaFuncSetAttribute(decode2d_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(csmem));
    if (e != cudaSuccess) return e;
    cconfigured = csmem;
  }
  cfg.gridDim = dim3(a.H, (a.B + kCombineUnits - 1) / kCombineUnits);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = csmem;
  return cudaLaunchKernelEx(&cfg, decode2d_combine_kernel, a);
}

}  // namespace lla
