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
// byte, so the call is bound by the tensor pipe, not by HBM.
//
// Design (CTA pairs, tcgen05 cta_group::2):
//  * Work is cut into blocks of 512 tokens of one sequence; each pair of CTAs
//    (a cluster of two on neighbouring SMs) takes a contiguous range of blocks.
//    CTA `rank` holds the block's K latent tiles at rows 256*rank + {0, 128}.
//  * For every head h and tile slot the pair MMA U = C_k Z_h^T runs with
//    M = 256 tokens (128 from each CTA), N = 128, K = r_k.  Z_h is the query
//    operand of the per-head kernel (the RoPE-rotated, scaled query folded into
//    W_up,k,t,h, built by decode2d_z_kernel); its rows are split between the two
//    CTAs, so each SM receives half of every head's operand.  The latent tiles
//    stay resident while the H operands stream through, which keeps both the
//    shared-memory read rate of the MMAs and the per-SM copy rate within bounds.
//  * Epilogue warps (one token per thread, fixed for the block) form the rotary
//    score s = sum_f cos(j th_f) (U_f + b_f) + sin(j th_f) (U_64+f + b_64+f) from
//    the token's cos/sin row held in registers (b = the mu_k term), and keep the
//    block's scores in TMEM.  At the end of a block an exact per-head
//    maximum over the CTA's 256 tokens sets the softmax reference (raised lazily,
//    by more than 2^8), P (bf16, heads x tokens) is written, and the value MMA
//    D_v += C_v^T P (M = r_v rows, N = heads; Appendix J) accumulates in TMEM over
//    the blocks of a sequence.  The value MMAs of block n run interleaved with
//    the score MMAs of block n + 1.
//  * When a CTA's run of a sequence ends it writes one record (m, l, acc_v) per
//    head; decode2d_combine_kernel merges the records of a sequence (log-sum-exp
//    merge) and applies the V up-projection once.
//
#include "lla_kernels.h"

#include <algorithm>
#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr float kRescaleLog2 = 8.f;                 // lazy reference threshold (log2 units)
constexpr int kNK = 3;        // latent tile slots (two per block)
constexpr int kNZ = 4;        // query-operand windows in flight (a group of four heads)
constexpr int kNV = 2;        // value chunk slots
constexpr int kNU = 3;        // TMEM score buffers (128 columns each)
constexpr int kVChunks = 8;   // 32-token value chunks of a CTA's 256 block tokens
constexpr int kVTok = 32;     // tokens per value chunk (two 16-token K steps)
constexpr uint32_t kScoreCol = 448;   // TMEM columns of the block's scores: 16 per warp group
constexpr uint32_t kDvCol = 384;   // TMEM column of the value accumulators (2 x 32)
constexpr int kZRowBytes = 128;    // one 64-wide bf16 chunk row

struct alignas(16) Misc2d {
  // full barriers: in the even CTA they also take the odd CTA's relay arrive (count
  // 2), so one wait covers both halves of a pair operand
  uint64_t kfull[kNK], kempty[kNK];
  uint64_t zfull[kNZ], zempty[kNZ];
  uint64_t vfull[kNV], vempty[kNV];
  // Score buffers: ufull per epilogue warp group (the group of a stage is its tile
  // slot), so that a group, which skips the other group's stages, never waits on a
  // barrier phase more than one completion ahead; uempty has one waiter (the issuer).
  uint64_t ufull[2][kNU], uempty[kNU];
  uint64_t pfull, vdone, mma_done[2];
  uint32_t tmem_base;
  int abort;
  int start_b, start_kb, count, total_blocks;
  float mx[8][kMax2dHeads];   // per epilogue warp: block maximum of each head
  float lp[8][kMax2dHeads];   // per epilogue warp: a run's sum of the weights of each head
  float m_ref[kMax2dHeads];   // softmax reference of each head (log2 units)
  float m_new[kMax2dHeads], alpha[kMax2dHeads];   // the block's new reference, rescale factor
  float m_rec[kMax2dHeads];   // reference of a finished run (for its record)
  int scan[kDecode2dThreads];
};
static_assert(sizeof(Misc2d) <= 4096, "misc region");

struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) { slot = 0; phase ^= 1u; }
  }
};

// Block of one sequence: tokens [512 kb, 512 kb + 512).
struct Walker2d {
  int b, kb, nb, L;
};

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

__device__ __forceinline__ int nblocks(int L) { return (L + kBlock2dTokens - 1) / kBlock2dTokens; }

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

// Score stages of a block: head by head, tile slot 0 then tile slot 1 (stage
// st = 2h + s), so the two epilogue warp groups (one per tile slot) take turns.
// Value chunk c of the previous block follows head vchunk_head(c) in every role's
// order (the first one two heads in, once that block's weights exist).
__device__ __forceinline__ int vchunk_head(int c, int H) { return min(2 * c + 2, H - 1); }

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
// them write the f16 copy of the RoPE table the epilogue reads (64 rows each).
constexpr int kZThreads = 256;
constexpr int kTrigRowsPerBlock = 64;
__global__ void __launch_bounds__(kZThreads) decode2d_z_kernel(const __grid_constant__ Decode2dArgs a) {
  // the decode grid may start its set-up now; it waits for this grid before it
  // copies an image
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float qs[2][64];
  const int u = blockIdx.x, tid = threadIdx.x;
  if (u >= a.B * a.H) {
    // RoPE rows as f16 pairs: row p = {cos(p th_2i), cos(p th_2i+1)} i < 32, then sin
    const int64_t r0 = static_cast<int64_t>(u - a.B * a.H) * kTrigRowsPerBlock;
    for (int i = tid; i < kTrigRowsPerBlock * 64; i += kZThreads) {
      const int64_t r = r0 + i / 64;
      const int c = i % 64;            // pair index: 0..31 cos, 32..63 sin
      if (r >= a.trig_rows) break;
      const float* src = (c < 32 ? a.rope_cos : a.rope_sin) + r * 64 + 2 * (c & 31);
      const __half2 v = __floats2half2_rn(src[0], src[1]);
      a.trig16[r * 64 + c] = *reinterpret_cast<const uint32_t*>(&v);
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

// Spinning form of mbar_wait_cluster (no suspend hint): for the issuer's waits on
// barriers whose arrivals come from the epilogue warps of both CTAs.
__device__ __forceinline__ bool mbar_spin_cluster(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(bar, parity, 0)) return true;
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kDecode2dThreads, 1)
decode2d_bf16_kernel(const __grid_constant__ Decode2dArgs a, const __grid_constant__ Decode2dMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Decode2dPlan& P = a.plan;
  const uint32_t sbase = smem_u32(sm);
  Misc2d* misc = reinterpret_cast<Misc2d*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_cta_rank();
  const int pair = static_cast<int>(blockIdx.x >> 1);

  // ---------------------------------------------------------- work range (same in both CTAs)
  {
    const int per_thr = (a.B + kDecode2dThreads - 1) / kDecode2dThreads;
    const int b0 = min(a.B, tid * per_thr), b1 = min(a.B, b0 + per_thr);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      const int L0 = __ldg(a.seq_lens + b);
      if ((L0 < 0 || L0 > a.L_max) && blockIdx.x == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
      local += nblocks(clamp_len(L0, a.L_max));
    }
    misc->scan[tid] = local;
    if (tid == 0) misc->abort = 0;
    __syncthreads();
    if (warp == 0) {
      constexpr int kPer = kDecode2dThreads / 32;
      int v[kPer];
      int s = 0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) { v[i] = misc->scan[lane * kPer + i]; s += v[i]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int excl = incl - s;
#pragma unroll
      for (int i = 0; i < kPer; ++i) { misc->scan[lane * kPer + i] = excl; excl += v[i]; }
      if (lane == 31) misc->total_blocks = incl;
    }
    __syncthreads();
    const long long NB = misc->total_blocks;
    const long long lo = pair * NB / a.pairs, hi = (pair + 1) * NB / a.pairs;
    long long P0 = misc->scan[tid];
    for (int b = b0; b < b1; ++b) {
      const int nb = nblocks(clamp_len(__ldg(a.seq_lens + b), a.L_max));
      if (nb > 0 && lo < hi && P0 <= lo && lo < P0 + nb) {
        misc->start_b = b;
        misc->start_kb = static_cast<int>(lo - P0);
      }
      P0 += nb;
    }
    if (tid == 0) misc->count = static_cast<int>(hi - lo);
    __syncthreads();
  }
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
    const uint32_t nfull = rank == 0 ? 2 : 1;   // + the odd CTA's relay in the even CTA
    for (int s = 0; s < kNK; ++s) {
      mbar_init(bar(misc->kfull[s]), nfull);
      mbar_init(bar(misc->kempty[s]), 4);       // the tile's warp group, after its last stage
    }
    for (int s = 0; s < kNZ; ++s) {
      mbar_init(bar(misc->zfull[s]), nfull);
      mbar_init(bar(misc->zempty[s]), 4);       // warp group 1, after the window's last stage
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(bar(misc->vfull[s]), nfull);
      mbar_init(bar(misc->vempty[s]), 1);
    }
    for (int s = 0; s < kNU; ++s) {
      mbar_init(bar(misc->ufull[0][s]), 1);
      mbar_init(bar(misc->ufull[1][s]), 1);
      mbar_init(bar(misc->uempty[s]), 8);        // 4 epilogue warps of each CTA
    }
    mbar_init(bar(misc->pfull), 16);             // 8 epilogue warps of each CTA
    mbar_init(bar(misc->vdone), 1);
    mbar_init(bar(misc->mma_done[0]), 1);
    mbar_init(bar(misc->mma_done[1]), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
  }
  // P rows of heads >= H stay zero
  for (int i = tid; i < 16 * 512 / 16; i += kDecode2dThreads)
    reinterpret_cast<uint4*>(sm + P.p)[i] = make_uint4(0, 0, 0, 0);
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
  // the combine grid may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = misc->tmem_base;

  // Zero value-chunk rows past the sequence end (they may hold anything; their
  // weights are 0, and 0 * x must stay 0 in the value MMA).
  auto zero_v_tail = [&](int sv, int valid) {
    if (valid >= kVTok) return;
    const int r0 = valid < 0 ? 0 : valid;
    uint8_t* vs = sm + P.v_ring + sv * P.v_stage;
    for (int bx = 0; bx < 2 * P.nvh; ++bx)
      for (int r = r0; r < kVTok; ++r)
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<uint4*>(vs + bx * 4096 + r * kZRowBytes + g * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  };

  if (warp == 0) {
    // ======================================================== TMA producer (each CTA)
    // Per block: both latent tiles, then per head its query window, with the value
    // chunks of the previous block after head vchunk_head(c) -- the issuers' order.
    if (lane == 0) {
      Walker2d w = start, wp = start;
      RingPos kr, zr, vr;
      int issued_k = 0, issued_z = 0, issued_v = 0;
      bool ok = true, images_ready = false;
      auto load_v = [&](const Walker2d& wb, int c) -> bool {
        const int sv = vr.slot;
        if (!mbar_wait(bar(misc->vempty[sv]), vr.phase ^ 1u, abort, a.status)) return false;
        const uint32_t fb = bar(misc->vfull[sv]);
        mbar_arrive_expect_tx(fb, P.nvh * 8192);
        const int y = wb.kb * kBlock2dTokens + static_cast<int>(rank) * 256 + kVTok * c;
        const uint32_t dst = sbase + P.v_ring + sv * P.v_stage;
        for (int bx = 0; bx < 2 * P.nvh; ++bx) tma_load_3d(dst + bx * 4096, &maps.v, fb, 64 * bx, y, wb.b);
        ++issued_v;
        vr.next(kNV);
        return true;
      };
      for (int n = 0; n < count && ok; ++n) {
        for (int s = 0; s < 2 && ok; ++s) {   // the block's two latent tiles
          const int sk = kr.slot;
          if (!(ok = mbar_wait(bar(misc->kempty[sk]), kr.phase ^ 1u, abort, a.status))) break;
          const uint32_t fb = bar(misc->kfull[sk]);
          mbar_arrive_expect_tx(fb, P.nkc * 16384);
          const int y = w.kb * kBlock2dTokens + static_cast<int>(rank) * 256 + kTile * s;
          for (int c = 0; c < P.nkc; ++c)
            tma_load_3d(sbase + P.k_ring + sk * P.k_stage + c * 16384, &maps.k, fb, 64 * c, y, w.b);
          ++issued_k;
          kr.next(kNK);
        }
        int vc = 0;
        for (int h = 0; h < a.H && ok; ++h) {
          const int sz = zr.slot;
          if (!(ok = mbar_wait(bar(misc->zempty[sz]), zr.phase ^ 1u, abort, a.status))) break;
          if (!images_ready) {
            asm volatile("griddepcontrol.wait;" ::: "memory");   // images written
            images_ready = true;
          }
          const uint32_t fb = bar(misc->zfull[sz]);
          mbar_arrive_expect_tx(fb, P.nkc * 8192 + 2048);
          const uint8_t* img = a.zimg + static_cast<int64_t>(w.b) * a.zimg_stride;
          const uint32_t dst = sbase + P.z_ring + sz * P.z_stage;
          const int64_t row0 = static_cast<int64_t>(h) * kHeadDim + 64 * rank;
          for (int c = 0; c < P.nkc; ++c)
            bulk_load(dst + c * 8192, img + c * a.zchunk_bytes + row0 * kZRowBytes, 8192, fb);
          bulk_load(dst + P.nkc * 8192, img + P.nkc * a.zchunk_bytes + row0 * 32, 2048, fb);
          ++issued_z;
          zr.next(kNZ);
          if (n > 0)
            while (ok && vc < kVChunks && vchunk_head(vc, a.H) == h) ok = load_v(wp, vc++);
        }
        wp = w;
        walk_advance(w, a);
      }
      for (int c = 0; ok && c < kVChunks; ++c) ok = load_v(wp, c);   // the last block's values
      // every copy this CTA issued lands before the CTA can exit
      auto drain = [&](uint64_t* full, int n, int issued) {
        for (int i = max(0, issued - n); i < issued; ++i) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar(full[i % n]), (i / n) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
      };
      drain(misc->kfull, kNK, issued_k);
      drain(misc->zfull, kNZ, issued_z);
      drain(misc->vfull, kNV, issued_v);
    }
  } else if (warp == 1 && rank == 1) {
    // ======================================================== relay (odd CTA)
    // Forwards each completed load of this CTA to the even CTA's full barrier, in
    // the producer's order.
    if (lane == 0) {
      Walker2d w = start, wp = start;
      RingPos kr, zr, vr;
      bool ok = true;
      auto relay_v = [&](const Walker2d& wb, int c) -> bool {
        const int sv = vr.slot;
        if (!mbar_wait(bar(misc->vfull[sv]), vr.phase, abort, a.status)) return false;
        zero_v_tail(sv, wb.L - (wb.kb * kBlock2dTokens + 256 + kVTok * c));
        mbar_arrive_cluster(bar(misc->vfull[sv]), 0);
        vr.next(kNV);
        return true;
      };
      for (int n = 0; n < count && ok; ++n) {
        for (int s = 0; s < 2 && ok; ++s) {
          if (!(ok = mbar_wait(bar(misc->kfull[kr.slot]), kr.phase, abort, a.status))) break;
          mbar_arrive_cluster(bar(misc->kfull[kr.slot]), 0);
          kr.next(kNK);
        }
        int vc = 0;
        for (int h = 0; h < a.H && ok; ++h) {
          if (!(ok = mbar_wait(bar(misc->zfull[zr.slot]), zr.phase, abort, a.status))) break;
          mbar_arrive_cluster(bar(misc->zfull[zr.slot]), 0);
          zr.next(kNZ);
          if (n > 0)
            while (ok && vc < kVChunks && vchunk_head(vc, a.H) == h) ok = relay_v(wp, vc++);
        }
        wp = w;
        walk_advance(w, a);
      }
      for (int c = 0; ok && c < kVChunks; ++c) ok = relay_v(wp, c);
    }
  } else if (warp == 1) {
    // ======================================================== pair MMA issuer (even CTA)
    // One thread issues every MMA of the pair.  Ring positions follow from global
    // counters (block n, head h): tiles 2n, 2n + 1, window nH + h, stage 2Hn + 2h + s.
    // The loop is kept lean (the issuing thread shares its sub-partition with two
    // epilogue warps): base descriptors per ring, K steps unrolled with constant offsets.
    if (lane == 0) {
      const uint32_t idesc_u = umma_idesc_bf16(256, 128, false, false);
      const uint32_t idesc_v = umma_idesc_bf16(256, 32, true, false);
      const int ksteps = a.r_k / 16;
      const uint64_t dA0 = umma_desc(sbase + P.k_ring, 16, 1024, kSw128);
      const uint64_t dZ0 = umma_desc(sbase + P.z_ring, 16, 1024, kSw128);
      const uint64_t dZb0 = umma_desc(sbase + P.z_ring + P.nkc * 8192, 16, 256, kSw32);
      const uint64_t daug = umma_desc(sbase + P.aug_a, 16, 256, kSw32);
      // MN-major value operand: 64-row r_v boxes 4 KB apart (LBO), 8 token rows 1 KB apart (SBO)
      const uint64_t dV0 = umma_desc(sbase + P.v_ring, 4096, 1024, kSw128);
      const uint64_t dP0 = umma_desc(sbase + P.p, 16, 256, kSw32);
      const uint32_t kst = static_cast<uint32_t>(P.k_stage) >> 4, zst = static_cast<uint32_t>(P.z_stage) >> 4,
                     vst = static_cast<uint32_t>(P.v_stage) >> 4;
      const uint32_t H = static_cast<uint32_t>(a.H);
      Walker2d w = start, wp = start;
      RingPos vr;
      bool ok = true, prev_run_start = true;
      // Value MMAs of chunk c of block `pblk` (walker wb): D_v[half] += C_v^T P over
      // the chunk's 16 tokens of each CTA; chunks wholly past the sequence end
      // (in both CTAs: the odd CTA's tokens come later) are skipped.
      auto issue_v = [&](const Walker2d& wb, bool run_start, int c, int pblk) -> bool {
        if (c == 0 && !mbar_wait_cluster(bar(misc->pfull), pblk & 1, abort, a.status)) return false;
        const int sv = vr.slot;
        if (!mbar_wait_cluster(bar(misc->vfull[sv]), vr.phase, abort, a.status)) return false;
        const int valid = wb.L - (wb.kb * kBlock2dTokens + kVTok * c);
        if (valid > 0) {
          zero_v_tail(sv, valid);
          tc_fence_after();
          const uint64_t av = dV0 + sv * vst, bp = dP0 + 2 * c * (512 >> 4);
#pragma unroll
          for (int k = 0; k < 2; ++k) {   // 16-token K steps: +2 KB in the chunk, +512 B in P
            if (16 * k >= valid) break;   // (wholly past the end in both CTAs)
            const uint32_t acc = (c > 0 || k > 0 || !run_start) ? 1u : 0u;
            umma_bf16_pair(tmem + kDvCol, av + k * (2048 >> 4), bp + k * (512 >> 4), idesc_v, acc);
            if (P.nvh > 1)
              umma_bf16_pair(tmem + kDvCol + 32, av + (8192 >> 4) + k * (2048 >> 4), bp + k * (512 >> 4), idesc_v,
                             acc);
          }
        }
        umma_commit_pair(bar(misc->vempty[sv]));
        if (c == kVChunks - 1) umma_commit_pair(bar(misc->vdone));
        vr.next(kNV);
        return true;
      };
      for (uint32_t n = 0; n < static_cast<uint32_t>(count) && ok; ++n) {
        const bool run_start = n == 0 || w.kb == 0;
        uint32_t ts[2];
        for (int s = 0; s < 2 && ok; ++s) {
          const uint32_t tile = 2 * n + s;
          ts[s] = tile % kNK;
          ok = mbar_wait_cluster(bar(misc->kfull[ts[s]]), (tile / kNK) & 1u, abort, a.status);
        }
        int vc = 0;
        for (uint32_t h = 0; h < H && ok; ++h) {
          const uint32_t zi = n * H + h, zs = zi & (kNZ - 1);
          if (!(ok = mbar_wait_cluster(bar(misc->zfull[zs]), (zi / kNZ) & 1u, abort, a.status))) break;
          const uint64_t b0 = dZ0 + zs * zst, bb = dZb0 + zs * zst;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint32_t G = 2 * H * n + 2 * h + s, su = G % kNU;
            if (!(ok = mbar_spin_cluster(bar(misc->uempty[su]), ((G / kNU) & 1u) ^ 1u, abort, a.status))) break;
            tc_fence_after();
            const uint64_t a0 = dA0 + ts[s] * kst;
            const uint32_t d = tmem + 128 * su;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              // 64-wide K chunks: A chunks 16 KB apart, Z chunks 8 KB apart; 32 B per K step
              if (k < ksteps)
                umma_bf16_pair(d, a0 + (k >> 2) * (16384 >> 4) + (k & 3) * 2,
                               b0 + (k >> 2) * (8192 >> 4) + (k & 3) * 2, idesc_u, k > 0 ? 1u : 0u);
            }
            umma_bf16_pair(d, daug, bb, idesc_u, 1u);   // + bias
            umma_commit_pair(bar(misc->ufull[s][su]));
          }
          if (!ok) break;
          if (n > 0)
            while (ok && vc < kVChunks && vchunk_head(vc, a.H) == static_cast<int>(h))
              ok = issue_v(wp, prev_run_start, vc++, n - 1);
        }
        prev_run_start = run_start;
        wp = w;
        walk_advance(w, a);
      }
      for (int c = 0; ok && c < kVChunks; ++c) ok = issue_v(wp, prev_run_start, c, count - 1);
      // this thread's MMAs complete before TMEM is released
      umma_commit_pair(bar(misc->mma_done[0]));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->mma_done[0]), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2 && warp < 10) {
    // ======================================================== epilogue (warps 2-9)
    // Warps 2-5 serve tile slot 0, warps 6-9 tile slot 1; one token per thread.
    const int we = warp - 2, wg = we >> 2, q = warp & 3;
    const int row = 32 * q + lane, tid_e = wg * kTile + row;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    uint8_t* pbuf = sm + P.p;
    const int H = a.H;

    // cos/sin(j th_f) of this thread's token j as f16 pairs: cs2[i] = (f = 2i, 2i + 1),
    // cos for i < 32, sin for i >= 32 (the f16 rounding error, 2^-12, is below the
    // bf16 query operand's)
    uint32_t cs2[64];
    auto load_trig = [&](const Walker2d& wb) {
      int64_t j = static_cast<int64_t>(wb.kb) * kBlock2dTokens + rank * 256 + wg * kTile + row;
      if (j >= a.trig_rows) j = a.trig_rows - 1;   // past the sequence end: masked anyway
      const uint4* t4 = reinterpret_cast<const uint4*>(a.trig16 + j * 64);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 v = __ldg(t4 + i);
        cs2[4 * i] = v.x; cs2[4 * i + 1] = v.y; cs2[4 * i + 2] = v.z; cs2[4 * i + 3] = v.w;
      }
    };
    auto epi_sync = []() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    auto arrive_even = [&](uint32_t b) {
      if (rank == 0) mbar_arrive(b); else mbar_arrive_cluster(b, 0);
    };
    // score-buffer release: this thread's TMEM reads completed (tcgen05.wait::ld) and
    // were fenced before the arrive, so the peer's later MMA into the buffer cannot
    // overtake them; nothing else needs to be made visible, so no cluster release
    auto release_u = [&](uint32_t b) {
      if (rank == 0) {
        mbar_arrive(b);
      } else {
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(map_to_rank(b, 0))
                     : "memory");
      }
    };
    // Each thread keeps its token's running sum of the weights of every head (lt);
    // the sums of the 256 tokens are reduced only when a run's record is written.
    float lt[kMax2dHeads];
#pragma unroll
    for (int h = 0; h < kMax2dHeads; ++h) lt[h] = 0.f;
    // One record per (run, head): m, l and this CTA's share of acc_v (the half of
    // r_v this warp group reads).  Called by all 256 epilogue threads (it syncs).
    auto write_record = [&](int b, bool live) {
      const int64_t rec = 2LL * (b + pair) + rank;
      if (live && wg < P.nvh) {
        float v[16];
        tmem_ld_x16(tmem + lane_base + kDvCol + 32 * wg + 16 * rank, v);
        tmem_wait_ld();
        const int r = kTile * wg + row;
        if (r < a.r_v) {
#pragma unroll
          for (int h = 0; h < kMax2dHeads; ++h)
            if (h < H) a.rec_acc[(rec * H + h) * a.r_v + r] = v[h];
        }
      }
#pragma unroll
      for (int h = 0; h < kMax2dHeads; ++h) {
        if (h < H) {
          const float ls = warp_sum(lt[h]);
          if (lane == 0) misc->lp[we][h] = ls;
        }
      }
      epi_sync();
      if (live && tid_e < H) {
        float l = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) l += misc->lp[ww][tid_e];
        a.rec_ml[(rec * H + tid_e) * 2] = misc->m_rec[tid_e];
        a.rec_ml[(rec * H + tid_e) * 2 + 1] = l;
      }
    };

    Walker2d w = start;
    int prev_b = start.b;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the f16 RoPE rows are written
    load_trig(w);
    bool ok = true;
    uint32_t uph = 0;   // this group's phase bit of each score buffer's ufull
    for (int n = 0; n < count; ++n) {
      const bool run_start = n == 0 || w.kb == 0;
      {
        const int jtok = w.kb * kBlock2dTokens + static_cast<int>(rank) * 256 + wg * kTile + row;
        const bool valid = jtok < w.L;
        // this warp group's stages of the block: st = 2 h + wg; score buffer (2 H n + st) mod 3
        const uint32_t gbase = static_cast<uint32_t>(2 * H) * n;
#pragma unroll 1
        for (int h = 0; h < H; ++h) {
          const uint32_t G = gbase + 2 * h + wg;
          const uint32_t uslot = G % kNU;
          if (ok) ok = warp_wait(bar(misc->ufull[wg][uslot]), (uph >> uslot) & 1u, abort, a.status);
          uph ^= 1u << uslot;
          float s = -INFINITY;
          if (ok) {
            tc_fence_after();
            const uint32_t tU = tmem + lane_base + 128 * uslot;
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {   // 64 columns per round, two loads in flight
              float u0[32], u1[32];
              tmem_ld_x32(tU + 64 * hf, u0);
              tmem_ld_x32(tU + 64 * hf + 32, u1);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 t0 = __half22float2(*reinterpret_cast<const __half2*>(&cs2[32 * hf + i]));
                const float2 t1 = __half22float2(*reinterpret_cast<const __half2*>(&cs2[32 * hf + 16 + i]));
                acc0 = fmaf(u0[2 * i], t0.x, acc0);
                acc1 = fmaf(u0[2 * i + 1], t0.y, acc1);
                acc0 = fmaf(u1[2 * i], t1.x, acc0);
                acc1 = fmaf(u1[2 * i + 1], t1.y, acc1);
              }
            }
            if (valid) s = acc0 + acc1;
            tc_fence_before();
          }
          tmem_st_x1(tmem + lane_base + kScoreCol + 16 * wg + h, __float_as_uint(s));
          const float wm = warp_max_redux(s);   // this warp's maximum of head h over its 32 tokens
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            release_u(bar(misc->uempty[uslot]));
            misc->mx[we][h] = wm;
            // the MMAs of this stage are complete: window h is free after group 1's
            // stage, the block's tile of this group after its last stage
            if (wg == 1) mbar_arrive(bar(misc->zempty[(static_cast<uint32_t>(H) * n + h) & (kNZ - 1)]));
            if (h == H - 1) mbar_arrive(bar(misc->kempty[(2u * n + wg) % kNK]));
          }
        }
      }
      Walker2d wn = w;
      walk_advance(wn, a);
      // this thread's token rows are no longer needed: fetch the next block's now
      if (n + 1 < count) load_trig(wn);

      // ---- end of block: exact per-head maximum over the CTA's 256 tokens sets the
      // reference (raised lazily: only when the block maximum exceeds it by 2^8)
      epi_sync();
      if (tid_e < H) {
        const int h = tid_e;
        float mb = misc->mx[0][h];
#pragma unroll
        for (int ww = 1; ww < 8; ++ww) mb = fmaxf(mb, misc->mx[ww][h]);
        const float mo = misc->m_ref[h];
        const float base = run_start ? -INFINITY : mo;
        const float mn = mb > base + kRescaleLog2 ? mb : base;
        misc->m_new[h] = mn;
        misc->alpha[h] = (run_start || mn == base) ? 1.f : exp2f(base - mn);
        if (run_start) misc->m_rec[h] = mo;   // the finished run's reference
        misc->m_ref[h] = mn;
      }
      epi_sync();
      // the previous block's value MMAs are complete: D_v and P may be touched
      if (n > 0) {
        if (ok) ok = warp_wait(bar(misc->vdone), (n - 1) & 1, abort, a.status);
        tc_fence_after();
      }
      // a run ended with the previous block: its record, before D_v is reused
      if (n > 0 && run_start) write_record(prev_b, ok);
      bool rescale = false;
      float sc[16];   // this token's scores of the block, one per head
      tmem_ld_x16(tmem + lane_base + kScoreCol + 16 * wg, sc);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < kMax2dHeads; ++h) {
        if (h < H) {
          const float mn = misc->m_new[h], al = misc->alpha[h];
          if (al != 1.f) rescale = true;
          const float p = mn == -INFINITY ? 0.f : exp2f(sc[h] - mn);
          const __nv_bfloat16 pb = __float2bfloat16_rn(p);
          *reinterpret_cast<__nv_bfloat16*>(pbuf + (tid_e >> 4) * 512 +
                                            swizzle_offset(h * 32 + (tid_e & 15) * 2, 32)) = pb;
          lt[h] = (run_start ? 0.f : lt[h] * al) + __bfloat162float(pb);
        }
      }
      // the reference of some head rose: rescale this CTA's accumulators (columns = heads)
      if (rescale && ok && wg < P.nvh) {
        const uint32_t dcol = tmem + lane_base + kDvCol + 32 * wg + 16 * rank;
        float v[16];
        tmem_ld_x16(dcol, v);
        tmem_wait_ld();
        uint32_t o[16];
#pragma unroll
        for (int h = 0; h < kMax2dHeads; ++h) o[h] = __float_as_uint(h < H ? v[h] * misc->alpha[h] : v[h]);
        tmem_st_x16(dcol, o);
        tmem_wait_st();
      }
      fence_proxy_async_smem();   // P visible to the value MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_even(bar(misc->pfull));
      prev_b = w.b;
      w = wn;
    }
    // the last run: its record once the last value MMAs are complete
    if (tid_e < H) misc->m_rec[tid_e] = misc->m_ref[tid_e];
    if (ok) {
      ok = warp_wait(bar(misc->vdone), (count - 1) & 1, abort, a.status);
      tc_fence_after();
    }
    write_record(prev_b, ok);
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

// Merge the run records of each (sequence, head) by log-sum-exp, apply the V
// up-projection once (Appendix J identity) and normalise:
//   out = (sum_c 2^(m_c - M) acc_c) W_up,v,t,h^T / (sum_c 2^(m_c - M) l_c) + mu_v,t,h.
// A sequence's records come from the pairs whose block ranges overlap it (both
// CTAs of each).  Block = (head h, two consecutive sequences); W_up,v,t,h is
// staged in shared memory (rows padded by one word) before the wait for the
// decode grid.
constexpr int kCombineUnits = 2;
constexpr int kCombineThreads = 128;

size_t combine_smem_bytes(int r_v) {
  return (static_cast<size_t>(128) * (r_v / 2 + 1) + kCombineUnits * 256 + 2 * kCombineUnits) * 4;
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
  int before = 0, all = 0;   // blocks of sequences [0, b0) and [0, B)
  for (int bb = tid; bb < a.B; bb += kCombineThreads) {
    const int n = nblocks(clamp_len(__ldg(a.seq_lens + bb), a.L_max));
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

  asm volatile("griddepcontrol.wait;" ::: "memory");   // records written

  float M = -INFINITY, Lt = 0.f;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  const int b = b0 + warp;
  if (warp < kCombineUnits && b < a.B) {
    long long B0 = pre;
    for (int bb = b0; bb < b; ++bb) B0 += nblocks(clamp_len(__ldg(a.seq_lens + bb), a.L_max));
    const int nb = nblocks(clamp_len(__ldg(a.seq_lens + b), a.L_max));
    if (nb > 0) {
      const long long NB = tot, NP = a.pairs;
      const long long p0 = ((B0 + 1) * NP - 1) / NB, p1 = ((B0 + nb) * NP - 1) / NB;
      for (long long p = p0; p <= p1; ++p) {
        const long long lo = p * NB / NP, hi = (p + 1) * NB / NP;
        if (max(lo, B0) >= min(hi, B0 + nb)) continue;   // the pair saw no block of b
        for (int r = 0; r < 2; ++r) {
          const long long rec = 2 * (b + p) + r;
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
    }
  }
  if (warp < kCombineUnits) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < a.r_v) accs[warp * 256 + lane + 32 * j] = acc[j];
    if (lane == 0) { Ms[warp] = M; Ls[warp] = Lt; }
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
  if (H < 4 || H > kMax2dHeads || H % 4 || r_k < 16 || r_k > 128 || r_v < 16 || r_v > 256 || r_k % 16 ||
      r_v % 16)
    return false;
  p->nkc = (r_k + 63) / 64;
  p->nvh = (r_v + 127) / 128;
  p->k_stage = p->nkc * 16384;
  p->z_stage = p->nkc * 8192 + 2048;   // half window rows, then their 16-wide bias operand
  p->v_stage = p->nvh * 8192;   // 32 tokens x (128 r_v) x 2 B per half
  int off = 0;
  p->k_ring = off; off += kNK * p->k_stage;
  p->z_ring = off; off += kNZ * p->z_stage;
  p->v_ring = off; off += kNV * p->v_stage;
  p->p = off;      off += 16 * 512;   // P: 16-token K chunks of 16 head rows
  p->aug_a = off;  off += 4096;
  p->misc = off;   off += 4096;
  p->bytes = off + 1024;
  return p->bytes <= kSmemLimit;
}

size_t decode2d_zimg_stride(int H, int r_k) {
  const size_t nkc = (r_k + 63) / 64;
  const size_t b = nkc * H * kHeadDim * kZRowBytes + static_cast<size_t>(H) * kHeadDim * 32;
  return (b + 1023) / 1024 * 1024;
}

int64_t decode2d_trig_rows(int64_t L_max, int64_t rope_len) {
  // positions a block can touch: up to L_max rounded up to a whole block
  const int64_t need = (L_max + kBlock2dTokens - 1) / kBlock2dTokens * kBlock2dTokens;
  return need < rope_len ? need : rope_len;
}

cudaError_t launch_decode2d_bf16(Decode2dArgs& a, const Decode2dMaps& maps, cudaStream_t s) {
  static int configured = 0;
  if (configured < a.plan.bytes) {
    cudaError_t e = cudaFuncSetAttribute(decode2d_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         a.plan.bytes);
    if (e != cudaSuccess) return e;
    configured = a.plan.bytes;
  }
  // pairs that can be resident at once (each CTA needs a whole SM)
  static int pairs_for = -1, max_pairs = 0;
  if (pairs_for != a.plan.bytes) {
    cudaLaunchConfig_t occ = {};
    occ.gridDim = dim3(2);
    occ.blockDim = dim3(kDecode2dThreads);
    occ.dynamicSmemBytes = a.plan.bytes;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, decode2d_bf16_kernel, &occ);
    if (e != cudaSuccess) return e;
    max_pairs = n;
    pairs_for = a.plan.bytes;
  }
  if (max_pairs < 1) return cudaErrorLaunchOutOfResources;
  a.pairs = std::min(a.pairs, std::min(max_pairs, kMaxPairs));
  if (a.pairs < 1) a.pairs = 1;

  const int trig_blocks = static_cast<int>((a.trig_rows + kTrigRowsPerBlock - 1) / kTrigRowsPerBlock);
  decode2d_z_kernel<<<a.B * a.H + trig_blocks, kZThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.pairs);
  cfg.blockDim = dim3(kDecode2dThreads);
  cfg.dynamicSmemBytes = a.plan.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode2d_bf16_kernel, a, maps);
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
