// lla_decode_small.cu — per-head latent decode attention of Looped Latent
// Attention at small latent ranks (r_k in {16, 32}, r_v in {32, 64}) on sm_103a
// ("Looped Latent Attention: Cross-Loop KV Compression for Looped Transformers",
// arXiv 2607.15456v2: §3 Eq. (2)-(3), "RoPE and reconstruction", §7 latent-store
// path, Appendix J "Absorbed attention").
//
// At small ranks a token carries few latent bytes (96 B per head at (16, 32)), so
// the per-token arithmetic has to shrink with them.  The rotary score
//   s_j = sum_f cos(j th_f) U_f + sin(j th_f) U_{64+f},   U = c_j Z^T + bias
// (Z folds the RoPE-rotated query into W_up,k,t, as in the per-head kernel) is
// regrouped as
//   s_j = sum_n c_j,n G_j,n + G_j,bias,    G_j = R_j [Z | bias],
// R_j = (cos(j th_0..63), sin(j th_0..63)), a row that depends on the position
// only.  G of a 128-token tile is one MMA chain per head set (nwg heads):
//   A = the tile's RoPE rows (f16, 128 x 128) in TMEM, written once per position
//       and shared by every head there,
//   B = the set's query image: each head's Z rows (r_k) and its bias rows (hi,
//       lo), N = nwg (r_k + 2) rounded up to 16 rows of 128 RoPE coordinates (f16,
//       K-major), resident in shared memory for the whole sequence,
//   D = G of the set's heads in TMEM (fp32).
// An M = 128, K = 16 MMA costs about the same for any N up to 128, so heads share
// one wide MMA rather than taking a narrow one each.  The latents never enter the
// tensor core: each epilogue thread takes an r_k-long dot product of its token's
// c_k row (shared memory) with its G row, and each warp forms sum_j p_j c_v,j over
// its 32 tokens with row-crossing 8-byte loads and a shuffle reduction.  K and V
// reconstructions never exist anywhere.
//
// Work: positions (sequence, 128-token tile) in contiguous ranges, one range per
// CTA, every head of a position inside it (heads inner).  Warps: 0 producer
// (bulk copies), 1 MMA issuer, 2-17 four epilogue groups of four warps (group g
// takes head g of every set; two groups when H mod 4 = 2), one token per epilogue
// thread.  Per (warp, head) the epilogue keeps a lazily raised reference max, the
// weight sum and sum_j p_j c_v,j in shared memory and writes them as a record
// when its run of the sequence ends; the combine kernel merges a unit's records
// and applies W_up,v,t once (Appendix J).
//
#include "lla_kernels.h"

#include <algorithm>
#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr float kRescaleLog2 = 8.f;                 // lazy rescale threshold (log2 units)
constexpr float kF16Max = 65504.f;
constexpr int kTrigCol = 0;                         // TMEM: 2 RoPE-row buffers of 64 columns
constexpr int kGCol = 128;                          // TMEM: G buffers from here
constexpr int kGCols = 512 - kGCol;
constexpr int kTrigRowsPerBlock = 64;
constexpr int kMaxG = 8;                            // G buffers at most
constexpr int kSmallMiscBytes = 4096;

struct alignas(16) SmallMisc {
  uint64_t full[kSmallMaxNS], empty[kSmallMaxNS];   // ring slots (K tile + V tile)
  uint64_t img_full[kSmallMaxHeads], img_empty[kSmallMaxHeads];   // per head set
  uint64_t trig_full[2];                            // RoPE-row buffers (position parity)
  uint64_t gfull[kMaxG], gempty[kMaxG];             // G buffers (one head set each)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int start_b, start_t, count;                      // first position of the range, positions
  int total_pos;
  int scan[kSmallThreads];
};
static_assert(sizeof(SmallMisc) <= kSmallMiscBytes, "misc region");

// Walk over positions (sequence b, tile t) in order, skipping empty sequences.
struct PosWalker {
  int b, t, nb, L;
};

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

__device__ __forceinline__ void pos_advance(PosWalker& w, const DecodeArgs& a) {
  if (++w.t < w.nb) return;
  w.t = 0;
  while (true) {
    ++w.b;
    if (w.b >= a.B) { w.nb = 0; return; }
    w.L = clamp_len(__ldg(a.seq_lens + w.b), a.L_max);
    w.nb = (w.L + kTile - 1) / kTile;
    if (w.nb > 0) return;
  }
}

// Ring position advanced by `step` (< n) slots at a time.
struct SlotPos {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void next(int step, int n) {
    slot += step;
    if (slot >= n) { slot -= n; phase ^= 1u; }
  }
};

__device__ __forceinline__ uint32_t half2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

// Query images of the small-rank kernel, one per (sequence, head set), written as
// the exact shared-memory image the decode kernel copies in: B operand rows of 128
// RoPE coordinates k (f16), two K chunks of 64 coordinates, each N rows x 128 B in
// the 128-byte swizzle.  Head hl of the set owns rows hl r_k + n (n < r_k) and the
// bias rows nwg r_k + 2 hl (the bias rounded to f16) and + 1 (its rounding
// remainder); rows from nwg (r_k + 2) up to N are zero.  With q' = RoPE(q, q_pos),
// sc = log2(e) / sqrt(d) and the frequency pair (i0, i1) of f < 64:
//   Z row n:  k = f      -> sc (q'_i0 W_i0,n + q'_i1 W_i1,n)
//             k = 64 + f -> sc (q'_i1 W_i0,n - q'_i0 W_i1,n)
//   bias:     k = f      -> sc (q'_i0 mu_i0 + q'_i1 mu_i1)
//             k = 64 + f -> sc (q'_i1 mu_i0 - q'_i0 mu_i1)
// so that sum_n c_j,n (R_j . Z row n) + R_j . (bias rows) equals
// log2(e) RoPE(q, q_pos).RoPE(k_j, j) / sqrt(d) for the key of Eq. (3).  A value
// beyond the f16 range records LLA_ERR_RANGE.  Block = (head h, kZSeqs sequences):
// W_up,k,t[h] is staged once and serves every sequence of the block, and the
// rotated queries of all of them are formed in one round of loads.  The first
// blocks write the f16 RoPE rows: row p = {cos(p th_2i), cos(p th_2i+1)} for
// i < 32, then the sines, two per 32-bit word (lower frequency in the low half).
constexpr int kSZThreads = 256;
constexpr int kZSeqs = 8;
__global__ void __launch_bounds__(kSZThreads) decode_small_z_kernel(const __grid_constant__ DecodeArgs a) {
  // launched as a programmatic dependent of whatever precedes the call on the
  // stream: nothing is read before that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the decode grid may start its set-up now; it waits for this grid before it
  // copies an image or reads a RoPE row
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ __align__(16) float qs[kZSeqs][2][64];  // sc q'_i0, sc q'_i1 per sequence and frequency
  __shared__ __align__(16) float bs[kZSeqs][128];    // bias per sequence and RoPE coordinate
  __shared__ float Ws[kHeadDim * 33];  // W_up,k,t[h] as fp32 [128][r_k] (row stride r_k + 1)
  __shared__ bool live[kZSeqs];        // sequence exists and is not empty
  const int ntb = static_cast<int>((a.trig_rows + kTrigRowsPerBlock - 1) / kTrigRowsPerBlock);
  const int tid = threadIdx.x;
  if (static_cast<int>(blockIdx.x) < ntb) {
    // RoPE rows first (the decode grid needs all of them): every load in flight at once
    constexpr int kPer = kTrigRowsPerBlock * 64 / kSZThreads;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTrigRowsPerBlock;
    float2 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kSZThreads, c = i % 64;
      const int64_t r = min(r0 + i / 64, a.trig_rows - 1);
      v[j] = *reinterpret_cast<const float2*>((c < 32 ? a.rope_cos : a.rope_sin) + r * 64 + 2 * (c & 31));
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kSZThreads;
      const int64_t r = r0 + i / 64;
      if (r < a.trig_rows) a.trig16[r * 64 + i % 64] = half2_bits(__floats2half2_rn(v[j].x, v[j].y));
    }
    return;
  }
  const int u = static_cast<int>(blockIdx.x) - ntb;
  const int h = u % a.H, b0 = (u / a.H) * kZSeqs;
  if (h == 0)
    for (int sb = 0; sb < kZSeqs && b0 + sb < a.B; ++sb) check_block_table(a, b0 + sb, tid, kSZThreads);
  const int rk = a.r_k, ws = rk + 1;
  const int nwg = a.splan.nwg, N = a.splan.N, hl = h % nwg;
  const __nv_bfloat16* W =
      static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * rk;
  for (int i = tid; i < kHeadDim * rk / 8; i += kSZThreads) {
    float w8[8];
    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(W) + i), w8);
    const int row = (8 * i) / rk, col = (8 * i) % rk;
#pragma unroll
    for (int e = 0; e < 8; ++e) Ws[row * ws + col + e] = w8[e];
  }
  const float* mu = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
  for (int i = tid; i < kZSeqs * 64; i += kSZThreads) {
    const int sb = i / 64, f = i % 64, b = b0 + sb;
    if (b >= a.B) break;
    int qp = __ldg(a.q_pos + b);
    if (qp < 0 || qp >= a.rope_len) {
      if (f == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
      qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
    }
    const int i0 = a.rope_style == 0 ? f : 2 * f;
    const int i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
    const __nv_bfloat16* qv =
        static_cast<const __nv_bfloat16*>(a.q) + (static_cast<int64_t>(b) * a.H + h) * kHeadDim;
    const float cq = __ldg(a.rope_cos + static_cast<int64_t>(qp) * 64 + f);
    const float sq = __ldg(a.rope_sin + static_cast<int64_t>(qp) * 64 + f);
    const float x0 = __bfloat162float(qv[i0]), x1 = __bfloat162float(qv[i1]);
    const float m0 = __ldg(mu + i0), m1 = __ldg(mu + i1);
    const float scale = kLog2e * kInvSqrtD;
    const float q0 = (x0 * cq - x1 * sq) * scale;
    const float q1 = (x0 * sq + x1 * cq) * scale;
    qs[sb][0][f] = q0;
    qs[sb][1][f] = q1;
    bs[sb][f] = q0 * m0 + q1 * m1;
    bs[sb][64 + f] = q1 * m0 - q0 * m1;
  }
  if (tid < kZSeqs) live[tid] = b0 + tid < a.B && clamp_len(__ldg(a.seq_lens + b0 + tid), a.L_max) > 0;
  __syncthreads();
  // Item = (row r of this head, 16-byte granule g = coordinates 8g..8g+7): its W
  // values and destination are set up once and serve every sequence of the block.
  // Rows: Z (r_k), bias hi, bias lo; head 0 of the set also zeroes the padding.
  const int rows = rk + 2 + (hl == 0 ? N - nwg * (rk + 2) : 0);
  float amax = 0.f;   // largest |value| written (f16 range check)
  for (int it = tid; it < rows * 16; it += kSZThreads) {
    const int r = it >> 4, g = it & 15, f0 = 8 * (g & 7);
    const bool sin_half = g >= 8;
    float w0[8], w1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int f = f0 + e;
      const int i0 = a.rope_style == 0 ? f : 2 * f;
      const int i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
      w0[e] = r < rk ? Ws[i0 * ws + r] : 0.f;
      w1[e] = r < rk ? Ws[i1 * ws + r] : 0.f;
    }
    const int n = r < rk ? hl * rk + r : r < rk + 2 ? nwg * rk + 2 * hl + (r - rk) : nwg * (rk + 2) + (r - rk - 2);
    const uint32_t off = (g >> 3) * (N * 128) + swizzle_offset(n * 128 + (g & 7) * 16, 128);
    for (int sb = 0; sb < kZSeqs; ++sb) {
      if (!live[sb]) continue;   // past the batch or an empty sequence: never read
      float v[8];
      if (r < rk) {
        const float4* q0p = reinterpret_cast<const float4*>(&qs[sb][0][f0]);
        const float4* q1p = reinterpret_cast<const float4*>(&qs[sb][1][f0]);
        const float4 a0 = q0p[0], a1 = q0p[1], c0 = q1p[0], c1 = q1p[1];
        const float q0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float q1[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          v[e] = sin_half ? q1[e] * w0[e] - q0[e] * w1[e] : q0[e] * w0[e] + q1[e] * w1[e];
      } else if (r < rk + 2) {
        const float4* bp = reinterpret_cast<const float4*>(&bs[sb][8 * g]);
        const float4 u0 = bp[0], u1 = bp[1];
        const float bb[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float hi = __half2float(__float2half_rn(bb[e]));
          v[e] = r == rk ? hi : bb[e] - hi;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
      const uint4 w = make_uint4(half2_bits(__floats2half2_rn(v[0], v[1])), half2_bits(__floats2half2_rn(v[2], v[3])),
                                 half2_bits(__floats2half2_rn(v[4], v[5])), half2_bits(__floats2half2_rn(v[6], v[7])));
      *reinterpret_cast<uint4*>(a.zimg + (static_cast<int64_t>(b0 + sb) * a.splan.nsets + h / nwg) * a.zimg_stride +
                                off) = w;
    }
  }
  if (amax > kF16Max) record_status(a.status, LLA_ERR_RANGE);   // (NaN queries stay NaN, as on every path)
}

// kPage: 0 dense cache, 1 page pool with pages of a multiple of 128 tokens (a
// head-tile inside one page: one pair of copies), 2 page pool of any other page size
// (a head-tile's rows copied page by page, the copies spread over the producer warp),
// 3 page pool with pages of 8..64 tokens in the set-page layout: a ring slot holds
// one head set's tile, [K: page][head][row] then [V: page][head][row], filled with
// one pair of copies per page (the set's heads are contiguous in a page), so the
// copies are nwg times fewer and larger; every epilogue group reads every slot.
template <int RK, int RV, int kPage>
__global__ void __launch_bounds__(kSmallThreads, 1) decode_small_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int KB = RK * 2, VB = RV * 2; // bytes of a latent K / V row
  constexpr int LPR = RV / 4;             // value step: lanes per V row, 4 columns each
  constexpr int RPL = 32 / LPR;           // V rows per warp-wide load
  extern __shared__ uint8_t smem_raw[];
  // swizzle atoms need 1024-byte alignment in the shared window itself
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const DecodeSmallPlan& P = a.splan;
  const uint32_t sbase = smem_u32(sm);
  SmallMisc* misc = reinterpret_cast<SmallMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, nwg = P.nwg, nsets = P.nsets;

  // ---------------------------------------------------------- work range
  // positions (sequence, tile) in order; CTA c takes [c per, (c + 1) per)
  {
    const int per_thr = (a.B + kSmallThreads - 1) / kSmallThreads;
    const int b0 = min(a.B, tid * per_thr), b1 = min(a.B, b0 + per_thr);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      const int L0 = __ldg(a.seq_lens + b);
      if ((L0 < 0 || L0 > a.L_max) && blockIdx.x == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
      local += (clamp_len(L0, a.L_max) + kTile - 1) / kTile;
    }
    misc->scan[tid] = local;
    if (tid == 0) misc->abort = 0;
    __syncthreads();
    if (warp == 0) {
      constexpr int kPer = kSmallThreads / 32;
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
      if (lane == 31) misc->total_pos = incl;
    }
    __syncthreads();
    const long long total = misc->total_pos;
    const long long per = max(1LL, (total + a.grid - 1) / a.grid);
    const long long f0 = static_cast<long long>(blockIdx.x) * per;
    const long long f1 = min(total, f0 + per);
    long long P0 = misc->scan[tid];
    for (int b = b0; b < b1; ++b) {
      const int nb = (clamp_len(__ldg(a.seq_lens + b), a.L_max) + kTile - 1) / kTile;
      if (nb > 0 && f0 < f1 && P0 <= f0 && f0 < P0 + nb) {
        misc->start_b = b;
        misc->start_t = static_cast<int>(f0 - P0);
      }
      P0 += nb;
    }
    if (tid == 0) misc->count = static_cast<int>(f1 > f0 ? f1 - f0 : 0);
    __syncthreads();
  }
  const int count = misc->count;
  if (count == 0) return;

  PosWalker start;
  start.b = misc->start_b;
  start.t = misc->start_t;
  start.L = clamp_len(__ldg(a.seq_lens + start.b), a.L_max);
  start.nb = (start.L + kTile - 1) / kTile;

  // ---------------------------------------------------------- set-up
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    for (int s = 0; s < P.NS; ++s) {
      mbar_init(bar(misc->full[s]), 1);
      mbar_init(bar(misc->empty[s]), kPage == 3 ? 4 * nwg : 4);
    }
    for (int s = 0; s < nsets; ++s) { mbar_init(bar(misc->img_full[s]), 1); mbar_init(bar(misc->img_empty[s]), 1); }
    mbar_init(bar(misc->trig_full[0]), 4 * nwg);
    mbar_init(bar(misc->trig_full[1]), 4 * nwg);
    for (int g = 0; g < P.NG; ++g) { mbar_init(bar(misc->gfull[g]), 1); mbar_init(bar(misc->gempty[g]), 4 * nwg); }
    mbar_init(bar(misc->mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&misc->tmem_base), 512);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the combine grid may be scheduled now; it waits for this grid to complete
  // before it reads a record
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    // ======================================================== producer
    // Per run (the CTA's positions of one sequence): the head-set images, each
    // once the MMAs of the previous run's image in that buffer are done.  Per
    // head-tile: its K and V rows (contiguous in the cache) into the next ring slot
    // with two plain bulk copies of the rows below the sequence length.  With a
    // paged cache the whole warp runs the loop (lane 0 waits, the warp follows its
    // decision) and lane i issues the copies of the tile's i-th page.
    constexpr bool kWarp = kPage >= 2;
    auto pwait = [&](uint32_t b, uint32_t parity) -> bool {
      if constexpr (kWarp) return warp_wait(b, parity, abort, a.status);
      else return mbar_wait(b, parity, abort, a.status);
    };
    if (lane == 0 || kWarp) {
      PosWalker w = start;
      SlotPos sp{0, 0u};
      int run = 0, issued = 0, imgs = 0;
      bool ok = true;
      for (int lp = 0; lp < count && ok; ++lp) {
        const bool run_start = lp == 0 || w.t == 0;
        if (run_start) {
          imgs = 0;
          for (int s = 0; s < nsets && ok; ++s) {
            if (run > 0 && !(ok = pwait(bar(misc->img_empty[s]), (run - 1) & 1))) break;
            if (lp == 0 && s == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // images written
            if (!kWarp || lane == 0) {
              const uint32_t fb = bar(misc->img_full[s]);
              mbar_arrive_expect_tx(fb, P.img);
              bulk_load(sbase + P.imgs + s * P.img,
                        a.zimg + (static_cast<int64_t>(w.b) * nsets + s) * a.zimg_stride, P.img, fb);
            }
            imgs = s + 1;
          }
          ++run;
        }
        const uint32_t rows = static_cast<uint32_t>(min(kTile, w.L - w.t * kTile));
        // rows of head h: (z0 + h) * zrows + y0 (dense: z0 = b H; whole pages: the tile's page)
        int64_t z0 = static_cast<int64_t>(w.b) * H, zrows = a.L_max, y0 = static_cast<int64_t>(w.t) * kTile;
        if constexpr (kPage == 1) {
          const int lp = static_cast<int>(y0 / a.page_size);
          z0 = static_cast<int64_t>(page_of(a, w.b, lp)) * H;
          zrows = a.page_size;
          y0 -= static_cast<int64_t>(lp) * a.page_size;
        }
        if constexpr (kPage == 3) {
          // one slot per head set: lane i copies page lp0 + i of the tile for the
          // set's heads (K and V), every copy completing on the slot's barrier
          const int lg = P.log2P, pg = 1 << lg;
          const int np = (static_cast<int>(rows) + pg - 1) >> lg;
          const int64_t lp0 = y0 >> lg;
          const uint32_t kbytes = static_cast<uint32_t>(nwg * KB) << lg, vbytes = static_cast<uint32_t>(nwg * VB) << lg;
          for (int s = 0; s < nsets && ok; ++s) {
            if (!(ok = pwait(bar(misc->empty[sp.slot]), sp.phase ^ 1u))) break;
            const uint32_t fb = bar(misc->full[sp.slot]);
            const uint32_t dst = sbase + P.ring + sp.slot * P.slot;
            if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(np) * (kbytes + vbytes));
            __syncwarp();
            for (int i = lane; i < np; i += 32) {
              const int64_t r0 = (static_cast<int64_t>(page_of(a, w.b, static_cast<int>(lp0 + i))) * H + s * nwg) << lg;
              bulk_load(dst + i * kbytes, static_cast<const uint8_t*>(a.cache_k) + r0 * KB, kbytes, fb);
              bulk_load(dst + nwg * P.k_tile + i * vbytes, static_cast<const uint8_t*>(a.cache_v) + r0 * VB, vbytes, fb);
            }
            ++issued;
            sp.next(1, P.NS);
          }
        } else
        for (int h = 0; h < H && ok; ++h) {
          if (!(ok = pwait(bar(misc->empty[sp.slot]), sp.phase ^ 1u))) break;
          const uint32_t fb = bar(misc->full[sp.slot]);
          const uint32_t dst = sbase + P.ring + sp.slot * P.slot;
          if constexpr (kWarp) {
            // one pair of copies per page the tile's rows lie in (pages of any size, a
            // page boundary possibly inside the tile): lane i takes page lp0 + i
            if (lane == 0) mbar_arrive_expect_tx(fb, rows * (KB + VB));
            __syncwarp();
            const int64_t pg = a.page_size;
            const int64_t lp0 = y0 / pg, np = (y0 + rows - 1) / pg - lp0 + 1;
            for (int64_t i = lane; i < np; i += 32) {
              const int64_t t0 = max(y0, (lp0 + i) * pg), t1 = min(y0 + rows, (lp0 + i + 1) * pg);
              const uint32_t j = static_cast<uint32_t>(t0 - y0), span = static_cast<uint32_t>(t1 - t0);
              const int64_t r0 = (static_cast<int64_t>(page_of(a, w.b, static_cast<int>(lp0 + i))) * H + h) * pg +
                                 (t0 - (lp0 + i) * pg);
              bulk_load(dst + j * KB, static_cast<const uint8_t*>(a.cache_k) + r0 * KB, span * KB, fb);
              bulk_load(dst + P.k_tile + j * VB, static_cast<const uint8_t*>(a.cache_v) + r0 * VB, span * VB, fb);
            }
          } else {
            mbar_arrive_expect_tx(fb, rows * (KB + VB));
            const int64_t r0 = (z0 + h) * zrows + y0;
            bulk_load(dst, static_cast<const uint8_t*>(a.cache_k) + r0 * KB, rows * KB, fb);
            bulk_load(dst + P.k_tile, static_cast<const uint8_t*>(a.cache_v) + r0 * VB, rows * VB, fb);
          }
          ++issued;
          sp.next(1, P.NS);
        }
        pos_advance(w, a);
      }
      // Let every copy this CTA issued land before the CTA can exit.
      if (lane == 0) {
        for (int i = max(0, issued - P.NS); i < issued; ++i) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar(misc->full[i % P.NS]), (i / P.NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
        for (int s = 0; s < imgs; ++s) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar(misc->img_full[s]), (run - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
      }
    }
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // Per position and head set: G = R_tile [set image], A = the position's RoPE
    // rows in TMEM (K-major f16, 8 columns per 16 coordinates), B = the set image
    // (K-major, 128B swizzle, two chunks of 64 coordinates), D = the next G buffer.
    // The whole warp runs the loop (warp-uniform descriptors); one elected lane
    // issues, every lane polls the barriers and the vote keeps the decision uniform.
    {
      auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
      const uint32_t idesc = umma_idesc_f16(128, P.N);
      const uint32_t chunk = static_cast<uint32_t>(P.N) * 128;
      PosWalker w = start;
      SlotPos gp{0, 0u};
      int run = 0;
      bool ok = true;
      for (int lp = 0; lp < count && ok; ++lp) {
        const bool run_start = lp == 0 || w.t == 0;
        const bool run_end = lp == count - 1 || w.t == w.nb - 1;
        const uint32_t tb = lp & 1;
        if (!(ok = agree(mbar_wait(bar(misc->trig_full[tb]), (lp >> 1) & 1, abort, a.status)))) break;
        for (int s = 0; s < nsets; ++s) {
          if (run_start && !(ok = agree(mbar_wait(bar(misc->img_full[s]), run & 1, abort, a.status)))) break;
          if (!(ok = agree(mbar_wait(bar(misc->gempty[gp.slot]), gp.phase ^ 1u, abort, a.status)))) break;
          tc_fence_after();
          const uint32_t d = tmem + kGCol + gp.slot * P.N;
          const uint32_t at = tmem + kTrigCol + tb * 64;
          const uint32_t ib = sbase + P.imgs + s * P.img;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = umma_desc(ib + (kk >> 2) * chunk, 16, 1024, kSw128) + 2 * (kk & 3);
            umma_bf16_ts_warp(d, at + 8 * kk, bd, idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit_warp(bar(misc->gfull[gp.slot]));
          if (run_end) umma_commit_warp(bar(misc->img_empty[s]));   // the set image is no longer read
          gp.next(1, P.NG);
        }
        if (run_start) ++run;
        pos_advance(w, a);
      }
      // this warp's MMAs complete before TMEM is released
      umma_commit_warp(bar(misc->mma_done));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->mma_done), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if ((warp - 2) >> 2 < nwg) {
    // ======================================================== epilogue (warps 2-17)
    // Group wg (warps 2 + 4 wg .. 5 + 4 wg) takes head wg of every set (heads
    // h = j nwg + wg); thread (TMEM quadrant q, lane) owns token row 32 q + lane.
    const int we = warp - 2, wg = we >> 2, q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float* accs = reinterpret_cast<float*>(sm + P.acc) + static_cast<size_t>(we) * nsets * RV;   // [nsets][RV]
    float2* mls = reinterpret_cast<float2*>(sm + P.ml) + we * nsets;                            // [nsets] (m, l)
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the f16 RoPE rows are written

    // The RoPE rows are the MMA's A operand in TMEM (buffer = position & 1): each
    // group writes 16-column quarters (quarter wg, and wg + 2 with two groups) of
    // its threads' rows, one position ahead.
    uint32_t tq[16];
    auto trig_load = [&](const PosWalker& pw, int quarter) {
      int64_t j = static_cast<int64_t>(pw.t) * kTile + row;
      if (j >= a.trig_rows) j = a.trig_rows - 1;   // past the sequence end: masked anyway
      const uint4* t4 = reinterpret_cast<const uint4*>(a.trig16 + j * 64 + 16 * quarter);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(t4 + i);
        tq[4 * i] = v.x; tq[4 * i + 1] = v.y; tq[4 * i + 2] = v.z; tq[4 * i + 3] = v.w;
      }
    };
    auto trig_store = [&](int lpos, int quarter) {
      tmem_st_x16(tmem + lane_base + kTrigCol + (lpos & 1) * 64 + 16 * quarter, tq);
    };
    auto trig_done = [&](int lpos) {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(misc->trig_full[lpos & 1]));
    };
    auto trig_write = [&](const PosWalker& pw, int lpos) {
      for (int qq = wg; qq < 4; qq += nwg) {
        trig_load(pw, qq);
        trig_store(lpos, qq);
      }
      trig_done(lpos);
    };

    PosWalker w = start;
    trig_write(w, 0);
    if (count > 1) {
      PosWalker w1 = w;
      pos_advance(w1, a);
      trig_write(w1, 1);
    }

    // ring slot of this group's next head-tile (every nwg-th; with set slots every one)
    SlotPos sp{kPage == 3 ? 0 : wg, 0u};
    // set-page layout: byte offset of this head's K row `row` and of V row r in a slot
    const int lgP = kPage == 3 ? P.log2P : 0;
    const uint32_t krow3 = kPage == 3 ? static_cast<uint32_t>(((row >> lgP) * nwg * KB << lgP) +
                                                              ((wg << lgP) + (row & ((1 << lgP) - 1))) * KB)
                                      : 0u;
    auto vrow3 = [&](int r) -> uint32_t {
      return static_cast<uint32_t>(nwg * P.k_tile + ((r >> lgP) * nwg * VB << lgP) +
                                   ((wg << lgP) + (r & ((1 << lgP) - 1))) * VB);
    };
    SlotPos gp{0, 0u};    // G buffer of the next head set
    const uint32_t gz = kGCol + wg * RK, gbias = kGCol + nwg * RK + 2 * wg;   // this head's G columns
    bool ok = true;
    for (int lp = 0; lp < count && ok; ++lp) {
      const bool run_start = lp == 0 || w.t == 0;
      const bool run_end = lp == count - 1 || w.t == w.nb - 1;
      const int nvalid = min(kTile, w.L - w.t * kTile);
      const bool valid = row < nvalid;
      PosWalker wn = w;
      pos_advance(wn, a);
      const bool writer = lp >= 1 && lp + 1 < count;   // RoPE rows of position lp + 1
      for (int j = 0; j < nsets; ++j) {
        const int h = j * nwg + wg;
        if (writer && j == 0) trig_load(wn, wg);   // stored once this head-tile is done
        // ---- G row of this token from TMEM; the buffer is free again once every
        // group has read its head's columns
        if (!(ok = warp_wait(bar(misc->gfull[gp.slot]), gp.phase, abort, a.status))) break;
        tc_fence_after();
        float g[RK + 2];
        {
          const uint32_t gb = tmem + lane_base + gp.slot * P.N;
          if constexpr (RK == 16) {
            float g0[16];
            tmem_ld_x16(gb + gz, g0);
#pragma unroll
            for (int c = 0; c < 16; ++c) g[c] = g0[c];
          } else {
            float g0[32];
            tmem_ld_x32(gb + gz, g0);
#pragma unroll
            for (int c = 0; c < 32; ++c) g[c] = g0[c];
          }
          float g1[2];
          tmem_ld_x2(gb + gbias, g1);
          g[RK] = g1[0];
          g[RK + 1] = g1[1];
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->gempty[gp.slot]));
        gp.next(1, P.NG);

        // ---- the head-tile's K and V latents
        if (!(ok = warp_wait(bar(misc->full[sp.slot]), sp.phase, abort, a.status))) break;
        const uint8_t* kt = sm + P.ring + sp.slot * P.slot;
        uint8_t* vt = sm + P.ring + sp.slot * P.slot + P.k_tile;

        // ---- score s_j = c_j . G_j[0, r_k) + bias hi + bias lo (log2 units)
        float s0 = g[RK], s1 = g[RK + 1];
#pragma unroll
        for (int c = 0; c < RK / 8; ++c) {
          float x[8];
          if constexpr (kPage == 3)
            unpack_bf16x8(*reinterpret_cast<const uint4*>(kt + krow3 + 16 * c), x);
          else
            unpack_bf16x8(*reinterpret_cast<const uint4*>(kt + row * KB + 16 * c), x);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            s0 = fmaf(x[e], g[8 * c + e], s0);
            s1 = fmaf(x[e + 1], g[8 * c + e + 1], s1);
          }
        }
        const float s = valid ? s0 + s1 : -INFINITY;

        // ---- online softmax per warp, reference raised lazily (by more than 2^8)
        float2 ml = run_start ? make_float2(-INFINITY, 0.f) : mls[j];
        const float mt = warp_max_redux(s);
        float alpha = 1.f;
        if (mt > ml.x + kRescaleLog2) {
          alpha = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mt);
          ml.x = mt;
        }
        if (run_start) alpha = 0.f;
        const float p = valid ? exp2f(s - ml.x) : 0.f;

        // ---- rows past the sequence end hold stale data: zero them (own row)
        if (nvalid < kTile) {
          if (!valid) {
            uint8_t* vr = kPage == 3 ? const_cast<uint8_t*>(kt) + vrow3(row) : vt + row * VB;
#pragma unroll
            for (int c = 0; c < VB / 16; ++c) *reinterpret_cast<uint4*>(vr + 16 * c) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }

        // ---- sum_j p_j c_v,j over the warp's 32 tokens: lane = (row group, 4 columns)
        const int cg = lane % LPR, rg = lane / LPR;
        float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < LPR; ++i) {
          const int tk = RPL * i + rg;
          const float pv = __shfl_sync(0xffffffffu, p, tk);
          const uint2 v = kPage == 3 ? *reinterpret_cast<const uint2*>(kt + vrow3(32 * q + tk) + 8 * cg)
                                     : *reinterpret_cast<const uint2*>(vt + (32 * q + tk) * VB + 8 * cg);
          a4[0] = fmaf(pv, __uint_as_float(v.x << 16), a4[0]);
          a4[1] = fmaf(pv, __uint_as_float(v.x & 0xFFFF0000u), a4[1]);
          a4[2] = fmaf(pv, __uint_as_float(v.y << 16), a4[2]);
          a4[3] = fmaf(pv, __uint_as_float(v.y & 0xFFFF0000u), a4[3]);
        }
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
          for (int c = 0; c < 4; ++c) a4[c] += __shfl_xor_sync(0xffffffffu, a4[c], o);
        const float ps = warp_sum(p);
        // the slot's latents are consumed (the shuffles above used every load)
        if (nvalid < kTile) fence_proxy_async_smem();   // zeroed rows before the next bulk copy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->empty[sp.slot]));
        sp.next(kPage == 3 ? 1 : nwg, P.NS);

        // ---- fold into the warp's state; a run's last tile writes the record
        // (m, l, -, -, acc) of (sequence, head, CTA, warp)
        float* rec = a.partials +
                     ((static_cast<int64_t>(w.b + blockIdx.x) * H + h) * kRecordsPerCta + (we & 3)) *
                         (RV + kRecordHead);
        if (lane < LPR) {
          float4* ap = reinterpret_cast<float4*>(accs + j * RV) + cg;
          float4 o = run_start ? make_float4(0.f, 0.f, 0.f, 0.f) : *ap;
          o.x = fmaf(o.x, alpha, a4[0]);
          o.y = fmaf(o.y, alpha, a4[1]);
          o.z = fmaf(o.z, alpha, a4[2]);
          o.w = fmaf(o.w, alpha, a4[3]);
          *ap = o;
          if (run_end) *reinterpret_cast<float4*>(rec + kRecordHead + 4 * cg) = o;
        }
        ml.y = fmaf(ml.y, alpha, ps);
        if (lane == 0) {
          mls[j] = ml;
          if (run_end) { rec[0] = ml.x; rec[1] = ml.y; }
        }
        __syncwarp();

        if (writer && j == 0) {
          // the G wait above saw an MMA of position lp complete, so every MMA of
          // position lp - 1 (the buffer's last reader) is complete too
          trig_store(lp + 1, wg);
          if (nwg == 2) {
            trig_load(wn, wg + 2);
            trig_store(lp + 1, wg + 2);
          }
          trig_done(lp + 1);
        }
      }
      w = wn;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int RK, int RV>
cudaError_t launch_small_instance(const DecodeArgs& a, cudaStream_t s) {
  // the dense-cache instantiation carries no page lookup in its producer, the
  // whole-page one no per-page loop
  const int page = a.block_table == nullptr ? 0 : a.page_size % kTile == 0 ? 1 : a.splan.log2P > 0 ? 3 : 2;
  auto kern = page == 0   ? decode_small_kernel<RK, RV, 0>
              : page == 1 ? decode_small_kernel<RK, RV, 1>
              : page == 2 ? decode_small_kernel<RK, RV, 2>
                          : decode_small_kernel<RK, RV, 3>;
  static int configured[4] = {0, 0, 0, 0};
  if (configured[page] < a.splan.bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, a.splan.bytes);
    if (e != cudaSuccess) return e;
    configured[page] = a.splan.bytes;
  }
  const int trig_blocks = static_cast<int>((a.trig_rows + kTrigRowsPerBlock - 1) / kTrigRowsPerBlock);
  const int z_blocks = a.H * ((a.B + kZSeqs - 1) / kZSeqs);
  cudaError_t e = launch_pdl(decode_small_z_kernel, dim3(z_blocks + trig_blocks), dim3(kSZThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the decode grid's set-up overlaps the image
  // kernel; it waits for that grid before the first image copy / RoPE row read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = a.splan.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool make_decode_small_plan(int H, int r_k, int r_v, DecodeSmallPlan* p) {
  *p = DecodeSmallPlan{};
  if (H < 2 || H % 2 || H > kSmallMaxHeads) return false;
  if ((r_k != 16 && r_k != 32) || (r_v != 32 && r_v != 64)) return false;
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  p->nwg = H % 4 == 0 ? 4 : 2;
  p->nsets = H / p->nwg;
  p->N = al(p->nwg * (r_k + 2), 16);
  p->img = 2 * p->N * 128;
  p->NG = std::min(kMaxG, kGCols / p->N);
  p->k_tile = kTile * r_k * 2;
  p->v_tile = kTile * r_v * 2;
  p->slot = al(p->k_tile + p->v_tile, 1024);
  const int imgs = p->nsets * p->img;
  const int acc = 4 * H * r_v * 4;                 // [4 nwg warps][nsets heads][r_v]
  const int ml = al(4 * H * 8, 1024);
  const int fixed = imgs + acc + ml + kSmallMiscBytes + 1024;
  int NS = std::min((kSmemLimit - fixed) / p->slot, kSmallMaxNS);
  NS -= NS % p->nwg;   // a slot always serves the same epilogue group
  if (NS < 2 * p->nwg || p->NG < 2) return false;
  p->NS = NS;
  int off = 0;
  p->imgs = off; off += imgs;
  p->ring = off; off += NS * p->slot;
  p->acc = off;  off += acc;
  p->ml = off;   off += ml;
  p->misc = off; off += kSmallMiscBytes;
  p->bytes = off + 1024;
  return p->bytes <= kSmemLimit;
}

bool make_decode_small_setpage_plan(int H, int r_k, int r_v, int page_size, DecodeSmallPlan* p) {
  if (page_size != 8 && page_size != 16 && page_size != 32 && page_size != 64) return false;
  if (!make_decode_small_plan(H, r_k, r_v, p)) return false;
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  const int fixed = p->bytes - p->NS * p->slot;   // everything but the ring
  const int slot = al(p->nwg * (p->k_tile + p->v_tile), 1024);
  const int NS = std::min((kSmemLimit - fixed) / slot, kSmallMaxNS);
  if (NS < 2) return false;
  const int shift = NS * slot - p->NS * p->slot;   // ring growth (the ring precedes acc, ml, misc)
  p->slot = slot;
  p->NS = NS;
  p->acc += shift;
  p->ml += shift;
  p->misc += shift;
  p->bytes += shift;
  int lg = 0;
  while ((1 << lg) < page_size) ++lg;
  p->log2P = lg;
  return p->bytes <= kSmemLimit;
}

size_t decode_small_img_stride(int H, int r_k) {
  const int nwg = H % 4 == 0 ? 4 : 2;
  return static_cast<size_t>(2) * ((nwg * (r_k + 2) + 15) / 16 * 16) * 128;
}

int64_t decode_small_trig_rows(int64_t L_max, int64_t rope_len) {
  const int64_t need = (L_max + kTile - 1) / kTile * kTile;   // positions a tile can touch
  return need < rope_len ? need : rope_len;
}

cudaError_t launch_decode_small_bf16(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e;
  if (a.r_k == 16 && a.r_v == 32) e = launch_small_instance<16, 32>(a, s);
  else if (a.r_k == 16 && a.r_v == 64) e = launch_small_instance<16, 64>(a, s);
  else if (a.r_k == 32 && a.r_v == 32) e = launch_small_instance<32, 32>(a, s);
  else if (a.r_k == 32 && a.r_v == 64) e = launch_small_instance<32, 64>(a, s);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, s);
}

}  // namespace lla
