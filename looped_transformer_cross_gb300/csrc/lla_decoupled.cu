// lla_decoupled.cu — absorbed decoupled-RoPE decode ("Looped Latent Attention:
// Cross-Loop KV Compression for Looped Transformers", arXiv 2607.15456v2,
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
// bf16 path, three launches:
//  1. decoupled_query_kernel, one block per (sequence, head), writes one query
//     record per 128-token tile of the unit: {sc w (r_k), (ua, ub) (32 + 32), sc b0,
//     three zeros}, where (ua, ub) is sc RoPE(q_r, q_pos) as the (i0, i1) halves of
//     the 32 frequency pairs, rotated further by -T theta_f (T the tile start), and
//     sc = log2(e) / sqrt(d + d_rope), so that scores come out in base-2 units.
//  2. decoupled_bf16_kernel<RK, NMM>: the tile-major split of the per-head tile
//     kernel (128-token tiles over (sequence, head), contiguous ranges per CTA), so
//     that the shared combine kernel merges the records.  Lane 0 of warp 0 copies
//     each tile's query record, K latent rows and rotary-key rows (contiguous in
//     their caches) with three plain bulk copies into a ring of NS slots, NS - 1
//     tiles ahead of its own scoring, and has L2 prefetch the tile's V latent rows.
//     All 16 warps work on the same tile: warp w owns tokens 8w..8w+7 with four
//     lanes per token, each lane taking a quarter of the r_k content dimensions and
//     8 of the 32 frequency pairs.  The rotary factor of the token at T + r is the
//     record's pair rotated by -r, a per-lane constant rotation (angle sum), so no
//     per-token trigonometry is read.  Each warp keeps its own online softmax and
//     adds sum_j p_j c_v,j for its 8 tokens from the V cache (lanes over column
//     pairs, NMM rounds of 64 columns; the loads are issued before the scores).  At
//     the end of a unit the 16 warp states are staged in shared memory and one warp
//     merges them (log-sum-exp), so one record (m, l, acc) per (unit, CTA) goes to
//     the combine kernel.
//  3. decode_combine_kernel (shared with the per-head decode paths).
//
// fp32 mode: one block per (unit, 128-token tile) writes the scores, then the shared
// fp32 softmax / V kernel finishes.
#include "lla_kernels.h"

#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRope = 64;                     // rotary branch width supported
constexpr int kHalf = kRope / 2;              // frequency pairs
constexpr int kQrecTail = 4;                  // b0 and three zeros after w, qa, qb
constexpr int kMaxNS = 8;                     // ring slots at most
constexpr int kQueryWarps = 8;                // query kernel: 256 threads per unit
constexpr int kComputeWarps = kDecoupledThreads / 32;       // 16: 8 tokens each

static_assert(kComputeWarps * 8 == kTile, "eight tokens per compute warp cover a tile");

__host__ __device__ constexpr int qrec_floats(int r_k) { return r_k + kRope + kQrecTail; }
// One ring slot: the query record (padded to 128 bytes), 128 K latent rows, 128
// rotary-key rows.
__host__ __device__ constexpr int slot_qbytes(int r_k) { return (qrec_floats(r_k) * 4 + 127) / 128 * 128; }
__host__ __device__ constexpr int slot_bytes(int r_k) { return slot_qbytes(r_k) + kTile * (2 * r_k + 2 * kRope); }

struct alignas(16) DecMisc {
  uint64_t full[kMaxNS], empty[kMaxNS];
  uint64_t staged;                            // 16 warps have staged their unit record
  uint64_t merged;                            // the merging warp has read the stage
  int abort;
  int start_b, start_h, start_t, count;
  int total_seq_tiles;
  int scan[kDecoupledThreads];
};

struct Walker {
  int b, h, t, nb, L;
};

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

__device__ __forceinline__ void walker_advance(Walker& w, const DecodeArgs& a) {
  if (++w.t < w.nb) return;
  w.t = 0;
  if (++w.h < a.H) return;
  w.h = 0;
  while (true) {
    ++w.b;
    if (w.b >= a.B) { w.nb = 0; return; }
    w.L = clamp_len(__ldg(a.seq_lens + w.b), a.L_max);
    w.nb = (w.L + kTile - 1) / kTile;
    if (w.nb > 0) return;
  }
}

// Rotary pair (i0, i1) of frequency f within the d_rope branch.
__host__ __device__ __forceinline__ void rope_pair(int style, int f, int& i0, int& i1) {
  i0 = style == 0 ? f : 2 * f;
  i1 = style == 0 ? f + kRope / 2 : 2 * f + 1;
}

// Ask L2 to fetch [src, src + bytes) (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// Bounded wait for a phase completed by other warps' arrivals (the staging
// barriers and the ring's empty slots): non-blocking test_wait polls, so the
// thread never sits suspended after the last warp has arrived.  After about one second,
// or when another role has raised *abort, it records LLA_ERR_TIMEOUT (first expiry
// only) and returns false.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_arrivals(uint32_t bar, uint32_t parity, volatile int* abort,
                                                   uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
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

// Warp-collective form: lane 0 polls, the warp leaves converged with its decision.
__device__ __forceinline__ bool warp_wait_arrivals(uint32_t bar, uint32_t parity, volatile int* abort,
                                                   uint32_t* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_arrivals(bar, parity, abort, status);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ------------------------------------------------------------------ query records
// Block = one (sequence, head) unit, 256 threads.  w_k = sum_e q_e W[e][k] is
// formed as 8 slices of 16 rows e (threads over (slice, k), coalesced along k),
// then summed; the rotary query is rotated to q_pos; b0 = q_c . mu_k,t.  Record
// (unit, tile t) = {w, (ua, ub), b0, 0, 0, 0} with (ua, ub) the RoPE'd query pair
// rotated further by -128 t theta_f, so that the main kernel only applies the
// rotation by the token's row within the tile.
__global__ void __launch_bounds__(kQueryWarps * 32) decoupled_query_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float qf[kHeadDim + kRope];
  __shared__ float part[8][128];
  __shared__ float qr[kRope];                   // RoPE(q_r, q_pos): i0 halves, then i1 halves
  __shared__ float wsh[128 + kQrecTail];
  const int u = blockIdx.x, tid = threadIdx.x;
  const int b = u / a.H, h = u - b * a.H;
  const int L = clamp_len(__ldg(a.seq_lens + b), a.L_max);
  const int nt = (L + kTile - 1) / kTile;       // tiles this unit has
  if (nt == 0) return;
  const __nv_bfloat16* qv = static_cast<const __nv_bfloat16*>(a.q) + static_cast<int64_t>(u) * (kHeadDim + kRope);
  for (int i = tid; i < kHeadDim + kRope; i += kQueryWarps * 32) qf[i] = __bfloat162float(qv[i]);
  __syncthreads();
  const float sc = kLog2e * rsqrtf(static_cast<float>(kHeadDim + kRope));
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * a.r_k;
  for (int idx = tid; idx < 8 * a.r_k; idx += kQueryWarps * 32) {
    const int sl = idx / a.r_k, k = idx - sl * a.r_k;
    const __nv_bfloat16* Wc = W + static_cast<int64_t>(16 * sl) * a.r_k + k;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) s = fmaf(qf[16 * sl + e], __bfloat162float(Wc[static_cast<int64_t>(e) * a.r_k]), s);
    part[sl][k] = s;
  }
  if (tid < kHalf) {
    int qp = __ldg(a.q_pos + b);
    if (qp < 0 || qp >= a.rope_len) {
      if (tid == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
      qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
    }
    int i0, i1;
    rope_pair(a.rope_style, tid, i0, i1);
    const float c = __ldg(a.rope_cos + static_cast<int64_t>(qp) * kHalf + tid);
    const float s = __ldg(a.rope_sin + static_cast<int64_t>(qp) * kHalf + tid);
    const float x0 = qf[kHeadDim + i0], x1 = qf[kHeadDim + i1];
    qr[tid] = (x0 * c - x1 * s) * sc;
    qr[kHalf + tid] = (x0 * s + x1 * c) * sc;
  } else if (tid < 64) {
    const float* mu = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
    float p = 0.f;
#pragma unroll
    for (int e = tid - 32; e < kHeadDim; e += 32) p = fmaf(qf[e], __ldg(mu + e), p);
    p = warp_sum(p);
    if (tid == 32) {
      wsh[a.r_k] = p * sc;
      wsh[a.r_k + 1] = 0.f;
      wsh[a.r_k + 2] = 0.f;
      wsh[a.r_k + 3] = 0.f;
    }
  }
  __syncthreads();
  for (int k = tid; k < a.r_k; k += kQueryWarps * 32) {
    float s = 0.f;
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) s += part[sl][k];
    wsh[k] = s * sc;
  }
  __syncthreads();
  const int QF = qrec_floats(a.r_k);
  const int64_t nt_max = (a.L_max + kTile - 1) / kTile;
  float* rec0 = reinterpret_cast<float*>(a.zimg) + static_cast<int64_t>(u) * nt_max * QF;
  // one warp per tile record, one frequency pair per lane; the table rows of four
  // tiles are read before any of their records is written
  const int wp = tid >> 5, ln = tid & 31;
  const float qa = qr[ln], qb = qr[kHalf + ln];
  for (int t0 = wp; t0 < nt; t0 += 4 * kQueryWarps) {
    float cT[4], sT[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = t0 + k * kQueryWarps;
      const int64_t T = static_cast<int64_t>(t < nt ? t : 0) * kTile;
      cT[k] = __ldg(a.rope_cos + T * kHalf + ln);
      sT[k] = __ldg(a.rope_sin + T * kHalf + ln);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = t0 + k * kQueryWarps;
      if (t >= nt) break;
      float* rec = rec0 + static_cast<int64_t>(t) * QF;
      for (int e = ln; e < a.r_k; e += 32) rec[e] = wsh[e];
      if (ln < kQrecTail) rec[a.r_k + kRope + ln] = wsh[a.r_k + ln];
      rec[a.r_k + ln] = fmaf(qa, cT[k], qb * sT[k]);
      rec[a.r_k + kHalf + ln] = fmaf(qb, cT[k], -qa * sT[k]);
    }
  }
}

// The merging warp of a unit: the 16 staged warp states {m, l, -, -, acc[r_v]}
// (rows rs floats apart) folded by log-sum-exp into the CTA's split record `rec`,
// then the stage released through `merged_bar`.  Kept out of line so that the
// main loop's code stays free of this warp-specific branch.
__device__ __noinline__ void merge_staged(const float* stage, int rs, int r_v, float* rec, uint32_t merged_bar) {
  const int lane = threadIdx.x & 31;
  constexpr int kW = kDecoupledThreads / 32;
  const float mw = lane < kW ? stage[lane * rs] : -INFINITY;
  const float M = warp_max_redux(mw);
  const float sw = (lane < kW && mw != -INFINITY) ? exp2f(mw - M) : 0.f;
  const float L = warp_sum(lane < kW ? stage[lane * rs + 1] * sw : 0.f);
  // every lane takes all 16 scales first: the column loop below runs a
  // lane-dependent number of rounds and holds no warp collective
  float f[kW];
#pragma unroll
  for (int w2 = 0; w2 < kW; ++w2) f[w2] = __shfl_sync(0xffffffffu, sw, w2);
  for (int c = 2 * lane; c < r_v; c += 64) {
    float2 o = make_float2(0.f, 0.f);
#pragma unroll
    for (int w2 = 0; w2 < kW; ++w2) {
      const float2 v = *reinterpret_cast<const float2*>(stage + w2 * rs + kRecordHead + c);
      o.x = fmaf(f[w2], v.x, o.x);
      o.y = fmaf(f[w2], v.y, o.y);
    }
    *reinterpret_cast<float2*>(rec + kRecordHead + c) = o;
  }
  if (lane == 0) { rec[0] = M; rec[1] = L; }
  __syncwarp();
  if (lane == 0) mbar_arrive(merged_bar);
}

// ------------------------------------------------------------------ main kernel
template <int RK, int NMM>
__global__ void __launch_bounds__(kDecoupledThreads, 1)
decoupled_bf16_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int KB = 2 * RK, RB = 2 * kRope;       // row bytes of a K latent / rotary key
  constexpr int QB = slot_qbytes(RK), SB = slot_bytes(RK);
  constexpr int QF = qrec_floats(RK);
  constexpr int NW = RK / 8;                       // 32-bit words of a K row per lane
  constexpr int VW = NW % 4 == 0 ? 4 : 2;          // words per shared load
  constexpr int NCH = NW / VW;
  // Rows of 64 or 128 latents would put the four lanes of a load phase on the
  // same banks: those ranks visit their chunks in a lane-rotated order.
  constexpr int kRotShift = RK == 64 ? 2 : (RK == 128 ? 1 : -1);
  static_assert(RK % 16 == 0 && RK >= 16 && RK <= 128, "r_k: multiple of 16 up to 128");
  static_assert(kRotShift < 0 || (NCH & (NCH - 1)) == 0, "rotation needs a power-of-two chunk count");
  static_assert(NMM >= 1 && NMM <= 4, "V rows of 64 NMM columns at most");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(smem_raw)) & 1023u)) & 1023u);
  const int NS = a.ring_slots;
  DecMisc* misc = reinterpret_cast<DecMisc*>(sm + NS * SB);
  float* stage = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(misc) + sizeof(DecMisc));
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------- work range (tile-major)
  {
    const int per_thr = (a.B + kDecoupledThreads - 1) / kDecoupledThreads;
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
      constexpr int kPer = kDecoupledThreads / 32;
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
      if (lane == 31) misc->total_seq_tiles = incl;
    }
    __syncthreads();
    const long long total = static_cast<long long>(a.H) * misc->total_seq_tiles;
    const long long per = max(1LL, (total + a.grid - 1) / a.grid);
    const long long f0 = static_cast<long long>(blockIdx.x) * per;
    const long long f1 = min(total, f0 + per);
    long long P0 = misc->scan[tid];
    for (int b = b0; b < b1; ++b) {
      const int nb = (clamp_len(__ldg(a.seq_lens + b), a.L_max) + kTile - 1) / kTile;
      if (nb > 0 && f0 < f1 && a.H * P0 <= f0 && f0 < a.H * (P0 + nb)) {
        const long long rem = f0 - a.H * P0;
        misc->start_b = b;
        misc->start_h = static_cast<int>(rem / nb);
        misc->start_t = static_cast<int>(rem % nb);
      }
      P0 += nb;
    }
    if (tid == 0) misc->count = static_cast<int>(f1 > f0 ? f1 - f0 : 0);
    __syncthreads();
  }
  // a CTA without tiles writes no record: the combine reads only the CTAs that
  // cover a unit's tiles
  const int count = misc->count;
  if (count == 0) return;
  Walker start;
  start.b = misc->start_b;
  start.h = misc->start_h;
  start.t = misc->start_t;
  start.L = clamp_len(__ldg(a.seq_lens + start.b), a.L_max);
  start.nb = (start.L + kTile - 1) / kTile;

  // ---------------------------------------------------------- set-up
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(misc->full[s]), 1);
      mbar_init(bar(misc->empty[s]), kComputeWarps);
    }
    mbar_init(bar(misc->staged), kComputeWarps);
    mbar_init(bar(misc->merged), 1);
    fence_mbar_init();
  }
  __syncthreads();
  // the combine grid may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t ring = smem_u32(sm);

  // ---------------------------------------------------------- copies (warp 0, lane 0)
  // Tile i goes to slot i mod NS.  Refilling the slot of tile k waits until all
  // 16 warps have scored tile k; warp 0 has, and every other warp gets there
  // without warp 0 (tiles up to k + NS - 1 are already issued), so the wait ends.
  const int64_t nt_max = (a.L_max + kTile - 1) / kTile;   // tile records per unit
  Walker pw = start;
  int issued = 0;
  bool pok = true;
  auto issue_upto = [&](int end) {
    for (; pok && issued < end && issued < count; ++issued) {
      const int i = issued, s = i % NS, lap = i / NS;
      if (lap > 0 && !(pok = mbar_wait_arrivals(bar(misc->empty[s]), (lap - 1) & 1, abort, a.status))) break;
      const uint32_t rows = static_cast<uint32_t>(min(kTile, pw.L - pw.t * kTile));
      const int64_t u = static_cast<int64_t>(pw.b) * a.H + pw.h;
      const int64_t r0 = u * a.L_max + static_cast<int64_t>(pw.t) * kTile;
      const uint32_t fb = bar(misc->full[s]);
      mbar_arrive_expect_tx(fb, QF * 4 + rows * (KB + RB));
      const uint32_t dst = ring + s * SB;
      bulk_load(dst, a.zimg + (u * nt_max + pw.t) * a.zimg_stride, QF * 4, fb);
      bulk_load(dst + QB, static_cast<const uint8_t*>(a.cache_k) + r0 * KB, rows * KB, fb);
      bulk_load(dst + QB + kTile * KB, static_cast<const uint8_t*>(a.k_rope) + r0 * RB, rows * RB, fb);
      bulk_prefetch_l2(static_cast<const uint8_t*>(a.cache_v) + r0 * (2 * a.r_v), rows * (2 * a.r_v));
      walker_advance(pw, a);
    }
  };
  const bool producer = tid == 0;
  if (producer) issue_upto(NS);

  // ---------------------------------------------------------- compute (all 16 warps)
  {
    const int cw = warp, tok = lane >> 2, q = lane & 3;
    const int row = 8 * cw + tok;                  // this lane's token row in every tile
    const bool odd = (tok & 1) != 0;
    const bool interleaved = a.rope_style != 0;
    // rotation by the row offset for this lane's frequencies 8q..8q+7 (rope_len >= 128)
    float cr[8], sr[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cr[e] = __ldg(a.rope_cos + static_cast<int64_t>(row) * kHalf + 8 * q + e);
      sr[e] = __ldg(a.rope_sin + static_cast<int64_t>(row) * kHalf + 8 * q + e);
    }
    const int rs = a.r_v + kRecordHead;

    Walker w = start;
    int cur_b = -1, cur_h = -1;
    float m = -INFINITY, l = 0.f;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    bool ok = true;

    // ---- end of a unit: every warp stages (m, l, acc); warp (n mod 16) merges the
    // 16 staged states of unit n by log-sum-exp into the CTA's one split record.
    // Staging for unit n waits until unit n - 1's stage has been read; a warp can
    // only reach unit n + 2 after that wait for unit n + 1, so neither barrier is
    // ever waited on two phases ahead.
    int nunit = 0;
    auto finish_unit = [&]() -> bool {
      bool fok = nunit == 0 || warp_wait_arrivals(bar(misc->merged), (nunit - 1) & 1, abort, a.status);
      if (fok) {
        float* st = stage + cw * rs;
        if (lane == 0) { st[0] = m; st[1] = l; }
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          const int c = 64 * mm + 2 * lane;
          if (c < a.r_v) *reinterpret_cast<float2*>(st + kRecordHead + c) = make_float2(acc[2 * mm], acc[2 * mm + 1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->staged));
      }
      if (fok && cw == nunit % kComputeWarps) {
        fok = warp_wait_arrivals(bar(misc->staged), nunit & 1, abort, a.status);
        if (fok) {
          const long long u = static_cast<long long>(cur_b) * a.H + cur_h;
          merge_staged(stage, rs, a.r_v, a.partials + (u + blockIdx.x) * rs, bar(misc->merged));
        }
      }
      ++nunit;
      return fok;
    };

    for (int i = 0; i < count; ++i) {
      // the slot of tile i - 2 takes tile i - 2 + NS: NS - 1 tiles ahead of warp 0,
      // which waits only for warps that are two tiles behind it
      if (producer && i >= 2) issue_upto(i - 2 + NS + 1);
      __syncwarp();
      if (w.b != cur_b || w.h != cur_h) {
        if (cur_b >= 0) ok = finish_unit();
        if (!ok) break;
        cur_b = w.b;
        cur_h = w.h;
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0.f;
      }
      const int T = w.t * kTile;
      const bool valid = T + row < w.L;

      // ---- V rows of this warp's 8 tokens (L2-prefetched), issued before the scores
      const int nval = min(8, max(0, w.L - (T + 8 * cw)));
      const __nv_bfloat16* vrow = static_cast<const __nv_bfloat16*>(a.cache_v) +
                                  ((static_cast<int64_t>(w.b) * a.H + w.h) * a.L_max + T + 8 * cw) * a.r_v;
      uint32_t vv[8][NMM];
#pragma unroll
      for (int t8 = 0; t8 < 8; ++t8)
#pragma unroll
        for (int mm = 0; mm < NMM; ++mm) {
          const int c = 64 * mm + 2 * lane;
          vv[t8][mm] = (t8 < nval && (mm < NMM - 1 || c < a.r_v))
                           ? __ldg(reinterpret_cast<const unsigned int*>(vrow + static_cast<int64_t>(t8) * a.r_v + c))
                           : 0u;
        }

      const int s_ = i % NS, lap = i / NS;
      if (!(ok = warp_wait(bar(misc->full[s_]), lap & 1, abort, a.status))) break;
      const uint8_t* slot = sm + s_ * SB;
      const float* qrec = reinterpret_cast<const float*>(slot);
      const uint8_t* kt = slot + QB + row * KB;
      const uint8_t* rt = slot + QB + kTile * KB + row * RB;

      // ---- content score: this lane's quarter of the r_k dimensions
      float s0 = q == 0 ? qrec[RK + kRope] : 0.f, s1 = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int cc = kRotShift >= 0 ? ((c + (lane >> (kRotShift < 0 ? 0 : kRotShift))) & (NCH - 1)) : c;
        const int wo = q * NW + VW * cc;           // word offset within the row
        if constexpr (VW == 4) {
          float x[8];
          unpack_bf16x8(*reinterpret_cast<const uint4*>(kt + 4 * wo), x);
          const float4 w0 = *reinterpret_cast<const float4*>(qrec + 2 * wo);
          const float4 w1 = *reinterpret_cast<const float4*>(qrec + 2 * wo + 4);
          s0 = fmaf(x[0], w0.x, s0); s1 = fmaf(x[1], w0.y, s1);
          s0 = fmaf(x[2], w0.z, s0); s1 = fmaf(x[3], w0.w, s1);
          s0 = fmaf(x[4], w1.x, s0); s1 = fmaf(x[5], w1.y, s1);
          s0 = fmaf(x[6], w1.z, s0); s1 = fmaf(x[7], w1.w, s1);
        } else {
          const uint2 kv = *reinterpret_cast<const uint2*>(kt + 4 * wo);
          const float4 w0 = *reinterpret_cast<const float4*>(qrec + 2 * wo);
          s0 = fmaf(__uint_as_float(kv.x << 16), w0.x, s0);
          s1 = fmaf(__uint_as_float(kv.x & 0xFFFF0000u), w0.y, s1);
          s0 = fmaf(__uint_as_float(kv.y << 16), w0.z, s0);
          s1 = fmaf(__uint_as_float(kv.y & 0xFFFF0000u), w0.w, s1);
        }
      }

      // ---- rotary score: frequencies 8q..8q+7 of this lane's token
      {
        // (ua, ub): the query pair already rotated by -T (per-tile record)
        const float4 ua0 = *reinterpret_cast<const float4*>(qrec + RK + 8 * q);
        const float4 ua1 = *reinterpret_cast<const float4*>(qrec + RK + 8 * q + 4);
        const float4 ub0 = *reinterpret_cast<const float4*>(qrec + RK + kHalf + 8 * q);
        const float4 ub1 = *reinterpret_cast<const float4*>(qrec + RK + kHalf + 8 * q + 4);
        const float ua[8] = {ua0.x, ua0.y, ua0.z, ua0.w, ua1.x, ua1.y, ua1.z, ua1.w};
        const float ub[8] = {ub0.x, ub0.y, ub0.z, ub0.w, ub1.x, ub1.y, ub1.z, ub1.w};
        // key components (i0, i1) of the 8 pairs: two 16-byte chunks of the row;
        // odd tokens read the second chunk first so that a load phase spans all banks
        const int offA = interleaved ? 32 * q : 16 * q;
        const int offB = interleaved ? 32 * q + 16 : 2 * kHalf + 16 * q;
        const uint4 first = *reinterpret_cast<const uint4*>(rt + (odd ? offB : offA));
        const uint4 second = *reinterpret_cast<const uint4*>(rt + (odd ? offA : offB));
        const uint4 A = odd ? second : first, B = odd ? first : second;
        float xa[8], xb[8], ka[8], kb[8];
        unpack_bf16x8(A, xa);
        unpack_bf16x8(B, xb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float ia = e < 4 ? xa[2 * e] : xb[2 * (e - 4)];
          const float ib = e < 4 ? xa[2 * e + 1] : xb[2 * (e - 4) + 1];
          ka[e] = interleaved ? ia : xa[e];
          kb[e] = interleaved ? ib : xb[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // (X, Y) = (ua, ub) rotated by -r: ka X + kb Y = RoPE(q_r) . RoPE(k_r, T + r)
          const float X = fmaf(ua[e], cr[e], ub[e] * sr[e]);
          const float Y = fmaf(ub[e], cr[e], -ua[e] * sr[e]);
          s1 = fmaf(ka[e], X, s1);
          s0 = fmaf(kb[e], Y, s0);
        }
      }
      float s = s0 + s1;
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s = valid ? s : -INFINITY;
      // the slot is no longer read
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(misc->empty[s_]));

      // ---- online softmax per warp (reference raised lazily, by more than 2^8)
      const float mt = warp_max_redux(s);
      if (mt > m + 8.f) {
        const float alpha = m == -INFINITY ? 0.f : exp2f(m - mt);
        l *= alpha;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= alpha;
        m = mt;
      }
      const float p = valid ? exp2f(s - m) : 0.f;
      float ps = p;                                // every token counted once per lane class
      ps += __shfl_xor_sync(0xffffffffu, ps, 4);
      ps += __shfl_xor_sync(0xffffffffu, ps, 8);
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);
      l += ps;

      // ---- sum_j p_j c_v,j over the warp's 8 tokens
#pragma unroll
      for (int t8 = 0; t8 < 8; ++t8) {
        const float pv = __shfl_sync(0xffffffffu, p, 4 * t8);
#pragma unroll
        for (int mm = 0; mm < NMM; ++mm) {
          acc[2 * mm] = fmaf(pv, __uint_as_float(vv[t8][mm] << 16), acc[2 * mm]);
          acc[2 * mm + 1] = fmaf(pv, __uint_as_float(vv[t8][mm] & 0xFFFF0000u), acc[2 * mm + 1]);
        }
      }
      walker_advance(w, a);
    }
    if (ok && cur_b >= 0) finish_unit();
  }
  // every issued copy lands before the CTA can exit (bounded: after an abort some
  // slots were never consumed)
  if (producer) {
    for (int i = max(0, issued - NS); i < issued; ++i) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->full[i % NS]), (i / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }
  __syncthreads();
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

int decoupled_qrec_floats(int r_k) { return qrec_floats(r_k); }

// shared memory besides the ring: barriers and scan, the 16 staged unit records,
// 1024 bytes of alignment slack
static size_t decoupled_fixed_bytes(int r_v) {
  return sizeof(DecMisc) + static_cast<size_t>(kComputeWarps) * (r_v + kRecordHead) * 4 + 1024;
}

int decoupled_ring_slots(int r_k, int r_v) {
  if (r_k < 16 || r_k > 128 || r_k % 16 != 0 || r_v < 16 || r_v > 256 || r_v % 16 != 0) return 0;
  const long long avail = kSmemLimit - static_cast<long long>(decoupled_fixed_bytes(r_v));
  const long long ns = avail / slot_bytes(r_k);
  return ns < 2 ? 0 : static_cast<int>(ns < kMaxNS ? ns : kMaxNS);
}

size_t decoupled_smem_bytes(int r_k, int r_v, int ns) {
  return static_cast<size_t>(ns) * slot_bytes(r_k) + decoupled_fixed_bytes(r_v);
}

namespace {

template <int RK, int NMM>
cudaError_t launch_main(const DecodeArgs& a, int bytes, cudaStream_t s) {
  static int configured = 0;
  if (configured < bytes) {
    cudaError_t e = cudaFuncSetAttribute(decoupled_bf16_kernel<RK, NMM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured = bytes;
  }
  decoupled_bf16_kernel<RK, NMM><<<a.grid, kDecoupledThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

template <int RK>
cudaError_t launch_main_v(const DecodeArgs& a, int bytes, cudaStream_t s) {
  switch ((a.r_v + 63) / 64) {
    case 1: return launch_main<RK, 1>(a, bytes, s);
    case 2: return launch_main<RK, 2>(a, bytes, s);
    case 3: return launch_main<RK, 3>(a, bytes, s);
    case 4: return launch_main<RK, 4>(a, bytes, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_main_rk(const DecodeArgs& a, int bytes, cudaStream_t s) {
  switch (a.r_k) {
    case 16: return launch_main_v<16>(a, bytes, s);
    case 32: return launch_main_v<32>(a, bytes, s);
    case 48: return launch_main_v<48>(a, bytes, s);
    case 64: return launch_main_v<64>(a, bytes, s);
    case 80: return launch_main_v<80>(a, bytes, s);
    case 96: return launch_main_v<96>(a, bytes, s);
    case 112: return launch_main_v<112>(a, bytes, s);
    case 128: return launch_main_v<128>(a, bytes, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decoupled_bf16(const DecodeArgs& a, cudaStream_t s) {
  if (a.ring_slots < 2 || a.ring_slots > kMaxNS) return cudaErrorInvalidValue;
  const int bytes = static_cast<int>(decoupled_smem_bytes(a.r_k, a.r_v, a.ring_slots));
  decoupled_query_kernel<<<a.B * a.H, kQueryWarps * 32, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_main_rk(a, bytes, s);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, s);
}

cudaError_t launch_decoupled_f32(const DecodeArgs& a, cudaStream_t s) {
  const dim3 g1(a.B * a.H, static_cast<unsigned>((a.L_max + kTile - 1) / kTile));
  decoupled_f32_scores_kernel<<<g1, 128, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_decode_f32_values(a, s);
}

}  // namespace lla
