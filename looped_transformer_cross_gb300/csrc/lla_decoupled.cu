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
// bf16 kernel: the tile-major work split of the per-head tile kernel (128-token
// tiles over (sequence, head), contiguous ranges per CTA) so that the shared combine
// kernel merges the records.  Warp 0 copies each tile's key side (K latent rows and
// rotary-key rows, contiguous in the caches) with two plain bulk copies into a
// 4-slot ring; warps 1-16 are four groups of four warps, group g taking tiles
// i = g mod 4, one token per thread.  Each warp recomputes its copy of the absorbed
// query when its unit changes (no barrier between warps); a thread scores its token
// from the slot (granules visited in a lane-rotated order, so that 8 lanes cover the
// 8 bank groups), the slot is released as soon as the scores exist, and each warp
// adds sum_j p_j c_v,j for its 32 tokens
// straight from the V cache (lanes over column pairs, coalesced rows).  One record
// (m, l, acc) per (unit, CTA, warp) goes to the combine kernel.
//
// fp32 mode: one block per (unit, 128-token tile) writes the scores, then the shared
// fp32 softmax / V kernel finishes.
#include "lla_kernels.h"

#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRope = 64;                     // rotary branch width supported
constexpr int kNS = 4;                        // ring slots = epilogue groups
constexpr int kGroups = 4;

struct alignas(16) DecMisc {
  uint64_t full[kNS], empty[kNS];
  int abort;
  int start_b, start_h, start_t, count;
  int total_seq_tiles;
  int scan[kDecoupledThreads];
};

struct WarpConst {                            // one per epilogue warp (no inter-warp sync)
  float w[256];                               // absorbed content query (scaled)
  float qr[kRope];                            // rotated rotary query (scaled)
  float b0;                                   // q_c . mu_k,t (scaled)
  float pad[3];
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
__device__ __forceinline__ void rope_pair(int style, int f, int& i0, int& i1) {
  i0 = style == 0 ? f : 2 * f;
  i1 = style == 0 ? f + kRope / 2 : 2 * f + 1;
}

__global__ void __launch_bounds__(kDecoupledThreads, 1)
decoupled_bf16_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(smem_raw)) & 1023u)) & 1023u);
  const int KB = a.r_k * 2, RB = kRope * 2;                 // row bytes of a K latent / rotary key
  const int slot_bytes = kTile * (KB + RB);
  DecMisc* misc = reinterpret_cast<DecMisc*>(sm + kNS * slot_bytes);
  WarpConst* wcs = reinterpret_cast<WarpConst*>(reinterpret_cast<uint8_t*>(misc) + sizeof(DecMisc));
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
  const int count = misc->count;
  if (count == 0) return;
  Walker start;
  start.b = misc->start_b;
  start.h = misc->start_h;
  start.t = misc->start_t;
  start.L = clamp_len(__ldg(a.seq_lens + start.b), a.L_max);
  start.nb = (start.L + kTile - 1) / kTile;

  // ---------------------------------------------------------- empty records
  // Every (unit, CTA, warp) record the combine will read exists: units this CTA
  // touches get m = -inf, l = 0, acc = 0 first; the warps that see the unit
  // overwrite theirs (same CTA, after the barrier below).
  {
    const int rs = a.r_v + kRecordHead;
    Walker w = start;
    int done = 0;
    while (done < count) {
      const long long u = static_cast<long long>(w.b) * a.H + w.h;
      float* rec = a.partials + (u + blockIdx.x) * kDecoupledRecords * rs;
      for (int i = tid; i < kDecoupledRecords * rs; i += kDecoupledThreads)
        rec[i] = (i % rs) == 0 ? -INFINITY : 0.f;
      const int left = w.nb - w.t;   // tiles of this unit from w on
      done += left;
      w.t = w.nb - 1;
      walker_advance(w, a);
    }
  }

  // ---------------------------------------------------------- set-up
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) { mbar_init(bar(misc->full[s]), 1); mbar_init(bar(misc->empty[s]), 4); }
    fence_mbar_init();
  }
  __syncthreads();
  // the combine grid may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t ring = smem_u32(sm);

  if (warp == 0) {
    // ======================================================== producer
    if (lane == 0) {
      Walker w = start;
      bool ok = true;
      for (int i = 0; i < count && ok; ++i) {
        const int s = i % kNS, lap = i / kNS;
        if (lap > 0 && !(ok = mbar_wait(bar(misc->empty[s]), (lap - 1) & 1, abort, a.status))) break;
        const uint32_t rows = static_cast<uint32_t>(min(kTile, w.L - w.t * kTile));
        const uint32_t fb = bar(misc->full[s]);
        mbar_arrive_expect_tx(fb, rows * (KB + RB));
        const int64_t r0 = (static_cast<int64_t>(w.b) * a.H + w.h) * a.L_max + static_cast<int64_t>(w.t) * kTile;
        const uint32_t dst = ring + s * slot_bytes;
        bulk_load(dst, static_cast<const uint8_t*>(a.cache_k) + r0 * KB, rows * KB, fb);
        bulk_load(dst + kTile * KB, static_cast<const uint8_t*>(a.k_rope) + r0 * RB, rows * RB, fb);
        walker_advance(w, a);
      }
      // every copy lands before the CTA can exit
      for (int i = max(0, count - kNS); i < count; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->full[i % kNS]), (i / kNS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ======================================================== groups (warps 1-16)
    const int g = (warp - 1) >> 2, wq = (warp - 1) & 3;
    const int row = 32 * wq + lane;
    WarpConst& gc = wcs[warp - 1];
    const int ng = a.r_k / 8;
    const float sc = kLog2e * rsqrtf(static_cast<float>(kHeadDim + kRope));

    Walker w = start;
    for (int k = 0; k < g; ++k) walker_advance(w, a);
    int cur_b = -1, cur_h = -1;
    float m = -INFINITY, l = 0.f;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    bool ok = true;

    auto write_record = [&]() {
      const long long u = static_cast<long long>(cur_b) * a.H + cur_h;
      float* rec = a.partials + ((u + blockIdx.x) * kDecoupledRecords + 4 * g + wq) * (a.r_v + kRecordHead);
      if (lane == 0) { rec[0] = m; rec[1] = l; }
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const int c = 64 * mm + 2 * lane;
        if (c < a.r_v) { rec[kRecordHead + c] = acc[2 * mm]; rec[kRecordHead + c + 1] = acc[2 * mm + 1]; }
      }
    };

    for (int i = g; i < count && ok; i += kGroups) {
      // ---- a new unit: the previous one's record, then the absorbed query
      if (w.b != cur_b || w.h != cur_h) {
        if (cur_b >= 0) write_record();
        const int h = w.h, b = w.b;
        const __nv_bfloat16* qv =
            static_cast<const __nv_bfloat16*>(a.q) + (static_cast<int64_t>(b) * a.H + h) * (kHeadDim + kRope);
        const __nv_bfloat16* W =
            static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * a.r_k;
        __syncwarp();   // this warp's previous constants are no longer read
        for (int k = lane; k < a.r_k; k += 32) {
          float s = 0.f;
          for (int e = 0; e < kHeadDim; ++e)
            s = fmaf(__bfloat162float(qv[e]), __bfloat162float(W[e * a.r_k + k]), s);
          gc.w[k] = s * sc;
        }
        {
          const float* mu = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
          float part = 0.f;
#pragma unroll
          for (int e = 0; e < kHeadDim / 32; ++e)
            part = fmaf(__bfloat162float(qv[lane + 32 * e]), __ldg(mu + lane + 32 * e), part);
          part = warp_sum(part);
          if (lane == 0) gc.b0 = part * sc;
        }
        {
          const int f = lane;   // one frequency pair per lane (d_rope / 2 = 32)
          int qp = __ldg(a.q_pos + b);
          if (qp < 0 || qp >= a.rope_len) {
            if (f == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
            qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
          }
          int i0, i1;
          rope_pair(a.rope_style, f, i0, i1);
          const float c = __ldg(a.rope_cos + static_cast<int64_t>(qp) * (kRope / 2) + f);
          const float s = __ldg(a.rope_sin + static_cast<int64_t>(qp) * (kRope / 2) + f);
          const float x0 = __bfloat162float(qv[kHeadDim + i0]), x1 = __bfloat162float(qv[kHeadDim + i1]);
          gc.qr[i0] = (x0 * c - x1 * s) * sc;
          gc.qr[i1] = (x0 * s + x1 * c) * sc;
        }
        __syncwarp();
        cur_b = b;
        cur_h = h;
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0.f;
      }

      // ---- scores of the tile's 128 tokens (this thread: token row `row`)
      const int s_ = i % kNS, lap = i / kNS;
      if (!(ok = warp_wait(bar(misc->full[s_]), lap & 1, abort, a.status))) break;
      const int j = w.t * kTile + row;
      const bool valid = j < w.L;
      const uint8_t* kt = sm + s_ * slot_bytes + row * KB;
      const uint8_t* rt = sm + s_ * slot_bytes + kTile * KB + row * RB;
      float s0 = gc.b0, s1 = 0.f;
      for (int c = 0; c < ng; ++c) {
        const int gq = (c + lane) % ng;   // lane-rotated granule: conflict-free rows
        float x[8];
        unpack_bf16x8(*reinterpret_cast<const uint4*>(kt + 16 * gq), x);
        const float4 w0 = *reinterpret_cast<const float4*>(gc.w + 8 * gq);
        const float4 w1 = *reinterpret_cast<const float4*>(gc.w + 8 * gq + 4);
        s0 = fmaf(x[0], w0.x, s0); s1 = fmaf(x[1], w0.y, s1);
        s0 = fmaf(x[2], w0.z, s0); s1 = fmaf(x[3], w0.w, s1);
        s0 = fmaf(x[4], w1.x, s0); s1 = fmaf(x[5], w1.y, s1);
        s0 = fmaf(x[6], w1.z, s0); s1 = fmaf(x[7], w1.w, s1);
      }
      {
        // rotary branch: 4 chunks of 8 frequencies; chunk cq takes granules
        // (cq, cq + 4) (rotate-half) or (2 cq, 2 cq + 1) (interleaved)
        const int64_t jr = valid ? j : 0;
        for (int c = 0; c < 4; ++c) {
          const int cq = (c + lane) & 3;
          const float4* cp = reinterpret_cast<const float4*>(a.rope_cos + jr * (kRope / 2) + 8 * cq);
          const float4* sp = reinterpret_cast<const float4*>(a.rope_sin + jr * (kRope / 2) + 8 * cq);
          const float4 ca = __ldg(cp), cb = __ldg(cp + 1), sa = __ldg(sp), sb = __ldg(sp + 1);
          const float cs[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
          const float sn[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
          float ka[8], kb[8];
          if (a.rope_style == 0) {
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rt + 16 * cq), ka);        // dims 8cq..
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rt + 16 * (cq + 4)), kb);  // dims 32+8cq..
          } else {
            float lo[8], hi[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rt + 32 * cq), lo);        // dims 16cq..16cq+7
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rt + 32 * cq + 16), hi);   // dims 16cq+8..
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              ka[e] = lo[2 * e]; kb[e] = lo[2 * e + 1];
              ka[4 + e] = hi[2 * e]; kb[4 + e] = hi[2 * e + 1];
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            int i0, i1;
            rope_pair(a.rope_style, 8 * cq + e, i0, i1);
            const float k0 = ka[e] * cs[e] - kb[e] * sn[e], k1 = ka[e] * sn[e] + kb[e] * cs[e];
            s0 = fmaf(gc.qr[i0], k0, s0);
            s1 = fmaf(gc.qr[i1], k1, s1);
          }
        }
      }
      const float s = valid ? s0 + s1 : -INFINITY;
      // the slot's keys are no longer needed
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
      l += warp_sum(p);

      // ---- sum_j p_j c_v,j for the warp's 32 tokens, rows read from the cache
      // (lane: column pairs 2 lane + 64 mm); tokens past the sequence end skipped
      const int nval = min(32, max(0, w.L - (w.t * kTile + 32 * wq)));
      const __nv_bfloat16* vrow = static_cast<const __nv_bfloat16*>(a.cache_v) +
                                  ((static_cast<int64_t>(w.b) * a.H + w.h) * a.L_max + w.t * kTile + 32 * wq) * a.r_v;
      for (int t0 = 0; t0 < nval; t0 += 8) {
        uint32_t vv[8][4];
#pragma unroll
        for (int u8 = 0; u8 < 8; ++u8)
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const int c = 64 * mm + 2 * lane;
            vv[u8][mm] = (t0 + u8 < nval && c < a.r_v)
                             ? __ldg(reinterpret_cast<const unsigned int*>(vrow + static_cast<int64_t>(t0 + u8) * a.r_v + c))
                             : 0u;
          }
#pragma unroll
        for (int u8 = 0; u8 < 8; ++u8) {
          const float pv = __shfl_sync(0xffffffffu, p, (t0 + u8) & 31);
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            acc[2 * mm] = fmaf(pv, __uint_as_float(vv[u8][mm] << 16), acc[2 * mm]);
            acc[2 * mm + 1] = fmaf(pv, __uint_as_float(vv[u8][mm] & 0xFFFF0000u), acc[2 * mm + 1]);
          }
        }
      }
      for (int k = 0; k < kGroups; ++k) walker_advance(w, a);
    }
    if (ok && cur_b >= 0) write_record();
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

size_t decoupled_smem_bytes(int r_k) {
  return static_cast<size_t>(kNS) * kTile * (2 * r_k + 2 * kRope) + sizeof(DecMisc) +
         (kDecoupledThreads / 32 - 1) * sizeof(WarpConst) + 1024;
}

cudaError_t launch_decoupled_bf16(const DecodeArgs& a, cudaStream_t s) {
  const int bytes = static_cast<int>(decoupled_smem_bytes(a.r_k));
  static int configured = 0;
  if (configured < bytes) {
    cudaError_t e = cudaFuncSetAttribute(decoupled_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured = bytes;
  }
  decoupled_bf16_kernel<<<a.grid, kDecoupledThreads, bytes, s>>>(a);
  cudaError_t e = cudaGetLastError();
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
