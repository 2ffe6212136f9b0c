// lla_decode.cu — latent-store decode attention of Looped Latent Attention on
// sm_103a ("Looped Latent Attention: Cross-Loop KV Compression for Looped
// Transformers", arXiv 2607.15456v2: §3 Eq. (2)-(3), "RoPE and
// reconstruction", §7 latent-store path, Appendix J "Absorbed attention").
//
// Per-head bf16 path, one persistent CTA per SM (7 warps):
//   * Work is the flat list of 128-token latent tiles over (sequence, head),
//     cut into equal contiguous ranges, one per CTA.  For each (sequence, head)
//     unit it touches a CTA writes one record (m, l, acc_v) per epilogue warp;
//     the combine kernel merges a unit's records (log-sum-exp merge) and applies
//     the V up-projection once (Appendix J identity).
//   * Warp 0 streams latent tiles with TMA into a K ring and a V ring (V tile i
//     requested after K tile i+1: it is needed only once tile i's weights exist).
//   * Warp 1 issues the score MMAs: U = C_k Z^T (+ bias) into TMEM, where Z folds
//     the RoPE-rotated query into W_up,k,t (exact rewrite of q'.R_j (W c + mu)).
//     Z of each unit comes ready-made from decode_z_kernel; the producer copies
//     the next unit's image in while the current one runs (two buffers).
//   * Warp 6 issues the value MMAs: D += P C_v, with the tile's softmax weights P
//     read from TMEM (written over the consumed scores) and the V latent tile as
//     an MN-major operand, accumulating over the whole unit in TMEM.
//   * Warps 2-5 (one per TMEM lane quadrant, one token per lane) turn U into the
//     rotary score s_j = sum_f cos(j th_f) U_f + sin(j th_f) U_{64+f}, run an
//     online softmax per warp and write P = diag(p): accumulator row j collects
//     p_j c_v,j over the unit's tiles and the rows are summed when the unit ends.
//     cos/sin(j th) come from the angle sum of the tile base row (a per-warp
//     shared-memory copy) and the lane's own row (registers).  A warp rescales its
//     accumulator row only when its running max grows by more than 2^8.
// Reconstructed keys and values never leave TMEM / registers.
//
#include "lla_kernels.h"

#include <algorithm>
#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr float kRescaleLog2 = 8.f;                 // lazy rescale threshold (log2 units)
constexpr int kDCol = 256;                          // TMEM columns of the value accumulator

struct alignas(16) DecodeMisc {
  uint64_t kfull[kMaxStages], kempty[kMaxStages];
  uint64_t vfull[kMaxStages], vempty[kMaxStages];
  uint64_t ufull[2], pfull[2], vdone[2];   // index = tile & 1
  uint64_t zfull[2], zfree[2];             // index = unit % NZ
  uint64_t mma_done[2];                    // score / value issuer drained
  uint32_t tmem_base;
  int abort;
  int start_b, start_h, start_t, count;
  int total_seq_tiles;
  int scan[kDecodeThreads];  // per-thread sequence-chunk tile counts
};
static_assert(sizeof(DecodeMisc) <= 2048, "misc region");

struct Walker {
  int b, h, t, nb, L;
};

// Position in a ring of n mbarrier-guarded slots: the slot index and the parity
// of the slot's current use, advanced without division (the role warps share
// their sub-partitions with the epilogue warps, so their per-tile scalar work
// is kept small).
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) { slot = 0; phase ^= 1u; }
  }
};

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

// TMA coordinates (y, z) of tile t of (sequence b, head h) in the 3-D map over the
// page pool (page_size a multiple of the tile): rows y within z = page H + h.
__device__ __forceinline__ void tile_yz(const DecodeArgs& a, int b, int h, int t, int& y, int& z) {
  const int j = t * kTile, lp = j / a.page_size;
  z = page_of(a, b, lp) * a.H + h;
  y = j - lp * a.page_size;
}

// One latent tile (K or V: chunk plan `cp`, map of chunk c from `map_of`) of (sequence
// b, head h, tile t; L tokens) from the page pool into `dst`, completing on `fb`.  A
// tile inside one page is one box per chunk; with pages of P < 128 tokens (P a
// multiple of 8 dividing 128, so every piece starts on a swizzle atom) it is one box
// of P rows per chunk and page, and only the pages holding tokens below L are read.
template <bool kPieces, typename MapOf>
__device__ __forceinline__ void paged_tile_load(const DecodeArgs& a, int b, int h, int t, int L, uint32_t dst,
                                                uint32_t fb, const ChunkPlan& cp, MapOf map_of) {
  if constexpr (!kPieces) {
    mbar_arrive_expect_tx(fb, cp.bytes);
    int y, z;
    tile_yz(a, b, h, t, y, z);
    for (int c = 0; c < cp.n; ++c) tma_load_3d(dst + cp.off[c], map_of(c), fb, cp.start[c], y, z);
    return;
  }
  // (called by the whole producer warp: lane i issues the boxes of page i)
  const int pg = a.page_size, lane = threadIdx.x & 31;
  const int np = (min(kTile, L - t * kTile) + pg - 1) / pg;
  if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(cp.bytes / kTile * pg * np));
  __syncwarp();
  const int lp0 = t * (kTile / pg);
  for (int i = lane; i < np; i += 32) {
    const int z = page_of(a, b, lp0 + i) * a.H + h;
    for (int c = 0; c < cp.n; ++c)
      tma_load_3d(dst + cp.off[c] + i * pg * cp.width[c] * 2, map_of(c), fb, cp.start[c], 0, z);
  }
}

// Row of token j of unit (b, h) for the fp32 kernels (LLA-2D: one latent per token).
__device__ __forceinline__ int64_t f32_row(const DecodeArgs& a, int b, int h, int64_t j) {
  if (a.shared_latent) return static_cast<int64_t>(b) * a.L_max + j;
  return latent_row(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max, a.H, b, h, j, a.status);
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

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}

// Query operand of the score MMA for every (sequence, head) unit, written as the
// exact shared-memory image the decode kernel copies in with one bulk transfer:
// Z in the K-chunk layout (swizzled like a latent K tile), then the bias operand
// (128 rows x 16 bf16, 32B swizzle).  With q' = RoPE(q, q_pos) and the frequency
// pair (i0, i1) of f < 64:
//   row f      :  Z_f    = sc * (q'_i0 W_i0 + q'_i1 W_i1),  bias sc * (q'_i0 mu_i0 + q'_i1 mu_i1)
//   row 64 + f :  Z_64+f = sc * (q'_i1 W_i0 - q'_i0 W_i1),  bias sc * (q'_i1 mu_i0 - q'_i0 mu_i1)
// so that s_j = sum_f cos(j th_f) U_f + sin(j th_f) U_{64+f} with U = c_j Z^T + bias,
// which equals log2(e) * RoPE(q,q_pos).RoPE(k_j, j) / sqrt(d) for k_j of Eq. (3)
// (sc = log2(e) / sqrt(d)).  The bias is split into bf16 hi (column 0) and lo
// (column 1).  Block = unit: threads 0..63 form sc * q' of each frequency pair and
// write the bias rows; then items (row pair f, 8-column group g), consecutive in g,
// so a warp loads contiguous W row segments and writes whole swizzled rows.
constexpr int kZThreads = 256;
__global__ void __launch_bounds__(kZThreads) decode_z_kernel(const __grid_constant__ DecodeArgs a) {
  // launched as a programmatic dependent of whatever precedes the call on the
  // stream: nothing is read before that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the decode kernel may start its set-up now; it waits for this grid before
  // it reads an image
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float qs[2][64];   // sc * q'_i0, sc * q'_i1 per frequency
  const DecodePlan& P = a.plan;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int b = u / a.H, h = u % a.H;
  if (h == 0) check_block_table(a, b, tid, kZThreads);
  if (clamp_len(__ldg(a.seq_lens + b), a.L_max) == 0) return;
  uint8_t* img = a.zimg + static_cast<int64_t>(u) * a.zimg_stride;
  const __nv_bfloat16* W =
      static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * a.r_k;
  const int ng = a.r_k / 8;
  constexpr int kItems = 64 * 32 / kZThreads;   // items per thread at r_k = 256
  uint4 ra[kItems], rb[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) {   // every load in flight before any use
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
    const float* mu = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
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
    uint8_t* ab = img + P.kplan.bytes;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int e = f + 64 * half;
      const __nv_bfloat16 zh = __float2bfloat16_rn(bias[half]);
      const __nv_bfloat16 zl = __float2bfloat16_rn(bias[half] - __bfloat162float(zh));
      const uint32_t pair = bf16x2_bits(__halves2bfloat162(zh, zl));
      *reinterpret_cast<uint4*>(ab + swizzle_offset(e * 32, 32)) = make_uint4(pair, 0, 0, 0);
      *reinterpret_cast<uint4*>(ab + swizzle_offset(e * 32 + 16, 32)) = make_uint4(0, 0, 0, 0);
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
    uint32_t z0[4], z1[4];   // rows f and 64 + f
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      z0[t] = bf16x2_bits(__floats2bfloat162_rn(q0 * wa[2 * t] + q1 * wb[2 * t],
                                                q0 * wa[2 * t + 1] + q1 * wb[2 * t + 1]));
      z1[t] = bf16x2_bits(__floats2bfloat162_rn(q1 * wa[2 * t] - q0 * wb[2 * t],
                                                q1 * wa[2 * t + 1] - q0 * wb[2 * t + 1]));
    }
    int c = 0;
    while (c + 1 < P.kplan.n && k >= P.kplan.start[c + 1]) ++c;
    const int rbytes = P.kplan.width[c] * 2;
    const int col = (k - P.kplan.start[c]) * 2;
    uint8_t* zc = img + P.kplan.off[c];
    *reinterpret_cast<uint4*>(zc + swizzle_offset(f * rbytes + col, rbytes)) = make_uint4(z0[0], z0[1], z0[2], z0[3]);
    *reinterpret_cast<uint4*>(zc + swizzle_offset((f + 64) * rbytes + col, rbytes)) =
        make_uint4(z1[0], z1[1], z1[2], z1[3]);
  }
}

// kPage: 0 dense cache, 1 page pool with a tile inside one page (pages of a multiple
// of 128 tokens), 2 page pool with tiles cut into page pieces (pages of 8..64 tokens)
template <int kPage>
__global__ void __launch_bounds__(kDecodeThreads, 1)
decode_bf16_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ DecodeMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  // swizzle atoms need 1024-byte alignment in the shared window itself
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const DecodePlan& P = a.plan;
  const uint32_t sbase = smem_u32(sm);
  DecodeMisc* misc = reinterpret_cast<DecodeMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------- work range
  {
    const int per_thr = (a.B + kDecodeThreads - 1) / kDecodeThreads;
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
      int v[kDecodeThreads / 32];
      int s = 0;
#pragma unroll
      for (int i = 0; i < kDecodeThreads / 32; ++i) { v[i] = misc->scan[lane * (kDecodeThreads / 32) + i]; s += v[i]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int excl = incl - s;
#pragma unroll
      for (int i = 0; i < kDecodeThreads / 32; ++i) { misc->scan[lane * (kDecodeThreads / 32) + i] = excl; excl += v[i]; }
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

  // ---------------------------------------------------------- set-up
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    // Test hook of the timeout path: while word 1 of the status block holds
    // LLA_TEST_STALL, the first weights barrier expects one arrival more than the four
    // epilogue warps give, so the value-MMA issuer's bounded wait on it expires (the
    // kernel records LLA_ERR_TIMEOUT and every role returns).
    const uint32_t stall = __ldcg(a.status + 1) == LLA_TEST_STALL ? 1u : 0u;
    for (int s = 0; s < P.SK; ++s) { mbar_init(bar(misc->kfull[s]), 1); mbar_init(bar(misc->kempty[s]), 1); }
    for (int s = 0; s < P.SV; ++s) { mbar_init(bar(misc->vfull[s]), 1); mbar_init(bar(misc->vempty[s]), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(misc->ufull[i]), 1);
      mbar_init(bar(misc->pfull[i]), 4 + (i == 0 ? stall : 0u));
      mbar_init(bar(misc->vdone[i]), 1);
      mbar_init(bar(misc->zfull[i]), 1);
      mbar_init(bar(misc->zfree[i]), 1);
    }
    mbar_init(bar(misc->mma_done[0]), 1);
    mbar_init(bar(misc->mma_done[1]), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 3; ++i) prefetch_tmap(&maps.k[i]);
    prefetch_tmap(&maps.v);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&misc->tmem_base), 512);
  }
  if (warp >= 2 && warp < 6) {
    // constant bias operand: columns 0 and 1 of every row are 1 (they meet bias hi / lo)
    const int et = tid - 64;
    const uint32_t ones = bf16x2_bits(__floats2bfloat162_rn(1.f, 1.f));
    *reinterpret_cast<uint4*>(sm + P.aug_a + swizzle_offset(et * 32, 32)) = make_uint4(ones, 0, 0, 0);
    *reinterpret_cast<uint4*>(sm + P.aug_a + swizzle_offset(et * 32 + 16, 32)) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the combine grid may be scheduled now; it waits for this grid to complete
  // before it reads a record
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = misc->tmem_base;
  const uint32_t v_ring = sbase + P.v_ring, k_ring = sbase + P.k_ring;

  if (warp == 0) {
    // ======================================================== TMA producer
    // Per unit: its query-operand image (built by decode_z_kernel) into Z buffer
    // unit % NZ once the score MMAs of the buffer's previous unit are done.  Per
    // tile: K tile i, then V tile i - vlag (a V stage is held until the tile's
    // softmax weights exist, so it is filled as late as still hides the load).
    // With page pieces the whole warp runs the loop (lane 0 waits and the warp
    // follows its decision) and each lane issues one page's boxes.
    constexpr bool kWarp = kPage == 2;
    auto pwait = [&](uint32_t b, uint32_t parity) -> bool {
      if constexpr (kWarp) return warp_wait(b, parity, abort, a.status);
      else return mbar_wait(b, parity, abort, a.status);
    };
    if (lane == 0 || kWarp) {
      Walker wk = start, wv = start;
      int issued_k = 0, issued_v = 0, issued_z = 0, unit = -1;
      RingPos kr, vr, zr;
      for (int i = 0; i < count + P.vlag; ++i) {
        if (i < count) {
          if (i == 0 || wk.t == 0) {
            if (++unit > 0) zr.next(P.NZ);
            const int zb = zr.slot;
            if (unit >= P.NZ && !pwait(bar(misc->zfree[zb]), zr.phase ^ 1u)) break;
            // images written.  Only the producer waits for decode_z_kernel's grid, so
            // nothing that grid writes (images, the status word) may be read by another
            // warp of this kernel: the others see its output only through these copies.
            if (unit == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
            if (!kWarp || lane == 0) {
              const uint32_t zf = bar(misc->zfull[zb]);
              mbar_arrive_expect_tx(zf, P.kplan.bytes + 4096);
              const uint8_t* img = a.zimg + static_cast<int64_t>(wk.b * a.H + wk.h) * a.zimg_stride;
              bulk_load(sbase + P.z + zb * P.z_stage, img, P.kplan.bytes, zf);
              bulk_load(sbase + P.aug_b + zb * 4096, img + P.kplan.bytes, 4096, zf);
            }
            issued_z = unit + 1;
          }
          const int sk = kr.slot;
          if (!pwait(bar(misc->kempty[sk]), kr.phase ^ 1u)) break;
          const uint32_t kb = bar(misc->kfull[sk]);
          if constexpr (kPage != 0) {
            paged_tile_load<kPage == 2>(a, wk.b, wk.h, wk.t, wk.L, k_ring + sk * P.k_stage, kb, P.kplan,
                            [&](int c) { return &maps.k[chunk_map_index(P.kplan.width[c])]; });
          } else {
            mbar_arrive_expect_tx(kb, P.kplan.bytes);
            const int y = wk.t * kTile, z = wk.b * a.H + wk.h;
            for (int c = 0; c < P.kplan.n; ++c)
              tma_load_3d(k_ring + sk * P.k_stage + P.kplan.off[c], &maps.k[chunk_map_index(P.kplan.width[c])],
                          kb, P.kplan.start[c], y, z);
          }
          issued_k = i + 1;
          kr.next(P.SK);
          walker_advance(wk, a);
        }
        const int j = i - P.vlag;
        if (j >= 0) {
          const int sv = vr.slot;
          if (!pwait(bar(misc->vempty[sv]), vr.phase ^ 1u)) break;
          const uint32_t vb = bar(misc->vfull[sv]);
          const uint32_t vs = v_ring + sv * P.v_stage;
          if constexpr (kPage == 2) {
            if (a.v_page_major) {
              // one box per page holding tokens below the length: [chunk][P rows][32],
              // page i of the tile at i * (chunks * P * 64) bytes (lane i issues page i)
              const int pg = a.page_size;
              const uint32_t region = static_cast<uint32_t>(P.vplan.n * pg * 64);
              const int np = (min(kTile, wv.L - wv.t * kTile) + pg - 1) / pg;
              if (lane == 0) mbar_arrive_expect_tx(vb, region * np);
              __syncwarp();
              const int lp0 = wv.t * (kTile / pg);
              for (int i = lane; i < np; i += 32)
                tma_load_4d(vs + i * region, &maps.v4, vb, 0, 0, 0, page_of(a, wv.b, lp0 + i) * a.H + wv.h);
            } else {
              paged_tile_load<true>(a, wv.b, wv.h, wv.t, wv.L, vs, vb, P.vplan, [&](int) { return &maps.v; });
            }
          } else if constexpr (kPage != 0) {
            paged_tile_load<false>(a, wv.b, wv.h, wv.t, wv.L, vs, vb, P.vplan, [&](int) { return &maps.v; });
          } else {
            mbar_arrive_expect_tx(vb, P.vplan.bytes);
            const int y = wv.t * kTile, z = wv.b * a.H + wv.h;
            for (int c = 0; c < P.vplan.n; ++c) tma_load_3d(vs + P.vplan.off[c], &maps.v, vb, P.vplan.start[c], y, z);
          }
          issued_v = j + 1;
          vr.next(P.SV);
          walker_advance(wv, a);
        }
      }
      // Let every copy this CTA issued land before the CTA can exit.
      auto drain = [&](uint64_t* full, int n, int issued) {
        for (int i = max(0, issued - n); i < issued; ++i) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar(full[i % n]), (i / n) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
      };
      if (lane == 0) {
        drain(misc->kfull, P.SK, issued_k);
        drain(misc->vfull, P.SV, issued_v);
        drain(misc->zfull, P.NZ, issued_z);
      }
    }
  } else if (warp == 1) {
    // ======================================================== score-MMA issuer
    // U[i & 1] = C_k(i) Z^T (+ bias).  The columns of U[i & 1] last held P(i-2),
    // the A operand of value MMA i-2 (issued by warp 6), so K(i) waits for it.
    // The whole warp runs the loop (warp-uniform descriptors); one elected lane
    // issues, and every lane polls the barriers (the vote keeps the decision uniform).
    {
      auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
      const uint32_t idesc_k = umma_idesc_bf16(128, 128, false, false);
      const uint64_t daa = umma_desc(sbase + P.aug_a, 16, 256, kSw32);
      const uint32_t kst = static_cast<uint32_t>(P.k_stage) >> 4;
      Walker w = start;
      int unit = -1;
      RingPos kr, zr;
      for (int i = 0; i < count; ++i, kr.next(P.SK)) {
        if (i == 0 || w.t == 0) {
          if (++unit > 0) zr.next(P.NZ);
          if (!agree(mbar_wait(bar(misc->zfull[zr.slot]), zr.phase, abort, a.status))) break;
        }
        const int sk = kr.slot, ub = i & 1, zb = zr.slot;
        if (!agree(mbar_wait(bar(misc->kfull[sk]), kr.phase, abort, a.status))) break;
        if (i >= 2 && !agree(mbar_wait(bar(misc->vdone[ub]), ((i - 2) >> 1) & 1, abort, a.status))) break;
        tc_fence_after();
        const uint32_t d = tmem + ub * 128;
        const uint32_t so = sk * kst;
        const uint32_t zreg = sbase + P.z + zb * P.z_stage;
        uint32_t acc = 0;
        for (int c = 0; c < P.kplan.n; ++c) {
          const int rb = P.kplan.width[c] * 2;
          const uint32_t lay = sw_mode_for_row_bytes(rb);
          const uint64_t a0 = umma_desc(k_ring + P.kplan.off[c], 16, 8 * rb, lay) + so;
          const uint64_t b0 = umma_desc(zreg + P.kplan.off[c], 16, 8 * rb, lay);
          for (int k = 0; k < P.kplan.width[c] / 16; ++k) {
            umma_bf16_warp(d, a0 + 2 * k, b0 + 2 * k, idesc_k, acc);
            acc = 1;
          }
        }
        umma_bf16_warp(d, daa, umma_desc(sbase + P.aug_b + zb * 4096, 16, 256, kSw32), idesc_k, 1);
        umma_commit_warp(bar(misc->kempty[sk]));
        umma_commit_warp(bar(misc->ufull[ub]));
        if (w.t == w.nb - 1) umma_commit_warp(bar(misc->zfree[zb]));   // unit's Z no longer read
        walker_advance(w, a);
      }
      // this warp's MMAs complete before TMEM is released
      umma_commit_warp(bar(misc->mma_done[0]));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->mma_done[0]), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == kWarpVMma) {
    // ======================================================== value-MMA issuer
    // D += P(j) C_v(j): P(j) from TMEM (written by the epilogue over U[j & 1]), the
    // V tile as the MN-major B operand.  The accumulator is never cleared by an
    // MMA: the epilogue zeroes it when a unit starts.  Whole warp, as above.
    {
      auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
      const uint32_t idesc_v = umma_idesc_bf16(128, a.r_v, false, true);
      // 32-column chunks 8 KB apart (LBO), 8 token rows 512 B apart (SBO); a
      // 16-token K step is +1 KB (+64 in the address field)
      const uint64_t dv0 = umma_desc(v_ring, kTile * 64, 512, kSw64);
      const uint32_t vst = static_cast<uint32_t>(P.v_stage) >> 4;
      Walker wv = start;
      RingPos vr;
      for (int j = 0; j < count; ++j, vr.next(P.SV)) {
        const int sv = vr.slot, jb = j & 1;
        if (!agree(mbar_wait(bar(misc->vfull[sv]), vr.phase, abort, a.status))) break;
        if (!agree(mbar_wait(bar(misc->pfull[jb]), (j >> 1) & 1, abort, a.status))) break;
        // rows past the sequence end: skip whole 16-token steps, zero the rest of a
        // partial step (they may hold anything; their weights are 0 and 0 * x stays 0)
        const int valid = wv.L - wv.t * kTile;
        const int steps = valid >= kTile ? kTile / 16 : (valid + 15) / 16;
        if (valid < steps * 16) {
          uint8_t* vs = sm + P.v_ring + sv * P.v_stage;
          const int per_c = (steps * 16 - valid) * 4;
          for (int x = lane; x < P.vplan.n * per_c; x += 32) {
            const int c = x / per_c, r = valid + (x - c * per_c) / 4, g = x & 3;
            if constexpr (kPage == 2) {
              if (a.v_page_major) {   // page-major: page r / P, chunk c, row r % P
                const int pg = a.page_size;
                *reinterpret_cast<uint4*>(vs + (r / pg) * (P.vplan.n * pg * 64) + c * pg * 64 +
                                          swizzle_offset((r % pg) * 64 + g * 16, 64)) = make_uint4(0, 0, 0, 0);
                continue;
              }
            }
            *reinterpret_cast<uint4*>(vs + P.vplan.off[c] + swizzle_offset(r * 64 + g * 16, 64)) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        const uint32_t pa = tmem + jb * 128;
        if constexpr (kPage == 2) {
          if (a.v_page_major) {
            // page-major V: chunks P * 64 B apart (LBO); 8-row groups 512 B apart within
            // a page of >= 16 rows, one page region apart with 8-row pages (SBO); the
            // 16-token K step k starts at page 16 k / P, row 16 k % P
            const int pg = a.page_size;
            const uint32_t region = static_cast<uint32_t>(P.vplan.n * pg * 64);
            const uint64_t dpm = umma_desc(v_ring + sv * P.v_stage, static_cast<uint32_t>(pg * 64),
                                           pg >= 16 ? 512u : region, kSw64);
            for (int k = 0; k < steps; ++k) {
              const uint32_t off = static_cast<uint32_t>((16 * k) / pg) * region + static_cast<uint32_t>((16 * k) % pg) * 64;
              umma_bf16_ts_warp(tmem + kDCol, pa + 8 * k, dpm + (off >> 4), idesc_v, 1u);
            }
          } else {
            const uint64_t b0 = dv0 + sv * vst;
            for (int k = 0; k < steps; ++k) umma_bf16_ts_warp(tmem + kDCol, pa + 8 * k, b0 + 64 * k, idesc_v, 1u);
          }
        } else {
          const uint64_t b0 = dv0 + sv * vst;
          for (int k = 0; k < steps; ++k) umma_bf16_ts_warp(tmem + kDCol, pa + 8 * k, b0 + 64 * k, idesc_v, 1u);
        }
        umma_commit_warp(bar(misc->vempty[sv]));
        umma_commit_warp(bar(misc->vdone[jb]));
        walker_advance(wv, a);
      }
      umma_commit_warp(bar(misc->mma_done[1]));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->mma_done[1]), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    // ======================================================== epilogue (warps 2-5)
    const int q = warp & 3;             // TMEM lane quadrant of this warp
    const int row = 32 * q + lane;      // token row within a tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // this warp's copy of the tile's RoPE base row: cos[64] then sin[64]
    float* trig = reinterpret_cast<float*>(sm + P.trig + q * 512);

    // cos/sin(row * th_f): the tile-local half of the angle-sum rotation
    float cl[64], sl[64];
#pragma unroll
    for (int f = 0; f < 64; f += 4) {
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(a.rope_cos + row * 64 + f));
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(a.rope_sin + row * 64 + f));
      cl[f] = c4.x; cl[f + 1] = c4.y; cl[f + 2] = c4.z; cl[f + 3] = c4.w;
      sl[f] = s4.x; sl[f + 1] = s4.y; sl[f + 2] = s4.z; sl[f + 3] = s4.w;
    }

    auto zero_acc = [&]() {
      float zf[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) zf[k] = 0.f;
      for (int c = 0; c < a.r_v; c += 32) tmem_st_x32(tmem + lane_base + kDCol + c, zf);
      tmem_wait_st();
    };
    auto load_trig = [&](int t, float (&v)[4]) {
      const int64_t o = static_cast<int64_t>(t) * kTile * 64;
      v[0] = __ldg(a.rope_cos + o + lane);
      v[1] = __ldg(a.rope_cos + o + 32 + lane);
      v[2] = __ldg(a.rope_sin + o + lane);
      v[3] = __ldg(a.rope_sin + o + 32 + lane);
    };
    auto store_trig = [&](const float (&v)[4]) {
      __syncwarp();
      trig[lane] = v[0]; trig[32 + lane] = v[1]; trig[64 + lane] = v[2]; trig[96 + lane] = v[3];
      __syncwarp();
    };

    Walker w = start;
    zero_acc();
    {
      float tv[4];
      load_trig(w.t, tv);
      store_trig(tv);
    }

    int cur_b = w.b, cur_h = w.h;
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;

    // Read out this warp's accumulator rows of a finished unit (its last value MMA
    // was tile `last`), sum them over the warp's 32 token rows and write the
    // warp's record (m, l, acc_v).
    auto finalize = [&](int last, int b, int h, float m, float l) -> bool {
      if (!warp_wait(bar(misc->vdone[last & 1]), (last >> 1) & 1, abort, a.status)) return false;
      tc_fence_after();
      const float lw = warp_sum(l);
      const long long u = static_cast<long long>(b) * a.H + h;
      float* rec = a.partials + ((u + blockIdx.x) * kRecordsPerCta + q) * (a.r_v + kRecordHead);
      if (lane == 0) { rec[0] = m; rec[1] = lw; }
      for (int c = 0; c < a.r_v; c += 32) {
        float v[32];
        tmem_ld_x32(tmem + lane_base + kDCol + c, v);
        tmem_wait_ld();
        const float col = warp_column_sum32(v);
        if (c + lane < a.r_v) rec[kRecordHead + c + lane] = col;
      }
      return true;
    };

    Walker wn = w;
    walker_advance(wn, a);
    for (int i = 0; i < count && ok; ++i) {
      const bool first = i > 0 && w.t == 0;   // a unit starts at tile i (not the CTA's first)
      float tn[4];
      if (i + 1 < count) load_trig(wn.t, tn);   // next tile's base row, used after this score
      const int ub = i & 1;
      if (!(ok = warp_wait(bar(misc->ufull[ub]), (i >> 1) & 1, abort, a.status))) break;
      tc_fence_after();

      // ---- rotary score from U, 32 frequencies at a time
      const float4* tcos = reinterpret_cast<const float4*>(trig);
      const float4* tsin = tcos + 16;
      const uint32_t tU = tmem + lane_base + ub * 128;
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float u1[32], u2[32];
        tmem_ld_x32(tU + 32 * h2, u1);
        tmem_ld_x32(tU + 64 + 32 * h2, u2);
        tmem_wait_ld();
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          const float4 cb = tcos[8 * h2 + k4], sb = tsin[8 * h2 + k4];
          const float cbv[4] = {cb.x, cb.y, cb.z, cb.w};
          const float sbv[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int f = 32 * h2 + 4 * k4 + kk, k = 4 * k4 + kk;
            const float c = fmaf(cbv[kk], cl[f], -sbv[kk] * sl[f]);   // cos((j0+row) th_f)
            const float sn = fmaf(sbv[kk], cl[f], cbv[kk] * sl[f]);   // sin((j0+row) th_f)
            s4[kk] = fmaf(c, u1[k], s4[kk]);
            s4[kk] = fmaf(sn, u2[k], s4[kk]);
          }
        }
      }
      if (i + 1 < count) store_trig(tn);

      // ---- a new unit: read out the finished one once its last value MMA is done
      // (no value MMA of the new unit can start before this warp's P arrives), then
      // clear the accumulator row for the new unit
      if (first) {
        if (!(ok = finalize(i - 1, cur_b, cur_h, m_ref, l_run))) break;
        zero_acc();
        cur_b = w.b; cur_h = w.h;
        m_ref = -INFINITY; l_run = 0.f;
      }

      // ---- online softmax (log2 domain, lazy per-warp reference)
      const bool valid = w.t * kTile + row < w.L;
      const float s = valid ? (s4[0] + s4[1]) + (s4[2] + s4[3]) : -INFINITY;
      const float m_tile = warp_max_redux(s);
      if (m_tile > m_ref + kRescaleLog2) {
        if (m_ref != -INFINITY) {
          // the accumulator row must be at rest: V(i-1) complete (V(i-2) already is,
          // as K(i) was issued after it and we hold U(i))
          if (!(ok = warp_wait(bar(misc->vdone[(i - 1) & 1]), ((i - 1) >> 1) & 1, abort, a.status))) break;
          tc_fence_after();
          const float alpha = exp2f(m_ref - m_tile);
          // (16 columns at a time: a small body keeps the per-tile loop compact)
          for (int c = 0; c < a.r_v; c += 16) {
            float v[16];
            tmem_ld_x16(tmem + lane_base + kDCol + c, v);
            tmem_wait_ld();
            uint32_t w16[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) w16[k] = __float_as_uint(v[k] * alpha);
            tmem_st_x16(tmem + lane_base + kDCol + c, w16);
          }
          tmem_wait_st();
          l_run *= alpha;
        }
        m_ref = m_tile;
      }
      const float p = valid ? exp2f(s - m_ref) : 0.f;
      const __nv_bfloat16 pb = __float2bfloat16_rn(p);
      l_run += __bfloat162float(pb);

      // ---- P = diag(p) over this warp's rows, into TMEM over the consumed scores:
      // row 32q + lane holds its own weight at token column 32q + lane (bf16 pairs:
      // column 16q + lane/2, low half for even lanes), every other entry is zero.
      // The value MMA then adds p_j c_v,j to accumulator row j; rows are summed
      // once per unit.
      {
        const uint32_t pbits = static_cast<uint32_t>(__bfloat16_as_ushort(pb)) << ((lane & 1) * 16);
        uint32_t mine[16], zero[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          mine[c] = c == (lane >> 1) ? pbits : 0u;
          zero[c] = 0u;
        }
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) tmem_st_x16(tU + 16 * blk, blk == q ? mine : zero);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(misc->pfull[ub]));

      walker_advance(w, a);
      walker_advance(wn, a);
    }
    if (ok) finalize(count - 1, cur_b, cur_h, m_ref, l_run);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge each (sequence, head) unit's split records (log-sum-exp merge of the
// per-CTA, per-warp (m, l, acc_v) triples), apply the V up-projection once
// (Appendix J identity) and normalise:
//   out = (sum_c 2^(m_c - M) acc_c) W_up,v,t^T / (sum_c 2^(m_c - M) l_c) + mu_v,t.
// Block = (head h, kCombineUnits consecutive sequences).  Before the wait for the
// decode grid it copies W_up,v,t[h] to shared memory (coalesced, rows padded by
// one word so that thread e reading row e is conflict-free) and derives the tile
// prefix of its sequences from seq_lens; after it, warp w merges the records of
// units w and w + 8 (one batch of loads per 8 records), and thread (half, e) forms
// output e of the half's 8 units.  Up to sixteen units per block (a.combine_units,
// sized by the launcher so that the grid still fills the GPU) share the W staging
// and keep the number of small, latency-bound blocks low at serving batch sizes.
constexpr int kCombineUnits = 16;

// W_up,v rows padded to r_v / 2 + 4 words: 16-byte aligned, and eight threads
// reading eight consecutive rows at one column touch 32 distinct banks.
size_t combine_smem_bytes(int r_v, int units) {
  return (static_cast<size_t>(128) * (r_v / 2 + 4) + units * 256 + 2 * units) * 4;
}

// d = a * b + d on a pair of fp32 lanes (one packed instruction).
__device__ __forceinline__ void fma_pair(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mov.b64 pd, {%0, %1};\n\tfma.rn.f32x2 pd, pa, pb, pd;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// kCombineThreads = 128: at most 4 units per block (small batches); 256: up to 16.
// NJ: record columns per lane (r_v <= 32 NJ).
template <int kCombineThreads, int NJ>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const __grid_constant__ DecodeArgs a) {
  // the next call's image grid may be scheduled now; it waits for this grid to
  // complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kCombineWarps = kCombineThreads / 32;
  extern __shared__ float csm[];
  __shared__ int red[kCombineThreads / 32];
  const int cu = a.combine_units;
  const int h = blockIdx.x, b0 = blockIdx.y * cu;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rw = a.r_v / 2, wpr = rw + 4;   // words per W row, per padded row
  uint32_t* Ws = reinterpret_cast<uint32_t*>(csm);
  float* accs = csm + 128 * wpr;                   // [cu][256]
  float* Ms = accs + cu * 256;
  float* Ls = Ms + cu;

  // ---- inputs only: W_up,v,t[h] -> shared memory; tiles of sequences < b0 and in total
  {
    const uint4* Wg = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w_up_v) +
                                                     static_cast<int64_t>(h) * kHeadDim * a.r_v);
    const int n16 = 128 * rw / 4;             // 16-byte pieces; a row holds rw / 4 of them
    constexpr int kMax = 128 * 128 / 4 / kCombineThreads;   // at r_v = 256
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
        *reinterpret_cast<uint4*>(Ws + e * wpr + k) = v[j];
      }
    }
  }
  int before = 0, all = 0;   // tiles of sequences [0, b0) and [0, B)
  for (int bb = tid; bb < a.B; bb += kCombineThreads) {
    const int n = (clamp_len(__ldg(a.seq_lens + bb), a.L_max) + kTile - 1) / kTile;
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

  // ---- inputs only: where each of this warp's units (b0 + w, h), (b0 + w + 8, h)
  // has its records, and this thread's mu
  // Tile-major split (per-head kernel): CTA ranges over the flat (sequence, head,
  // tile) list, records ((b H + h) + c) R + warp.  Position-major split (small-rank
  // kernels): ranges over (sequence, tile) with every head inner, records
  // ((b + c) H + h) R + warp.  R = 4 (one per epilogue warp), 8 (decoupled tile-major
  // tensor-core kernel: two groups of four) or 1 (decoupled CUDA-core kernel: its
  // warps are merged within the CTA).  A unit's records: one per (CTA c
  // in [c0, c1], epilogue warp); a warp that saw no token of the unit in that CTA
  // wrote m = -inf, l = 0, acc = 0.  (CTA ranges are [c per, (c + 1) per): only CTAs
  // past the last tile are empty, never one between c0 and c1.)
  constexpr int kUPW = kCombineThreads == 256 ? 2 : 1;   // units per warp (cu <= 16 / <= 4)
  const int R = a.records_per_cta, rsh = R == 8 ? 3 : R == 4 ? 2 : 0;   // R is 8, 4 or 1
  const int rs = a.r_v + kRecordHead;
  const long long cstride = a.pos_major ? static_cast<long long>(R) * a.H : R;
  long long ubase[kUPW];
  int unrec[kUPW];
#pragma unroll
  for (int q = 0; q < kUPW; ++q) {
    const int ui = warp + q * kCombineWarps, b = b0 + ui;
    ubase[q] = 0;
    unrec[q] = 0;
    if (ui >= cu || b >= a.B) continue;
    int pb = pre;   // tiles of sequences before b
    for (int bb = b0; bb < b; ++bb) pb += (clamp_len(__ldg(a.seq_lens + bb), a.L_max) + kTile - 1) / kTile;
    const int nb = (clamp_len(__ldg(a.seq_lens + b), a.L_max) + kTile - 1) / kTile;
    if (nb == 0) continue;
    const long long total = a.pos_major ? tot : static_cast<long long>(a.H) * tot;
    const long long per = max(1LL, (total + a.grid - 1) / a.grid);
    const long long F0 = a.pos_major ? pb : static_cast<long long>(a.H) * pb + static_cast<long long>(h) * nb;
    const long long F1 = F0 + nb - 1;
    const int c0 = static_cast<int>(F0 / per), c1 = static_cast<int>(F1 / per);
    const long long u = static_cast<long long>(b) * a.H + h;
    ubase[q] = a.pos_major ? ((b + c0) * static_cast<long long>(a.H) + h) * R : (u + c0) * R;
    unrec[q] = R * (c1 - c0 + 1);
  }
  const int e = tid & (kHeadDim - 1);
  const float mu = __ldg(a.mu_v + static_cast<int64_t>(h) * a.mu_hstride + e);

  asm volatile("griddepcontrol.wait;" ::: "memory");   // records written

  // ---- warp w merges the records of its units
#pragma unroll
  for (int q = 0; q < kUPW; ++q) {
    const int ui = warp + q * kCombineWarps;
    if (ui >= cu) break;
    float M = -INFINITY, Lt = 0.f;
    float acc[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) acc[j] = 0.f;
    const long long base = ubase[q];
    const int nrec = unrec[q];
    // record r of the unit: CTA c0 + r / R, warp r % R
    auto rec_at = [&](int r) { return a.partials + (base + (r >> rsh) * cstride + (r & (R - 1))) * rs; };
    for (int cb = 0; cb < nrec; cb += 8) {
      // heads (m, l) of records cb..cb+7 in lanes 0..7, and this lane's columns
      // lane + 32 j of each, all in one round of loads
      const int cl = cb + (lane & 7);
      const float mh = cl < nrec ? rec_at(cl)[0] : -INFINITY;
      const float lh = cl < nrec ? rec_at(cl)[1] : 0.f;
      float x[8][NJ];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int col = lane + 32 * j;
          x[r][j] = cb + r < nrec && col < a.r_v ? rec_at(cb + r)[kRecordHead + col] : 0.f;
        }
      const float Mn = fmaxf(M, warp_max(mh));
      if (Mn != -INFINITY) {
        const float alpha = M == -INFINITY ? 0.f : exp2f(M - Mn);
        Lt *= alpha;
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[j] *= alpha;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float mr = __shfl_sync(0xffffffffu, mh, r), lr = __shfl_sync(0xffffffffu, lh, r);
          const float w = mr == -INFINITY ? 0.f : exp2f(mr - Mn);
          Lt = fmaf(lr, w, Lt);
#pragma unroll
          for (int j = 0; j < NJ; ++j) acc[j] = fmaf(x[r][j], w, acc[j]);
        }
        M = Mn;
      }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (lane + 32 * j < a.r_v) accs[ui * 256 + lane + 32 * j] = acc[j];
    if (lane == 0) { Ms[ui] = M; Ls[ui] = Lt; }
  }
  __syncthreads();

  // ---- out[b][h][e] = acc_b . W_e / Lt_b + mu_e, thread (half, e) reading row e of W
  // once; even and odd columns summed in the two lanes of a packed FMA
  constexpr int kHalf = kCombineThreads == 256 ? kCombineUnits / 2 : 4;
  const int j0 = (tid >> 7) * kHalf;
  float ox[kHalf], oy[kHalf];
#pragma unroll
  for (int j = 0; j < kHalf; ++j) { ox[j] = 0.f; oy[j] = 0.f; }
  const uint4* wr = reinterpret_cast<const uint4*>(Ws + e * wpr);
#pragma unroll 2
  for (int k4 = 0; k4 < rw / 4; ++k4) {   // columns 8 k4 .. 8 k4 + 7
    float wf[8];
    unpack_bf16x8(wr[k4], wf);
#pragma unroll
    for (int j = 0; j < kHalf; ++j) {
      if (j0 + j < cu) {   // accs holds cu units
        const float4* ap = reinterpret_cast<const float4*>(accs + (j0 + j) * 256) + 2 * k4;
        const float4 a0 = ap[0], a1 = ap[1];
        fma_pair(ox[j], oy[j], a0.x, a0.y, wf[0], wf[1]);
        fma_pair(ox[j], oy[j], a0.z, a0.w, wf[2], wf[3]);
        fma_pair(ox[j], oy[j], a1.x, a1.y, wf[4], wf[5]);
        fma_pair(ox[j], oy[j], a1.z, a1.w, wf[6], wf[7]);
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < kHalf; ++jj) {
    const int j = j0 + jj;
    const int bb = b0 + j;
    if (j >= cu || bb >= a.B) continue;
    const int64_t uu = static_cast<int64_t>(bb) * a.H + h;
    const bool empty = Ms[j] == -INFINITY;
    a.out[uu * kHeadDim + e] = empty ? 0.f : (ox[jj] + oy[jj]) / Ls[j] + mu;
    if (e == 0) a.lse[uu] = empty ? -INFINITY : (Ms[j] + log2f(Ls[j])) * kLn2;
  }
}

// ------------------------------------------------------------------ fp32 path

// Element loads of the plain path: fp32 storage, or bf16 storage widened to fp32
// (the LLA-2D shapes the CTA-pair kernels do not take).
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Scores s_j = RoPE(q).RoPE(k_j)/sqrt(d), k_j reconstructed per Eq. (3) in fp32.
// Block = (unit, 128-token tile); thread = token.
template <typename T>
__global__ void __launch_bounds__(128)
decode_f32_scores_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float qrot[kHeadDim];
  __shared__ float ct[kTile][33];       // latent tile chunk [token][32 ranks]
  __shared__ float wt[kHeadDim][33];    // W_up chunk [dim][32 ranks]
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
  const T* qv = static_cast<const T*>(a.q) + static_cast<int64_t>(u) * kHeadDim;
  if (tid < 64) {
    const int f = tid;
    const int i0 = a.rope_style == 0 ? f : 2 * f, i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
    const float c = a.rope_cos[static_cast<int64_t>(qp) * 64 + f], s = a.rope_sin[static_cast<int64_t>(qp) * 64 + f];
    const float x0 = ldf(qv + i0), x1 = ldf(qv + i1);
    qrot[i0] = x0 * c - x1 * s;
    qrot[i1] = x0 * s + x1 * c;
  }
  // token rows j0.. of the unit (paged: possibly across pages; LLA-2D: every head
  // reads the sequence's latent); rows past L are not read
  const T* C = static_cast<const T*>(a.cache_k);
  const T* W = static_cast<const T*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * a.r_k;
  const int rows = min(kTile, L - j0);
  float kh[kHeadDim];
#pragma unroll
  for (int e = 0; e < kHeadDim; ++e) kh[e] = 0.f;
  for (int k0 = 0; k0 < a.r_k; k0 += 32) {
    const int kw = min(32, a.r_k - k0);
    __syncthreads();
    for (int idx = tid; idx < kTile * 32; idx += 128) {
      const int r = idx / 32, k = idx % 32;
      ct[r][k] = (r < rows && k < kw) ? ldf(C + f32_row(a, b, h, j0 + r) * a.r_k + k0 + k) : 0.f;
      wt[r][k] = (k < kw) ? ldf(W + static_cast<int64_t>(r) * a.r_k + k0 + k) : 0.f;
    }
    __syncthreads();
    for (int k = 0; k < 32; ++k) {
      const float c = ct[tid][k];
#pragma unroll
      for (int e = 0; e < kHeadDim; ++e) kh[e] = fmaf(c, wt[e][k], kh[e]);
    }
  }
  const int j = j0 + tid;
  if (j < L) {
    const float* mu = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
    float s = 0.f;
#pragma unroll
    for (int f = 0; f < 64; ++f) {
      const int i0 = a.rope_style == 0 ? f : 2 * f, i1 = a.rope_style == 0 ? f + 64 : 2 * f + 1;
      const float k0v = kh[i0] + mu[i0], k1v = kh[i1] + mu[i1];
      const float c = a.rope_cos[static_cast<int64_t>(j) * 64 + f], sn = a.rope_sin[static_cast<int64_t>(j) * 64 + f];
      s = fmaf(qrot[i0], k0v * c - k1v * sn, s);
      s = fmaf(qrot[i1], k0v * sn + k1v * c, s);
    }
    a.scores[static_cast<int64_t>(u) * a.L_max + j] = s * kInvSqrtD;
  }
}

__device__ float block_reduce(float v, float* red, bool is_max) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < nw; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// Softmax over the unit's scores, then out = (sum_j p_j c_v,j) W_up,v,t^T / Z + mu_v,t.
template <typename T>
__global__ void __launch_bounds__(256)
decode_f32_values_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float red[8];
  __shared__ float accs[kMaxRank2d];
  const int u = blockIdx.x, tid = threadIdx.x;
  const int b = u / a.H, h = u % a.H;
  const int L = clamp_len(__ldg(a.seq_lens + b), a.L_max);
  float* out = a.out + static_cast<int64_t>(u) * kHeadDim;
  if (L == 0) {
    if (tid < kHeadDim) out[tid] = 0.f;
    if (tid == 0) a.lse[u] = -INFINITY;
    return;
  }
  float* sc = a.scores + static_cast<int64_t>(u) * a.L_max;
  float m = -INFINITY;
  for (int j = tid; j < L; j += 256) m = fmaxf(m, sc[j]);
  m = block_reduce(m, red, true);
  float z = 0.f;
  for (int j = tid; j < L; j += 256) {
    const float p = expf(sc[j] - m);
    sc[j] = p;
    z += p;
  }
  z = block_reduce(z, red, false);   // also orders the p writes before the reads below
  const T* Cv = static_cast<const T*>(a.cache_v);
  for (int rr = tid; rr < a.r_v; rr += 256) {
    float v = 0.f;
    for (int j = 0; j < L; ++j) v = fmaf(sc[j], ldf(Cv + f32_row(a, b, h, j) * a.r_v + rr), v);
    accs[rr] = v;
  }
  __syncthreads();
  if (tid < kHeadDim) {
    const T* Wv = static_cast<const T*>(a.w_up_v) + (static_cast<int64_t>(h) * kHeadDim + tid) * a.r_v;
    float o = 0.f;
    for (int i = 0; i < a.r_v; ++i) o = fmaf(accs[i], ldf(Wv + i), o);
    out[tid] = o / z + a.mu_v[static_cast<int64_t>(h) * a.mu_hstride + tid];
  }
  if (tid == 0) a.lse[u] = m + logf(z);
}

}  // namespace

bool make_decode_plan(int r_k, int r_v, DecodePlan* p) {
  *p = DecodePlan{};
  p->kplan = make_chunk_plan(r_k, kTile);
  p->vplan = make_chunk_plan_32(r_v, kTile);
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  p->k_stage = al(p->kplan.bytes, 1024);
  p->v_stage = al(p->vplan.bytes, 1024);
  p->z_stage = al(p->kplan.bytes, 1024);
  p->vlag = 1;
  // (Z buffers, K stages, V stages) in order of preference: Z built one unit
  // ahead and double-buffered rings first; single buffers only for the largest ranks.
  const int tries[5][3] = {{2, 2, 2}, {1, 2, 2}, {1, 1, 2}, {1, 2, 1}, {1, 1, 1}};
  int SK = 0, SV = 0, fixed = 0;
  for (const auto& t : tries) {
    p->NZ = t[0];
    fixed = p->NZ * p->z_stage + 4096 + 8192 + 2048 + 2048 + 1024;
    SK = t[1];
    SV = t[2];
    if (fixed + SK * p->k_stage + SV * p->v_stage <= kSmemLimit) break;
    SK = 0;
  }
  if (SK == 0) return false;
  auto fits = [&](int sk, int sv) { return fixed + sk * p->k_stage + sv * p->v_stage <= kSmemLimit; };
  // The V stage is held longest (until the value MMA, after the softmax), so
  // deepen the V ring first.
  while (true) {
    const bool tryv = SV <= SK;
    if (tryv && SV < kMaxStages && fits(SK, SV + 1)) { ++SV; continue; }
    if (SK < kMaxStages && fits(SK + 1, SV)) { ++SK; continue; }
    if (!tryv && SV < kMaxStages && fits(SK, SV + 1)) { ++SV; continue; }
    break;
  }
  p->SK = SK;
  p->SV = SV;
  int off = 0;
  p->v_ring = off; off += SV * p->v_stage;
  p->k_ring = off; off += SK * p->k_stage;
  p->z = off;      off += p->NZ * p->z_stage;
  p->aug_a = off;  off += 4096;
  p->aug_b = off;  off += 8192;
  p->trig = off;   off += 2048;
  p->misc = off;   off += 2048;
  p->bytes = off + 1024;
  return true;
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t s) {
  // the dense-cache instantiation carries no page lookup in its producer, the
  // whole-page one no piece loop
  const int page = a.block_table == nullptr ? 0 : a.page_size >= kTile ? 1 : 2;
  auto kern = page == 0 ? decode_bf16_kernel<0> : page == 1 ? decode_bf16_kernel<1> : decode_bf16_kernel<2>;
  static int configured[3] = {0, 0, 0};
  if (configured[page] < a.plan.bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, a.plan.bytes);
    if (e != cudaSuccess) return e;
    configured[page] = a.plan.bytes;
  }
  // programmatic dependent launches: the image grid is scheduled while the previous
  // grid on the stream drains (it waits for it before reading anything); the decode
  // grid's set-up overlaps the image grid; its producer waits for that grid before
  // the first image copy
  cudaError_t e = launch_pdl(decode_z_kernel, dim3(a.B * a.H), dim3(kZThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = a.plan.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a, maps);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, s);
}

int decode_combine_units(int B, int H, int sms) {
  // two units per block (128 threads) unless the batch gives more than about two
  // blocks per SM that way; then up to 16 per block (256 threads)
  const long long u = static_cast<long long>(B) * H / (2LL * (sms > 0 ? sms : 1));
  return u <= 2 ? 2 : static_cast<int>(std::min<long long>(kCombineUnits, u));
}

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t s) {
  // the combine grid, a programmatic dependent of the decode grid, copies W_up,v
  // while the decode grid drains
  const bool wide = a.combine_units > 4, narrow_v = a.r_v <= 64;
  const int which = (wide ? 2 : 0) + (narrow_v ? 1 : 0);
  void (*const kern[4])(DecodeArgs) = {decode_combine_kernel<128, 8>, decode_combine_kernel<128, 2>,
                                       decode_combine_kernel<256, 8>, decode_combine_kernel<256, 2>};
  // at least 76 KB: two blocks per SM, so the blocks, placed as the decode grid's CTAs
  // leave their SMs, spread over more of them
  const size_t csmem = std::max<size_t>(combine_smem_bytes(a.r_v, a.combine_units), 76 * 1024);
  static size_t cconfigured[4] = {0, 0, 0, 0};
  if (cconfigured[which] < csmem) {
    cudaError_t e = cudaFuncSetAttribute(kern[which], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(csmem));
    if (e != cudaSuccess) return e;
    cconfigured[which] = csmem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H, (a.B + a.combine_units - 1) / a.combine_units);
  cfg.blockDim = dim3(wide ? 256 : 128);
  cfg.dynamicSmemBytes = csmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern[which], a);
}

cudaError_t launch_decode_f32_values(const DecodeArgs& a, cudaStream_t s) {
  decode_f32_values_kernel<float><<<a.B * a.H, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t s) {
  const dim3 g1(a.B * a.H, static_cast<unsigned>((a.L_max + kTile - 1) / kTile));
  decode_f32_scores_kernel<float><<<g1, 128, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_f32_values_kernel<float><<<a.B * a.H, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_plain_bf16(const DecodeArgs& a, cudaStream_t s) {
  const dim3 g1(a.B * a.H, static_cast<unsigned>((a.L_max + kTile - 1) / kTile));
  decode_f32_scores_kernel<__nv_bfloat16><<<g1, 128, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_f32_values_kernel<__nv_bfloat16><<<a.B * a.H, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lla
