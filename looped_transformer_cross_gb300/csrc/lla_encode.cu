// lla_encode.cu — the cross-loop encode of Looped Latent Attention on sm_103a
// ("Looped Latent Attention: Cross-Loop KV Compression for Looped
// Transformers", arXiv 2607.15456v2, §3 Eq. (1)-(2)):
//     c = (x - mu) W_down ,  x = [x_1; ...; x_T] in R^{T d}
// for every token and head, written into the token's cache slot.
//
// bf16 path: a persistent grid (one CTA per SM) over units of (128-token tile,
// head, axis K/V).  TMA streams 64-wide K-slices of x (K-major) and W_down
// (MN-major) through a ring that runs on across units; warp 1 issues tcgen05
// MMAs accumulating x W_down in one of two TMEM accumulators; four epilogue warps
// (one token per TMEM lane) subtract mu W_down (computed once per call by a small
// kernel), round to bf16 and store the latent row while the next unit's MMAs
// fill the other accumulator.  Computing x W - mu W
// instead of (x - mu) W is exact in real arithmetic.
//
// fp32 path: one block per (token, head, axis), the literal sum in fp32.
#include "lla_kernels.h"

namespace lla {

namespace {

struct alignas(16) EncodeMisc {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t dfull[2], dempty[2];     // accumulator full (MMA commit) / drained (epilogue)
  uint64_t mdone;                    // every MMA of the CTA complete
  uint32_t tmem_base;
  int abort;
};

// bias[axis][h][k] = sum_u mu[h][u] * W_down[h][u][k]  (fp32).  Block = (head,
// axis, 256-column half): warp w sums rows u = w, w + 8, ...; lane l covers columns
// 8l..8l+7 of the half with 16-byte loads, sixteen rows in flight; the eight warps'
// partial sums are added in shared memory.
__global__ void __launch_bounds__(256) encode_bias_kernel(const __grid_constant__ EncodeArgs a) {
  __shared__ float part[8][256];
  const int h = blockIdx.x, axis = blockIdx.y, k0 = 256 * blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = axis == 0 ? a.r_k : a.r_v;
  if (k0 >= r) return;
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(axis == 0 ? a.w_down_k : a.w_down_v) +
                           static_cast<int64_t>(h) * a.Td * r;
  const float* mu = (axis == 0 ? a.mu_k : a.mu_v) + static_cast<int64_t>(h) * a.Td;
  const int k = k0 + 8 * lane;
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
    for (int t = 0; t < 8; ++t) part[warp][8 * lane + t] = acc[t];
  }
  __syncthreads();
  const int t = threadIdx.x;
  if (k0 + t < r) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][t];
    a.bias[(static_cast<int64_t>(axis) * a.H + h) * kMaxRank2d + k0 + t] = s;
  }
}

__device__ __forceinline__ bool slot_ok(const EncodeArgs& a, int sid, int p) {
  return sid >= 0 && sid < a.B && p >= 0 && p < a.L_max;
}

// Unit u of the persistent schedule: (token tile, head, axis), heads fastest, then
// the axis, then the tile, so the CTAs running at one time read neighbouring rows
// of x (one token's heads are contiguous).
struct EncodeUnit {
  int tile, h, axis;
};

__device__ __forceinline__ EncodeUnit encode_unit(int64_t u, int H) {
  EncodeUnit e;
  e.h = static_cast<int>(u % H);
  const int64_t q = u / H;
  e.axis = static_cast<int>(q & 1);
  e.tile = static_cast<int>(q >> 1);
  return e;
}

// MMA runs per axis: 64-wide W chunks grouped up to N = 256, then a 32- and a
// 16-wide chunk (ranks up to 512 need four).
constexpr int kRuns = 4;

// Persistent: one CTA per SM walks units blockIdx.x, blockIdx.x + gridDim.x, ...
// The x / W_down ring runs on across units (its position is the count of k-blocks
// this CTA has issued), and two TMEM accumulators alternate between units, so
// the epilogue of one unit overlaps the copies and MMAs of the next; ranks above
// 256 (LLA-2D) use one 512-column accumulator.
__global__ void __launch_bounds__(kEncodeThreads, 1)
encode_bf16_kernel(const __grid_constant__ EncodeArgs a, const __grid_constant__ EncodePlan P,
                   const __grid_constant__ EncodeMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  EncodeMisc* misc = reinterpret_cast<EncodeMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = a.Td / 64;
  const uint32_t S = static_cast<uint32_t>(P.S);
  const int64_t nunits = static_cast<int64_t>((a.N + 127) / 128) * a.H * 2;
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  // accumulator buffer of this CTA's j-th unit, and how often it was used before
  auto acc_buf = [&](int64_t j) { return P.nacc == 2 ? static_cast<int>(j & 1) : 0; };
  auto acc_use = [&](int64_t j) { return P.nacc == 2 ? (j >> 1) : j; };

  if (tid == 0) {
    for (int s = 0; s < P.S; ++s) { mbar_init(bar(misc->full[s]), 1); mbar_init(bar(misc->empty[s]), 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(misc->dfull[b]), 1);
      mbar_init(bar(misc->dempty[b]), 4);   // one arrive per epilogue warp
    }
    mbar_init(bar(misc->mdone), 1);
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
      uint32_t g = 0;   // k-blocks issued by this CTA: the ring position
      bool ok = true;
      for (int64_t u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const EncodeUnit e = encode_unit(u, a.H);
        const ChunkPlan& bp = e.axis == 0 ? P.bk : P.bv;
        const CUtensorMap* xmap = e.axis == 0 ? &maps.xk : &maps.xv;
        const CUtensorMap* wmaps = e.axis == 0 ? maps.wk : maps.wv;
        const uint32_t bytes = 128 * 64 * 2 + bp.bytes;
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const uint32_t s = g % S;
          if (!(ok = mbar_wait(bar(misc->empty[s]), ((g / S) & 1) ^ 1, abort, a.status))) break;
          const uint32_t fb = bar(misc->full[s]);
          mbar_arrive_expect_tx(fb, bytes);
          const uint32_t st = sbase + P.ring + s * P.stage;
          tma_load_3d(st + P.a_off, xmap, fb, kb * 64, e.h, e.tile * 128);
          for (int c = 0; c < bp.n; ++c)
            tma_load_3d(st + P.b_off + bp.off[c], &wmaps[chunk_map_index(bp.width[c])], fb, bp.start[c],
                        kb * 64, e.h);
        }
      }
      // the copies still in flight land before the CTA exits
      for (uint32_t k = g > S ? g - S : 0; k < g; ++k) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->full[k % S]), (k / S) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform descriptors); one elected lane
    // issues, every lane polls the barriers and the vote keeps the decision uniform.
    {
      auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
      // MMA runs of each axis: all 64-wide W chunks in one MMA (N up to 256), then the
      // 32- and 16-wide chunk alone.  Descriptors are built once, for ring stage 0; a
      // stage and a k-step only add offsets (building a descriptor per MMA made the
      // issuing thread, not the tensor pipe, set the rate).
      uint64_t rdesc[2][kRuns];
      uint32_t ridesc[2][kRuns], rcol[2][kRuns], rkstep[2][kRuns];
      int nrun[2];
#pragma unroll
      for (int ax = 0; ax < 2; ++ax) {
        const ChunkPlan& bp = ax == 0 ? P.bk : P.bv;
        int c = 0, n = 0;
#pragma unroll
        for (int r = 0; r < kRuns; ++r) {
          rdesc[ax][r] = 0; ridesc[ax][r] = 0; rcol[ax][r] = 0; rkstep[ax][r] = 0;
          if (c < bp.n) {
            const int w = bp.width[c];
            int nch = 1;
            if (w == 64) while (c + nch < bp.n && bp.width[c + nch] == 64 && nch < 4) ++nch;
            const int rb = w * 2;
            rdesc[ax][r] = umma_desc(sbase + P.ring + P.b_off + bp.off[c], 64 * rb, 8 * rb, sw_mode_for_row_bytes(rb));
            ridesc[ax][r] = umma_idesc_bf16(128, w * nch, false, true);
            rcol[ax][r] = static_cast<uint32_t>(bp.start[c]);
            rkstep[ax][r] = static_cast<uint32_t>(16 * rb) >> 4;
            c += nch;
            n = r + 1;
          }
        }
        nrun[ax] = n;
      }
      const uint64_t adesc = umma_desc(sbase + P.ring + P.a_off, 16, 1024, kSw128);
      const uint32_t stage16 = static_cast<uint32_t>(P.stage) >> 4;
      uint32_t g = 0;
      bool ok = true;
      int64_t j = 0;
      for (int64_t u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++j) {
        const EncodeUnit e = encode_unit(u, a.H);
        const int nr = e.axis == 0 ? nrun[0] : nrun[1];
        uint64_t bdesc[kRuns];
        uint32_t idesc[kRuns], col[kRuns], kstep[kRuns];
#pragma unroll
        for (int r = 0; r < kRuns; ++r) {
          bdesc[r] = e.axis == 0 ? rdesc[0][r] : rdesc[1][r];
          idesc[r] = e.axis == 0 ? ridesc[0][r] : ridesc[1][r];
          col[r] = e.axis == 0 ? rcol[0][r] : rcol[1][r];
          kstep[r] = e.axis == 0 ? rkstep[0][r] : rkstep[1][r];
        }
        const int ab = acc_buf(j);
        // the epilogue has read this accumulator's previous unit out of TMEM
        if (!(ok = agree(mbar_wait(bar(misc->dempty[ab]), (acc_use(j) & 1) ^ 1, abort, a.status)))) break;
        tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(ab * P.acc_stride);
        uint32_t s = g % S;
        for (int kb = 0; kb < KB; ++kb, ++g) {
          if (!(ok = agree(mbar_wait(bar(misc->full[s]), (g / S) & 1, abort, a.status)))) break;
          tc_fence_after();
          const uint32_t so = s * stage16;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int r = 0; r < kRuns; ++r)
              if (r < nr)
                umma_bf16_warp(acc + col[r], adesc + so + 2 * k, bdesc[r] + so + k * kstep[r], idesc[r],
                               (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit_warp(bar(misc->empty[s]));
          s = s + 1 == S ? 0 : s + 1;
        }
        if (ok) umma_commit_warp(bar(misc->dfull[ab]));
      }
      // every MMA this warp issued is complete before TMEM is released
      if (g > 0) {
        umma_commit_warp(bar(misc->mdone));
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->mdone), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int64_t j = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, ++j) {
      const EncodeUnit e = encode_unit(u, a.H);
      const int r = e.axis == 0 ? a.r_k : a.r_v;
      const int ab = acc_buf(j);
      // this lane's token slot is read before the accumulator wait, so the load's
      // latency hides behind the unit's MMAs
      const int n = e.tile * 128 + row;
      int sid = -1, p = -1;
      if (n < a.N) {
        sid = __ldg(a.seq_idx + n);
        p = __ldg(a.pos + n);
      }
      if (!warp_wait(bar(misc->dfull[ab]), acc_use(j) & 1, abort, a.status)) break;
      tc_fence_after();
      if (n < a.N && !slot_ok(a, sid, p)) record_status(a.status, LLA_ERR_DEVICE_ARG);
      const int64_t drow = n < a.N && slot_ok(a, sid, p)
                               ? latent_row_for_write(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max,
                                                      a.H, sid, e.h, p, a.status)
                               : -1;
      const bool write = drow >= 0;
      const float4* bias4 = reinterpret_cast<const float4*>(a.bias + (static_cast<int64_t>(e.axis) * a.H + e.h) * kMaxRank2d);
      __nv_bfloat16* dst =
          static_cast<__nv_bfloat16*>(e.axis == 0 ? a.cache_k : a.cache_v) + (write ? drow : 0) * r;
      const uint32_t acc = tmem + static_cast<uint32_t>(ab * P.acc_stride) + lane_base;
      // 32 columns per TMEM load (a 16-column tail when r is an odd multiple of 16);
      // the bias columns load while the TMEM load is in flight
      for (int c0 = 0; c0 < r; c0 += 32) {
        const bool full32 = r - c0 >= 32;
        float v[32], v16[16], bb[32];
        if (full32)
          tmem_ld_x32(acc + c0, v);   // every lane of the warp takes part
        else
          tmem_ld_x16(acc + c0, v16);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 t = (full32 || i < 4) ? __ldg(bias4 + (c0 >> 2) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          bb[4 * i] = t.x; bb[4 * i + 1] = t.y; bb[4 * i + 2] = t.z; bb[4 * i + 3] = t.w;
        }
        tmem_wait_ld();
        if (!full32) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = v16[i];
        }
        if (write) {
          uint32_t wds[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i] - bb[2 * i], v[2 * i + 1] - bb[2 * i + 1]);
            wds[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
          d4[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
          d4[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
          if (full32) {
            d4[2] = make_uint4(wds[8], wds[9], wds[10], wds[11]);
            d4[3] = make_uint4(wds[12], wds[13], wds[14], wds[15]);
          }
        }
      }
      // this warp's rows are out of the accumulator: the MMA thread may reuse it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(misc->dempty[ab]));
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

// CTA-pair form of the encode for ranks that are multiples of 32 up to 256 (both
// axes): a unit is (pair of 128-token tiles, head, axis); CTA `rank` of the pair
// holds tile 2 t + rank of x and half of the W_down columns, [rank r/2, rank r/2 +
// r/2), as 16-column boxes, and one pair MMA per K step (M = 256 tokens, N = r)
// covers both tiles.  Each CTA's ring stage is then 16 KB of x + 64 r bytes of W
// instead of 16 KB + 128 r, so about a third more x is in flight per SM (the
// single-CTA encode holds six 36 KB stages and is bound by the copies' latency).
// Both CTAs' copies complete on the even CTA's full barrier (cta_group::2 copies);
// the even CTA's warp 1 issues; each CTA's epilogue writes its own tile's latents.
__global__ void __launch_bounds__(kEncodeThreads, 1)
encode_pair_kernel(const __grid_constant__ EncodeArgs a, const __grid_constant__ EncodePlan P,
                   const __grid_constant__ EncodeMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  EncodeMisc* misc = reinterpret_cast<EncodeMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_cta_rank();
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int KB = a.Td / 64;
  const uint32_t S = static_cast<uint32_t>(P.S);
  const int64_t nunits = static_cast<int64_t>((a.N + 255) / 256) * a.H * 2;
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };

  if (tid == 0) {
    for (int s = 0; s < P.S; ++s) {
      mbar_init(bar(misc->full[s]), 1);    // the even producer's expect_tx (both CTAs' bytes)
      mbar_init(bar(misc->empty[s]), 1);   // MMA commit (multicast)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(misc->dfull[b]), 1);
      mbar_init(bar(misc->dempty[b]), 8);  // the epilogue warps of both CTAs
    }
    mbar_init(bar(misc->mdone), 1);
    misc->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any remote arrive or copy
  if (warp == 1) {
    __syncwarp();
    tmem_alloc_pair(smem_u32(&misc->tmem_base), P.tmem_cols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t g = 0;   // k-blocks issued by this CTA: the ring position
      bool ok = true;
      // x streams through once; W_down is read by every tile of its head
      const uint64_t pol_x = l2_policy_evict_first(), pol_w = l2_policy_evict_last();
      for (int64_t u = pair; u < nunits && ok; u += npairs) {
        const EncodeUnit e = encode_unit(u, a.H);
        const int r = e.axis == 0 ? a.r_k : a.r_v;
        const CUtensorMap* xmap = e.axis == 0 ? &maps.xk : &maps.xv;
        const CUtensorMap* wmap = e.axis == 0 ? &maps.wk[2] : &maps.wv[2];   // 16-column boxes
        const int c0 = static_cast<int>(rank) * (r / 2), nbox = r / 32;
        const int tile = 2 * e.tile + static_cast<int>(rank);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const uint32_t s = g % S;
          if (!(ok = mbar_wait(bar(misc->empty[s]), ((g / S) & 1) ^ 1, abort, a.status))) break;
          const uint32_t fb = bar(misc->full[s]);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (128 * 64 * 2 + 64 * r));
          const uint32_t fbe = map_to_rank(fb, 0);
          const uint32_t st = sbase + P.ring + s * P.stage;
          tma_load_3d_pair(st + P.a_off, xmap, fbe, kb * 64, e.h, tile * 128, pol_x);
          for (int c = 0; c < nbox; ++c)
            tma_load_3d_pair(st + P.b_off + c * 2048, wmap, fbe, c0 + 16 * c, kb * 64, e.h, pol_w);
        }
      }
      // the copies still in flight land before the CTAs exit (they count on the even
      // CTA's barriers; the final cluster barrier holds the odd CTA)
      if (rank == 0) {
        for (uint32_t k = g > S ? g - S : 0; k < g; ++k) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar(misc->full[k % S]), (k / S) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
      }
    }
  } else if (warp == 1 && rank == 0) {
    // One warp issues the pair MMAs (warp-uniform loop, elected lane, all-lane polls).
    auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
    // A: 128 x 64 x tile (K-major, 128B swizzle); B: the W half, MN-major 16-column
    // boxes of 64 K rows (32B swizzle): next box 2 KB on (LBO), next 8 rows 256 B on (SBO)
    const uint64_t adesc = umma_desc(sbase + P.ring + P.a_off, 16, 1024, kSw128);
    const uint64_t bdesc = umma_desc(sbase + P.ring + P.b_off, 2048, 256, kSw32);
    const uint32_t idesc_k = umma_idesc_bf16(256, a.r_k, false, true), idesc_v = umma_idesc_bf16(256, a.r_v, false, true);
    const uint32_t stage16 = static_cast<uint32_t>(P.stage) >> 4;
    uint32_t g = 0;
    bool ok = true;
    int64_t j = 0;
    for (int64_t u = pair; u < nunits && ok; u += npairs, ++j) {
      const EncodeUnit e = encode_unit(u, a.H);
      const uint32_t idesc = e.axis == 0 ? idesc_k : idesc_v;
      const int ab = static_cast<int>(j & 1);
      // both CTAs' epilogues have read this accumulator's previous unit out of TMEM
      if (!(ok = agree(mbar_wait(bar(misc->dempty[ab]), ((j >> 1) & 1) ^ 1, abort, a.status)))) break;
      tc_fence_after();
      const uint32_t acc = tmem + static_cast<uint32_t>(ab * P.acc_stride);
      uint32_t s = g % S;
      for (int kb = 0; kb < KB; ++kb, ++g) {
        if (!(ok = agree(mbar_wait(bar(misc->full[s]), (g / S) & 1, abort, a.status)))) break;
        tc_fence_after();
        const uint32_t so = s * stage16;
#pragma unroll
        for (int k = 0; k < 4; ++k)   // 16-row K steps: +32 B in x rows, +512 B in the W boxes
          umma_bf16_pair_warp(acc, adesc + so + 2 * k, bdesc + so + k * (512 >> 4), idesc, (kb > 0 || k > 0) ? 1u : 0u);
        umma_commit_pair_warp(bar(misc->empty[s]));
        s = s + 1 == S ? 0 : s + 1;
      }
      if (ok) umma_commit_pair_warp(bar(misc->dfull[ab]));
    }
    // every MMA this warp issued is complete before TMEM is released
    if (g > 0) {
      umma_commit_pair_warp(bar(misc->mdone));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(misc->mdone), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2) {
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int64_t j = 0;
    for (int64_t u = pair; u < nunits; u += npairs, ++j) {
      const EncodeUnit e = encode_unit(u, a.H);
      const int r = e.axis == 0 ? a.r_k : a.r_v;
      const int ab = static_cast<int>(j & 1);
      // this lane's token slot is read before the accumulator wait
      const int n = (2 * e.tile + static_cast<int>(rank)) * 128 + row;
      int sid = -1, p = -1;
      if (n < a.N) {
        sid = __ldg(a.seq_idx + n);
        p = __ldg(a.pos + n);
      }
      if (!warp_wait(bar(misc->dfull[ab]), (j >> 1) & 1, abort, a.status)) break;
      tc_fence_after();
      if (n < a.N && !slot_ok(a, sid, p)) record_status(a.status, LLA_ERR_DEVICE_ARG);
      const int64_t drow = n < a.N && slot_ok(a, sid, p)
                               ? latent_row_for_write(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max,
                                                      a.H, sid, e.h, p, a.status)
                               : -1;
      const bool write = drow >= 0;
      const float4* bias4 = reinterpret_cast<const float4*>(a.bias + (static_cast<int64_t>(e.axis) * a.H + e.h) * kMaxRank2d);
      __nv_bfloat16* dst =
          static_cast<__nv_bfloat16*>(e.axis == 0 ? a.cache_k : a.cache_v) + (write ? drow : 0) * r;
      const uint32_t acc = tmem + static_cast<uint32_t>(ab * P.acc_stride) + lane_base;
      // 32 columns per TMEM load (r is a multiple of 32 here); the bias columns load
      // while the TMEM load is in flight
      for (int c0 = 0; c0 < r; c0 += 32) {
        float v[32], bb[32];
        tmem_ld_x32(acc + c0, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 t = __ldg(bias4 + (c0 >> 2) + i);
          bb[4 * i] = t.x; bb[4 * i + 1] = t.y; bb[4 * i + 2] = t.z; bb[4 * i + 3] = t.w;
        }
        tmem_wait_ld();
        if (write) {
          uint32_t wds[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i] - bb[2 * i], v[2 * i + 1] - bb[2 * i + 1]);
            wds[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
          d4[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
          d4[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
          d4[2] = make_uint4(wds[8], wds[9], wds[10], wds[11]);
          d4[3] = make_uint4(wds[12], wds[13], wds[14], wds[15]);
        }
      }
      // this warp's rows are out of the accumulator: the pair may reuse it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(bar(misc->dempty[ab]));
        else asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(map_to_rank(bar(misc->dempty[ab]), 0))
                          : "memory");
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's MMAs, copies and arrives are done with this CTA's memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, P.tmem_cols);
  }
}

// fp32: literal c[k] = sum_u (x[u] - mu[u]) W[u][k]; block = (token, head, axis).
__global__ void __launch_bounds__(256) encode_f32_kernel(const __grid_constant__ EncodeArgs a) {
  const int n = blockIdx.x, h = blockIdx.y, axis = blockIdx.z;
  const int r = axis == 0 ? a.r_k : a.r_v;
  const int sid = __ldg(a.seq_idx + n), p = __ldg(a.pos + n);
  if (!slot_ok(a, sid, p)) {
    if (threadIdx.x == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
    return;
  }
  const int64_t row =
      latent_row_for_write(a.block_table, a.page_size, a.max_pages, a.num_pages, a.L_max, a.H, sid, h, p, a.status);
  if (row < 0) return;
  const float* x = static_cast<const float*>(axis == 0 ? a.x_k : a.x_v) + (static_cast<int64_t>(n) * a.H + h) * a.Td;
  const float* mu = (axis == 0 ? a.mu_k : a.mu_v) + static_cast<int64_t>(h) * a.Td;
  const float* W = static_cast<const float*>(axis == 0 ? a.w_down_k : a.w_down_v) + static_cast<int64_t>(h) * a.Td * r;
  float* dst = static_cast<float*>(axis == 0 ? a.cache_k : a.cache_v);
  for (int k = threadIdx.x; k < r; k += blockDim.x) {
    float s = 0.f;
    for (int u = 0; u < a.Td; ++u) s = fmaf(x[u] - mu[u], W[static_cast<int64_t>(u) * r + k], s);
    dst[row * r + k] = s;
  }
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
  // two accumulators of 256 columns (every rank the host checks admit), else one of 512
  p->nacc = rmax <= 256 ? 2 : 1;
  p->acc_stride = 256;
  p->tmem_cols = 512;
  return true;
}

bool make_encode_pair_plan(int r_k, int r_v, int Td, EncodePlan* p) {
  *p = EncodePlan{};
  if (Td % 64 != 0 || r_k % 32 || r_v % 32 || r_k > 256 || r_v > 256) return false;
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  const int rmax = r_k > r_v ? r_k : r_v;
  p->a_off = 0;
  p->b_off = 128 * 64 * 2;
  p->stage = al(p->b_off + 64 * rmax, 1024);   // x tile, then the W half (16-column boxes)
  const int fixed = 1024 + 1024;
  int S = kMaxStages;
  while (S > 2 && fixed + S * p->stage > kSmemLimit) --S;
  if (fixed + S * p->stage > kSmemLimit) return false;
  p->S = S;
  p->ring = 0;
  p->misc = S * p->stage;
  p->bytes = p->misc + 1024 + 1024;
  p->nacc = 2;
  p->acc_stride = 256;
  p->tmem_cols = 512;
  return true;
}

cudaError_t launch_encode_pair(const EncodeArgs& a, const EncodePlan& plan, const EncodeMaps& m, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  encode_bias_kernel<<<dim3(a.H, 2, 2), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static int configured = 0;
  if (configured < plan.bytes) {
    e = cudaFuncSetAttribute(encode_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.bytes);
    if (e != cudaSuccess) return e;
    configured = plan.bytes;
  }
  // as many pairs as can be resident at once (each CTA takes a whole SM), no more
  // pairs than units
  static int pairs_for = -1, max_pairs = 0;
  if (pairs_for != plan.bytes) {
    cudaLaunchConfig_t occ = {};
    occ.gridDim = dim3(2);
    occ.blockDim = dim3(kEncodeThreads);
    occ.dynamicSmemBytes = plan.bytes;
    cudaLaunchAttribute oat[1];
    oat[0].id = cudaLaunchAttributeClusterDimension;
    oat[0].val.clusterDim.x = 2;
    oat[0].val.clusterDim.y = 1;
    oat[0].val.clusterDim.z = 1;
    occ.attrs = oat;
    occ.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, encode_pair_kernel, &occ);
    if (e != cudaSuccess) return e;
    max_pairs = n;
    pairs_for = plan.bytes;
  }
  if (max_pairs < 1) return cudaErrorLaunchOutOfResources;
  const int64_t units = static_cast<int64_t>((a.N + 255) / 256) * a.H * 2;
  int pairs = plan.sms / 2 < max_pairs ? plan.sms / 2 : max_pairs;
  if (units < pairs) pairs = static_cast<int>(units);
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kEncodeThreads);
  cfg.dynamicSmemBytes = plan.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, encode_pair_kernel, a, plan, m);
}

cudaError_t launch_encode_bf16(const EncodeArgs& a, const EncodePlan& plan, const EncodeMaps& m,
                               cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  encode_bias_kernel<<<dim3(a.H, 2, 2), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static int configured = 0;
  if (configured < plan.bytes) {
    e = cudaFuncSetAttribute(encode_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.bytes);
    if (e != cudaSuccess) return e;
    configured = plan.bytes;
  }
  // persistent: one CTA per SM (or per unit, when there are fewer units)
  const int64_t units = static_cast<int64_t>((a.N + 127) / 128) * a.H * 2;
  const int grid = static_cast<int>(units < plan.sms ? units : plan.sms);
  encode_bf16_kernel<<<grid, kEncodeThreads, plan.bytes, s>>>(a, plan, m);
  return cudaGetLastError();
}

cudaError_t launch_encode_f32(const EncodeArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  encode_f32_kernel<<<dim3(a.N, a.H, 2), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lla
