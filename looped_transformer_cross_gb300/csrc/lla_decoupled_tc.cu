// lla_decoupled_tc.cu — absorbed decoupled-RoPE decode in bf16 storage with the
// rotary branch and the content score on the tensor cores ("Looped Latent
// Attention: Cross-Loop KV Compression for Looped Transformers", arXiv
// 2607.15456v2, Appendix J "Absorbed attention", Tables 13-14): a position-major
// kernel for small ranks (r_k in {16, 32}, r_v in {32, 64}, even H <= 16) and a
// tile-major one for the other ranks up to (128, 256), both fed by one image kernel.
//
// At small ranks the 64-wide rotary key is most of a token's bytes (128 of 224 B
// per head at (16, 32)), so the rotary score has to cost the CUDA cores next to
// nothing.  With q' = sc RoPE(q_r, q_pos) and (i0, i1) the pair of frequency f,
//   RoPE(q_r, q_pos) . RoPE(r_j, j) sc = sum_f cos(j th_f) U_f,j + sin(j th_f) V_f,j,
//   U_f,j = r_j,i0 q'_i0 + r_j,i1 q'_i1,    V_f,j = r_j,i0 q'_i1 - r_j,i1 q'_i0.
// U and V are linear in the stored (unrotated) key, so for a 128-token head-tile
// one MMA chain gives every token's 64 of them:
//   A = the head-tile's rotary keys as stored (bf16, 128 x 64, 128-byte swizzle),
//   B = the head's coefficient rows (bf16, K-major, 32-byte swizzle).  Row (U_f)
//       and row (V_f) have their two nonzeros at keys i0(f) and i1(f), so the 64
//       output columns split into two groups of 16 frequencies whose pairs lie in
//       two K-steps of 16 keys: {G, G + 2} for the halves pairing, {2G, 2G + 1} for
//       the interleaved one.  Four 32 x 16 blocks per head, four MMAs (N = 32).
//   D = (U_0, V_0, U_1, V_1, ..., U_31, V_31) in TMEM (fp32).
// A second chain gives the content score w . c_k,j (A = the K latent tile, B = a
// row sc w rounded to bf16 and a row of its rounding remainder; N = 16).  The
// epilogue thread of token j holds cos / sin(j th_f) of its position in registers
// (fp32, loaded once per position and used for every head of its group) and
// finishes the score with 32 paired FMAs:
//   s_j = sc b0 + D_64 + D_65 + sum_f (D_2f cos(j th_f) + D_2f+1 sin(j th_f)),
// in base-2 units (sc = log2(e) / sqrt(d + d_rope)).  Neither the rotary keys nor
// the K latents pass through the CUDA cores.  The value side is the small-rank
// kernel's: each warp forms sum_j p_j c_v,j over its 32 tokens from the V tile in
// shared memory, records go out per (sequence + CTA, head, warp), and the shared
// combine applies W_up,v,t once.
//
// Work: positions (sequence, 128-token tile) in contiguous ranges, one range per
// CTA, every head of a position inside it.  Warps: 0 producer (TMA copies of the
// rotary and K tiles, a bulk copy of the V rows, the sequence's B images once per
// run), 1 MMA issuer, 2-9 two epilogue groups of four warps (group g takes the
// heads h = g mod 2), one token per epilogue thread.
#include "lla_kernels.h"

#include <algorithm>
#include <cmath>

namespace lla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtDR = 0.07216878364870322f;   // 1 / sqrt(d + d_rope) = 1 / sqrt(192)
constexpr float kRescaleLog2 = 8.f;                  // lazy rescale threshold (log2 units)
constexpr int kRope = 64;                            // rotary branch width
constexpr int kEpiGroups = 2;
constexpr int kDsThreads = 64 + kEpiGroups * 128;    // producer, MMA issuer, 2 x 4 epilogue warps
constexpr int kDCols = 80;                           // TMEM columns per head-tile: 64 (U, V), 16 content
constexpr int kNG = 6;                               // D buffers (6 x 80 columns)
constexpr int kMaxNS = 8;
constexpr int kRotBlock = 1024;                      // B block: 32 rows x 32 B
constexpr int kConBlock = 512;                       // content B block: 16 rows x 32 B
constexpr int kRTile = kTile * kRope * 2;            // rotary tile: 128 rows x 128 B
constexpr int kCkBox = kTile * 32;                   // K latent box: 128 rows x 16 columns
constexpr int kDzThreads = 256;
constexpr int kDzSeqs = 8;                           // sequences per image block at most (a.z_seqs)
constexpr int kTrigJ = 64;                           // positions per trig-table block

static_assert(kNG * kDCols <= 512, "TMEM columns");
static_assert(kNG % kEpiGroups == 0, "a D buffer always serves the same group");

struct alignas(16) DsMisc {
  uint64_t full[kMaxNS], empty[kMaxNS];   // ring slots (rotary + K tiles, V rows)
  uint64_t img_full, img_empty;           // the run's B images
  uint64_t gfull[kNG], gempty[kNG];       // D buffers (one head-tile each)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int start_b, start_t, count;
  int total_pos;
  int scan[kDsThreads];
};

struct DsPlan {
  int nk;           // content K-steps (r_k / 16)
  int img;          // bytes of one head's B image
  int k_tile;       // rotary tile + K latent boxes
  int slot;         // ring slot: k_tile + V rows, 1024-aligned
  int NS;           // ring slots
  int imgs, ring, acc, ml, misc, bytes;
};

__host__ __device__ inline int al_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline bool make_ds_plan(int H, int r_k, int r_v, DsPlan* p) {
  if (H < 2 || H % 2 || H > kSmallMaxHeads) return false;
  if ((r_k != 16 && r_k != 32) || (r_v != 32 && r_v != 64)) return false;
  p->nk = r_k / 16;
  p->img = 4 * kRotBlock + p->nk * kConBlock;
  p->k_tile = kRTile + p->nk * kCkBox;
  p->slot = al_up(p->k_tile + kTile * r_v * 2, 1024);
  const int imgs = al_up(H * p->img, 1024);
  const int acc = 8 * (H / 2) * r_v * 4;                  // [8 warps][H / 2 heads][r_v]
  const int ml = al_up(8 * (H / 2) * 8, 16);             // [8 warps][H / 2 heads] (m, l)
  const int misc = al_up(static_cast<int>(sizeof(DsMisc)), 16);
  const int fixed = imgs + acc + ml + misc + 1024;
  int NS = (kSmemLimit - fixed) / p->slot;
  NS = NS < kMaxNS ? NS : kMaxNS;
  // a slot always serves the same epilogue group: a group's consecutive uses of a
  // slot are then consecutive phases of its barriers (a parity wait must never be
  // more than one phase ahead)
  NS -= NS % kEpiGroups;
  if (NS < 2) return false;
  p->NS = NS;
  int off = 0;
  p->imgs = off; off += imgs;
  p->ring = off; off += NS * p->slot;
  p->acc = off;  off += acc;
  p->ml = off;   off += ml;
  p->misc = off; off += misc;
  p->bytes = off + 1024;
  return p->bytes <= kSmemLimit;
}

__device__ __forceinline__ int clamp_len(int L, int64_t L_max) {
  return L < 0 ? 0 : (L > L_max ? static_cast<int>(L_max) : L);
}

// Rotary pair (i0, i1) of frequency f (f < 32) within the 64-wide branch.
__host__ __device__ __forceinline__ void rope_pair(int style, int f, int& i0, int& i1) {
  i0 = style == 0 ? f : 2 * f;
  i1 = style == 0 ? f + kRope / 2 : 2 * f + 1;
}

// K-step (16 keys) of the rotary tile that block (G, kk) of the B image multiplies.
__host__ __device__ __forceinline__ int rot_kstep(int style, int G, int kk) {
  return style == 0 ? G + 2 * kk : 2 * G + kk;
}

// d = a * b + d on a pair of fp32 lanes (one packed instruction).
__device__ __forceinline__ void fma_pair(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mov.b64 pd, {%0, %1};\n\tfma.rn.f32x2 pd, pa, pb, pd;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Walk over positions (sequence b, tile t) in order, skipping empty sequences.
struct PosWalker {
  int b, t, nb, L;
};

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

// Ring position advanced by `step` (< n, or = n) slots at a time.
struct SlotPos {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void next(int step, int n) {
    slot += step;
    if (slot >= n) { slot -= n; phase ^= 1u; }
  }
};

// Query side, one launch before the decode grid.
//  * The first blocks write the transposed fp32 RoPE table of the rotary branch,
//    trigT[2f][j] = cos(j th_f), trigT[2f + 1][j] = sin(j th_f) for j < trig_rows
//    (rows past the caller's table repeat its last row; only masked tokens read
//    them), so that a warp reading one column for 32 consecutive tokens reads one
//    128-byte line.
//  * Block (head h, a.z_seqs <= kDzSeqs sequences; fewer when the batch is small, so
//    that the grid still covers the SMs): W_up,k,t[h] is staged once; per sequence
//    w = W_up,k,t[h]^T q_c, b0 = q_c . mu_k,t[h] and q' = RoPE(q_r, q_pos), all
//    times sc, then the head's B image at zimg + (b H + h) zimg_stride: rotary
//    block (G, kk) at (2 G + kk) 1 KB, row 2 f' + v of frequency f = 16 G + f'
//    (v = 0: U_f, 1: V_f), column c = key 16 rot_kstep(G, kk) + c; content block kb
//    at 4 KB + kb 512 B, row 0 = sc w rounded to bf16, row 1 = its remainder,
//    rows 2-15 zero; each block in the 32-byte swizzle.  sc b0 goes to qb0[b H + h].
//    Empty sequences are skipped (never read).
__global__ void __launch_bounds__(kDzThreads) decoupled_small_z_kernel(const __grid_constant__ DecodeArgs a) {
  // launched as a programmatic dependent of whatever precedes the call on the
  // stream: nothing is read before that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the decode grid may start its set-up now; it waits for this grid before it
  // copies an image or reads the table
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // W_up,k,t[h] as bf16 [128][r_k] (row stride r_k + 2, r_k <= 128); the table
  // blocks use the same bytes as an fp32 [64][kTrigJ + 1] transpose tile
  __shared__ __align__(16) uint8_t wraw[kHeadDim * (128 + 2) * 2];
  __shared__ __align__(16) float qc[kDzSeqs][kHeadDim];
  __shared__ float qa[kDzSeqs][kRope / 2], qb[kDzSeqs][kRope / 2];   // sc q'_i0, sc q'_i1
  __shared__ float wsc[kDzSeqs][128];            // sc w
  __shared__ bool live[kDzSeqs];
  const int tid = threadIdx.x;
  const int ntb = static_cast<int>((a.trig_rows + kTrigJ - 1) / kTrigJ);
  if (static_cast<int>(blockIdx.x) < ntb) {
    float* tile = reinterpret_cast<float*>(wraw);   // [64 columns][kTrigJ + 1]
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kTrigJ;
    for (int i = tid; i < kTrigJ * 64; i += kDzThreads) {
      const int jj = i / 64, c = i % 64, f = c >> 1;
      int64_t j = j0 + jj;
      if (j >= a.rope_len) j = a.rope_len - 1;
      tile[c * (kTrigJ + 1) + jj] =
          __ldg(((c & 1) ? a.rope_sin : a.rope_cos) + j * (kRope / 2) + f);
    }
    __syncthreads();
    for (int i = tid; i < kTrigJ * 64; i += kDzThreads) {
      const int c = i / kTrigJ, jj = i % kTrigJ;
      if (j0 + jj < a.trig_rows) a.trigT[c * a.trig_rows + j0 + jj] = tile[c * (kTrigJ + 1) + jj];
    }
    return;
  }
  const int u = static_cast<int>(blockIdx.x) - ntb;
  const int zs = a.z_seqs;
  const int h = u % a.H, b0 = (u / a.H) * zs;
  const int rk = a.r_k, ws = rk + 2, nk = rk / 16;
  __nv_bfloat16* Wb = reinterpret_cast<__nv_bfloat16*>(wraw);
  const float sc = kLog2e * kInvSqrtDR;
  const __nv_bfloat16* W =
      static_cast<const __nv_bfloat16*>(a.w_up_k) + static_cast<int64_t>(h) * kHeadDim * rk;
  for (int i = tid; i < kHeadDim * rk / 8; i += kDzThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(W) + i);
    const __nv_bfloat16* v8 = reinterpret_cast<const __nv_bfloat16*>(&v);
    const int row = (8 * i) / rk, col = (8 * i) % rk;
#pragma unroll
    for (int e = 0; e < 8; ++e) Wb[row * ws + col + e] = v8[e];
  }
  const int qrow = kHeadDim + kRope;
  for (int i = tid; i < kDzSeqs * kHeadDim; i += kDzThreads) {
    const int sb = i / kHeadDim, e = i % kHeadDim, b = b0 + sb;
    qc[sb][e] = sb < zs && b < a.B ? __bfloat162float(static_cast<const __nv_bfloat16*>(
                              a.q)[(static_cast<int64_t>(b) * a.H + h) * qrow + e])
                        : 0.f;
  }
  for (int i = tid; i < zs * (kRope / 2); i += kDzThreads) {
    const int sb = i / (kRope / 2), f = i % (kRope / 2), b = b0 + sb;
    if (b >= a.B) break;
    int qp = __ldg(a.q_pos + b);
    if (qp < 0 || qp >= a.rope_len) {
      if (f == 0) record_status(a.status, LLA_ERR_DEVICE_ARG);
      qp = qp < 0 ? 0 : static_cast<int>(a.rope_len - 1);
    }
    int i0, i1;
    rope_pair(a.rope_style, f, i0, i1);
    const __nv_bfloat16* qr =
        static_cast<const __nv_bfloat16*>(a.q) + (static_cast<int64_t>(b) * a.H + h) * qrow + kHeadDim;
    const float c = __ldg(a.rope_cos + static_cast<int64_t>(qp) * (kRope / 2) + f);
    const float s = __ldg(a.rope_sin + static_cast<int64_t>(qp) * (kRope / 2) + f);
    const float x0 = __bfloat162float(qr[i0]), x1 = __bfloat162float(qr[i1]);
    qa[sb][f] = (x0 * c - x1 * s) * sc;
    qb[sb][f] = (x0 * s + x1 * c) * sc;
  }
  if (tid < kDzSeqs)
    live[tid] = tid < zs && b0 + tid < a.B && clamp_len(__ldg(a.seq_lens + b0 + tid), a.L_max) > 0;
  __syncthreads();
  for (int i = tid; i < zs * rk; i += kDzThreads) {
    const int sb = i / rk, n = i % rk;
    float s = 0.f;
#pragma unroll 8
    for (int e = 0; e < kHeadDim; ++e) s = fmaf(qc[sb][e], __bfloat162float(Wb[e * ws + n]), s);
    wsc[sb][n] = s * sc;
  }
  {
    // warp sb: sc q_c . mu_k,t[h]
    const int warp = tid >> 5, lane = tid & 31;
    const float* mu = a.mu_k + static_cast<int64_t>(h) * a.mu_hstride;
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < kHeadDim / 32; ++k) part = fmaf(qc[warp][lane + 32 * k], __ldg(mu + lane + 32 * k), part);
    part = warp_sum(part);
    if (lane == 0 && live[warp]) a.qb0[static_cast<int64_t>(b0 + warp) * a.H + h] = part * sc;
  }
  __syncthreads();
  // image granules (16 B = 8 columns of one row): 4 rotary blocks x 32 rows x 2,
  // then nk content blocks x 16 rows x 2
  const int ng = 256 + 32 * nk;
  for (int it = tid; it < zs * ng; it += kDzThreads) {
    const int sb = it / ng, gi = it % ng;
    if (!live[sb]) continue;
    float v[8];
    uint32_t off;
    if (gi < 256) {
      const int blk = gi >> 6, n = (gi >> 1) & 31, half = gi & 1;
      const int G = blk >> 1, kk = blk & 1;
      const int f = 16 * G + (n >> 1);
      const bool vrow = n & 1;
      int i0, i1;
      rope_pair(a.rope_style, f, i0, i1);
      const float q0 = qa[sb][f], q1 = qb[sb][f];
      const int e0 = 16 * rot_kstep(a.rope_style, G, kk) + 8 * half;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int key = e0 + e;
        v[e] = key == i0 ? (vrow ? q1 : q0) : key == i1 ? (vrow ? -q0 : q1) : 0.f;
      }
      off = blk * kRotBlock + swizzle_offset(n * 32 + 16 * half, 32);
    } else {
      const int ci = gi - 256, kb = ci >> 5, n = (ci >> 1) & 15, half = ci & 1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = wsc[sb][16 * kb + 8 * half + e];
        const float hi = __bfloat162float(__float2bfloat16_rn(x));
        v[e] = n == 0 ? hi : n == 1 ? x - hi : 0.f;
      }
      off = 4 * kRotBlock + kb * kConBlock + swizzle_offset(n * 32 + 16 * half, 32);
    }
    const uint4 w = make_uint4(bf16x2_bits(v[0], v[1]), bf16x2_bits(v[2], v[3]), bf16x2_bits(v[4], v[5]),
                               bf16x2_bits(v[6], v[7]));
    *reinterpret_cast<uint4*>(a.zimg + (static_cast<int64_t>(b0 + sb) * a.H + h) * a.zimg_stride + off) = w;
  }
}

template <int RK, int RV>
__global__ void __launch_bounds__(kDsThreads, 1)
    decoupled_small_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ DecoupledMaps maps) {
  constexpr int NK = RK / 16;
  constexpr int VB = RV * 2;              // bytes of a latent V row
  constexpr int LPR = RV / 4;             // value step: lanes per V row, 4 columns each
  constexpr int RPL = 32 / LPR;           // V rows per warp-wide load
  extern __shared__ uint8_t smem_raw[];
  // swizzle atoms need 1024-byte alignment in the shared window itself
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  DsPlan P;
  make_ds_plan(a.H, RK, RV, &P);
  const uint32_t sbase = smem_u32(sm);
  DsMisc* misc = reinterpret_cast<DsMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, NS = P.NS;

  // ---------------------------------------------------------- work range
  // positions (sequence, tile) in order; CTA c takes [c per, (c + 1) per)
  {
    const int per_thr = (a.B + kDsThreads - 1) / kDsThreads;
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
      constexpr int kPer = kDsThreads / 32;
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
    for (int s = 0; s < NS; ++s) { mbar_init(bar(misc->full[s]), 1); mbar_init(bar(misc->empty[s]), 4); }
    mbar_init(bar(misc->img_full), 1);
    mbar_init(bar(misc->img_empty), 1);
    for (int g = 0; g < kNG; ++g) { mbar_init(bar(misc->gfull[g]), 1); mbar_init(bar(misc->gempty[g]), 4); }
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
    // Per run (the CTA's positions of one sequence): the H B images in one bulk
    // copy, once the MMAs of the previous run are done with them.  Per head-tile:
    // the rotary tile and the K latent boxes (TMA, swizzled as the MMA reads them;
    // rows past the cache end read as zero, rows past the sequence end are masked),
    // and the V rows below the sequence length (one bulk copy).
    if (lane == 0) {
      prefetch_tmap(&maps.kr);
      prefetch_tmap(&maps.ck);
      const uint64_t pol = l2_policy_evict_first();
      PosWalker w = start;
      SlotPos sp{0, 0u};
      int run = 0, issued = 0;
      bool ok = true;
      for (int lp = 0; lp < count && ok; ++lp) {
        if (lp == 0 || w.t == 0) {
          if (run > 0 && !(ok = mbar_wait(bar(misc->img_empty), (run - 1) & 1, abort, a.status))) break;
          if (lp == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // images written
          const uint32_t fb = bar(misc->img_full);
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(H * P.img));
          bulk_load(sbase + P.imgs, a.zimg + static_cast<int64_t>(w.b) * H * a.zimg_stride,
                    static_cast<uint32_t>(H * P.img), fb);
          ++run;
        }
        const uint32_t rows = static_cast<uint32_t>(min(kTile, w.L - w.t * kTile));
        const int y = w.t * kTile;
        for (int h = 0; h < H && ok; ++h) {
          if (!(ok = mbar_wait(bar(misc->empty[sp.slot]), sp.phase ^ 1u, abort, a.status))) break;
          const uint32_t fb = bar(misc->full[sp.slot]);
          const uint32_t dst = sbase + P.ring + sp.slot * P.slot;
          const int z = w.b * H + h;
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(P.k_tile) + rows * VB);
          tma_load_3d_hint(dst, &maps.kr, fb, 0, y, z, pol);
#pragma unroll
          for (int kb = 0; kb < NK; ++kb) tma_load_3d_hint(dst + kRTile + kb * kCkBox, &maps.ck, fb, 16 * kb, y, z, pol);
          bulk_load_hint(dst + P.k_tile,
                         static_cast<const uint8_t*>(a.cache_v) + (static_cast<int64_t>(z) * a.L_max + y) * VB,
                         rows * VB, fb, pol);
          ++issued;
          sp.next(1, NS);
        }
        pos_advance(w, a);
      }
      // Let every copy this CTA issued land before the CTA can exit.
      for (int i = max(0, issued - NS); i < issued; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->full[i % NS]), (i / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
      if (run > 0) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->img_full), (run - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // Per head-tile, into the next D buffer: four rotary MMAs (two column groups of
    // 32, two K-steps each) and the content MMAs (N = 16, one per 16 K latents).
    // The whole warp runs the loop; one elected lane issues, every lane polls and
    // the vote keeps the decision uniform.
    auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
    const uint32_t idesc_rot = umma_idesc_bf16(128, 32, false, false);
    const uint32_t idesc_con = umma_idesc_bf16(128, 16, false, false);
    const int style = a.rope_style;
    PosWalker w = start;
    SlotPos sp{0, 0u}, gp{0, 0u};
    int run = 0;
    bool ok = true;
    for (int lp = 0; lp < count && ok; ++lp) {
      const bool run_start = lp == 0 || w.t == 0;
      const bool run_end = lp == count - 1 || w.t == w.nb - 1;
      if (run_start) {
        if (!(ok = agree(mbar_wait(bar(misc->img_full), run & 1, abort, a.status)))) break;
        ++run;
      }
      for (int h = 0; h < H; ++h) {
        if (!(ok = agree(mbar_wait(bar(misc->full[sp.slot]), sp.phase, abort, a.status)))) break;
        if (!(ok = agree(mbar_wait(bar(misc->gempty[gp.slot]), gp.phase ^ 1u, abort, a.status)))) break;
        tc_fence_after();
        const uint32_t d = tmem + gp.slot * kDCols;
        const uint32_t ra = sbase + P.ring + sp.slot * P.slot;
        const uint32_t ib = sbase + P.imgs + h * P.img;
        const uint64_t a_rot = umma_desc(ra, 16, 1024, kSw128);
#pragma unroll
        for (int G = 0; G < 2; ++G)
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            umma_bf16_warp(d + 32 * G, a_rot + 2 * rot_kstep(style, G, kk),
                           umma_desc(ib + (2 * G + kk) * kRotBlock, 16, 256, kSw32), idesc_rot, kk);
#pragma unroll
        for (int kb = 0; kb < NK; ++kb)
          umma_bf16_warp(d + 64, umma_desc(ra + kRTile + kb * kCkBox, 16, 256, kSw32),
                         umma_desc(ib + 4 * kRotBlock + kb * kConBlock, 16, 256, kSw32), idesc_con, kb);
        umma_commit_warp(bar(misc->gfull[gp.slot]));
        if (run_end && h == H - 1) umma_commit_warp(bar(misc->img_empty));   // the images are no longer read
        gp.next(1, kNG);
        sp.next(1, NS);
      }
      pos_advance(w, a);
    }
    // this warp's MMAs complete before TMEM is released
    umma_commit_warp(bar(misc->mma_done));
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar(misc->mma_done), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
  } else {
    // ======================================================== epilogue (warps 2-9)
    // Group g (warps 2 + 4 g .. 5 + 4 g) takes heads h = 2 jj + g; thread (TMEM
    // quadrant q, lane) owns token row 32 q + lane.
    const int we = warp - 2, g = we >> 2, q = warp & 3;
    const int row = 32 * q + lane;
    const int HG = H / 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float* accs = reinterpret_cast<float*>(sm + P.acc) + static_cast<size_t>(we) * HG * RV;   // [HG][RV]
    float2* mls = reinterpret_cast<float2*>(sm + P.ml) + we * HG;                            // [HG] (m, l)
    asm volatile("griddepcontrol.wait;" ::: "memory");   // table and sc b0 written

    SlotPos sp{g, 0u};   // ring slot of this group's next head-tile (every other one)
    SlotPos gp{g, 0u};   // D buffer of the same
    PosWalker w = start;
    bool ok = true;
    for (int lp = 0; lp < count && ok; ++lp) {
      const bool run_start = lp == 0 || w.t == 0;
      const bool run_end = lp == count - 1 || w.t == w.nb - 1;
      const int nvalid = min(kTile, w.L - w.t * kTile);
      const bool valid = row < nvalid;
      // cos / sin of this token's position, kept for every head of the position
      float cs[kRope];
      {
        int64_t j = static_cast<int64_t>(w.t) * kTile + row;
        if (j >= a.trig_rows) j = a.trig_rows - 1;   // past the cache end: masked anyway
        const float* tp = a.trigT + j;
#pragma unroll
        for (int c = 0; c < kRope; ++c) cs[c] = __ldg(tp + c * a.trig_rows);
      }
      for (int jj = 0; jj < HG; ++jj) {
        const int h = 2 * jj + g;
        const float qb0 = __ldg(a.qb0 + static_cast<int64_t>(w.b) * H + h);
        // ---- (U, V) and the content products of this token from TMEM; the buffer
        // is free again once the group's four warps have read it
        if (!(ok = warp_wait(bar(misc->gfull[gp.slot]), gp.phase, abort, a.status))) break;
        tc_fence_after();
        float u0[32], u1[32], uc[2];
        {
          const uint32_t gb = tmem + lane_base + gp.slot * kDCols;
          tmem_ld_x32(gb, u0);
          tmem_ld_x32(gb + 32, u1);
          tmem_ld_x2(gb + 64, uc);
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->gempty[gp.slot]));
        gp.next(kEpiGroups, kNG);

        // ---- s_j = sc b0 + content (hi + lo) + sum_f U_f cos + V_f sin (log2 units)
        float x0 = 0.f, x1 = 0.f, y0 = 0.f, y1 = 0.f, z0 = 0.f, z1 = 0.f, t0 = 0.f, t1 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          fma_pair(x0, x1, u0[2 * i], u0[2 * i + 1], cs[2 * i], cs[2 * i + 1]);
          fma_pair(y0, y1, u0[2 * i + 2], u0[2 * i + 3], cs[2 * i + 2], cs[2 * i + 3]);
          fma_pair(z0, z1, u0[2 * i + 4], u0[2 * i + 5], cs[2 * i + 4], cs[2 * i + 5]);
          fma_pair(t0, t1, u0[2 * i + 6], u0[2 * i + 7], cs[2 * i + 6], cs[2 * i + 7]);
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          fma_pair(x0, x1, u1[2 * i], u1[2 * i + 1], cs[32 + 2 * i], cs[32 + 2 * i + 1]);
          fma_pair(y0, y1, u1[2 * i + 2], u1[2 * i + 3], cs[32 + 2 * i + 2], cs[32 + 2 * i + 3]);
          fma_pair(z0, z1, u1[2 * i + 4], u1[2 * i + 5], cs[32 + 2 * i + 4], cs[32 + 2 * i + 5]);
          fma_pair(t0, t1, u1[2 * i + 6], u1[2 * i + 7], cs[32 + 2 * i + 6], cs[32 + 2 * i + 7]);
        }
        const float sr = ((x0 + x1) + (y0 + y1)) + ((z0 + z1) + (t0 + t1));
        const float s = valid ? (qb0 + (uc[0] + uc[1])) + sr : -INFINITY;

        // ---- the head-tile's V rows
        if (!(ok = warp_wait(bar(misc->full[sp.slot]), sp.phase, abort, a.status))) break;
        uint8_t* vt = sm + P.ring + sp.slot * P.slot + P.k_tile;

        // ---- online softmax per warp, reference raised lazily (by more than 2^8)
        float2 ml = run_start ? make_float2(-INFINITY, 0.f) : mls[jj];
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
#pragma unroll
            for (int c = 0; c < VB / 16; ++c) *reinterpret_cast<uint4*>(vt + row * VB + 16 * c) = make_uint4(0, 0, 0, 0);
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
          const uint2 v = *reinterpret_cast<const uint2*>(vt + (32 * q + tk) * VB + 8 * cg);
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
        // the slot is consumed: its MMAs completed before the D wait above, and the
        // shuffles used every V load
        if (nvalid < kTile) fence_proxy_async_smem();   // zeroed rows before the next bulk copy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->empty[sp.slot]));
        sp.next(kEpiGroups, NS);

        // ---- fold into the warp's state; a run's last tile writes the record
        // (m, l, -, -, acc) of (sequence + CTA, head, warp)
        float* rec = a.partials +
                     ((static_cast<int64_t>(w.b + blockIdx.x) * H + h) * kRecordsPerCta + (we & 3)) *
                         (RV + kRecordHead);
        if (lane < LPR) {
          float4* ap = reinterpret_cast<float4*>(accs + jj * RV) + cg;
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
          mls[jj] = ml;
          if (run_end) { rec[0] = ml.x; rec[1] = ml.y; }
        }
        __syncwarp();
      }
      pos_advance(w, a);
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
cudaError_t launch_instance(const DecodeArgs& a, const DecoupledMaps& m, int bytes, cudaStream_t s) {
  auto kern = decoupled_small_kernel<RK, RV>;
  static int configured = 0;
  if (configured < bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured = bytes;
  }
  // programmatic dependent launch: the decode grid's set-up overlaps the image
  // kernel; it waits for that grid before the first image copy / table read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kDsThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, m);
}


// ================================================================ tile-major kernel
// Larger ranks (r_k up to 128, r_v up to 256).  A unit's B image stays small (4 KB +
// r_k / 16 x 512 B), but a head-tile's rotary and K rows grow (16 KB + r_k x 256 B)
// and a position's head-tiles no longer fit beside every head's image, so the work
// is tile-major as in the per-head tile kernel: 128-token tiles over (sequence,
// head) in contiguous ranges per CTA, the unit's image copied once per unit into
// one of two buffers.  The MMA chain is the small-rank kernel's.  The V rows do not
// pass through shared memory: the producer asks L2 for each tile's V rows as it
// issues the tile's copies, and each epilogue warp reads its 32 tokens' rows with
// coalesced 4-byte loads (lane = pairs of V columns), keeping sum_j p_j c_v,j for
// its columns in registers while the unit lasts.  Two epilogue groups take
// alternate tiles; both walk every tile and close every unit, so each warp writes
// one record per (unit, CTA): eight per (unit, CTA).
constexpr int kDtThreads = 320;
constexpr int kDtMaxNS = 8;

struct alignas(16) DtMisc {
  uint64_t full[kDtMaxNS], empty[kDtMaxNS];   // ring slots (rotary + K tiles), consumed by the MMAs
  uint64_t img_full[2], img_empty[2];         // unit images (unit parity)
  uint64_t gfull[kNG], gempty[kNG];           // D buffers (one head-tile each)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int start_b, start_h, start_t, count;
  int total_seq_tiles;
  int scan[kDtThreads];
};

struct DtPlan {
  int nk;           // content K-steps (r_k / 16)
  int img;          // bytes of one image buffer (1024-aligned)
  int slot;         // ring slot: rotary tile + K latent boxes
  int NS;           // ring slots
  int imgs, ring, misc, bytes;
};

__host__ __device__ inline bool make_dt_plan(int r_k, int r_v, DtPlan* p) {
  if (r_k < 16 || r_k > 128 || r_k % 16 || r_v < 16 || r_v > 256 || r_v % 16) return false;
  p->nk = r_k / 16;
  p->img = al_up(4 * kRotBlock + p->nk * kConBlock, 1024);
  p->slot = al_up(kRTile + p->nk * kCkBox, 1024);
  const int misc = al_up(static_cast<int>(sizeof(DtMisc)), 16);
  int NS = (kSmemLimit - 2 * p->img - misc - 1024) / p->slot;
  NS = NS < kDtMaxNS ? NS : kDtMaxNS;
  if (NS < 2) return false;
  p->NS = NS;
  int off = 0;
  p->imgs = off; off += 2 * p->img;
  p->ring = off; off += NS * p->slot;
  p->misc = off; off += misc;
  p->bytes = off + 1024;
  return p->bytes <= kSmemLimit;
}

// Walk over head-tiles (sequence b, head h, tile t) in order, skipping empty sequences.
struct TileWalker {
  int b, h, t, nb, L;
};

__device__ __forceinline__ void tile_advance(TileWalker& w, const DecodeArgs& a) {
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

// NPL: pairs of V columns per lane, ceil(r_v / 64)
template <int NPL>
__global__ void __launch_bounds__(kDtThreads, 1)
    decoupled_tile_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ DecoupledMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  DtPlan P;
  make_dt_plan(a.r_k, a.r_v, &P);
  const uint32_t sbase = smem_u32(sm);
  DtMisc* misc = reinterpret_cast<DtMisc*>(sm + P.misc);
  volatile int* abort = &misc->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, NS = P.NS, NK = P.nk;
  const int VB = a.r_v * 2;   // bytes of a latent V row

  // ---------------------------------------------------------- work range
  // head-tiles (sequence, head, tile) in order; CTA c takes [c per, (c + 1) per)
  {
    const int per_thr = (a.B + kDtThreads - 1) / kDtThreads;
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
      constexpr int kPer = kDtThreads / 32;
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
    const long long total = static_cast<long long>(H) * misc->total_seq_tiles;
    const long long per = max(1LL, (total + a.grid - 1) / a.grid);
    const long long f0 = static_cast<long long>(blockIdx.x) * per;
    const long long f1 = min(total, f0 + per);
    long long P0 = misc->scan[tid];
    for (int b = b0; b < b1; ++b) {
      const int nb = (clamp_len(__ldg(a.seq_lens + b), a.L_max) + kTile - 1) / kTile;
      if (nb > 0 && f0 < f1 && H * P0 <= f0 && f0 < H * (P0 + nb)) {
        const long long rem = f0 - H * P0;
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

  TileWalker start;
  start.b = misc->start_b;
  start.h = misc->start_h;
  start.t = misc->start_t;
  start.L = clamp_len(__ldg(a.seq_lens + start.b), a.L_max);
  start.nb = (start.L + kTile - 1) / kTile;

  // ---------------------------------------------------------- set-up
  auto bar = [&](const uint64_t& m) { return smem_u32(&m); };
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) { mbar_init(bar(misc->full[s]), 1); mbar_init(bar(misc->empty[s]), 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(bar(misc->img_full[i]), 1); mbar_init(bar(misc->img_empty[i]), 1); }
    for (int g = 0; g < kNG; ++g) { mbar_init(bar(misc->gfull[g]), 1); mbar_init(bar(misc->gempty[g]), 4); }
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
    // Per unit: its image into buffer unit & 1, once the MMAs of the unit two back
    // are done with it.  Per head-tile: the rotary tile and the K latent boxes (TMA,
    // swizzled as the MMA reads them; rows past the cache end read as zero, rows
    // past the sequence end are masked), and an L2 prefetch of its V rows.
    if (lane == 0) {
      prefetch_tmap(&maps.kr);
      prefetch_tmap(&maps.ck);
      const uint64_t pol = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      TileWalker w = start;
      SlotPos sp{0, 0u};
      int unit = -1, issued = 0;
      bool ok = true;
      for (int lp = 0; lp < count && ok; ++lp) {
        const int z = w.b * H + w.h;
        if (lp == 0 || w.t == 0) {
          ++unit;
          const int ib = unit & 1;
          if (unit >= 2 && !(ok = mbar_wait(bar(misc->img_empty[ib]), ((unit >> 1) - 1) & 1, abort, a.status))) break;
          if (unit == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // images written
          const uint32_t fb = bar(misc->img_full[ib]);
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(a.zimg_stride));
          bulk_load(sbase + P.imgs + ib * P.img, a.zimg + static_cast<int64_t>(z) * a.zimg_stride,
                    static_cast<uint32_t>(a.zimg_stride), fb);
        }
        if (!(ok = mbar_wait(bar(misc->empty[sp.slot]), sp.phase ^ 1u, abort, a.status))) break;
        const uint32_t fb = bar(misc->full[sp.slot]);
        const uint32_t dst = sbase + P.ring + sp.slot * P.slot;
        const int y = w.t * kTile;
        const uint32_t rows = static_cast<uint32_t>(min(kTile, w.L - y));
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(kRTile + NK * kCkBox));
        tma_load_3d_hint(dst, &maps.kr, fb, 0, y, z, pol);
        for (int kb = 0; kb < NK; ++kb) tma_load_3d_hint(dst + kRTile + kb * kCkBox, &maps.ck, fb, 16 * kb, y, z, pol);
        // the V rows stay in L2 until the epilogue reads them (it reads them with an
        // evict-first policy, so they leave once used)
        prefetch_l2_bulk_hint(static_cast<const uint8_t*>(a.cache_v) + (static_cast<int64_t>(z) * a.L_max + y) * VB,
                              rows * VB, pol_keep);
        ++issued;
        sp.next(1, NS);
        tile_advance(w, a);
      }
      // Let every copy this CTA issued land before the CTA can exit.
      for (int i = max(0, issued - NS); i < issued; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->full[i % NS]), (i / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
      for (int u = max(0, unit - 1); u <= unit; ++u) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar(misc->img_full[u & 1]), (u >> 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // Per head-tile, into the next D buffer: the four rotary MMAs and the content
    // MMAs (as the small-rank kernel); its commit frees the ring slot and, at the
    // unit's last tile here, the image buffer.
    auto agree = [](bool r) { return __all_sync(0xffffffffu, r); };
    const uint32_t idesc_rot = umma_idesc_bf16(128, 32, false, false);
    const uint32_t idesc_con = umma_idesc_bf16(128, 16, false, false);
    const int style = a.rope_style;
    TileWalker w = start;
    SlotPos sp{0, 0u}, gp{0, 0u};
    int unit = -1;
    bool ok = true;
    for (int lp = 0; lp < count && ok; ++lp) {
      const bool unit_end = lp == count - 1 || w.t == w.nb - 1;
      if (lp == 0 || w.t == 0) {
        ++unit;
        if (!(ok = agree(mbar_wait(bar(misc->img_full[unit & 1]), (unit >> 1) & 1, abort, a.status)))) break;
      }
      if (!(ok = agree(mbar_wait(bar(misc->full[sp.slot]), sp.phase, abort, a.status)))) break;
      if (!(ok = agree(mbar_wait(bar(misc->gempty[gp.slot]), gp.phase ^ 1u, abort, a.status)))) break;
      tc_fence_after();
      const uint32_t d = tmem + gp.slot * kDCols;
      const uint32_t ra = sbase + P.ring + sp.slot * P.slot;
      const uint32_t ib = sbase + P.imgs + (unit & 1) * P.img;
      const uint64_t a_rot = umma_desc(ra, 16, 1024, kSw128);
#pragma unroll
      for (int G = 0; G < 2; ++G)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          umma_bf16_warp(d + 32 * G, a_rot + 2 * rot_kstep(style, G, kk),
                         umma_desc(ib + (2 * G + kk) * kRotBlock, 16, 256, kSw32), idesc_rot, kk);
      for (int kb = 0; kb < NK; ++kb)
        umma_bf16_warp(d + 64, umma_desc(ra + kRTile + kb * kCkBox, 16, 256, kSw32),
                       umma_desc(ib + 4 * kRotBlock + kb * kConBlock, 16, 256, kSw32), idesc_con, kb);
      umma_commit_warp(bar(misc->gfull[gp.slot]));
      umma_commit_warp(bar(misc->empty[sp.slot]));                       // the slot's rows are read
      if (unit_end) umma_commit_warp(bar(misc->img_empty[unit & 1]));   // the image is no longer read
      gp.next(1, kNG);
      sp.next(1, NS);
      tile_advance(w, a);
    }
    // this warp's MMAs complete before TMEM is released
    umma_commit_warp(bar(misc->mma_done));
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar(misc->mma_done), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
  } else {
    // ======================================================== epilogue (warps 2-9)
    // Group g takes the CTA's head-tiles lp = g mod 2 (D buffers g, g + 2, g + 4);
    // thread (TMEM quadrant q, lane) owns token row 32 q + lane of a tile, and lane
    // the V column pairs lane + 32 i of its warp's sum.
    const int we = warp - 2, g = we >> 2, q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int npairs = a.r_v / 2;
    const uint64_t pol_v = l2_policy_evict_first();   // V rows: read once
    asm volatile("griddepcontrol.wait;" ::: "memory");   // table and sc b0 written
    SlotPos gp{g, 0u};
    TileWalker w = start;
    float m = -INFINITY, l = 0.f, qb0 = 0.f;
    float acc[2 * NPL];
    bool ok = true;
    for (int lp = 0; lp < count && ok; ++lp) {
      const bool unit_start = lp == 0 || w.t == 0;
      const bool unit_end = lp == count - 1 || w.t == w.nb - 1;
      const int64_t u = static_cast<int64_t>(w.b) * H + w.h;
      if (unit_start) {
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < 2 * NPL; ++i) acc[i] = 0.f;
        qb0 = __ldg(a.qb0 + u);
      }
      if ((lp & 1) == g) {
        const int nvalid = min(kTile, w.L - w.t * kTile);
        const bool valid = row < nvalid;
        // V rows of the warp's tokens (valid ones only; lane = column pairs): the first
        // 8 tokens' loads go out before anything else of the tile, the other 24 once
        // the score is formed, so both wait behind other work
        const int nv = min(32, max(0, nvalid - 32 * q));
        const uint32_t* vrows = static_cast<const uint32_t*>(a.cache_v) +
                                (u * a.L_max + static_cast<int64_t>(w.t) * kTile + 32 * q) * npairs;
        uint32_t va[8][NPL];
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
          for (int i = 0; i < NPL; ++i) {
            const int pr = lane + 32 * i;
            va[k][i] = k < nv && pr < npairs ? ldg_hint(vrows + static_cast<int64_t>(k) * npairs + pr, pol_v) : 0u;
          }
        // cos / sin of this token's position
        float cs[kRope];
        {
          int64_t j = static_cast<int64_t>(w.t) * kTile + row;
          if (j >= a.trig_rows) j = a.trig_rows - 1;   // past the cache end: masked anyway
          const float* tp = a.trigT + j;
#pragma unroll
          for (int c = 0; c < kRope; ++c) cs[c] = __ldg(tp + c * a.trig_rows);
        }
        if (!(ok = warp_wait(bar(misc->gfull[gp.slot]), gp.phase, abort, a.status))) break;
        tc_fence_after();
        // ---- s_j = sc b0 + content (hi + lo) + sum_f U_f cos + V_f sin (log2 units),
        // the 64 (U, V) columns read from TMEM in two halves
        float x0 = 0.f, x1 = 0.f, y0 = 0.f, y1 = 0.f, z0 = 0.f, z1 = 0.f, t0 = 0.f, t1 = 0.f;
        float uc[2];
        {
          const uint32_t gb = tmem + lane_base + gp.slot * kDCols;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float uu[32];
            tmem_ld_x32(gb + 32 * hf, uu);
            if (hf == 1) tmem_ld_x2(gb + 64, uc);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              fma_pair(x0, x1, uu[2 * i], uu[2 * i + 1], cs[32 * hf + 2 * i], cs[32 * hf + 2 * i + 1]);
              fma_pair(y0, y1, uu[2 * i + 2], uu[2 * i + 3], cs[32 * hf + 2 * i + 2], cs[32 * hf + 2 * i + 3]);
              fma_pair(z0, z1, uu[2 * i + 4], uu[2 * i + 5], cs[32 * hf + 2 * i + 4], cs[32 * hf + 2 * i + 5]);
              fma_pair(t0, t1, uu[2 * i + 6], uu[2 * i + 7], cs[32 * hf + 2 * i + 6], cs[32 * hf + 2 * i + 7]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(misc->gempty[gp.slot]));
        gp.next(kEpiGroups, kNG);
        const float sr = ((x0 + x1) + (y0 + y1)) + ((z0 + z1) + (t0 + t1));
        const float s = valid ? (qb0 + (uc[0] + uc[1])) + sr : -INFINITY;

        // ---- online softmax per warp, reference raised lazily (by more than 2^8)
        const float mt = warp_max_redux(s);
        if (mt > m + kRescaleLog2) {
          const float alpha = m == -INFINITY ? 0.f : exp2f(m - mt);
          l *= alpha;
#pragma unroll
          for (int i = 0; i < 2 * NPL; ++i) acc[i] *= alpha;
          m = mt;
        }
        const float p = valid ? exp2f(s - m) : 0.f;
        l += warp_sum(p);

        // ---- sum_j p_j c_v,j (a token past the sequence end has p = 0 and v = 0)
        if (nv > 8) {
          uint32_t vb[24][NPL];
#pragma unroll
          for (int k = 0; k < 24; ++k)
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
              const int pr = lane + 32 * i;
              vb[k][i] = 8 + k < nv && pr < npairs ? ldg_hint(vrows + static_cast<int64_t>(8 + k) * npairs + pr, pol_v) : 0u;
            }
#pragma unroll
          for (int k = 0; k < 24; ++k) {
            const float pv = __shfl_sync(0xffffffffu, p, 8 + k);
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
              acc[2 * i] = fmaf(pv, __uint_as_float(vb[k][i] << 16), acc[2 * i]);
              acc[2 * i + 1] = fmaf(pv, __uint_as_float(vb[k][i] & 0xFFFF0000u), acc[2 * i + 1]);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float pv = __shfl_sync(0xffffffffu, p, k);
#pragma unroll
          for (int i = 0; i < NPL; ++i) {
            acc[2 * i] = fmaf(pv, __uint_as_float(va[k][i] << 16), acc[2 * i]);
            acc[2 * i + 1] = fmaf(pv, __uint_as_float(va[k][i] & 0xFFFF0000u), acc[2 * i + 1]);
          }
        }
      }
      if (unit_end) {
        // record (m, l, -, -, acc) of (unit, CTA, group, warp); a group that took no
        // tile of the unit here writes m = -inf, l = 0, acc = 0
        float* rec = a.partials +
                     ((u + blockIdx.x) * kDecoupledTileRecords + g * 4 + q) * (a.r_v + kRecordHead);
        if (lane == 0) { rec[0] = m; rec[1] = l; }
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int pr = lane + 32 * i;
          if (pr < npairs) *reinterpret_cast<float2*>(rec + kRecordHead + 2 * pr) = make_float2(acc[2 * i], acc[2 * i + 1]);
        }
      }
      tile_advance(w, a);
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

template <int NPL>
cudaError_t launch_tile_instance(const DecodeArgs& a, const DecoupledMaps& m, int bytes, cudaStream_t s) {
  auto kern = decoupled_tile_kernel<NPL>;
  static int configured = 0;
  if (configured < bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured = bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kDtThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, m);
}

}  // namespace

bool decoupled_small_supported(int H, int r_k, int r_v) {
  DsPlan p;
  return make_ds_plan(H, r_k, r_v, &p);
}

size_t decoupled_small_img_stride(int r_k) { return static_cast<size_t>(4 * kRotBlock + (r_k / 16) * kConBlock); }

int64_t decoupled_small_trig_rows(int64_t L_max) { return (L_max + kTile - 1) / kTile * kTile; }

bool decoupled_tile_supported(int r_k, int r_v) {
  DtPlan p;
  return make_dt_plan(r_k, r_v, &p);
}

cudaError_t launch_decoupled_tile(const DecodeArgs& a, const DecoupledMaps& m, cudaStream_t s) {
  DtPlan P;
  if (!make_dt_plan(a.r_k, a.r_v, &P) || a.records_per_cta != kDecoupledTileRecords) return cudaErrorInvalidValue;
  const int trig_blocks = static_cast<int>((a.trig_rows + kTrigJ - 1) / kTrigJ);
  if (a.z_seqs < 1 || a.z_seqs > kDzSeqs) return cudaErrorInvalidValue;
  const int z_blocks = a.H * ((a.B + a.z_seqs - 1) / a.z_seqs);
  cudaError_t e = launch_pdl(decoupled_small_z_kernel, dim3(z_blocks + trig_blocks), dim3(kDzThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  switch ((a.r_v + 63) / 64) {
    case 1: e = launch_tile_instance<1>(a, m, P.bytes, s); break;
    case 2: e = launch_tile_instance<2>(a, m, P.bytes, s); break;
    case 3: e = launch_tile_instance<3>(a, m, P.bytes, s); break;
    default: e = launch_tile_instance<4>(a, m, P.bytes, s); break;
  }
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, s);
}

cudaError_t launch_decoupled_small(const DecodeArgs& a, const DecoupledMaps& m, cudaStream_t s) {
  DsPlan P;
  if (!make_ds_plan(a.H, a.r_k, a.r_v, &P)) return cudaErrorInvalidValue;
  const int trig_blocks = static_cast<int>((a.trig_rows + kTrigJ - 1) / kTrigJ);
  if (a.z_seqs < 1 || a.z_seqs > kDzSeqs) return cudaErrorInvalidValue;
  const int z_blocks = a.H * ((a.B + a.z_seqs - 1) / a.z_seqs);
  cudaError_t e = launch_pdl(decoupled_small_z_kernel, dim3(z_blocks + trig_blocks), dim3(kDzThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  if (a.r_k == 16 && a.r_v == 32) e = launch_instance<16, 32>(a, m, P.bytes, s);
  else if (a.r_k == 16 && a.r_v == 64) e = launch_instance<16, 64>(a, m, P.bytes, s);
  else if (a.r_k == 32 && a.r_v == 32) e = launch_instance<32, 32>(a, m, P.bytes, s);
  else e = launch_instance<32, 64>(a, m, P.bytes, s);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, s);
}

}  // namespace lla
