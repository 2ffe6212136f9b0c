// lla_kernels.h — parameter blocks and launchers shared by the host API
// (lla_api.cu) and the kernels (lla_decode.cu, lla_encode.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "lla_sm103.cuh"

namespace lla {

constexpr int kMaxStages = 8;
constexpr int kMaxGrid = 1024;          // upper bound on decode CTAs (workspace sizing)
constexpr int kMaxRankPerHead = 256;    // r_k, r_v of the per-head variant
constexpr int kMaxRank2d = 512;         // r_k, r_v of LLA-2D
constexpr int kDecodeThreads = 224;     // producer, score-MMA, 4 epilogue, value-MMA warps
constexpr int kWarpVMma = 6;            // decode warp issuing the value MMAs
constexpr int kRecordsPerCta = 4;       // split records per (unit, CTA): one per epilogue warp
constexpr int kRecordHead = 4;          // record = {m, l, -, -, acc[r_v]}: acc 16-byte aligned
constexpr int kEncodeThreads = 192;     // producer warp, MMA warp, 4 epilogue warps
constexpr int kSmemLimit = 232448;      // dynamic shared memory per block on sm_100/103

// Shared-memory plan of the per-head bf16 decode kernel (byte offsets from a
// 1024-aligned base).
struct DecodePlan {
  ChunkPlan kplan;                   // K latent chunks (64/32/16 wide, 128 rows)
  ChunkPlan vplan;                   // V latent chunks, 32 wide (64B swizzle)
  int SK, SV;                        // ring depths
  int NZ;                            // query-operand (Z) buffers: 2 = built one unit ahead
  int vlag;                          // V tile i is requested after K tile i + vlag
  int k_stage, v_stage, z_stage;     // stage strides
  int v_ring, k_ring, z, aug_a, aug_b, trig, misc;
  int bytes;                         // total dynamic smem incl. alignment slack
};

// Shared-memory plan of the per-head small-rank kernel (byte offsets from a
// 1024-aligned base): the query images of the current sequence, a ring of
// (K tile, V tile) slots, per-warp softmax state and the barriers.  Heads are
// taken nwg at a time ("head sets", one head per epilogue group): a set's image
// stacks its heads' Z rows and bias rows as one MMA B operand of N rows.
struct DecodeSmallPlan {
  int nwg;                           // epilogue warp groups in use = heads per set (4 if H % 4 == 0, else 2)
  int nsets;                         // head sets per position (H / nwg)
  int N;                             // set image rows = G columns (MMA N): nwg (r_k + 2) rounded up to 16
  int img;                           // bytes of one set image (2 chunks of N rows x 128 B)
  int NG;                            // G buffers in TMEM (one set each)
  int k_tile, v_tile, slot;          // bytes of a K tile, a V tile, a ring slot
  int NS;                            // ring slots (a multiple of nwg)
  int imgs, ring, acc, ml, misc;
  int bytes;                         // total dynamic smem incl. alignment slack
  int log2P;                         // set-page layout (pages of 8..64 tokens): log2 of the page
                                     // size, each ring slot one head set's tile; 0 otherwise
};

constexpr int kSmallThreads = 576;      // producer, MMA issuer, 4 x 4 epilogue warps
constexpr int kSmallMaxHeads = 16;      // every head's query image stays resident
constexpr int kSmallMaxNS = 8;

struct DecodeArgs {
  int B, H, r_k, r_v, rope_style, grid;
  int shared_latent;                 // fp32 path: 1 = LLA-2D cache [B][L_max][r] read by every head
  int64_t L_max, rope_len, mu_hstride;
  const void* q;                     // [B][H][128]
  const int32_t* seq_lens;           // [B]
  const int32_t* q_pos;              // [B]
  const void* cache_k;               // fp32 path only (bf16 path reads via TMA)
  const void* cache_v;
  const void* w_up_k;                // loop-t slice [H][128][r_k]
  const void* w_up_v;                // loop-t slice [H][128][r_v]
  const float* mu_k;                 // loop-t slice: element (h, e) at mu_k[h*mu_hstride + e]
  const float* mu_v;
  const float* rope_cos;             // [rope_len][64]
  const float* rope_sin;
  float* out;                        // [B][H][128]
  float* lse;                        // [B][H]
  uint32_t* status;                  // workspace status word
  float* partials;                   // [(B*H + kMaxGrid) * 4][r_v + 4] records per (unit, CTA, warp)
  float* scores;                     // fp32 path: [B][H][L_max]
  uint8_t* zimg;                     // bf16 path: per-unit query-operand images
  int64_t zimg_stride;               // bytes per unit image (Z chunks, then 4 KB bias operand)
  uint32_t* trig16;                  // small-rank path: f16 RoPE rows [trig_rows][64 pairs] (cos, then sin)
  int64_t trig_rows;
  int pos_major;                     // records indexed ((b + cta) H + h) 4 + warp (small-rank path)
  int combine_units;                 // sequences per combine block (1..16)
  int records_per_cta;               // records per (unit, CTA): 4, or 1 (decoupled kernel)
  const void* k_rope;                // decoupled path: rotary keys [B][H][L_max][d_rope]
  int d_rope;                        // decoupled path: rotary branch width (0: full-RoPE path)
  int z_seqs;                        // decoupled tensor-core paths: sequences per image block (1..8)
  float* trigT;                      // decoupled small-rank path: fp32 RoPE table [64][trig_rows]
  float* qb0;                        // decoupled small-rank path: sc q_c . mu_k per (sequence, head)
  // Paged cache (per-head variant): cache_k / cache_v are page pools
  // [num_pages][H][page_size][r]; logical page p of sequence b is physical page
  // block_table[b * max_pages + p].  block_table == nullptr: dense [B][H][L_max][r].
  const int32_t* block_table;
  int page_size;
  int max_pages;
  int64_t num_pages;
  DecodePlan plan;
  DecodeSmallPlan splan;
  int v_page_major;                  // tile kernel, page pieces: V tile stored page-major (maps.v4)
};

// Launch `kern` as a programmatic dependent of the previous grid on stream `s`: its
// blocks may be scheduled while that grid drains, so the kernel must execute
// griddepcontrol.wait before it reads or writes anything that grid (or an earlier
// one) produces or consumes.
template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Validation of the block-table entries a paged decode reads: the decode kernels
// clamp an entry into the pool without checking it, and the query-image kernels
// (one block per sequence here) record LLA_ERR_DEVICE_ARG for any entry of a
// logical page holding one of sequence b's tokens that lies outside [0, num_pages).
__device__ __forceinline__ void check_block_table(const DecodeArgs& a, int b, int tid, int nthreads) {
  if (a.block_table == nullptr) return;
  int L = __ldg(a.seq_lens + b);
  L = L < 0 ? 0 : (L > a.L_max ? static_cast<int>(a.L_max) : L);
  const int used = (L + a.page_size - 1) / a.page_size;
  for (int lp = tid; lp < used; lp += nthreads) {
    const int pg = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + lp);
    if (pg < 0 || pg >= a.num_pages) record_status(a.status, LLA_ERR_DEVICE_ARG);
  }
}

// Physical page of logical page lp of sequence b for the bf16 decode producers,
// clamped into the pool (entries were checked by check_block_table).
__device__ __forceinline__ int page_of(const DecodeArgs& a, int b, int lp) {
  const int pg = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + lp);
  return min(max(pg, 0), static_cast<int>(a.num_pages) - 1);
}

// Token eviction (sink + window budget) over a dense latent cache.
struct EvictArgs {
  int B;
  int units_per_seq;                 // H (per-head) or 1 (LLA-2D)
  int r_k, r_v, esize;
  int sink, window;
  int64_t L_max;
  void* cache_k;                     // [B][units_per_seq][L_max][r] rows
  void* cache_v;
  int32_t* seq_lens;                 // [B], updated to sink + window where over budget
  uint32_t* status;
};
cudaError_t launch_evict_window(const EvictArgs& a, cudaStream_t s);

struct DecodeMaps {
  CUtensorMap k[3];                  // latent K boxes of width 64 / 32 / 16
  CUtensorMap v;                     // latent V boxes of width 32
  // page pool with pages of 8..64 tokens and r_v a multiple of 32: one page of V as
  // one box [chunk][P rows][32 columns] (4-D view: columns, rows, 32-column chunks,
  // page-head), the page-major V layout of the tile kernel (DecodeArgs::v_page_major)
  CUtensorMap v4;
};

bool make_decode_plan(int r_k, int r_v, DecodePlan* p);
bool make_decode_small_plan(int H, int r_k, int r_v, DecodeSmallPlan* p);
// The small-rank kernel over a page pool with pages of 8, 16, 32 or 64 tokens:
// ring slots of a whole head set, filled with one copy per page for the set's heads
// (contiguous in the pool).  False if two such slots do not fit.
bool make_decode_small_setpage_plan(int H, int r_k, int r_v, int page_size, DecodeSmallPlan* p);
size_t decode_small_img_stride(int H, int r_k);   // bytes per (sequence, head set) image
int64_t decode_small_trig_rows(int64_t L_max, int64_t rope_len);
cudaError_t launch_decode_small_bf16(const DecodeArgs& a, cudaStream_t s);
// Merge a unit's split records, apply W_up,v once and normalise (both per-head paths).
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t s);
// Sequences per combine block: as many as keep about two blocks per SM, at most 16.
int decode_combine_units(int B, int H, int sms);

// Absorbed decoupled-RoPE decode (content path on the latents + rotary branch).
// Small ranks (r_k in {16, 32}, r_v in {32, 64}, H even <= 16): rotary branch and
// content score on the tensor cores, position-major split (a.pos_major = 1, four
// records per CTA).  Needs a.zimg (B images per (sequence, head),
// decoupled_small_img_stride bytes apart), a.qb0 [B H], a.trigT [64][a.trig_rows].
struct DecoupledMaps {
  CUtensorMap kr;                    // rotary keys [B H][L_max][64], boxes 64 x 128 (128-byte swizzle)
  CUtensorMap ck;                    // K latents [B H][L_max][r_k], boxes 16 x 128 (32-byte swizzle)
};
bool decoupled_small_supported(int H, int r_k, int r_v);
size_t decoupled_small_img_stride(int r_k);
int64_t decoupled_small_trig_rows(int64_t L_max);
cudaError_t launch_decoupled_small(const DecodeArgs& a, const DecoupledMaps& m, cudaStream_t s);
// Other bf16 shapes with r_k <= 128, r_v <= 256: the same MMA chain over 128-token
// tiles of one (sequence, head) (tile-major split, a.pos_major = 0, eight records
// per CTA), V read from L2 by the epilogue.  Same workspace regions as above.
constexpr int kDecoupledTileRecords = 8;
bool decoupled_tile_supported(int r_k, int r_v);
cudaError_t launch_decoupled_tile(const DecodeArgs& a, const DecoupledMaps& m, cudaStream_t s);
// fp32 softmax over a.scores and the V path (shared by the fp32 decode paths).
cudaError_t launch_decode_f32_values(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decoupled_f32(const DecodeArgs& a, cudaStream_t s);

cudaError_t launch_decode_bf16(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t s);
cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t s);
// The same plain kernels over bf16 storage (fp32 arithmetic): the LLA-2D shapes
// the CTA-pair kernels do not take (ranks above 128 / 256, odd or > 16 heads).
cudaError_t launch_decode_plain_bf16(const DecodeArgs& a, cudaStream_t s);

// Page sizes the tile kernel's copy path takes: whole tiles inside a page (a multiple
// of 128 tokens) or a tile as 128/P pieces of P tokens (P a multiple of 8 dividing 128).
__host__ __device__ inline bool tile_kernel_page_size(int P) {
  return P > 0 && (P % 128 == 0 || (P % 8 == 0 && 128 % P == 0));
}
// bf16 decode over a paged cache of any page size (the tile kernel's other page sizes):
// one CTA per (sequence, head), rows gathered through the block table.
cudaError_t launch_decode_paged_generic(const DecodeArgs& a, cudaStream_t s);
size_t decode_paged_generic_smem(int r_k, int r_v);

// ----------------------------------------------------------------- exact window

struct WindowArgs {
  int B, H, W, rope_style;
  int64_t rope_len;
  const void* q;                     // [B][H][128] (storage dtype)
  const void* k_win;                 // [B][H][W][128] exact keys of the loop, before RoPE
  const void* v_win;                 // [B][H][W][128]
  const int32_t* win_len;            // [B] valid window tokens
  const int32_t* win_pos;            // [B] position of window token 0
  const int32_t* q_pos;              // [B]
  const float* rope_cos;             // [rope_len][64]
  const float* rope_sin;
  float* out;                        // [B][H][128] in: latent part, out: merged
  float* lse;                        // [B][H]      likewise (natural log)
  uint32_t* status;
};

cudaError_t launch_window_attn(const WindowArgs& a, bool bf16, cudaStream_t s);

// ----------------------------------------------------------------- LLA-2D decode

constexpr int kScore2dThreads = 320;    // producer, MMA issuer / relay, 8 epilogue warps
constexpr int kBlock2dTokens = 256;     // tokens of a pair block: one 128-token tile per CTA
constexpr int kMax2dHeads = 16;         // heads of one shared latent (value MMA N = 16)
constexpr int kMaxPairs = kMaxGrid / 2;
constexpr int kValue2dThreads = 192;    // producer, MMA issuer, 4 scaling / record warps

// Shared-memory plans (byte offsets from a 1024-aligned base) of the LLA-2D score
// kernel (CTA pairs) and value kernel (one CTA per SM).
struct Decode2dPlan {
  int nkc;                           // 64-wide K chunks of a latent / query-operand row (r_k <= 128)
  int k_stage, z_stage;              // ring stage strides
  int k_ring, z_ring, aug_a, misc;
  int bytes;
  int nvb;                           // 64-wide r_v boxes of a value tile (r_v <= 256)
  int nvc;                           // 128-row r_v chunks (value MMA M = 128)
  int v_stage;                       // value ring stage: V tile, then the weight tile
  int v_ring, v_p, v_misc;
  int v_bytes;
};

struct Decode2dArgs {
  int B, H, r_k, r_v, rope_style, pairs, units;
  int64_t L_max, rope_len;
  int64_t ntiles;                    // 128-token tiles per sequence slot: ceil(L_max / 128)
  const void* q;                     // [B][H][128]
  const int32_t* seq_lens;           // [B]
  const int32_t* q_pos;              // [B]
  const void* w_up_k;                // loop-t slice [H*128][r_k]
  const void* w_up_v;                // loop-t slice [H*128][r_v]
  const float* mu_k;                 // loop-t slice [H*128]
  const float* mu_v;
  const float* rope_cos;             // [rope_len][64]
  const float* rope_sin;
  float* out;                        // [B][H][128]
  float* lse;                        // [B][H]
  uint32_t* status;
  float* rec_acc;                    // [B + units][H][r_v] run records of the value kernel
  float* rec_ml;                     // [B + units][H][2]   (m, l) of each record
  uint8_t* zimg;                     // per sequence: nkc chunks of [H*128 rows][128 B], then the bias
                                     // operand [H*128 rows][16 bf16] (32 B rows)
  int64_t zimg_stride;               // bytes per sequence image
  int64_t zchunk_bytes;              // H * 128 * 128
  float* trigT;                      // [128][trig_rows]: cos(j th_c) for c < 64, then sin(j th_c-64)
  int64_t trig_rows;                 // positions of trigT: L_max rounded up to a whole block
  uint16_t* pw;                      // softmax weights, bf16 [B][H][ntiles * 128], each 32-token group
                                     // relative to 2^m of that group
  float* grp_m;                      // [B][H][ntiles * 4]: m of each 32-token group (an integer in
                                     // log2 units, -inf for a group past the sequence end)
  Decode2dPlan plan;
};

struct Decode2dMaps {
  CUtensorMap k;                     // latent K: box (64, 128, 1) over (r_k, L_max, B), 128B swizzle
  CUtensorMap z;                     // query-operand images, copied as stored (already swizzled):
                                     // box (64, 128, 1) over (64, nkc * H * 128 rows, B)
  CUtensorMap zb;                    // their bias operand: box (16, 128, 1) over (16, H * 128 rows, B)
  CUtensorMap v;                     // latent V: box (64, 128, 1) over (r_v, L_max, B), 128B swizzle
  CUtensorMap p;                     // weights: box (64, H, 1) over (ntiles * 128, H, B), 128B swizzle
};

bool make_decode2d_plan(int H, int r_k, int r_v, Decode2dPlan* p);
size_t decode2d_zimg_stride(int H, int r_k);
int64_t decode2d_trig_rows(int64_t L_max);
cudaError_t launch_decode2d_bf16(Decode2dArgs& a, const Decode2dMaps& maps, cudaStream_t s);

// ----------------------------------------------------------------- encode

struct EncodeArgs {
  int N, H, Td, r_k, r_v, B;
  int64_t L_max;
  const void* x_k;                   // [N][H][Td]
  const void* x_v;
  const int32_t* seq_idx;
  const int32_t* pos;
  const void* w_down_k;              // [H][Td][r_k]
  const void* w_down_v;
  const float* mu_k;                 // [H][Td]
  const float* mu_v;
  void* cache_k;
  void* cache_v;
  uint32_t* status;
  float* bias;                       // workspace [2][H][512]: mu W_down per head/axis
  const int32_t* block_table;        // paged cache (as DecodeArgs), or nullptr
  int page_size;
  int max_pages;
  int64_t num_pages;
};

struct EncodePlan {
  ChunkPlan bk, bv;                  // W_down chunks (64 K-rows per stage)
  int S;                             // ring depth
  int stage;                         // stage stride
  int a_off, b_off;                  // inside a stage
  int ring, misc, bytes;
  int tmem_cols;
  int nacc, acc_stride;              // TMEM accumulators (1 or 2) and their column stride
  int sms;                           // persistent grid size (set by the caller)
};

struct EncodeMaps {
  CUtensorMap xk, xv;                // box (64, 1, 128)
  CUtensorMap wk[3], wv[3];          // box (w, 64, 1)
};

bool make_encode_plan(int r_k, int r_v, int Td, EncodePlan* p);
// CTA-pair encode (ranks multiples of 32 up to 256): one pair MMA covers two tiles
bool make_encode_pair_plan(int r_k, int r_v, int Td, EncodePlan* p);
cudaError_t launch_encode_pair(const EncodeArgs& a, const EncodePlan& plan, const EncodeMaps& m, cudaStream_t s);
cudaError_t launch_encode_bf16(const EncodeArgs& a, const EncodePlan& plan, const EncodeMaps& m,
                               cudaStream_t s);
cudaError_t launch_encode_f32(const EncodeArgs& a, cudaStream_t s);

// ----------------------------------------------------------------- scratch without allocation

// Device address of the library's fixed scratch array on the current device (looked
// up once per device, defined in lla_noalloc.cu).
lla_status noalloc_scratch_address(void** out);
// lla_decode_attn that zeroes the status word on `stream` after every host check has
// passed and before its first launch (a call the host checks reject enqueues nothing).
lla_status decode_attn_status_cleared(const lla_dims* dims, int loop_t, const void* q, lla_cache cache,
                                      const int32_t* seq_lens, const int32_t* q_pos, const void* w_up_k,
                                      const void* w_up_v, const float* mu_k, const float* mu_v,
                                      const float* rope_cos, const float* rope_sin, int64_t rope_len,
                                      float* out, float* lse, void* workspace, size_t ws_bytes, void* stream);

}  // namespace lla
