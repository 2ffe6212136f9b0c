// lla_api.cu — the C ABI of liblla.so (declared in include/lla.h): host-side
// argument checks, workspace layout, TMA descriptors and kernel launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>

#include "lla_kernels.h"

using namespace lla;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D tiled map over a dense row-major tensor [d2][d1][d0] of `esize`-byte elements.
// Swizzle = the atom matching the box row bytes (128 / 64 / 32 B).
// 3-D map with explicit byte strides of dimensions 1 and 2 and an explicit swizzle.
bool make_map_3d_strided(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t d0, uint64_t d1,
                         uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
                         CUtensorMapSwizzle sw) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t d0,
                 uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  const int row_bytes = static_cast<int>(b0) * esize;
  const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t partials, rec_ml, bias, scores, zimg, zimg_stride, trig16, pw, grp_m, total;
};

// Bytes of one unit's query-operand image: Z (128 rows x r_k bf16, K-chunk
// layout) followed by the 4 KB bias operand, padded to 128 bytes.
size_t zimg_stride(int r_k) {
  return (static_cast<size_t>(make_chunk_plan(r_k, kTile).bytes) + 4096 + 127) / 128 * 128;
}

// Per-head bf16 decode at small ranks runs the small-rank kernel (its shapes and
// shared-memory plan decide); every other per-head bf16 shape the tile kernel.
bool small_path(const lla_dims* d) {
  DecodeSmallPlan p;
  return d->variant == LLA_PER_HEAD && d->dtype == LLA_BF16 && make_decode_small_plan(d->H, d->r_k, d->r_v, &p);
}

WsLayout ws_layout(const lla_dims* d, int B, int64_t L_max) {
  WsLayout w{};
  size_t off = 256;  // status word
  if (d->variant == LLA_2D) {
    // run records of the value kernel, encode bias (one "head" of width T*H*d),
    // fp32 scores, per-sequence query-operand images
    const size_t nrec = static_cast<size_t>(2) * (static_cast<size_t>(B) + kMaxPairs);
    w.partials = off; off += al256(nrec * d->H * d->r_v * 4);
    w.rec_ml = off;   off += al256(nrec * d->H * 2 * 4);
    w.bias = off;     off += al256(static_cast<size_t>(2) * kMaxRank2d * 4);
    // fp32 scores of the plain kernels (fp32 storage, and bf16 shapes the CTA-pair
    // kernels do not take)
    w.scores = off;
    Decode2dPlan pp;
    if (d->dtype == LLA_F32 || !make_decode2d_plan(d->H, d->r_k, d->r_v, &pp))
      off += al256(static_cast<size_t>(B) * d->H * L_max * 4);
    w.zimg = off;
    if (d->dtype == LLA_BF16 && d->r_k <= 128) {
      w.zimg_stride = decode2d_zimg_stride(d->H, d->r_k);
      off += al256(static_cast<size_t>(B) * w.zimg_stride);
    }
    // softmax weights (bf16 [B][H][tiles * 128]) and per-32-token-group m of the
    // score kernel
    const size_t tiles = static_cast<size_t>((L_max + kTile - 1) / kTile);
    // the transposed RoPE table [128][positions] fp32, positions up to L_max rounded
    // up to a whole 256-token block
    w.trig16 = off;
    if (d->dtype == LLA_BF16) off += al256(static_cast<size_t>(128) * decode2d_trig_rows(L_max) * 4);
    w.pw = off;
    if (d->dtype == LLA_BF16) off += al256(static_cast<size_t>(B) * d->H * tiles * kTile * 2);
    w.grp_m = off;
    if (d->dtype == LLA_BF16) off += al256(static_cast<size_t>(B) * d->H * tiles * 4 * 4);
    w.total = off;
    return w;
  }
  if (small_path(d)) {
    // small-rank kernel: records per (sequence + CTA, head, warp), per-unit query
    // images, f16 RoPE rows
    // (a CTA index is below min(kMaxGrid, positions): the grid never exceeds either)
    const size_t max_pos = static_cast<size_t>(B) * ((L_max + kTile - 1) / kTile);
    w.partials = off;
    off += al256((static_cast<size_t>(B) + std::min<size_t>(kMaxGrid, std::max<size_t>(1, max_pos))) * d->H *
                 kRecordsPerCta * (d->r_v + kRecordHead) * 4);
    w.bias = off; off += al256(static_cast<size_t>(2) * d->H * kMaxRank2d * 4);
    w.scores = off;
    w.zimg = off;
    // one image per (sequence, head set) of 4 heads (2 when H mod 4 = 2)
    w.zimg_stride = decode_small_img_stride(d->H, d->r_k);
    off += al256(static_cast<size_t>(B) * (d->H % 4 == 0 ? d->H / 4 : d->H / 2) * w.zimg_stride);
    w.trig16 = off;
    off += al256(static_cast<size_t>(decode_small_trig_rows(L_max, INT64_MAX)) * 256);
    w.total = off;
    return w;
  }
  w.partials = off; off += al256((static_cast<size_t>(B) * d->H + kMaxGrid) * kRecordsPerCta * (d->r_v + kRecordHead) * 4);
  w.bias = off; off += al256(static_cast<size_t>(2) * d->H * kMaxRank2d * 4);
  w.scores = off;
  if (d->dtype == LLA_F32) off += al256(static_cast<size_t>(B) * d->H * L_max * 4);
  w.zimg = off;
  w.zimg_stride = zimg_stride(d->r_k);
  if (d->dtype == LLA_BF16) off += al256(static_cast<size_t>(B) * d->H * w.zimg_stride);
  w.total = off;
  return w;
}

lla_status check_dims(const lla_dims* d) {
  if (!d) return LLA_ERR_INVALID_ARG;
  if (d->T < 1 || d->H < 1 || d->d_head < 2 || d->r_k < 1 || d->r_v < 1) return LLA_ERR_INVALID_ARG;
  if (d->variant != LLA_PER_HEAD && d->variant != LLA_2D) return LLA_ERR_INVALID_ARG;
  if (d->dtype != LLA_BF16 && d->dtype != LLA_F32) return LLA_ERR_INVALID_ARG;
  if (d->rope_style != LLA_ROPE_HALF && d->rope_style != LLA_ROPE_INTERLEAVED) return LLA_ERR_INVALID_ARG;
  if (!(d->rope_base > 0.f) || !std::isfinite(d->rope_base)) return LLA_ERR_INVALID_ARG;
  if (d->d_head != kHeadDim) return LLA_ERR_UNSUPPORTED;
  const int rmax = d->variant == LLA_2D ? kMaxRank2d : kMaxRankPerHead;
  if (d->r_k % 16 || d->r_v % 16 || d->r_k > rmax || d->r_v > rmax) return LLA_ERR_UNSUPPORTED;
  return LLA_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

extern "C" {

int lla_abi_version(void) { return LLA_ABI_VERSION; }

const char* lla_status_string(lla_status s) {
  switch (s) {
    case LLA_OK: return "ok";
    case LLA_ERR_INVALID_ARG: return "invalid argument";
    case LLA_ERR_UNSUPPORTED: return "unsupported shape, variant or dtype";
    case LLA_ERR_CUDA: return "CUDA error";
    case LLA_ERR_TIMEOUT: return "a kernel wait timed out";
    case LLA_ERR_DEVICE_ARG: return "out-of-range seq_lens/q_pos/seq_idx/pos seen on the device";
    case LLA_ERR_RANGE: return "a folded query operand exceeded the f16 range (small-rank decode)";
  }
  return "unknown status";
}

const char* lla_decode_kernel(const lla_dims* dims) {
  if (check_dims(dims) != LLA_OK) return nullptr;
  if (dims->dtype == LLA_F32) return "fp32";
  if (dims->variant == LLA_2D) {
    Decode2dPlan p;
    return make_decode2d_plan(dims->H, dims->r_k, dims->r_v, &p) ? "pair-2d" : "plain-2d";
  }
  if (small_path(dims)) return "small-rank";
  DecodePlan p;
  return make_decode_plan(dims->r_k, dims->r_v, &p) ? "tile" : nullptr;
}

const char* lla_decoupled_kernel(const lla_dims* dims, int d_rope) {
  if (check_dims(dims) != LLA_OK || dims->variant != LLA_PER_HEAD || d_rope != 64) return nullptr;
  if (dims->dtype == LLA_F32) return "fp32";
  if (decoupled_small_supported(dims->H, dims->r_k, dims->r_v)) return "small-rank";
  return decoupled_tile_supported(dims->r_k, dims->r_v) ? "tile" : nullptr;
}

size_t lla_workspace_size(const lla_dims* dims, int B, int64_t L_max, int max_N) {
  (void)max_N;
  if (check_dims(dims) != LLA_OK || B < 0 || L_max < 0) return 0;
  return ws_layout(dims, B, L_max).total;
}

lla_status lla_rope_table(const lla_dims* dims, int64_t n_pos, float* cos_out, float* sin_out) {
  if (!dims || dims->d_head < 2 || dims->d_head % 2 || !(dims->rope_base > 0.f) || n_pos < 0 ||
      (n_pos > 0 && (!cos_out || !sin_out)))
    return LLA_ERR_INVALID_ARG;
  const int half = dims->d_head / 2;
  for (int f = 0; f < half; ++f) {
    const double theta = std::pow(static_cast<double>(dims->rope_base), -2.0 * f / dims->d_head);
    for (int64_t p = 0; p < n_pos; ++p) {
      const double ang = static_cast<double>(p) * theta;
      cos_out[p * half + f] = static_cast<float>(std::cos(ang));
      sin_out[p * half + f] = static_cast<float>(std::sin(ang));
    }
  }
  return LLA_OK;
}

lla_status lla_device_status(void* workspace, void* stream, int clear) {
  if (!workspace) {
    // no workspace: the status word of lla_decode_attn_noalloc's scratch on this device
    const lla_status st = noalloc_scratch_address(&workspace);
    if (st != LLA_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LLA_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LLA_ERR_CUDA;
  if (clear && v != 0 && cudaMemset(workspace, 0, 4) != cudaSuccess) return LLA_ERR_CUDA;
  return static_cast<lla_status>(v);
}

}  // extern "C"

namespace {

// The cache a call reads or writes: dense [B][H][L_max][r] rows, or a page pool
// [num_pages][H][page_size][r] with a block table (L_max = max_pages * page_size).
struct CacheView {
  void* k;
  void* v;
  int B;
  int64_t L_max;
  const int32_t* bt;
  int page_size;
  int max_pages;
  int64_t num_pages;
};

CacheView dense_view(const lla_cache& c) { return CacheView{c.k, c.v, c.B, c.L_max, nullptr, 0, 0, 0}; }

// Host checks of a paged cache description; LLA_OK also for B == 0.
lla_status paged_view(const lla_dims* dims, const lla_paged_cache& c, CacheView* v) {
  if (c.B < 0 || c.max_pages < 1 || c.page_size < 1 || c.num_pages < 1) return LLA_ERR_INVALID_ARG;
  if (dims->variant != LLA_PER_HEAD) return LLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(c.max_pages) * c.page_size > (int64_t(1) << 30) ||
      c.num_pages * static_cast<int64_t>(dims->H) >= (int64_t(1) << 31) ||
      static_cast<int64_t>(c.B) * c.max_pages >= (int64_t(1) << 31))
    return LLA_ERR_UNSUPPORTED;
  if (c.B > 0 && (!c.block_table || (reinterpret_cast<uintptr_t>(c.block_table) & 3u) != 0)) return LLA_ERR_INVALID_ARG;
  *v = CacheView{c.k, c.v, c.B, static_cast<int64_t>(c.max_pages) * c.page_size, c.block_table, c.page_size,
                 c.max_pages, c.num_pages};
  return LLA_OK;
}

lla_status decode_impl(const lla_dims* dims, int loop_t, const void* q, const CacheView& cache,
                       const int32_t* seq_lens, const int32_t* q_pos, const void* w_up_k,
                       const void* w_up_v, const float* mu_k, const float* mu_v,
                       const float* rope_cos, const float* rope_sin, int64_t rope_len, float* out,
                       float* lse, void* workspace, size_t ws_bytes, void* stream,
                       bool clear_status = false) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  if (loop_t < 0 || loop_t >= dims->T || cache.B < 0 || cache.L_max < 1) return LLA_ERR_INVALID_ARG;
  if (cache.B == 0) return LLA_OK;
  if (cache.L_max > (int64_t(1) << 30) || static_cast<int64_t>(cache.B) * dims->H > (int64_t(1) << 30))
    return LLA_ERR_UNSUPPORTED;
  if (rope_len < cache.L_max || rope_len < kTile) return LLA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, cache.k, cache.v, seq_lens, q_pos, w_up_k, w_up_v, mu_k,
                        mu_v, rope_cos, rope_sin, out, lse, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LLA_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(dims, cache.B, cache.L_max);
  if (ws_bytes < wl.total) return LLA_ERR_INVALID_ARG;

  const int H = dims->H, d = dims->d_head;
  const int esize = dims->dtype == LLA_BF16 ? 2 : 4;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every host check has passed: zero the status word first when asked to (the
  // entry point without a workspace), then launch
  auto ready = [&]() { return !clear_status || cudaMemsetAsync(ws, 0, 256, s) == cudaSuccess; };
  Decode2dPlan plan2d;
  const bool pair2d = dims->variant == LLA_2D && dims->dtype == LLA_BF16 &&
                      make_decode2d_plan(H, dims->r_k, dims->r_v, &plan2d);
  if (pair2d) {
    // LLA-2D: one latent per token shared by the H heads (CTA-pair score kernel,
    // value kernel)
    Decode2dArgs a{};
    a.plan = plan2d;
    a.B = cache.B;
    a.H = H;
    a.r_k = dims->r_k;
    a.r_v = dims->r_v;
    a.rope_style = dims->rope_style;
    a.L_max = cache.L_max;
    a.rope_len = rope_len;
    a.q = q;
    a.seq_lens = seq_lens;
    a.q_pos = q_pos;
    a.w_up_k = static_cast<const uint8_t*>(w_up_k) + static_cast<size_t>(loop_t) * H * d * dims->r_k * esize;
    a.w_up_v = static_cast<const uint8_t*>(w_up_v) + static_cast<size_t>(loop_t) * H * d * dims->r_v * esize;
    a.mu_k = mu_k + static_cast<size_t>(loop_t) * H * d;
    a.mu_v = mu_v + static_cast<size_t>(loop_t) * H * d;
    a.rope_cos = rope_cos;
    a.rope_sin = rope_sin;
    a.out = out;
    a.lse = lse;
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.rec_acc = reinterpret_cast<float*>(ws + wl.partials);
    a.rec_ml = reinterpret_cast<float*>(ws + wl.rec_ml);
    a.zimg = ws + wl.zimg;
    a.zimg_stride = static_cast<int64_t>(wl.zimg_stride);
    a.zchunk_bytes = static_cast<int64_t>(H) * d * 128;
    a.ntiles = (cache.L_max + kTile - 1) / kTile;
    a.trig_rows = decode2d_trig_rows(cache.L_max);
    a.trigT = reinterpret_cast<float*>(ws + wl.trig16);
    a.pw = reinterpret_cast<uint16_t*>(ws + wl.pw);
    a.grp_m = reinterpret_cast<float*>(ws + wl.grp_m);
    const int sms = sm_count();
    if (sms <= 1) return LLA_ERR_CUDA;
    const int64_t max_blocks = static_cast<int64_t>(cache.B) * ((cache.L_max + kBlock2dTokens - 1) / kBlock2dTokens);
    a.pairs = static_cast<int>(std::min<int64_t>(std::min<int64_t>(sms / 2, kMaxPairs), std::max<int64_t>(1, max_blocks)));
    a.units = static_cast<int>(std::min<int64_t>(std::min<int64_t>(sms, kMaxGrid),
                                                 std::max<int64_t>(1, static_cast<int64_t>(cache.B) * a.ntiles)));
    Decode2dMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const uint64_t rows = static_cast<uint64_t>(cache.L_max), seqs = static_cast<uint64_t>(cache.B);
    if (!make_map_3d(&maps.k, cache.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims->r_k, rows, seqs, 64, kTile, 1))
      return LLA_ERR_CUDA;
    if (!make_map_3d(&maps.v, cache.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims->r_v, rows, seqs, 64, kTile, 1))
      return LLA_ERR_CUDA;
    // query-operand images as stored (pre-swizzled rows of 128 B, then the 32-byte
    // bias rows), one image per sequence
    const uint64_t zrows = static_cast<uint64_t>(a.plan.nkc) * H * d;
    if (!make_map_3d_strided(&maps.z, a.zimg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, zrows, seqs, 128,
                             static_cast<uint64_t>(a.zimg_stride), 64, kTile, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return LLA_ERR_CUDA;
    if (!make_map_3d_strided(&maps.zb, a.zimg + zrows * 128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 16,
                             static_cast<uint64_t>(H) * d, seqs, 32, static_cast<uint64_t>(a.zimg_stride), 16,
                             kTile, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return LLA_ERR_CUDA;
    if (!make_map_3d(&maps.p, a.pw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.ntiles) * kTile,
                     static_cast<uint64_t>(H), seqs, 64, static_cast<uint32_t>(H), 1))
      return LLA_ERR_CUDA;
    if (!ready()) return LLA_ERR_CUDA;
    return launch_decode2d_bf16(a, maps, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  }
  DecodeArgs a{};
  a.B = cache.B;
  a.H = H;
  a.r_k = dims->r_k;
  a.r_v = dims->r_v;
  a.rope_style = dims->rope_style;
  a.L_max = cache.L_max;
  a.rope_len = rope_len;
  // per-head mu [H][T*d]; LLA-2D mu [T*H*d] with the loop-t slice [H][d]
  a.mu_hstride = dims->variant == LLA_2D ? d : static_cast<int64_t>(dims->T) * d;
  a.shared_latent = dims->variant == LLA_2D ? 1 : 0;
  a.q = q;
  a.seq_lens = seq_lens;
  a.q_pos = q_pos;
  a.cache_k = cache.k;
  a.cache_v = cache.v;
  a.block_table = cache.bt;
  a.page_size = cache.page_size;
  a.max_pages = cache.max_pages;
  a.num_pages = cache.num_pages;
  a.w_up_k = static_cast<const uint8_t*>(w_up_k) + static_cast<size_t>(loop_t) * H * d * dims->r_k * esize;
  a.w_up_v = static_cast<const uint8_t*>(w_up_v) + static_cast<size_t>(loop_t) * H * d * dims->r_v * esize;
  const size_t mu_loop = dims->variant == LLA_2D ? static_cast<size_t>(H) * d : d;
  a.mu_k = mu_k + loop_t * mu_loop;
  a.mu_v = mu_v + loop_t * mu_loop;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.out = out;
  a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.partials = reinterpret_cast<float*>(ws + wl.partials);
  a.scores = reinterpret_cast<float*>(ws + wl.scores);
  a.zimg = ws + wl.zimg;
  a.zimg_stride = static_cast<int64_t>(wl.zimg_stride);

  if (dims->dtype == LLA_F32) {
    if (!ready()) return LLA_ERR_CUDA;
    return launch_decode_f32(a, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  }
  if (dims->variant == LLA_2D) {
    // LLA-2D shapes outside the CTA-pair kernels' range: the plain kernels over bf16
    if (cache.bt) return LLA_ERR_UNSUPPORTED;
    if (!ready()) return LLA_ERR_CUDA;
    return launch_decode_plain_bf16(a, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  }

  const int sms = sm_count();
  if (sms <= 0) return LLA_ERR_CUDA;
  a.combine_units = decode_combine_units(cache.B, H, sms);
  a.records_per_cta = kRecordsPerCta;
  // 3-D maps over the dense cache (rows L_max, z = b H + h) or the page pool (rows
  // page_size, z = page H + h)
  const uint64_t rows = static_cast<uint64_t>(cache.bt ? cache.page_size : cache.L_max);
  const uint64_t units = cache.bt ? static_cast<uint64_t>(cache.num_pages) * H : static_cast<uint64_t>(cache.B) * H;
  // a TMA box is one tile, or one page when pages are smaller than a tile
  const uint32_t box_rows = static_cast<uint32_t>(cache.bt && cache.page_size < kTile ? cache.page_size : kTile);
  if (small_path(dims)) {
    // small ranks: positions split over the CTAs, every head of a position in one CTA
    // pages of 8..64 tokens: one copy per page for a whole head set, if it fits
    if (!(cache.bt && make_decode_small_setpage_plan(H, dims->r_k, dims->r_v, cache.page_size, &a.splan)))
      make_decode_small_plan(H, dims->r_k, dims->r_v, &a.splan);
    a.pos_major = 1;
    a.trig16 = reinterpret_cast<uint32_t*>(ws + wl.trig16);
    a.trig_rows = decode_small_trig_rows(cache.L_max, rope_len);
    const int64_t max_pos = static_cast<int64_t>(cache.B) * ((cache.L_max + kTile - 1) / kTile);
    a.grid = static_cast<int>(std::min<int64_t>(std::min<int64_t>(sms, kMaxGrid), std::max<int64_t>(1, max_pos)));
    if (!ready()) return LLA_ERR_CUDA;
    return launch_decode_small_bf16(a, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  }
  if (!make_decode_plan(dims->r_k, dims->r_v, &a.plan)) return LLA_ERR_UNSUPPORTED;
  if (cache.bt && !tile_kernel_page_size(cache.page_size)) {
    // pages the tile kernel's copies do not take: rows gathered one by one
    if (!ready()) return LLA_ERR_CUDA;
    return launch_decode_paged_generic(a, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  }
  const int64_t max_tiles = static_cast<int64_t>(cache.B) * H * ((cache.L_max + kTile - 1) / kTile);
  a.grid = static_cast<int>(std::min<int64_t>(std::min<int64_t>(sms, kMaxGrid), std::max<int64_t>(1, max_tiles)));
  DecodeMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  for (int c = 0; c < a.plan.kplan.n; ++c) {
    const int w = a.plan.kplan.width[c];
    if (!make_map_3d(&maps.k[chunk_map_index(w)], cache.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims->r_k, rows,
                     units, w, box_rows, 1))
      return LLA_ERR_CUDA;
  }
  // V latents: 32-column boxes (a tail box zero-filled past r_v), 64B swizzle
  if (!make_map_3d(&maps.v, cache.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims->r_v, rows, units, 32, box_rows, 1))
    return LLA_ERR_CUDA;
  // pages of 8..64 tokens with whole 32-column chunks: one box per page for all of V
  // (rows, chunks and page-heads as the outer dimensions of a 4-D view of the pool)
  if (cache.bt && cache.page_size < kTile && dims->r_v % 32 == 0) {
    auto enc = tensor_map_encoder();
    const cuuint64_t d4[4] = {32, static_cast<cuuint64_t>(cache.page_size), static_cast<cuuint64_t>(dims->r_v / 32), units};
    const cuuint64_t s4[3] = {static_cast<cuuint64_t>(dims->r_v) * 2, 64,
                              static_cast<cuuint64_t>(cache.page_size) * dims->r_v * 2};
    const cuuint32_t b4[4] = {32, static_cast<cuuint32_t>(cache.page_size), static_cast<cuuint32_t>(dims->r_v / 32), 1};
    const cuuint32_t e4[4] = {1, 1, 1, 1};
    if (enc && enc(&maps.v4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache.v), d4, s4, b4, e4,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      a.v_page_major = 1;
  }
  if (!ready()) return LLA_ERR_CUDA;
  return launch_decode_bf16(a, maps, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

}  // namespace

extern "C" {

lla_status lla_decode_attn(const lla_dims* dims, int loop_t, const void* q, lla_cache cache,
                           const int32_t* seq_lens, const int32_t* q_pos, const void* w_up_k,
                           const void* w_up_v, const float* mu_k, const float* mu_v,
                           const float* rope_cos, const float* rope_sin, int64_t rope_len, float* out,
                           float* lse, void* workspace, size_t ws_bytes, void* stream) {
  return decode_impl(dims, loop_t, q, dense_view(cache), seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v, rope_cos,
                     rope_sin, rope_len, out, lse, workspace, ws_bytes, stream);
}

lla_status lla_decode_attn_paged(const lla_dims* dims, int loop_t, const void* q, lla_paged_cache cache,
                                 const int32_t* seq_lens, const int32_t* q_pos, const void* w_up_k,
                                 const void* w_up_v, const float* mu_k, const float* mu_v,
                                 const float* rope_cos, const float* rope_sin, int64_t rope_len, float* out,
                                 float* lse, void* workspace, size_t ws_bytes, void* stream) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  CacheView v{};
  if ((st = paged_view(dims, cache, &v)) != LLA_OK) return st;
  return decode_impl(dims, loop_t, q, v, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v, rope_cos, rope_sin,
                     rope_len, out, lse, workspace, ws_bytes, stream);
}

}  // extern "C"

namespace lla {

lla_status decode_attn_status_cleared(const lla_dims* dims, int loop_t, const void* q, lla_cache cache,
                                      const int32_t* seq_lens, const int32_t* q_pos, const void* w_up_k,
                                      const void* w_up_v, const float* mu_k, const float* mu_v,
                                      const float* rope_cos, const float* rope_sin, int64_t rope_len,
                                      float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  return decode_impl(dims, loop_t, q, dense_view(cache), seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v, rope_cos,
                     rope_sin, rope_len, out, lse, workspace, ws_bytes, stream, true);
}

}  // namespace lla

extern "C" {

size_t lla_decoupled_workspace_size(const lla_dims* dims, int d_rope, int B, int64_t L_max) {
  if (check_dims(dims) != LLA_OK || dims->variant != LLA_PER_HEAD || d_rope != 64 || B < 0 || L_max < 0) return 0;
  size_t off = 256;   // status word
  const bool small = dims->dtype == LLA_BF16 && decoupled_small_supported(dims->H, dims->r_k, dims->r_v);
  if (small || (dims->dtype == LLA_BF16 && decoupled_tile_supported(dims->r_k, dims->r_v))) {
    // tensor-core kernels: records per (sequence + CTA, head, warp) (small ranks; a
    // CTA index is below min(kMaxGrid, positions)) or per (unit + CTA, warp) (tile
    // kernel, eight warps), B images per (sequence, head), sc b0 per (sequence,
    // head), the fp32 RoPE table [64][trig_rows]
    const size_t max_pos = static_cast<size_t>(B) * ((L_max + kTile - 1) / kTile);
    if (small)
      off += al256((static_cast<size_t>(B) + std::min<size_t>(kMaxGrid, std::max<size_t>(1, max_pos))) * dims->H *
                   kRecordsPerCta * (dims->r_v + kRecordHead) * 4);
    else
      off += al256((static_cast<size_t>(B) * dims->H + kMaxGrid) * kDecoupledTileRecords *
                   (dims->r_v + kRecordHead) * 4);
    off += al256(static_cast<size_t>(B) * dims->H * decoupled_small_img_stride(dims->r_k));
    off += al256(static_cast<size_t>(B) * dims->H * 4);
    off += al256(static_cast<size_t>(decoupled_small_trig_rows(L_max)) * 64 * 4);
    return off;
  }
  if (dims->dtype == LLA_BF16) return 0;   // bf16 shapes neither tensor-core kernel takes
  // fp32 mode: scores [B][H][L_max]
  off += al256(static_cast<size_t>(B) * dims->H * L_max * 4);
  return off;
}

lla_status lla_decode_attn_decoupled(const lla_dims* dims, int loop_t, int d_rope, const void* q, lla_cache cache,
                                     const void* k_rope, const int32_t* seq_lens, const int32_t* q_pos,
                                     const void* w_up_k, const void* w_up_v, const float* mu_k, const float* mu_v,
                                     const float* rope_cos, const float* rope_sin, int64_t rope_len, float* out,
                                     float* lse, void* workspace, size_t ws_bytes, void* stream) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  if (dims->variant != LLA_PER_HEAD || d_rope != 64) return LLA_ERR_UNSUPPORTED;
  if (loop_t < 0 || loop_t >= dims->T || cache.B < 0 || cache.L_max < 1) return LLA_ERR_INVALID_ARG;
  if (cache.B == 0) return LLA_OK;
  if (cache.L_max > (int64_t(1) << 30) || static_cast<int64_t>(cache.B) * dims->H > (int64_t(1) << 30))
    return LLA_ERR_UNSUPPORTED;
  if (rope_len < cache.L_max || rope_len < kTile) return LLA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, cache.k, cache.v, k_rope, seq_lens, q_pos, w_up_k, w_up_v, mu_k,
                        mu_v, rope_cos, rope_sin, out, lse, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LLA_ERR_INVALID_ARG;
  const size_t need = lla_decoupled_workspace_size(dims, d_rope, cache.B, cache.L_max);
  if (ws_bytes < need) return LLA_ERR_INVALID_ARG;
  const int H = dims->H, d = dims->d_head;
  const int esize = dims->dtype == LLA_BF16 ? 2 : 4;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeArgs a{};
  a.B = cache.B;
  a.H = H;
  a.r_k = dims->r_k;
  a.r_v = dims->r_v;
  a.rope_style = dims->rope_style;
  a.L_max = cache.L_max;
  a.rope_len = rope_len;
  a.mu_hstride = static_cast<int64_t>(dims->T) * d;
  a.q = q;
  a.seq_lens = seq_lens;
  a.q_pos = q_pos;
  a.cache_k = cache.k;
  a.cache_v = cache.v;
  a.k_rope = k_rope;
  a.d_rope = d_rope;
  a.w_up_k = static_cast<const uint8_t*>(w_up_k) + static_cast<size_t>(loop_t) * H * d * dims->r_k * esize;
  a.w_up_v = static_cast<const uint8_t*>(w_up_v) + static_cast<size_t>(loop_t) * H * d * dims->r_v * esize;
  a.mu_k = mu_k + static_cast<size_t>(loop_t) * d;
  a.mu_v = mu_v + static_cast<size_t>(loop_t) * d;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.out = out;
  a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.partials = reinterpret_cast<float*>(ws + 256);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool small = dims->dtype == LLA_BF16 && decoupled_small_supported(H, dims->r_k, dims->r_v);
  if (small || (dims->dtype == LLA_BF16 && decoupled_tile_supported(dims->r_k, dims->r_v))) {
    // rotary branch and content score on the tensor cores: small ranks with positions
    // split over the CTAs and every head of a position in one CTA, other ranks with
    // 128-token tiles of one (sequence, head) split over the CTAs
    const int sms = sm_count();
    if (sms <= 0) return LLA_ERR_CUDA;
    const int64_t max_pos = static_cast<int64_t>(cache.B) * ((cache.L_max + kTile - 1) / kTile);
    uint8_t* p = ws + 256 +
                 (small ? al256((static_cast<size_t>(cache.B) +
                                 std::min<size_t>(kMaxGrid, std::max<int64_t>(1, max_pos))) *
                                H * kRecordsPerCta * (dims->r_v + kRecordHead) * 4)
                        : al256((static_cast<size_t>(cache.B) * H + kMaxGrid) * kDecoupledTileRecords *
                                (dims->r_v + kRecordHead) * 4));
    a.zimg = p;
    a.zimg_stride = static_cast<int64_t>(decoupled_small_img_stride(dims->r_k));
    p += al256(static_cast<size_t>(cache.B) * H * a.zimg_stride);
    a.qb0 = reinterpret_cast<float*>(p);
    p += al256(static_cast<size_t>(cache.B) * H * 4);
    a.trigT = reinterpret_cast<float*>(p);
    a.trig_rows = decoupled_small_trig_rows(cache.L_max);
    a.pos_major = small ? 1 : 0;
    a.records_per_cta = small ? kRecordsPerCta : kDecoupledTileRecords;
    const int64_t work = small ? max_pos : max_pos * H;   // positions, or head-tiles
    a.grid = static_cast<int>(std::min<int64_t>(std::min<int64_t>(sms, kMaxGrid), std::max<int64_t>(1, work)));
    a.combine_units = decode_combine_units(cache.B, H, sms);
    // image blocks of up to 8 sequences, fewer when that leaves SMs idle
    a.z_seqs = static_cast<int>(std::min<int64_t>(
        8, std::max<int64_t>(1, (static_cast<int64_t>(cache.B) * H + 2 * sms - 1) / (2 * sms))));
    const uint64_t units = static_cast<uint64_t>(cache.B) * H, rows = static_cast<uint64_t>(cache.L_max);
    DecoupledMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!make_map_3d(&maps.kr, k_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, rows, units, 64, kTile, 1) ||
        !make_map_3d(&maps.ck, cache.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims->r_k, rows, units, 16, kTile, 1))
      return LLA_ERR_CUDA;
    return (small ? launch_decoupled_small(a, maps, s) : launch_decoupled_tile(a, maps, s)) == cudaSuccess
               ? LLA_OK
               : LLA_ERR_CUDA;
  }
  if (dims->dtype != LLA_F32) return LLA_ERR_UNSUPPORTED;   // bf16 shapes neither tensor-core kernel takes
  a.scores = reinterpret_cast<float*>(ws + 256);
  return launch_decoupled_f32(a, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

lla_status lla_evict_window(const lla_dims* dims, lla_cache cache, int32_t* seq_lens, int sink, int window,
                            void* workspace, size_t ws_bytes, void* stream) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  if (cache.B < 0 || cache.L_max < 1 || sink < 0 || window < 0 || sink + window < 1) return LLA_ERR_INVALID_ARG;
  if (cache.B == 0) return LLA_OK;
  if (cache.L_max > (int64_t(1) << 30) || static_cast<int64_t>(cache.B) * dims->H > (int64_t(1) << 30))
    return LLA_ERR_UNSUPPORTED;
  const void* ptrs[] = {cache.k, cache.v, seq_lens, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LLA_ERR_INVALID_ARG;
  if (ws_bytes < 256) return LLA_ERR_INVALID_ARG;
  EvictArgs a{};
  a.B = cache.B;
  a.units_per_seq = dims->variant == LLA_2D ? 1 : dims->H;
  a.r_k = dims->r_k;
  a.r_v = dims->r_v;
  a.esize = dims->dtype == LLA_BF16 ? 2 : 4;
  a.sink = sink;
  a.window = window;
  a.L_max = cache.L_max;
  a.cache_k = cache.k;
  a.cache_v = cache.v;
  a.seq_lens = seq_lens;
  a.status = static_cast<uint32_t*>(workspace);
  return launch_evict_window(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

lla_status lla_window_attn(const lla_dims* dims, int B, int W, const void* q, const void* k_win,
                           const void* v_win, const int32_t* win_len, const int32_t* win_pos,
                           const int32_t* q_pos, const float* rope_cos, const float* rope_sin, int64_t rope_len,
                           float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  if (B < 0 || W < 0 || rope_len < kTile) return LLA_ERR_INVALID_ARG;
  if (B == 0 || W == 0) return LLA_OK;
  if (static_cast<int64_t>(B) * dims->H > (int64_t(1) << 30)) return LLA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_win, v_win, win_len, win_pos, q_pos, rope_cos, rope_sin, out, lse, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LLA_ERR_INVALID_ARG;
  if (ws_bytes < 256) return LLA_ERR_INVALID_ARG;
  WindowArgs a{};
  a.B = B;
  a.H = dims->H;
  a.W = W;
  a.rope_style = dims->rope_style;
  a.rope_len = rope_len;
  a.q = q;
  a.k_win = k_win;
  a.v_win = v_win;
  a.win_len = win_len;
  a.win_pos = win_pos;
  a.q_pos = q_pos;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.out = out;
  a.lse = lse;
  a.status = static_cast<uint32_t*>(workspace);
  return launch_window_attn(a, dims->dtype == LLA_BF16, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LLA_OK
             : LLA_ERR_CUDA;
}

}  // extern "C"

namespace {

lla_status encode_impl(const lla_dims* dims, const void* x_k, const void* x_v, int N, const int32_t* seq_idx,
                       const int32_t* pos, const void* w_down_k, const void* w_down_v, const float* mu_k,
                       const float* mu_v, const CacheView& cache, void* workspace, size_t ws_bytes, void* stream) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  if (N < 0 || cache.B < 0 || cache.L_max < 1) return LLA_ERR_INVALID_ARG;
  if (N == 0) return LLA_OK;
  const void* ptrs[] = {x_k, x_v, seq_idx, pos, w_down_k, w_down_v, mu_k, mu_v, cache.k, cache.v, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LLA_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(dims, cache.B, cache.L_max);
  if (ws_bytes < wl.total) return LLA_ERR_INVALID_ARG;

  EncodeArgs a{};
  a.N = N;
  // LLA-2D: one latent per token from the whole stack x in R^{T*H*d} (one "head")
  a.H = dims->variant == LLA_2D ? 1 : dims->H;
  a.Td = dims->T * dims->d_head * (dims->variant == LLA_2D ? dims->H : 1);
  a.r_k = dims->r_k;
  a.r_v = dims->r_v;
  a.B = cache.B;
  a.L_max = cache.L_max;
  a.x_k = x_k;
  a.x_v = x_v;
  a.seq_idx = seq_idx;
  a.pos = pos;
  a.w_down_k = w_down_k;
  a.w_down_v = w_down_v;
  a.mu_k = mu_k;
  a.mu_v = mu_v;
  a.cache_k = cache.k;
  a.cache_v = cache.v;
  a.block_table = cache.bt;
  a.page_size = cache.page_size;
  a.max_pages = cache.max_pages;
  a.num_pages = cache.num_pages;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.bias = reinterpret_cast<float*>(ws + wl.bias);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dims->dtype == LLA_F32) return launch_encode_f32(a, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;

  EncodeMaps m;
  std::memset(&m, 0, sizeof(m));
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  EncodePlan plan;
  if (make_encode_pair_plan(dims->r_k, dims->r_v, a.Td, &plan)) {
    // CTA pairs: x tiles and 16-column W_down boxes
    plan.sms = sm_count();
    if (plan.sms <= 1) return LLA_ERR_CUDA;
    if (!make_map_3d(&m.xk, x_k, BF, 2, a.Td, a.H, N, 64, 1, 128)) return LLA_ERR_CUDA;
    if (!make_map_3d(&m.xv, x_v, BF, 2, a.Td, a.H, N, 64, 1, 128)) return LLA_ERR_CUDA;
    if (!make_map_3d(&m.wk[2], w_down_k, BF, 2, a.r_k, a.Td, a.H, 16, 64, 1)) return LLA_ERR_CUDA;
    if (!make_map_3d(&m.wv[2], w_down_v, BF, 2, a.r_v, a.Td, a.H, 16, 64, 1)) return LLA_ERR_CUDA;
    return launch_encode_pair(a, plan, m, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  }
  if (!make_encode_plan(dims->r_k, dims->r_v, a.Td, &plan)) return LLA_ERR_UNSUPPORTED;
  plan.sms = sm_count();
  if (plan.sms <= 0) return LLA_ERR_CUDA;
  if (!make_map_3d(&m.xk, x_k, BF, 2, a.Td, a.H, N, 64, 1, 128)) return LLA_ERR_CUDA;
  if (!make_map_3d(&m.xv, x_v, BF, 2, a.Td, a.H, N, 64, 1, 128)) return LLA_ERR_CUDA;
  for (int c = 0; c < plan.bk.n; ++c) {
    const int w = plan.bk.width[c];
    if (!make_map_3d(&m.wk[chunk_map_index(w)], w_down_k, BF, 2, a.r_k, a.Td, a.H, w, 64, 1)) return LLA_ERR_CUDA;
  }
  for (int c = 0; c < plan.bv.n; ++c) {
    const int w = plan.bv.width[c];
    if (!make_map_3d(&m.wv[chunk_map_index(w)], w_down_v, BF, 2, a.r_v, a.Td, a.H, w, 64, 1)) return LLA_ERR_CUDA;
  }
  return launch_encode_bf16(a, plan, m, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

}  // namespace

extern "C" {

lla_status lla_encode(const lla_dims* dims, const void* x_k, const void* x_v, int N, const int32_t* seq_idx,
                      const int32_t* pos, const void* w_down_k, const void* w_down_v, const float* mu_k,
                      const float* mu_v, lla_cache cache, void* workspace, size_t ws_bytes, void* stream) {
  return encode_impl(dims, x_k, x_v, N, seq_idx, pos, w_down_k, w_down_v, mu_k, mu_v, dense_view(cache), workspace,
                     ws_bytes, stream);
}

lla_status lla_encode_paged(const lla_dims* dims, const void* x_k, const void* x_v, int N, const int32_t* seq_idx,
                            const int32_t* pos, const void* w_down_k, const void* w_down_v, const float* mu_k,
                            const float* mu_v, lla_paged_cache cache, void* workspace, size_t ws_bytes,
                            void* stream) {
  lla_status st = check_dims(dims);
  if (st != LLA_OK) return st;
  CacheView v{};
  if ((st = paged_view(dims, cache, &v)) != LLA_OK) return st;
  return encode_impl(dims, x_k, x_v, N, seq_idx, pos, w_down_k, w_down_v, mu_k, mu_v, v, workspace, ws_bytes,
                     stream);
}

}  // extern "C"
