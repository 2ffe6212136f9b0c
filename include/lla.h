/*
 * lla.h — C ABI of the Looped Latent Attention (LLA) GPU library (liblla.so).
 *
 * LLA ("Looped Latent Attention: Cross-Loop KV Compression for Looped
 * Transformers", arXiv 2607.15456v2) replaces the per-loop K/V cache of a
 * weight-tied looped decoder (T loops, D layers, H heads of width d) by one K
 * latent and one V latent per token, layer and head, and rebuilds the loop-t
 * K/V only when attention reads them (§1, §3; §7 "latent-store path").  This
 * library is the data-parallel hot path of that latent-store decode:
 *
 *   lla_encode       Eq. (2)  c = (x - mu) W_down, written into cache slots
 *   lla_decode_attn  Eq. (3)  k_t = c_k W_up,k,t^T + mu_k,t (v likewise),
 *                    RoPE after reconstruction (§3 "RoPE and reconstruction"),
 *                    softmax(q.k/sqrt(d)) v over each sequence's history,
 *                    for one layer and one loop, all heads and sequences.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked "device" are CUDA device pointers owned by the caller;
 *   the library allocates nothing and keeps no per-call state.  "host"
 *   pointers are ordinary CPU memory.
 * - Arrays are dense and row-major, with the shapes given below.  Storage
 *   types follow lla_dims.dtype: LLA_BF16 stores latents, W, x and q as
 *   bfloat16 (mu always fp32); LLA_F32 stores everything as fp32.
 * - Every device pointer must be 16-byte aligned.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream).  Argument errors found on the host return before any launch.
 *   Values that live on the device (seq_lens, q_pos, seq_idx, pos) are
 *   checked by the kernels: an out-of-range value is clamped or its token
 *   skipped, and LLA_ERR_DEVICE_ARG is recorded in the workspace status word
 *   (read it with lla_device_status).  Every wait inside a kernel is bounded
 *   (about one second); on expiry the kernel records LLA_ERR_TIMEOUT and
 *   returns.
 * - The workspace is caller-allocated device memory of at least
 *   lla_workspace_size() bytes.  Its first 256 bytes hold the status word and
 *   must be zero before the first call; the rest is scratch.  Calls that
 *   share a workspace must be ordered on one stream.
 * - Test hook of the timeout path: while the 32-bit word at byte 4 of the
 *   workspace holds LLA_TEST_STALL, the per-head bf16 tile decode kernel
 *   ("tile" in lla_decode_kernel) waits on a barrier that one arrival short
 *   never completes; the wait expires after about one second and the call's
 *   status becomes LLA_ERR_TIMEOUT (outputs undefined).  Zero the word to
 *   resume normal calls.
 * - Constraints: d_head == 128; r_k and r_v multiples of 16 in [16, 256]
 *   (LLA_PER_HEAD) or [16, 512] (LLA_2D, one latent per token, "The LLA-2D
 *   variant"); T >= 1; H >= 1.  Other shapes return LLA_ERR_UNSUPPORTED.
 */
#ifndef LLA_H
#define LLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LLA_ABI_VERSION 1

/* Value of workspace word 1 (byte offset 4) that makes the next tile decode
 * kernel's bounded wait expire (see the test hook above). */
#define LLA_TEST_STALL 0x4C415453u

typedef enum {
    LLA_OK = 0,
    LLA_ERR_INVALID_ARG = 1,   /* bad host-side argument: nothing launched       */
    LLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented shape/variant/dtype  */
    LLA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed              */
    LLA_ERR_TIMEOUT = 4,       /* a kernel's bounded wait expired (device word)  */
    LLA_ERR_DEVICE_ARG = 5,    /* out-of-range seq_lens/q_pos/seq_idx/pos seen
                                  by a kernel (device word)                       */
    LLA_ERR_RANGE = 6          /* a folded query operand left the f16 range of
                                  the small-rank decode path (device word)        */
} lla_status;

typedef enum { LLA_BF16 = 0, LLA_F32 = 1 } lla_dtype;

/* LLA_PER_HEAD: one latent per (token, layer, head) (§3 "Cross-loop codec").
 * LLA_2D: one latent per (token, layer) shared by all heads, reconstructing
 * every head (§3 "The LLA-2D variant"). */
typedef enum { LLA_PER_HEAD = 0, LLA_2D = 1 } lla_variant;

/* RoPE pairing: LLA_ROPE_HALF rotates (i, i + d/2); LLA_ROPE_INTERLEAVED
 * rotates (2i, 2i+1).  Frequencies theta_f = rope_base^(-2f/d). */
typedef enum { LLA_ROPE_HALF = 0, LLA_ROPE_INTERLEAVED = 1 } lla_rope_style;

typedef struct {
    int T;                      /* loops                                   */
    int H;                      /* heads                                   */
    int d_head;                 /* head width (must be 128)                */
    int r_k, r_v;               /* latent ranks                            */
    lla_variant variant;
    lla_dtype dtype;
    float rope_base;            /* e.g. 10000                              */
    lla_rope_style rope_style;
} lla_dims;

/* One layer's latent cache (device).  Per-head: k [B][H][L_max][r_k],
 * v [B][H][L_max][r_v]; element (b,h,j,i) of k at ((b*H+h)*L_max+j)*r_k+i.
 * LLA-2D: k [B][L_max][r_k], v [B][L_max][r_v]. */
typedef struct {
    void* k;
    void* v;
    int B;
    int64_t L_max;
} lla_cache;

/*
 * lla_encode — Eq. (2) of §3: for each of N tokens and each head,
 *     c_k = (x_k - mu_k) W_down,k ,  c_v = (x_v - mu_v) W_down,v
 * rounded to the cache dtype (round-to-nearest-even) and stored in cache slot
 * (seq_idx[n], pos[n]).  x is the loop stack of Eq. (1): index t*d+i.
 *   x_k, x_v        device  [N][H][T*d]      (LLA-2D: [N][T*H*d], index (t*H+h)*d+i)
 *   seq_idx, pos    device  int32 [N]        slot of token n; entries outside
 *                                            [0,B) x [0,L_max) are skipped and
 *                                            flagged LLA_ERR_DEVICE_ARG
 *   w_down_k/_v     device  [H][T*d][r]      (LLA-2D: [T*H*d][r])
 *   mu_k, mu_v      device  fp32 [H][T*d]    (LLA-2D: [T*H*d])
 * Used both for a decode step's new token and for prefill (N = all prompt
 * tokens of a layer).  Two tokens writing the same slot race.
 */
lla_status lla_encode(const lla_dims* dims, const void* x_k, const void* x_v, int N,
                      const int32_t* seq_idx, const int32_t* pos,
                      const void* w_down_k, const void* w_down_v,
                      const float* mu_k, const float* mu_v,
                      lla_cache cache, void* workspace, size_t ws_bytes, void* stream);

/*
 * lla_decode_attn — one layer, one loop t (0-based; the paper counts t=1..T),
 * all heads and all B sequences.  For sequence b with L = seq_lens[b] cached
 * tokens (positions 0..L-1) and a query at position q_pos[b]:
 *     k_j = c_k,j W_up,k,t^T + mu_k,t ,  v_j = c_v,j W_up,v,t^T + mu_v,t   (Eq. (3))
 *     s_j = RoPE(q, q_pos) . RoPE(k_j, j) / sqrt(d)   for j < L
 *     out = sum_j softmax(s)_j v_j ,  lse = ln sum_j exp(s_j)
 * mu_t is the t-th d-slice of the codec mean mu of Eq. (2).
 *   q              device  [B][H][d]               pre-RoPE query
 *   seq_lens       device  int32 [B]                0 <= L <= L_max (L=0: out=0, lse=-inf)
 *   q_pos          device  int32 [B]                0 <= q_pos < rope_len
 *   w_up_k, w_up_v device  [T][H][d][r]             all loops (LLA-2D: [T][H*d][r])
 *   mu_k, mu_v     device  fp32 [H][T*d]            (LLA-2D: [T*H*d])
 *   rope_cos/_sin  device  fp32 [rope_len][d/2]     cos/sin(p*theta_f) as made by
 *                                                   lla_rope_table; rope_len >=
 *                                                   max(L_max, 128)
 *   out            device  fp32 [B][H][d]
 *   lse            device  fp32 [B][H]              natural log
 * The new token's own K/V are attended only if the caller has encoded them
 * into slot q_pos (the paper's latent-store decoder reads every cached token
 * back through its latent); lse lets a caller merge further exact terms.
 * LLA_2D (§3 "The LLA-2D variant"): every head h reads the sequence's one latent
 * and reconstructs with rows h*d .. h*d+d-1 of W_up,t; mu_t is the loop-t slice
 * [H*d] of mu [T*H*d] (index (t*H + h)*d + e).  The bf16 kernel runs on pairs of
 * CTAs (thread-block clusters of two).
 */
lla_status lla_decode_attn(const lla_dims* dims, int loop_t, const void* q,
                           lla_cache cache, const int32_t* seq_lens, const int32_t* q_pos,
                           const void* w_up_k, const void* w_up_v,
                           const float* mu_k, const float* mu_v,
                           const float* rope_cos, const float* rope_sin, int64_t rope_len,
                           float* out, float* lse,
                           void* workspace, size_t ws_bytes, void* stream);

/* A paged per-head latent cache (device), as the page tables of "Enabling
 * dynamic computation in Looped LMs" (arXiv 2610.09013, §"Ragged KV" and
 * Appendix A.1 "Page-table aliases for compact K/V storage"): a pool of physical
 * pages and a logical-to-physical table per sequence.
 *   k, v         device  pools [num_pages][H][page_size][r_k / r_v]
 *   block_table  device  int32 [B][max_pages]: logical page p of sequence b
 *                        (tokens p*page_size .. (p+1)*page_size-1) is physical
 *                        page block_table[b*max_pages + p]; several entries may
 *                        name the same page (aliased reads)
 * The logical capacity per sequence is L_max = max_pages * page_size.  Only the
 * entries of pages that hold written or read tokens are looked at; an entry
 * outside [0, num_pages) records LLA_ERR_DEVICE_ARG (reads then use a page
 * inside the pool, writes are skipped), so no access leaves the pool.  Per-head variant only;
 * any page_size >= 1 in both storage types.  In bf16 the tile kernel copies a
 * 128-token tile whole when page_size is a multiple of 128, as 128/P page pieces when
 * P is 8, 16, 32 or 64 (with r_v a multiple of 32, one copy per page holds all of its
 * V columns), and other page sizes (one-token pages, as vLLM's) run a kernel that
 * gathers token rows one by one (correct, much slower); the small-rank kernel copies
 * one page for a whole set of heads when P is 8, 16, 32 or 64, else each tile's rows
 * page by page (any page size). */
typedef struct {
    void* k;
    void* v;
    const int32_t* block_table;
    int B;
    int max_pages;
    int page_size;
    int64_t num_pages;
} lla_paged_cache;

/*
 * lla_encode_paged / lla_decode_attn_paged — lla_encode and lla_decode_attn over
 * a paged cache: token j of (sequence b, head h) lives in row j mod page_size of
 * head h of page block_table[b][j / page_size].  Every other argument, result
 * and rule is that of the dense call with L_max = max_pages * page_size (the
 * workspace is lla_workspace_size(dims, B, max_pages * page_size, N)).
 * LLA_ERR_UNSUPPORTED: LLA-2D.
 */
lla_status lla_encode_paged(const lla_dims* dims, const void* x_k, const void* x_v, int N,
                            const int32_t* seq_idx, const int32_t* pos,
                            const void* w_down_k, const void* w_down_v,
                            const float* mu_k, const float* mu_v,
                            lla_paged_cache cache, void* workspace, size_t ws_bytes, void* stream);
lla_status lla_decode_attn_paged(const lla_dims* dims, int loop_t, const void* q,
                                 lla_paged_cache cache, const int32_t* seq_lens, const int32_t* q_pos,
                                 const void* w_up_k, const void* w_up_v,
                                 const float* mu_k, const float* mu_v,
                                 const float* rope_cos, const float* rope_sin, int64_t rope_len,
                                 float* out, float* lse,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * lla_evict_window — token eviction composed with LLA (LLA paper, Appendix D
 * "Token-eviction composition table" and Appendix J "Eviction and long-context
 * prefill"): a StreamingLLM/H2O-style budget keeps each sequence's first `sink`
 * tokens and its `window` newest, and only their latents stay in the cache.
 * For every sequence with L = seq_lens[b] > sink + window, the latent rows of
 * tokens L-window .. L-1 move, in order, to slots sink .. sink+window-1 (every
 * head, K and V, in place) and seq_lens[b] becomes sink + window; sequences at
 * or below the budget are untouched.  A later lla_decode_attn rotates slot j at
 * position j, i.e. positions within the kept cache (StreamingLLM's re-indexing);
 * the query's position is then its slot in the kept cache.  Rows past the new
 * length keep stale latents.
 *   cache      dense cache, as for lla_decode_attn (any variant, dtype)
 *   seq_lens   device int32 [B], read and rewritten; a length outside
 *              [0, L_max] is left alone and records LLA_ERR_DEVICE_ARG
 *   sink, window  >= 0, sink + window >= 1
 *   workspace  device, >= 256 bytes: the status word
 * Asynchronous on `stream`; decode calls after it on the same stream see the new
 * lengths.
 */
lla_status lla_evict_window(const lla_dims* dims, lla_cache cache, int32_t* seq_lens, int sink,
                            int window, void* workspace, size_t ws_bytes, void* stream);

/*
 * lla_window_attn — exact attention over each sequence's window of recent
 * tokens, merged into a latent-store result ("Hybrid Latent Attention for Looped
 * Language Models", §3.4 "Exact sliding window", Eq. (4), and Appendix I
 * "Serving Implementation").  Eq. (4) takes one softmax over the latent tokens
 * before the window and the window's exact keys; with `out`/`lse` holding
 * lla_decode_attn's result for the latent tokens (seq_lens = their count) at
 * loop t, this call computes the window's own softmax and merges the two by
 * log-sum-exp, which equals that single softmax.  Any lla_dims variant; the
 * window is per head in both.
 *   q         device  [B][H][d]        the query lla_decode_attn took
 *   k_win     device  [B][H][W][d]     exact keys of loop t, BEFORE RoPE
 *   v_win     device  [B][H][W][d]     exact values of loop t
 *   win_len   device  int32 [B]        window tokens in use, 0..W
 *   win_pos   device  int32 [B]        position of window token 0; token w is
 *                                      rotated at win_pos[b] + w
 *   q_pos     device  int32 [B]        as for lla_decode_attn
 *   rope_cos/_sin, rope_len            as for lla_decode_attn (rope_len >= 128);
 *                                      every window position must be < rope_len
 *   out, lse  device  fp32 [B][H][d], [B][H]   in: latent part; out: merged
 *                                      (rows with win_len 0 are left as they are)
 *   workspace device  >= 256 bytes: the status word (lla_device_status)
 * q, k_win and v_win use the storage dtype (bf16 or fp32).  A win_len outside
 * [0, W] or a window reaching past rope_len skips that sequence's window, a
 * q_pos outside [0, rope_len) is clamped; both record LLA_ERR_DEVICE_ARG.
 * W == 0 or B == 0 launches nothing.
 */
lla_status lla_window_attn(const lla_dims* dims, int B, int W, const void* q,
                           const void* k_win, const void* v_win, const int32_t* win_len,
                           const int32_t* win_pos, const int32_t* q_pos,
                           const float* rope_cos, const float* rope_sin, int64_t rope_len,
                           float* out, float* lse, void* workspace, size_t ws_bytes, void* stream);

/*
 * lla_decode_attn_decoupled — absorbed decoupled-RoPE decode (LLA paper,
 * Appendix J "Absorbed attention"; the path its Table 13 times).  The K
 * up-projection moves to the query side (an MLA-style content path on the
 * latents without RoPE) and position enters through a small explicit rotary
 * branch of d_rope = 64 dimensions per token and head, stored once for all loops:
 *   s_j = (q_c . (c_k,j W_up,k,t^T + mu_k,t) + RoPE(q_r, q_pos) . RoPE(r_j, j))
 *         / sqrt(d + d_rope),
 *   out = sum_j softmax(s)_j (c_v,j W_up,v,t^T + mu_v,t),  lse = ln sum_j exp(s_j).
 * This is a different function from lla_decode_attn (no RoPE on the content
 * keys); a model must have been trained or adapted for it (Appendix J, Table 14).
 * LLA_PER_HEAD only; d_rope must be 64; r_k <= 128 on the bf16 kernel.
 *   q          device  [B][H][d + d_rope]   content part then rotary part
 *   k_rope     device  [B][H][L_max][d_rope] rotary keys before RoPE (storage dtype)
 *   rope_cos/_sin      [rope_len][d_rope/2] for the rotary branch: lla_rope_table
 *                      with lla_dims.d_head = d_rope (theta_f = base^(-2f/d_rope));
 *                      rope_len >= max(L_max, 128)
 *   workspace          >= lla_decoupled_workspace_size() bytes, first 256 zero
 * Everything else as lla_decode_attn (cache, seq_lens, q_pos, W_up, mu, out, lse).
 */
size_t lla_decoupled_workspace_size(const lla_dims* dims, int d_rope, int B, int64_t L_max);
lla_status lla_decode_attn_decoupled(const lla_dims* dims, int loop_t, int d_rope, const void* q,
                                     lla_cache cache, const void* k_rope,
                                     const int32_t* seq_lens, const int32_t* q_pos,
                                     const void* w_up_k, const void* w_up_v,
                                     const float* mu_k, const float* mu_v,
                                     const float* rope_cos, const float* rope_sin, int64_t rope_len,
                                     float* out, float* lse,
                                     void* workspace, size_t ws_bytes, void* stream);

/* Size of the fixed scratch array behind lla_decode_attn_noalloc (64 MiB). */
#define LLA_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * lla_decode_attn_noalloc — lla_decode_attn without a caller workspace, for
 * callers that cannot allocate device memory (for example a plugin inside a
 * host framework whose memory pool owns the GPU, or a serving path that must
 * never call cudaMalloc).  The paper has no counterpart: this is a deployment
 * convenience.  Arguments and results are those of lla_decode_attn, minus
 * `workspace` and `ws_bytes`.
 *   - Scratch lives in a fixed __device__ array of LLA_NOALLOC_SCRATCH_BYTES
 *     inside this library; every GPU that loads the library keeps it until
 *     the process exits.  The call allocates nothing.
 *   - Shapes whose workspace (lla_workspace_size) exceeds that size return
 *     LLA_ERR_UNSUPPORTED before any launch (e.g. beyond about 2,000 sequence-heads
 *     at r_k = 96, r_v = 160).
 *   - The first call on each device looks up the array's device address with
 *     the device current; make that first call before any stream capture.
 *   - The array is shared by every call and keeps the last call's contents;
 *     once the host checks have passed, the status word is cleared on `stream`
 *     before the first launch (a call rejected on the host enqueues nothing).
 *     Calls that overlap on the GPU race and must be serialised by the caller.
 *   - The kernels' device status (LLA_ERR_DEVICE_ARG, LLA_ERR_TIMEOUT,
 *     LLA_ERR_RANGE) is read with lla_device_status(NULL, stream, clear) on
 *     the same device.
 */
lla_status lla_decode_attn_noalloc(const lla_dims* dims, int loop_t, const void* q,
                                   lla_cache cache, const int32_t* seq_lens, const int32_t* q_pos,
                                   const void* w_up_k, const void* w_up_v,
                                   const float* mu_k, const float* mu_v,
                                   const float* rope_cos, const float* rope_sin, int64_t rope_len,
                                   float* out, float* lse, void* stream);

/* Name of the kernel family lla_decode_attn runs for `dims` (host-only, no
 * launch): "fp32" (LLA_F32), "pair-2d" (LLA_2D bf16 with an even H <= 16,
 * r_k <= 128 and r_v <= 256: CTA-pair score kernel on the tensor cores, then a
 * tensor-core value kernel), "plain-2d" (every other LLA_2D bf16 shape: the
 * plain per-(sequence, head) kernels in fp32 arithmetic over the bf16 storage;
 * correct, not tuned), "small-rank"
 * (LLA_PER_HEAD bf16 with r_k in {16, 32}, r_v in {32, 64} and an even H <= 16
 * whose H query images and a 4-slot latent ring fit in shared memory:
 * positions split over CTAs, RoPE applied by the tensor cores), "tile"
 * (every other LLA_PER_HEAD bf16 shape: 128-token tiles over (sequence, head)
 * split over CTAs), or NULL for invalid or unsupported dims. */
const char* lla_decode_kernel(const lla_dims* dims);

/* Name of the kernel family lla_decode_attn_decoupled runs for `dims` and
 * d_rope (host-only, no launch): "fp32" (LLA_F32), "small-rank" (bf16 with r_k in
 * {16, 32}, r_v in {32, 64} and an even H <= 16: positions split over CTAs,
 * rotary branch and content score on the tensor cores, fp32 cos/sin per token),
 * "tile" (every other bf16 shape with r_k <= 128 and r_v <= 256: 128-token
 * tiles over (sequence, head), the same tensor-core score, V read from L2), or
 * NULL for invalid or unsupported dims (LLA_2D, d_rope != 64, larger ranks). */
const char* lla_decoupled_kernel(const lla_dims* dims, int d_rope);

/* Workspace bytes for calls with at most B sequences of L_max slots and
 * encode batches of at most max_N tokens, on the current CUDA device.
 * Returns 0 for invalid dims. */
size_t lla_workspace_size(const lla_dims* dims, int B, int64_t L_max, int max_N);

/* Host-side RoPE table: cos_out/sin_out (host, fp32 [n_pos][d/2]) get
 * cos(p*theta_f), sin(p*theta_f) for p < n_pos, computed in fp64 and rounded
 * once to fp32. */
lla_status lla_rope_table(const lla_dims* dims, int64_t n_pos, float* cos_out, float* sin_out);

/* Synchronise `stream`, then return the status word the kernels recorded in
 * `workspace` (LLA_OK if none); clear it when `clear` is non-zero.  With
 * workspace == NULL the word read is that of lla_decode_attn_noalloc's fixed
 * scratch on the current device. */
lla_status lla_device_status(void* workspace, void* stream, int clear);

/* Static description of a status code. */
const char* lla_status_string(lla_status status);

/* LLA_ABI_VERSION of the loaded library. */
int lla_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LLA_H */
