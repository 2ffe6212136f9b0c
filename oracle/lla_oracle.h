/*
 * lla_oracle.h — the oracle for Looped Latent Attention (LLA): a plain, slow,
 * fp64 CPU statement of what the cache codec and the latent-store decode
 * compute.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never includes, links or
 * calls anything declared here; only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped
 * Transformers" (arXiv 2607.15456v2), §3 Eq. (1)-(4) and "RoPE and
 * reconstruction", §3 "The LLA-2D variant", Appendix J "Absorbed attention".
 * Matrices follow the row-vector convention of the paper's slides
 * ("Store one code; reconstruct the requested loop").
 *
 * All arrays are dense, row-major, fp64.  Return value 0 = ok, non-zero =
 * invalid argument or a failed internal check (see each function).
 */
#ifndef LLA_ORACLE_H
#define LLA_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int T;             /* loops (recurrence steps)                          */
    int H;             /* attention heads                                   */
    int d;             /* head width d_head (even)                          */
    int r_k, r_v;      /* latent ranks of the K and V codecs                */
    int variant;       /* 0 = per-head LLA, 1 = LLA-2D (heads folded)       */
    double rope_base;  /* RoPE base, theta_f = base^(-2f/d)                 */
    int rope_style;    /* 0 = rotate-half pairs (f, f+d/2); 1 = interleaved
                          pairs (2f, 2f+1)                                 */
} oracle_dims;

/* Eq. (4): rho = 2*T*d / (r_k + r_v) (per-head).  LLA-2D: the latent covers
 * all heads, rho = 2*T*H*d / (r_k + r_v). */
double oracle_compression_ratio(const oracle_dims* dm);

/* Cached scalars per token for a D-layer stack: the teacher stores 2*T*H*d
 * per layer, per-head LLA (r_k+r_v)*H, LLA-2D (r_k+r_v) (§3 "Teacher cache",
 * "Cross-loop codec", "The LLA-2D variant"). */
long long oracle_teacher_scalars_per_token(const oracle_dims* dm, int D);
long long oracle_latent_scalars_per_token(const oracle_dims* dm, int D);

/* Round an fp64 value to the nearest bfloat16 value (ties to even),
 * returned widened to fp64.  Storage conversion for the encode output. */
double oracle_round_bf16(double x);

/* Eq. (2): c = (x - mu) W_down for N tokens of one axis (K or V) with rank r,
 * written to cache slot (seq_idx[n], pos[n]).
 *   per-head: x [N][H][T*d], w_down [H][T*d][r], mu [H][T*d],
 *             cache [B][H][L_max][r]
 *   LLA-2D:   x [N][T*H*d], w_down [T*H*d][r], mu [T*H*d],
 *             cache [B][L_max][r]
 * (x index t*d+i per head follows Eq. (1); LLA-2D stacks loop-major,
 * index (t*H+h)*d+i.)  round_bf16 != 0 rounds each latent to bf16. */
int oracle_encode(const oracle_dims* dm, int N, const double* x,
                  const int* seq_idx, const int* pos, const double* w_down,
                  const double* mu, int r, double* cache, int B, long L_max,
                  int round_bf16);

/* Decode attention at loop t (0-based) for every sequence and head, the
 * literal definition:
 *   Eq. (3)  k_j = c_k,j W_up,k,t^T + mu_k,t ; v_j likewise,
 *   RoPE applied after reconstruction (key at position j+pos_offset, query
 *   at q_pos[b]+pos_offset),
 *   s_j = q'.k'_j / sqrt(d) over j < seq_lens[b], two-pass softmax,
 *   out = sum_j p_j v_j, lse = ln sum_j exp(s_j).
 * Layouts: q [B][H][d]; cache_k [B][H][L_max][r_k] (2D: [B][L_max][r_k]);
 * w_up_k [T][H][d][r_k] (2D: [T][H*d][r_k], the same memory order);
 * mu_k [H][T*d] (2D: [T*H*d]); v likewise; out [B][H][d]; lse [B][H];
 * scores [B][H][L_max] (may be NULL; unused slots untouched).
 * v_mode 0 reconstructs every v_j; v_mode 1 uses the Appendix J identity
 * sum_j p_j (c_v,j W^T + mu) = (sum_j p_j c_v,j) W^T + (sum_j p_j) mu.
 * seq_lens[b] == 0 gives out = 0 and lse = -inf.  Returns 2 if a softmax
 * row fails to sum to 1 within 1e-12. */
int oracle_decode(const oracle_dims* dm, int t, int B, long L_max,
                  const double* q, const double* cache_k, const double* cache_v,
                  const int* seq_lens, const int* q_pos, long pos_offset,
                  const double* w_up_k, const double* w_up_v,
                  const double* mu_k, const double* mu_v,
                  double* out, double* lse, double* scores, int v_mode);

/* The same attention over given uncompressed pre-RoPE K and V
 * ([B][H][L_max][d] each): the teacher's computation. */
int oracle_sdpa(const oracle_dims* dm, int B, long L_max, const double* q,
                const double* k, const double* v, const int* seq_lens,
                const int* q_pos, long pos_offset, double* out, double* lse);

/* Hybrid attention with an exact window ("Hybrid Latent Attention for Looped
 * Language Models", §3.4 "Exact sliding window", Eq. (4)): one softmax over
 *   latent scores  s_j  for cached tokens j < n_lat[b] (keys and values
 *                  reconstructed by Eq. (3) of the LLA page, key rotated at j),
 *   exact scores   s_w  for window tokens w < n_win[b] (pre-RoPE keys k_win and
 *                  values v_win given, key rotated at win_pos[b] + w),
 * query rotated at q_pos[b]; out = sum of p times the token's value (latent:
 * reconstructed, window: exact), lse = ln sum exp(s).  Per-head variant only.
 * Layouts as oracle_decode, plus k_win / v_win [B][H][W][d].  An empty row
 * (n_lat + n_win == 0) gives out = 0 and lse = -inf.  Returns 2 if a softmax row
 * fails to sum to 1 within 1e-12. */
int oracle_hybrid(const oracle_dims* dm, int t, int B, long L_max, long W,
                  const double* q, const double* cache_k, const double* cache_v,
                  const int* n_lat, const int* q_pos,
                  const double* w_up_k, const double* w_up_v,
                  const double* mu_k, const double* mu_v,
                  const double* k_win, const double* v_win, const int* n_win,
                  const int* win_pos, double* out, double* lse);

/* Absorbed decoupled-RoPE decode at loop t (LLA page, Appendix J "Absorbed
 * attention": an MLA-style NoPE content path on the latents plus a small explicit
 * rotary branch shared across the loops), per-head variant, written out:
 *   content key   k_j = c_k,j W_up,k,t^T + mu_k,t           (Eq. (3), no rotation)
 *   rotary key    r_j = k_rope[b][h][j] (d_rope values, one per token for all loops)
 *   query         q = [q_c (d) ; q_r (d_rope)]
 *   s_j = (q_c . k_j + RoPE(q_r, q_pos) . RoPE(r_j, j)) / sqrt(d + d_rope)
 * with the rotary branch's frequencies theta_f = base^(-2f/d_rope) and the
 * dimension pairs of dm->rope_style over d_rope; out = sum_j p_j v_j with
 * v_j = c_v,j W_up,v,t^T + mu_v,t, lse = ln sum_j exp(s_j).  Layouts: q
 * [B][H][d + d_rope]; k_rope [B][H][L_max][d_rope]; the rest as oracle_decode.
 * Returns 2 if a softmax row fails to sum to 1 within 1e-12. */
int oracle_decoupled(const oracle_dims* dm, int t, int d_rope, int B, long L_max,
                     const double* q, const double* cache_k, const double* cache_v,
                     const double* k_rope, const int* seq_lens, const int* q_pos,
                     long pos_offset, const double* w_up_k, const double* w_up_v,
                     const double* mu_k, const double* mu_v, double* out, double* lse);

/* Threads the oracle's OpenMP loops use. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
