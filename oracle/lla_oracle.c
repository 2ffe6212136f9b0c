/*
 * lla_oracle.c — fp64 oracle for Looped Latent Attention.
 *
 * TEST INFRASTRUCTURE ONLY (see lla_oracle.h).  Plain loops in the order the
 * paper states the computation; no blocking, fusion or reordering beyond the
 * definitions.  Parallel over (sequence, head) with OpenMP only: each
 * (b, h) row is computed exactly as the serial loop would.
 *
 * Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped
 * Transformers" (arXiv 2607.15456v2).
 */
#include "lla_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int dims_ok(const oracle_dims* dm) {
    if (!dm) return 0;
    if (dm->T < 1 || dm->H < 1 || dm->d < 2 || (dm->d % 2) != 0) return 0;
    if (dm->r_k < 1 || dm->r_v < 1) return 0;
    if (dm->variant != 0 && dm->variant != 1) return 0;
    if (dm->rope_style != 0 && dm->rope_style != 1) return 0;
    if (!(dm->rope_base > 0.0)) return 0;
    return 1;
}

/* §3 Eq. (4). */
double oracle_compression_ratio(const oracle_dims* dm) {
    double teacher = 2.0 * dm->T * dm->d;            /* per head */
    if (dm->variant == 1) teacher *= dm->H;          /* one latent for all heads */
    return teacher / (double)(dm->r_k + dm->r_v);
}

/* §3 "Teacher cache": 2*T*H*d scalars per token per layer. */
long long oracle_teacher_scalars_per_token(const oracle_dims* dm, int D) {
    return 2LL * dm->T * dm->H * dm->d * (long long)D;
}

/* §3 "Cross-loop codec": (r_k+r_v)*H per token per layer; LLA-2D: (r_k+r_v). */
long long oracle_latent_scalars_per_token(const oracle_dims* dm, int D) {
    long long per_layer = (long long)(dm->r_k + dm->r_v);
    if (dm->variant == 0) per_layer *= dm->H;
    return per_layer * D;
}

/* Nearest bf16 (8 significant bits), ties to even, from the binary
 * representation's definition: scale x into [2^7, 2^8) and round the
 * integer part. */
double oracle_round_bf16(double x) {
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    int e;
    (void)frexp(fabs(x), &e);                /* |x| = m * 2^e, m in [0.5, 1) */
    if (e < -125) e = -125;                  /* below 2^-126 the spacing stays 2^-133 */
    double scaled = ldexp(fabs(x), 8 - e);   /* in [128, 256) for normal x */
    double fl = floor(scaled);
    double frac = scaled - fl;
    double rounded;
    if (frac > 0.5) rounded = fl + 1.0;
    else if (frac < 0.5) rounded = fl;
    else rounded = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double y = ldexp(rounded, e - 8);
    if (y > 3.3895313892515355e38) y = INFINITY;   /* above bf16 max */
    return x < 0 ? -y : y;
}

/* theta_f = base^(-2f/d): the standard rotary frequencies (Su et al.), which
 * the paper applies unchanged after reconstruction (§3 "RoPE and
 * reconstruction"). */
static double rope_theta(const oracle_dims* dm, int f) {
    return pow(dm->rope_base, -2.0 * (double)f / (double)dm->d);
}

/* Index pair rotated by frequency f. */
static void rope_pair(const oracle_dims* dm, int f, int* i0, int* i1) {
    if (dm->rope_style == 0) { *i0 = f; *i1 = f + dm->d / 2; }
    else                     { *i0 = 2 * f; *i1 = 2 * f + 1; }
}

/* y = R(position) x : each pair (x0, x1) is rotated by angle position*theta_f. */
static void rope_rotate(const oracle_dims* dm, const double* x, double pos,
                        double* y) {
    for (int f = 0; f < dm->d / 2; ++f) {
        int i0, i1;
        rope_pair(dm, f, &i0, &i1);
        double ang = pos * rope_theta(dm, f);
        double c = cos(ang), s = sin(ang);
        y[i0] = x[i0] * c - x[i1] * s;
        y[i1] = x[i0] * s + x[i1] * c;
    }
}

/* §3 Eq. (2). */
int oracle_encode(const oracle_dims* dm, int N, const double* x,
                  const int* seq_idx, const int* pos, const double* w_down,
                  const double* mu, int r, double* cache, int B, long L_max,
                  int round_bf16) {
    if (!dims_ok(dm) || N < 0 || r < 1 || B < 0 || L_max < 0) return 1;
    const int T = dm->T, H = dm->H, d = dm->d;
    for (int n = 0; n < N; ++n)
        if (seq_idx[n] < 0 || seq_idx[n] >= B || pos[n] < 0 || pos[n] >= L_max)
            return 1;
    if (dm->variant == 0) {
        const long Td = (long)T * d;
        for (int n = 0; n < N; ++n)
            for (int h = 0; h < H; ++h) {
                const double* xv = x + ((long)n * H + h) * Td;
                const double* m = mu + (long)h * Td;
                const double* W = w_down + (long)h * Td * r;
                double* c = cache + (((long)seq_idx[n] * H + h) * L_max + pos[n]) * r;
                for (int k = 0; k < r; ++k) {
                    double acc = 0.0;
                    for (long u = 0; u < Td; ++u) acc += (xv[u] - m[u]) * W[u * r + k];
                    c[k] = round_bf16 ? oracle_round_bf16(acc) : acc;
                }
            }
    } else {
        const long THd = (long)T * H * d;
        for (int n = 0; n < N; ++n) {
            const double* xv = x + (long)n * THd;
            double* c = cache + ((long)seq_idx[n] * L_max + pos[n]) * r;
            for (int k = 0; k < r; ++k) {
                double acc = 0.0;
                for (long u = 0; u < THd; ++u) acc += (xv[u] - mu[u]) * w_down[u * r + k];
                c[k] = round_bf16 ? oracle_round_bf16(acc) : acc;
            }
        }
    }
    return 0;
}

/* Eq. (3) for one token: xhat[e] = sum_k c[k] * W[e][k] + mu_t[e]. */
static void reconstruct(const double* c, const double* W, const double* mu_t,
                        int d, int r, double* xhat) {
    for (int e = 0; e < d; ++e) {
        double acc = 0.0;
        for (int k = 0; k < r; ++k) acc += c[k] * W[(long)e * r + k];
        xhat[e] = acc + mu_t[e];
    }
}

/* Softmax over s[0..L) with the max subtracted; returns m and sum exp(s-m),
 * writes normalised weights into p. */
static void softmax(const double* s, long L, double* p, double* m_out,
                    double* z_out) {
    double m = -INFINITY;
    for (long j = 0; j < L; ++j) if (s[j] > m) m = s[j];
    double z = 0.0;
    for (long j = 0; j < L; ++j) { p[j] = exp(s[j] - m); z += p[j]; }
    for (long j = 0; j < L; ++j) p[j] /= z;
    *m_out = m; *z_out = z;
}

int oracle_decode(const oracle_dims* dm, int t, int B, long L_max,
                  const double* q, const double* cache_k, const double* cache_v,
                  const int* seq_lens, const int* q_pos, long pos_offset,
                  const double* w_up_k, const double* w_up_v,
                  const double* mu_k, const double* mu_v,
                  double* out, double* lse, double* scores, int v_mode) {
    if (!dims_ok(dm) || t < 0 || t >= dm->T || B < 0 || L_max < 0) return 1;
    if (v_mode != 0 && v_mode != 1) return 1;
    const int T = dm->T, H = dm->H, d = dm->d, rk = dm->r_k, rv = dm->r_v;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > L_max) return 1;
    int bad = 0;
    (void)T;
#pragma omp parallel for schedule(dynamic, 1) reduction(|:bad)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        const long L = seq_lens[b];
        double* o = out + bh * d;
        if (L == 0) {
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            lse[bh] = -INFINITY;
            continue;
        }
        /* Per-loop maps and means (Eq. (3)): W_up,t and mu_t = slice t of mu. */
        const double *Wk, *Wv, *muk_t, *muv_t;
        if (dm->variant == 0) {
            Wk = w_up_k + (((long)t * H + h) * d) * rk;
            Wv = w_up_v + (((long)t * H + h) * d) * rv;
            muk_t = mu_k + (long)h * dm->T * d + (long)t * d;
            muv_t = mu_v + (long)h * dm->T * d + (long)t * d;
        } else {
            Wk = w_up_k + ((long)t * H * d + (long)h * d) * rk;
            Wv = w_up_v + ((long)t * H * d + (long)h * d) * rv;
            muk_t = mu_k + ((long)t * H + h) * d;
            muv_t = mu_v + ((long)t * H + h) * d;
        }
        double* qr = (double*)malloc(sizeof(double) * d);
        double* kh = (double*)malloc(sizeof(double) * d);
        double* kr = (double*)malloc(sizeof(double) * d);
        double* vh = (double*)malloc(sizeof(double) * d);
        double* s = (double*)malloc(sizeof(double) * L);
        double* p = (double*)malloc(sizeof(double) * L);
        double* av = (double*)malloc(sizeof(double) * rv);

        rope_rotate(dm, q + bh * d, (double)(q_pos[b] + pos_offset), qr);
        const double scale = 1.0 / sqrt((double)d);
        for (long j = 0; j < L; ++j) {
            const double* ck = (dm->variant == 0)
                ? cache_k + (bh * L_max + j) * rk
                : cache_k + ((long)b * L_max + j) * rk;
            reconstruct(ck, Wk, muk_t, d, rk, kh);
            rope_rotate(dm, kh, (double)(j + pos_offset), kr);
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += qr[e] * kr[e];
            s[j] = acc * scale;
            if (scores) scores[bh * L_max + j] = s[j];
        }
        double m, z;
        softmax(s, L, p, &m, &z);
        double psum = 0.0;
        for (long j = 0; j < L; ++j) psum += p[j];
        if (fabs(psum - 1.0) > 1e-12) bad |= 1;

        for (int e = 0; e < d; ++e) o[e] = 0.0;
        if (v_mode == 0) {
            for (long j = 0; j < L; ++j) {
                const double* cv = (dm->variant == 0)
                    ? cache_v + (bh * L_max + j) * rv
                    : cache_v + ((long)b * L_max + j) * rv;
                reconstruct(cv, Wv, muv_t, d, rv, vh);
                for (int e = 0; e < d; ++e) o[e] += p[j] * vh[e];
            }
        } else {
            /* Appendix J "Absorbed attention": the V up-projection moves out
             * of the sum over tokens. */
            for (int k = 0; k < rv; ++k) av[k] = 0.0;
            for (long j = 0; j < L; ++j) {
                const double* cv = (dm->variant == 0)
                    ? cache_v + (bh * L_max + j) * rv
                    : cache_v + ((long)b * L_max + j) * rv;
                for (int k = 0; k < rv; ++k) av[k] += p[j] * cv[k];
            }
            for (int e = 0; e < d; ++e) {
                double acc = 0.0;
                for (int k = 0; k < rv; ++k) acc += av[k] * Wv[(long)e * rv + k];
                o[e] = acc + psum * muv_t[e];
            }
        }
        lse[bh] = m + log(z);
        free(qr); free(kh); free(kr); free(vh); free(s); free(p); free(av);
    }
    return bad ? 2 : 0;
}

/* "Hybrid Latent Attention for Looped Language Models" §3.4 Eq. (4), written out:
 * the latent tokens' scores and the window tokens' scores form one vector, one
 * softmax normalises it, and each weight multiplies its own token's value. */
int oracle_hybrid(const oracle_dims* dm, int t, int B, long L_max, long W,
                  const double* q, const double* cache_k, const double* cache_v,
                  const int* n_lat, const int* q_pos,
                  const double* w_up_k, const double* w_up_v,
                  const double* mu_k, const double* mu_v,
                  const double* k_win, const double* v_win, const int* n_win,
                  const int* win_pos, double* out, double* lse) {
    if (!dims_ok(dm) || dm->variant != 0 || t < 0 || t >= dm->T || B < 0 || L_max < 0 || W < 0)
        return 1;
    const int H = dm->H, d = dm->d, rk = dm->r_k, rv = dm->r_v;
    for (int b = 0; b < B; ++b)
        if (n_lat[b] < 0 || n_lat[b] > L_max || n_win[b] < 0 || n_win[b] > W) return 1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(|:bad)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        const long nl = n_lat[b], nw = n_win[b], n = nl + nw;
        double* o = out + bh * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        if (n == 0) {
            lse[bh] = -INFINITY;
            continue;
        }
        const double* Wk = w_up_k + (((long)t * H + h) * d) * rk;
        const double* Wv = w_up_v + (((long)t * H + h) * d) * rv;
        const double* muk_t = mu_k + (long)h * dm->T * d + (long)t * d;
        const double* muv_t = mu_v + (long)h * dm->T * d + (long)t * d;
        double* qr = (double*)malloc(sizeof(double) * d);
        double* kh = (double*)malloc(sizeof(double) * d);
        double* kr = (double*)malloc(sizeof(double) * d);
        double* vh = (double*)malloc(sizeof(double) * d);
        double* s = (double*)malloc(sizeof(double) * n);
        double* p = (double*)malloc(sizeof(double) * n);
        rope_rotate(dm, q + bh * d, (double)q_pos[b], qr);
        const double scale = 1.0 / sqrt((double)d);
        for (long j = 0; j < n; ++j) {
            if (j < nl) {   /* latent token j */
                reconstruct(cache_k + (bh * L_max + j) * rk, Wk, muk_t, d, rk, kh);
                rope_rotate(dm, kh, (double)j, kr);
            } else {        /* window token w = j - nl */
                const long w = j - nl;
                rope_rotate(dm, k_win + (bh * W + w) * d, (double)(win_pos[b] + w), kr);
            }
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += qr[e] * kr[e];
            s[j] = acc * scale;
        }
        double m, z;
        softmax(s, n, p, &m, &z);
        double psum = 0.0;
        for (long j = 0; j < n; ++j) psum += p[j];
        if (fabs(psum - 1.0) > 1e-12) bad |= 1;
        for (long j = 0; j < n; ++j) {
            const double* v;
            if (j < nl) {
                reconstruct(cache_v + (bh * L_max + j) * rv, Wv, muv_t, d, rv, vh);
                v = vh;
            } else {
                v = v_win + (bh * W + (j - nl)) * d;
            }
            for (int e = 0; e < d; ++e) o[e] += p[j] * v[e];
        }
        lse[bh] = m + log(z);
        free(qr); free(kh); free(kr); free(vh); free(s); free(p);
    }
    return bad ? 2 : 0;
}

/* RoPE over a d_rope-wide branch: frequencies base^(-2f/d_rope), f < d_rope/2,
 * pairs (f, f + d_rope/2) or (2f, 2f + 1) as dm->rope_style. */
static void rope_rotate_branch(const oracle_dims* dm, int d_rope, const double* x, double pos,
                               double* y) {
    for (int f = 0; f < d_rope / 2; ++f) {
        const int i0 = dm->rope_style == 0 ? f : 2 * f;
        const int i1 = dm->rope_style == 0 ? f + d_rope / 2 : 2 * f + 1;
        const double ang = pos * pow(dm->rope_base, -2.0 * f / d_rope);
        const double c = cos(ang), s = sin(ang);
        y[i0] = x[i0] * c - x[i1] * s;
        y[i1] = x[i0] * s + x[i1] * c;
    }
}

/* LLA page, Appendix J "Absorbed attention" (decoupled rotary branch). */
int oracle_decoupled(const oracle_dims* dm, int t, int d_rope, int B, long L_max,
                     const double* q, const double* cache_k, const double* cache_v,
                     const double* k_rope, const int* seq_lens, const int* q_pos,
                     long pos_offset, const double* w_up_k, const double* w_up_v,
                     const double* mu_k, const double* mu_v, double* out, double* lse) {
    if (!dims_ok(dm) || dm->variant != 0 || t < 0 || t >= dm->T || B < 0 || L_max < 0 ||
        d_rope < 2 || d_rope % 2)
        return 1;
    const int H = dm->H, d = dm->d, rk = dm->r_k, rv = dm->r_v, dq = d + d_rope;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > L_max) return 1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(|:bad)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        const long L = seq_lens[b];
        double* o = out + bh * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        if (L == 0) {
            lse[bh] = -INFINITY;
            continue;
        }
        const double* Wk = w_up_k + (((long)t * H + h) * d) * rk;
        const double* Wv = w_up_v + (((long)t * H + h) * d) * rv;
        const double* muk_t = mu_k + (long)h * dm->T * d + (long)t * d;
        const double* muv_t = mu_v + (long)h * dm->T * d + (long)t * d;
        const double* qv = q + bh * dq;
        double* kh = (double*)malloc(sizeof(double) * d);
        double* vh = (double*)malloc(sizeof(double) * d);
        double* qr = (double*)malloc(sizeof(double) * d_rope);
        double* kr = (double*)malloc(sizeof(double) * d_rope);
        double* s = (double*)malloc(sizeof(double) * L);
        double* p = (double*)malloc(sizeof(double) * L);
        rope_rotate_branch(dm, d_rope, qv + d, (double)(q_pos[b] + pos_offset), qr);
        const double scale = 1.0 / sqrt((double)dq);
        for (long j = 0; j < L; ++j) {
            reconstruct(cache_k + (bh * L_max + j) * rk, Wk, muk_t, d, rk, kh);
            rope_rotate_branch(dm, d_rope, k_rope + (bh * L_max + j) * d_rope, (double)(j + pos_offset), kr);
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += qv[e] * kh[e];
            for (int e = 0; e < d_rope; ++e) acc += qr[e] * kr[e];
            s[j] = acc * scale;
        }
        double m, z;
        softmax(s, L, p, &m, &z);
        double psum = 0.0;
        for (long j = 0; j < L; ++j) psum += p[j];
        if (fabs(psum - 1.0) > 1e-12) bad |= 1;
        for (long j = 0; j < L; ++j) {
            reconstruct(cache_v + (bh * L_max + j) * rv, Wv, muv_t, d, rv, vh);
            for (int e = 0; e < d; ++e) o[e] += p[j] * vh[e];
        }
        lse[bh] = m + log(z);
        free(kh); free(vh); free(qr); free(kr); free(s); free(p);
    }
    return bad ? 2 : 0;
}

int oracle_sdpa(const oracle_dims* dm, int B, long L_max, const double* q,
                const double* k, const double* v, const int* seq_lens,
                const int* q_pos, long pos_offset, double* out, double* lse) {
    if (!dims_ok(dm) || B < 0 || L_max < 0) return 1;
    const int H = dm->H, d = dm->d;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > L_max) return 1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(|:bad)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H);
        const long L = seq_lens[b];
        double* o = out + bh * d;
        if (L == 0) {
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            lse[bh] = -INFINITY;
            continue;
        }
        double* qr = (double*)malloc(sizeof(double) * d);
        double* kr = (double*)malloc(sizeof(double) * d);
        double* s = (double*)malloc(sizeof(double) * L);
        double* p = (double*)malloc(sizeof(double) * L);
        rope_rotate(dm, q + bh * d, (double)(q_pos[b] + pos_offset), qr);
        const double scale = 1.0 / sqrt((double)d);
        for (long j = 0; j < L; ++j) {
            rope_rotate(dm, k + (bh * L_max + j) * d, (double)(j + pos_offset), kr);
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += qr[e] * kr[e];
            s[j] = acc * scale;
        }
        double m, z;
        softmax(s, L, p, &m, &z);
        double psum = 0.0;
        for (long j = 0; j < L; ++j) psum += p[j];
        if (fabs(psum - 1.0) > 1e-12) bad |= 1;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        for (long j = 0; j < L; ++j)
            for (int e = 0; e < d; ++e) o[e] += p[j] * v[(bh * L_max + j) * d + e];
        lse[bh] = m + log(z);
        free(qr); free(kr); free(s); free(p);
    }
    return bad ? 2 : 0;
}
