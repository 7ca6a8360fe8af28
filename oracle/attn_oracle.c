/*
 * attn_oracle.c -- plain fp64 CPU oracle for multi-head scaled-dot-product
 * attention in the three forms the attention pages use.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline / reference arm load this library.  It shares no code, header,
 * table or helper with the CUDA library; it is written to be checked by eye.
 *
 * Every entry point computes, for each query row i and its admitted key set
 * K(i) (all keys; the first seq_len keys; or the 3D neighborhood window):
 *
 *     s_j = scale * sum_d q[i,d] * k[j,d]          for j in K(i)
 *     m   = max_j s_j
 *     p_j = exp(s_j - m) / sum_{j' in K(i)} exp(s_j' - m)
 *     o_i = sum_j p_j * v[j, :]
 *
 * in double precision with libm's exp, cos, sin and pow.  This is the
 * attention the pages name: "cuBLAS matmuls for ... attention scores" plus a
 * custom softmax kernel (iris.c issue #15 "CUDA codepath !", the cuBLAS reply),
 * the naive decode attention over a device-resident KV cache (fak "GPU - the
 * in-kernel forward pass", sections 0 and 4) and the windowed
 * score/softmax/accumulate of candle's neighborhood attention (candle PR #11,
 * the "Line-for-line port of neighborhood_attention.metal" commit).
 *
 * Layouts (all contiguous, row-major, D innermost):
 *   full / joint / na3d : q, k, v, o  [B, H, N, D]
 *   decode              : q, o [B, Hq, D];  k, v [B, Hkv, Lmax, D]
 *   positions           : pos [N, 4] int32
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math), so
 * the result does not depend on the host ISA's FMA contraction.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * One query row against an explicit list of admitted keys.
 * kbase/vbase point at the [N, D] key/value matrix of this (batch, head);
 * keys[] holds row indices into it.  On return o[0..D) is the output row and,
 * if p != NULL, p[j] is the normalised probability of keys[j].
 * s[] is caller-provided scratch of length nkeys.
 */
static void attend_row(const double *qi, const double *kbase, const double *vbase,
                       const int64_t *keys, int64_t nkeys, int D, double scale,
                       double *o, double *p, double *s)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        const double *kj = kbase + keys[j] * (int64_t)D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const double pj = s[j] / l;
        const double *vj = vbase + keys[j] * (int64_t)D;
        for (int d = 0; d < D; ++d) o[d] += pj * vj[d];
        if (p) p[j] = pj;
    }
}

/* ------------------------------------------------------------------ full -- */

/*
 * Full (unmasked) attention of query row `row` (flattened b*H*Nq + h*Nq + i)
 * over all Nkv keys of the same (b, h).  p (optional) receives Nkv values.
 */
static void full_one(const double *q, const double *k, const double *v, double *o, double *p,
                     int H, int Nq, int Nkv, int D, double scale, int64_t row,
                     int64_t *keys, double *s)
{
    const int64_t bh = row / Nq;
    (void)H;
    for (int64_t j = 0; j < Nkv; ++j) keys[j] = j;
    attend_row(q + row * D, k + bh * (int64_t)Nkv * D, v + bh * (int64_t)Nkv * D,
               keys, Nkv, D, scale, o, p, s);
}

/* All rows.  p (optional) is [B, H, Nq, Nkv]. */
void oracle_full_fwd(const double *q, const double *k, const double *v, double *o, double *p,
                     int B, int H, int Nq, int Nkv, int D, double scale, int nthreads)
{
    set_threads(nthreads);
    const int64_t rows = (int64_t)B * H * Nq;
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Nkv > 0 ? Nkv : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r)
            full_one(q, k, v, o + r * D, p ? p + r * (int64_t)Nkv : NULL, H, Nq, Nkv, D, scale,
                     r, keys, s);
        free(keys);
        free(s);
    }
}

/* Selected rows only: o_rows is [nrows, D], rows[] are flattened row ids. */
void oracle_full_rows(const double *q, const double *k, const double *v, double *o_rows,
                      int B, int H, int Nq, int Nkv, int D, double scale,
                      const int64_t *rows, int64_t nrows, int nthreads)
{
    (void)B;
    set_threads(nthreads);
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Nkv > 0 ? Nkv : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r)
            full_one(q, k, v, o_rows + r * D, NULL, H, Nq, Nkv, D, scale, rows[r], keys, s);
        free(keys);
        free(s);
    }
}

/* ------------------------------------------------------------------ RoPE -- */

/*
 * FLUX-style multi-axis rotary embedding, in place on x [BH, N, D].
 * The D channels are cut into consecutive axis blocks of axes_dim[0..3]
 * channels ("[32,32,32,32]", iris.c issue #15, GGML lessons item 3).  Inside
 * the block of axis a (width n_a, starting at channel c_a), adjacent channel
 * pair (c_a + 2i, c_a + 2i + 1), i = 0 .. n_a/2 - 1, is rotated by the angle
 *     phi = pos[t, a] * theta^(-2i / n_a)
 * so both members of a pair share one angle (the "repeat_interleave" of the
 * per-pair frequency):
 *     x0' = x0 cos(phi) - x1 sin(phi)
 *     x1' = x0 sin(phi) + x1 cos(phi)
 * Requires sum(axes_dim) == D and every axes_dim even (checked by the caller).
 */
void oracle_rope_rotate(double *x, const int32_t *pos, int BH, int N, int D,
                        const int32_t *axes_dim, double theta)
{
    int64_t total = (int64_t)BH * N;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < total; ++r) {
        const int64_t t = r % N;
        double *xr = x + r * D;
        int c = 0;
        for (int a = 0; a < 4; ++a) {
            const int na = axes_dim[a];
            for (int i = 0; i < na / 2; ++i) {
                const double freq = pow(theta, -2.0 * (double)i / (double)na);
                const double phi = (double)pos[t * 4 + a] * freq;
                const double cs = cos(phi), sn = sin(phi);
                const double x0 = xr[c + 2 * i], x1 = xr[c + 2 * i + 1];
                xr[c + 2 * i] = x0 * cs - x1 * sn;
                xr[c + 2 * i + 1] = x0 * sn + x1 * cs;
            }
            c += na;
        }
    }
    (void)D;
}

/*
 * Joint text+image attention: rotate copies of q and k (never v), then full
 * attention over the whole concatenated sequence.  If rows != NULL only those
 * rows are produced into o ([nrows, D]); otherwise o is [B, H, N, D].
 */
int oracle_joint_fwd(const double *q, const double *k, const double *v, double *o,
                     int B, int H, int N, int D, const int32_t *pos, const int32_t *axes_dim,
                     double theta, double scale, const int64_t *rows, int64_t nrows,
                     int nthreads)
{
    set_threads(nthreads);
    const size_t n = (size_t)B * H * N * D;
    double *qr = (double *)malloc(n * sizeof(double));
    double *kr = (double *)malloc(n * sizeof(double));
    if (!qr || !kr) { free(qr); free(kr); return 1; }
    memcpy(qr, q, n * sizeof(double));
    memcpy(kr, k, n * sizeof(double));
    oracle_rope_rotate(qr, pos, B * H, N, D, axes_dim, theta);
    oracle_rope_rotate(kr, pos, B * H, N, D, axes_dim, theta);
    if (rows)
        oracle_full_rows(qr, kr, v, o, B, H, N, N, D, scale, rows, nrows, nthreads);
    else
        oracle_full_fwd(qr, kr, v, o, NULL, B, H, N, N, D, scale, nthreads);
    free(qr);
    free(kr);
    return 0;
}

/* ------------------------------------------------------ causal prefill -- */

/*
 * Causal grouped-query prefill (Llama prefill, the pp64..pp512 workloads of
 * fak "GPU - the in-kernel forward pass", section 3): q [B, Hq, N, D],
 * k, v [B, Hkv, N, D]; query head hq reads KV head hq / (Hq / Hkv) and query
 * position i attends to key positions j <= i.  If rows != NULL only those
 * flattened rows (b*Hq*N + hq*N + i) are produced into o ([nrows, D]).
 */
void oracle_causal_gqa_fwd(const double *q, const double *k, const double *v, double *o,
                           int B, int Hq, int Hkv, int N, int D, double scale,
                           const int64_t *rows, int64_t nrows, int nthreads)
{
    set_threads(nthreads);
    const int group = Hq / Hkv;
    const int64_t total = rows ? nrows : (int64_t)B * Hq * N;
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < total; ++r) {
            const int64_t row = rows ? rows[r] : r;
            const int64_t i = row % N, bh = row / N;
            const int64_t b = bh / Hq, hq = bh % Hq;
            const int64_t kvbase = (b * Hkv + hq / group) * (int64_t)N * D;
            for (int64_t j = 0; j < N; ++j) keys[j] = j;
            attend_row(q + row * D, k + kvbase, v + kvbase, keys, i + 1,
                       D, scale, o + r * D, NULL, s);
        }
        free(keys);
        free(s);
    }
}

/* ---------------------------------------------------------------- decode -- */

/*
 * Single-token GQA decode over a KV cache of capacity Lmax.  Query head hq of
 * batch b reads KV head hq / (Hq / Hkv) (contiguous groups of query heads share
 * one KV head) and attends to cache rows j < seq_len[b]; rows at or beyond
 * seq_len[b] are never read.
 */
void oracle_decode_gqa(const double *q, const double *kc, const double *vc,
                       const int32_t *seq_len, double *o, int B, int Hq, int Hkv, int Lmax,
                       int D, double scale, int nthreads)
{
    set_threads(nthreads);
    const int group = Hq / Hkv;
    const int64_t rows = (int64_t)B * Hq;
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Lmax > 0 ? Lmax : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < rows; ++r) {
            const int64_t b = r / Hq, hq = r % Hq;
            const int64_t kvh = hq / group;
            const int64_t L = seq_len[b];
            for (int64_t j = 0; j < L; ++j) keys[j] = j;
            const int64_t base = (b * Hkv + kvh) * (int64_t)Lmax * D;
            attend_row(q + r * D, kc + base, vc + base, keys, L, D, scale, o + r * D, NULL, s);
        }
        free(keys);
        free(s);
    }
}

/* ------------------------------------------------------------------ NA3D -- */

/*
 * NATTEN boundary window along one axis of extent n for a requested (odd)
 * kernel k: the effective kernel is k_eff = min(k, n) ("effective_kernel()"
 * in candle PR #11's "kernel exceeds grid extent" commit) and the window of
 * position i is [start, start + k_eff) with
 *     start = clamp(i - floor(k / 2), 0, n - k_eff)
 * i.e. centred on i and shifted to stay inside the axis.
 */
int oracle_na_window_start(int i, int n, int k)
{
    const int keff = k < n ? k : n;
    int st = i - k / 2;
    if (st < 0) st = 0;
    if (st > n - keff) st = n - keff;
    return st;
}

/* Per-query start triple, starts[N*3] = (t, h, w) starts, for the window test. */
void oracle_na3d_window_starts(int T, int Hg, int W, const int32_t *kernel, int32_t *starts)
{
    const int64_t N = (int64_t)T * Hg * W;
    for (int64_t i = 0; i < N; ++i) {
        const int t = (int)(i / ((int64_t)Hg * W));
        const int h = (int)((i / W) % Hg);
        const int w = (int)(i % W);
        starts[i * 3 + 0] = oracle_na_window_start(t, T, kernel[0]);
        starts[i * 3 + 1] = oracle_na_window_start(h, Hg, kernel[1]);
        starts[i * 3 + 2] = oracle_na_window_start(w, W, kernel[2]);
    }
}

/* Admitted keys of query i (row-major t, h, w), in increasing index order. */
static int64_t na3d_keys(int64_t i, int T, int Hg, int W, const int32_t *kernel, int64_t *keys)
{
    const int t = (int)(i / ((int64_t)Hg * W));
    const int h = (int)((i / W) % Hg);
    const int w = (int)(i % W);
    const int kt = kernel[0] < T ? kernel[0] : T;
    const int kh = kernel[1] < Hg ? kernel[1] : Hg;
    const int kw = kernel[2] < W ? kernel[2] : W;
    const int st = oracle_na_window_start(t, T, kernel[0]);
    const int sh = oracle_na_window_start(h, Hg, kernel[1]);
    const int sw = oracle_na_window_start(w, W, kernel[2]);
    int64_t n = 0;
    for (int a = st; a < st + kt; ++a)
        for (int b = sh; b < sh + kh; ++b)
            for (int c = sw; c < sw + kw; ++c)
                keys[n++] = ((int64_t)a * Hg + b) * W + c;
    return n;
}

/*
 * 3D neighborhood attention, B batches x H heads over a T x Hg x W grid
 * (N = T*Hg*W tokens, row-major t, h, w).  If rows != NULL only those
 * flattened rows are produced into o ([nrows, D]).  If p != NULL (full run
 * only) it receives the dense [B, H, N, N] probability matrix with zeros
 * outside each window.
 */
void oracle_na3d_fwd(const double *q, const double *k, const double *v, double *o, double *p,
                     int B, int H, int T, int Hg, int W, int D, const int32_t *kernel,
                     double scale, const int64_t *rows, int64_t nrows, int nthreads)
{
    set_threads(nthreads);
    const int64_t N = (int64_t)T * Hg * W;
    const int64_t kt = kernel[0] < T ? kernel[0] : T;
    const int64_t kh = kernel[1] < Hg ? kernel[1] : Hg;
    const int64_t kw = kernel[2] < W ? kernel[2] : W;
    const int64_t win = kt * kh * kw;
    const int64_t total = rows ? nrows : (int64_t)B * H * N;
    if (p && !rows) memset(p, 0, sizeof(double) * (size_t)((int64_t)B * H * N * N));
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)win);
        double *s = (double *)malloc(sizeof(double) * (size_t)win);
        double *pw = (double *)malloc(sizeof(double) * (size_t)win);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < total; ++r) {
            const int64_t row = rows ? rows[r] : r;
            const int64_t bh = row / N, i = row % N;
            const int64_t nk = na3d_keys(i, T, Hg, W, kernel, keys);
            attend_row(q + row * D, k + bh * N * D, v + bh * N * D, keys, nk, D, scale,
                       o + r * D, pw, s);
            if (p && !rows)
                for (int64_t j = 0; j < nk; ++j) p[row * N + keys[j]] = pw[j];
        }
        free(keys);
        free(s);
        free(pw);
    }
    (void)B;
    (void)H;
}
