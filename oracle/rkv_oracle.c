/*
 * rkv_oracle.c -- plain, slow, single-threaded fp64 reference of the ResidualKV
 * cache-write path and its sparse read path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or helper with the CUDA path.
 *
 * Citations name sections of the reading-notes page "ResidualKV：基于参考向量与
 * 残差的 KV Cache 压缩" (on "ResidualKV: Residual-Based KV Cache Compression for
 * Efficient Long-Context Inference", arXiv 2602.08005v2); after "=" comes the paper
 * section the note summarises.  Where the page is silent, the reading taken is
 * stated at the function.
 *
 * All inputs are the stored values (fp32 / bf16 / FP8 bytes decoded exactly to
 * double by the caller); every sum and product below is in double, in the order
 * the formula is written, with no blocking or reordering.
 *
 * Pins (tests/test_oracle_*.py): every function below is checked against
 * brute force, closed forms, a library routine or an exact identity.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Reference schedule.  §2.6 = Sec. IV-A: a fixed stride keeps every s-th token
 * as a reference.  Reading: the first reference is token `first`, then every
 * `stride` tokens.  Returns the number of references written to ref_pos.      */
int rkvo_fixed_schedule(int T, int stride, int first, int32_t *ref_pos)
{
    int n = 0;
    for (int t = first; t < T; t += stride)
        ref_pos[n++] = t;
    return n;
}

/* §2.6 = Sec. IV-A, dynamic stride: p_{m+1} = p_m + s0 + floor(alpha (p_m - n_sink)),
 * starting at p_0 = first.  Writes positions < T (at most cap) and returns the count. */
int rkvo_dynamic_schedule(int T, int s0, double alpha, int n_sink, int first,
                          int32_t *ref_pos, int cap)
{
    int n = 0;
    long long p = first;
    while (p < T && n < cap) {
        ref_pos[n++] = (int32_t)p;
        p = p + s0 + (long long)floor(alpha * (double)(p - n_sink));
    }
    return n;
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 as defined by the OCP 8-bit floating point specification (OFP8):
 * sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; the only
 * NaN encodings are S.1111.111; largest finite magnitude 448 = 1.75 * 2^8;
 * subnormals m * 2^-9.  §2.4 = Sec. IV-A / V-A: deployed references are FP8.
 * Reading: round to nearest, ties to even; magnitudes above 448 saturate to 448.  */
double rkvo_fp8_decode(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* round half to even of a non-negative double */
static double rne(double q)
{
    double f = floor(q);
    double r = q - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

uint8_t rkvo_fp8_encode(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t s = (signbit(x) ? 0x80 : 0x00);
    double a = fabs(x);
    if (a >= 448.0)
        return s | 0x7E;                         /* 1.75 * 2^8 */
    if (a < ldexp(1.0, -6)) {                    /* subnormal range: step 2^-9 */
        double q = rne(ldexp(a, 9));             /* 0..8; 8 is the smallest normal */
        return s | (uint8_t)q;
    }
    int e2;
    frexp(a, &e2);                               /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                              /* a in [2^e, 2^(e+1)) */
    double q = rne(ldexp(a, 3 - e));             /* in [8, 16] */
    if (q >= 16.0) { q = 8.0; e += 1; }
    if (e > 8 || (e == 8 && q > 14.0))
        return s | 0x7E;
    return s | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* ------------------------------------------------------------------------- */
/* Squared L2 distance ||x - r||^2, summed in index order. */
double rkvo_sqdist(const double *x, const double *r, int W)
{
    double d = 0.0;
    for (int c = 0; c < W; c++) {
        double u = x[c] - r[c];
        d += u * u;
    }
    return d;
}

typedef struct { double d; int32_t slot; } cand_t;

static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->d < b->d) return -1;
    if (a->d > b->d) return 1;
    return (a->slot > b->slot) - (a->slot < b->slot);     /* tie -> lower slot */
}

static int int_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* §2.2 = Sec. IV-A, retrieval: R_i = arg top-k_i over the pool of -||kv_i - kv_j||^2,
 * k_i = min(k, |pool|) (§2.1 symbol table).  The pool is refs[0 .. n_pool-1], the
 * references strictly before token i (reading of "historical reference set").
 * Reading: equal distances are broken towards the lower slot (earlier position).
 * Output: idx[0..k_i-1] in ascending slot order, idx[k_i..k-1] = -1.
 * If dk != NULL: dk[0] = k_i-th smallest distance, dk[1] = (k_i+1)-th (or INFINITY).
 * Returns k_i.                                                                   */
int rkvo_retrieve(const double *x, const double *refs, int n_pool, int W, int k,
                  int32_t *idx, double *dk)
{
    int ki = n_pool < k ? n_pool : k;
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(n_pool > 0 ? n_pool : 1));
    for (int j = 0; j < n_pool; j++) {
        c[j].d = rkvo_sqdist(x, refs + (size_t)j * W, W);
        c[j].slot = j;
    }
    qsort(c, (size_t)n_pool, sizeof(cand_t), cand_cmp);
    for (int m = 0; m < k; m++)
        idx[m] = m < ki ? c[m].slot : -1;
    qsort(idx, (size_t)ki, sizeof(int32_t), int_cmp);
    if (dk) {
        dk[0] = ki > 0 ? c[ki - 1].d : 0.0;
        dk[1] = n_pool > ki ? c[ki].d : INFINITY;
    }
    free(c);
    return ki;
}

/* §2.2 = Sec. IV-A: mean_i = (1/k_i) sum_{j in R_i} kv_j, taken in KV space.
 * The sum runs over idx in the given (ascending) order.  k_i = 0 gives the zero
 * vector (reading: an empty pool has mean 0).                                    */
void rkvo_mean(const double *refs, const int32_t *idx, int ki, int W, double *mean)
{
    for (int c = 0; c < W; c++) {
        double s = 0.0;
        for (int m = 0; m < ki; m++)
            s += refs[(size_t)idx[m] * W + c];
        mean[c] = ki > 0 ? s / (double)ki : 0.0;
    }
}

/* Swish with beta = 1 (reading: the page writes Swish without a parameter). */
double rkvo_swish(double u)
{
    return u / (1.0 + exp(-u));
}

/* §2.3 = Sec. IV-A, compressor: f_c(x) = (Swish(x W_c1) ⊙ x W_c2) W_c3, with
 * W_c1, W_c2 in R^{2dk x dff} and W_c3 in R^{dff x dc}.  The weights arrive
 * out-major: W1t[f][c] = W_c1[c][f], W2t[f][c] = W_c2[c][f], W3t[j][f] = W_c3[f][j].
 * If h != NULL it receives the d_ff-wide gated hidden vector.                    */
void rkvo_fc(const double *x, const double *W1t, const double *W2t, const double *W3t,
             int W, int d_ff, int d_c, double *out, double *h)
{
    double *hv = (double *)malloc(sizeof(double) * (size_t)d_ff);
    for (int f = 0; f < d_ff; f++) {
        double a1 = 0.0, a2 = 0.0;
        for (int c = 0; c < W; c++) {
            a1 += x[c] * W1t[(size_t)f * W + c];
            a2 += x[c] * W2t[(size_t)f * W + c];
        }
        hv[f] = rkvo_swish(a1) * a2;
    }
    for (int j = 0; j < d_c; j++) {
        double s = 0.0;
        for (int f = 0; f < d_ff; f++)
            s += hv[f] * W3t[(size_t)j * d_ff + f];
        out[j] = s;
    }
    if (h)
        memcpy(h, hv, sizeof(double) * (size_t)d_ff);
    free(hv);
}

/* §2.4 = Sec. IV-A, per-token group quantisation.  For each group G of at most
 * `group` consecutive latent coordinates (groups never span tokens):
 *   delta = (z_max - z_min) / (2^b - 1),  q = round((z - z_min) / delta),
 *   z~ = q delta + z_min.
 * Readings: groups are [g*group, min(d_c, (g+1)*group)); round() is half-up,
 * floor(u + 1/2), clamped to [0, 2^b - 1]; a constant group (z_max == z_min) is
 * stored exactly as delta = 0, q = 0, z_min = the constant.                      */
void rkvo_quantize(const double *z, int d_c, int group, int bits,
                   uint8_t *q, double *zmin, double *delta)
{
    int qmax = (1 << bits) - 1;
    int ng = (d_c + group - 1) / group;
    for (int g = 0; g < ng; g++) {
        int c0 = g * group, c1 = c0 + group < d_c ? c0 + group : d_c;
        double lo = z[c0], hi = z[c0];
        for (int c = c0 + 1; c < c1; c++) {
            if (z[c] < lo) lo = z[c];
            if (z[c] > hi) hi = z[c];
        }
        zmin[g] = lo;
        if (hi == lo) {
            delta[g] = 0.0;
            for (int c = c0; c < c1; c++) q[c] = 0;
            continue;
        }
        double dl = (hi - lo) / (double)qmax;
        delta[g] = dl;
        for (int c = c0; c < c1; c++) {
            double v = floor((z[c] - lo) / dl + 0.5);
            if (v < 0) v = 0;
            if (v > qmax) v = qmax;
            q[c] = (uint8_t)v;
        }
    }
}

/* §2.4: z~ = q delta + z_min, per group. */
void rkvo_dequantize(const uint8_t *q, const double *zmin, const double *delta,
                     int d_c, int group, double *zq)
{
    for (int c = 0; c < d_c; c++)
        zq[c] = (double)q[c] * delta[c / group] + zmin[c / group];
}

/* ------------------------------------------------------------------------- */
/* The write path for a list of tokens of one (layer, sequence).
 *   kv    [T][W]      stored token vectors
 *   refs  [n_ref][W]  stored reference vectors (after the storage round trip:
 *                     §2.5 = Sec. IV-B, encoder and decoder use the same numerical
 *                     references), refs[m] belongs to position ref_pos[m]
 * For a non-reference token t (§2.2-§2.4):
 *   pool = references with position < t;  R = retrieve;  mean = mean(R);
 *   z = f_c(kv_t) - f_c(mean)   (§2.3: encode each, then subtract);
 *   (q, z_min, delta) = quantize(z).
 * Reading for a reference token t (stored uncompressed): idx = [own slot, -1..],
 * z = 0, q = 0, z_min = delta = 0, so that a read returns the reference itself.
 * forced_idx (nullable, [n_tok][k]): use these reference slots (-1 padded,
 * ascending) instead of retrieving.
 * Outputs (all nullable except idx): idx [n_tok][k], ki [n_tok],
 * dk [n_tok][2] (k-th and (k+1)-th distance), z [n_tok][d_c], q [n_tok][d_c],
 * zmin/delta [n_tok][ceil(d_c/group)], mean [n_tok][W].                          */
void rkvo_compress_tokens(int T, int W, int d_ff, int d_c, int k, int group, int bits,
                          const double *kv, const double *refs, const int32_t *ref_pos,
                          int n_ref, const double *W1t, const double *W2t,
                          const double *W3t, const int32_t *tokens, int n_tok,
                          const int32_t *forced_idx, int32_t *idx, int32_t *ki_out,
                          double *dk, double *z, uint8_t *q, double *zmin,
                          double *delta, double *mean_out)
{
    int ng = (d_c + group - 1) / group;
    double *mean = (double *)malloc(sizeof(double) * (size_t)W);
    double *f1 = (double *)malloc(sizeof(double) * (size_t)d_c);
    double *f2 = (double *)malloc(sizeof(double) * (size_t)d_c);
    double *zz = (double *)malloc(sizeof(double) * (size_t)d_c);
    uint8_t *qq = (uint8_t *)malloc((size_t)d_c);
    double *mn = (double *)malloc(sizeof(double) * (size_t)ng);
    double *dl = (double *)malloc(sizeof(double) * (size_t)ng);
    (void)T;
    for (int n = 0; n < n_tok; n++) {
        int t = tokens[n];
        int32_t *ix = idx + (size_t)n * k;
        int own = -1, n_pool = 0;
        for (int m = 0; m < n_ref; m++) {
            if (ref_pos[m] == t) own = m;
            if (ref_pos[m] < t) n_pool++;
        }
        int ki;
        double d2[2] = {0.0, INFINITY};
        if (own >= 0) {
            ix[0] = own;
            for (int m = 1; m < k; m++) ix[m] = -1;
            ki = 1;
            memcpy(mean, refs + (size_t)own * W, sizeof(double) * (size_t)W);
            for (int c = 0; c < d_c; c++) { zz[c] = 0.0; qq[c] = 0; }
            for (int g = 0; g < ng; g++) { mn[g] = 0.0; dl[g] = 0.0; }
        } else {
            if (forced_idx) {
                ki = 0;
                for (int m = 0; m < k; m++) {
                    ix[m] = forced_idx[(size_t)n * k + m];
                    if (ix[m] >= 0) ki++;
                }
            } else {
                ki = rkvo_retrieve(kv + (size_t)t * W, refs, n_pool, W, k, ix, d2);
            }
            rkvo_mean(refs, ix, ki, W, mean);
            rkvo_fc(kv + (size_t)t * W, W1t, W2t, W3t, W, d_ff, d_c, f1, NULL);
            rkvo_fc(mean, W1t, W2t, W3t, W, d_ff, d_c, f2, NULL);
            for (int c = 0; c < d_c; c++) zz[c] = f1[c] - f2[c];
            rkvo_quantize(zz, d_c, group, bits, qq, mn, dl);
        }
        if (ki_out) ki_out[n] = ki;
        if (dk) { dk[2 * n] = d2[0]; dk[2 * n + 1] = d2[1]; }
        if (z) memcpy(z + (size_t)n * d_c, zz, sizeof(double) * (size_t)d_c);
        if (q) memcpy(q + (size_t)n * d_c, qq, (size_t)d_c);
        if (zmin) memcpy(zmin + (size_t)n * ng, mn, sizeof(double) * (size_t)ng);
        if (delta) memcpy(delta + (size_t)n * ng, dl, sizeof(double) * (size_t)ng);
        if (mean_out) memcpy(mean_out + (size_t)n * W, mean, sizeof(double) * (size_t)W);
    }
    free(mean); free(f1); free(f2); free(zz); free(qq); free(mn); free(dl);
}

/* §2.7 = Sec. IV-C, sparse read: for each selected token, read only its own codes,
 * group extremes and reference relation, plus the referenced vectors; return
 *   z~_t = dequantize(q_t)   and   mean_t = (1/k_t) sum_{j in idx_t} refs[j].
 * idx entries < 0 are padding.  Records are [T][...] of one sequence.             */
void rkvo_gather(int W, int d_c, int group, int k, const double *refs,
                 const uint8_t *q, const double *zmin, const double *delta,
                 const int32_t *idx, const int32_t *sel, int n_sel,
                 double *zq_out, double *mean_out)
{
    int ng = (d_c + group - 1) / group;
    for (int n = 0; n < n_sel; n++) {
        int t = sel[n];
        rkvo_dequantize(q + (size_t)t * d_c, zmin + (size_t)t * ng, delta + (size_t)t * ng,
                        d_c, group, zq_out + (size_t)n * d_c);
        const int32_t *ix = idx + (size_t)t * k;
        int ki = 0;
        for (int m = 0; m < k; m++)
            if (ix[m] >= 0) ki++;
        rkvo_mean(refs, ix, ki, W, mean_out + (size_t)n * W);
    }
}

/* Retrieval alone (§2.2) for a list of tokens of one sequence: idx [n_tok][k]
 * (reference tokens get {own slot, -1, ...}), k_i [n_tok], dk [n_tok][2].        */
void rkvo_retrieve_tokens(int W, int k, const double *kv, const double *refs,
                          const int32_t *ref_pos, int n_ref, const int32_t *tokens, int n_tok,
                          int32_t *idx, int32_t *ki_out, double *dk)
{
    for (int n = 0; n < n_tok; n++) {
        int t = tokens[n], own = -1, n_pool = 0;
        for (int m = 0; m < n_ref; m++) {
            if (ref_pos[m] == t) own = m;
            if (ref_pos[m] < t) n_pool++;
        }
        int32_t *ix = idx + (size_t)n * k;
        if (own >= 0) {
            ix[0] = own;
            for (int m = 1; m < k; m++) ix[m] = -1;
            ki_out[n] = 1;
            dk[2 * n] = 0.0;
            dk[2 * n + 1] = INFINITY;
            continue;
        }
        ki_out[n] = rkvo_retrieve(kv + (size_t)t * W, refs, n_pool, W, k, ix, dk + 2 * n);
    }
}

/* ------------------------------------------------------------------------- */
/* Rotary position embedding of one head of dimension D at position pos.  §2.1
 * (implementation requirement) says the restored pre-RoPE key must be rotated at the
 * token's own position before RoPE attention; the page does not fix the RoPE variant.
 * Reading: the rotary embedding as first defined (RoFormer): consecutive coordinate
 * pairs (x_{2i}, x_{2i+1}), i = 0 .. D/2-1, rotated by the angle pos * theta_i with
 * theta_i = base^(-2i/D):
 *   x'_{2i}   = x_{2i} cos(a) - x_{2i+1} sin(a)
 *   x'_{2i+1} = x_{2i} sin(a) + x_{2i+1} cos(a).                                   */
void rkvo_rope(double *x, int D, double pos, double base)
{
    for (int i = 0; i < D / 2; i++) {
        double theta = pow(base, -2.0 * (double)i / (double)D);
        double a = pos * theta;
        double c = cos(a), s = sin(a);
        double x0 = x[2 * i], x1 = x[2 * i + 1];
        x[2 * i] = x0 * c - x1 * s;
        x[2 * i + 1] = x0 * s + x1 * c;
    }
}

/* §2.5 = Sec. IV-B, linear decoder without bias: f_d(z) = z W_d, W_d in R^{d_c x 2d_k},
 * stored out-major: Wd[c][j] = W_d[j][c], c < 2 d_k.                               */
void rkvo_decode(const double *z, const double *Wd, int d_c, int W, double *out)
{
    for (int c = 0; c < W; c++) {
        double s = 0.0;
        for (int j = 0; j < d_c; j++) s += z[j] * Wd[(size_t)c * d_c + j];
        out[c] = s;
    }
}

/* §2.5 = Sec. IV-B and §2.7 = Sec. IV-C, restoring the selected tokens of one sequence:
 *   KV^_t = f_d(z~_t) + mean_t,   then split: K^ = KV^[0, N D), V^ = KV^[N D, 2 N D),
 *   heads in order (head h = coordinates [h D, (h+1) D) of each half);
 * the key of every head is rotated at the token's own position t (rkvo_rope);
 * z~_t and mean_t are the sparse read of rkvo_gather.  Outputs [n_sel][N D] each.     */
void rkvo_restore(int N, int D, int d_c, int group, int k, double rope_base,
                  const double *refs, const uint8_t *q, const double *zmin, const double *delta,
                  const int32_t *idx, const double *Wd, const int32_t *sel, int n_sel,
                  double *k_out, double *v_out)
{
    int dk = N * D, W = 2 * dk;
    double *zq = malloc(sizeof(double) * d_c);
    double *mean = malloc(sizeof(double) * W);
    double *dec = malloc(sizeof(double) * W);
    for (int n = 0; n < n_sel; n++) {
        int32_t one = sel[n];
        rkvo_gather(W, d_c, group, k, refs, q, zmin, delta, idx, &one, 1, zq, mean);
        rkvo_decode(zq, Wd, d_c, W, dec);
        double *ko = k_out + (size_t)n * dk, *vo = v_out + (size_t)n * dk;
        for (int c = 0; c < dk; c++) {
            ko[c] = dec[c] + mean[c];
            vo[c] = dec[dk + c] + mean[dk + c];
        }
        for (int h = 0; h < N; h++) rkvo_rope(ko + (size_t)h * D, D, (double)one, rope_base);
    }
    free(zq); free(mean); free(dec);
}

/* §2.7 = Sec. IV-C, sparse attention of one decode step over the restored set:
 *   o_j = softmax( q_j K^_I^T / sqrt(D) ) V^_I
 * for each query head j.  Reading (the page writes the formula per head): H query
 * heads share the N key/value heads in groups of H/N, query head j reading KV head
 * floor(j / (H/N)).  Rows n with valid[n] == 0 (padding) are not part of I.
 * q [H][D]; K, V [n][N D] (head h = [h D, (h+1) D)); o [H][D].  The softmax is taken
 * as exp(s - max s) / sum exp(s - max s), which equals the definition.            */
void rkvo_attention(int H, int N, int D, const double *q, const double *K, const double *V,
                    const int32_t *valid, int n, double *o)
{
    int G = H / N;
    double *s = malloc(sizeof(double) * (n > 0 ? n : 1));
    for (int j = 0; j < H; j++) {
        int h = j / G;
        double mx = -INFINITY;
        for (int t = 0; t < n; t++) {
            if (!valid[t]) continue;
            double d = 0.0;
            for (int c = 0; c < D; c++) d += q[(size_t)j * D + c] * K[(size_t)t * N * D + (size_t)h * D + c];
            s[t] = d / sqrt((double)D);
            if (s[t] > mx) mx = s[t];
        }
        double den = 0.0;
        for (int t = 0; t < n; t++)
            if (valid[t]) den += exp(s[t] - mx);
        for (int c = 0; c < D; c++) {
            double acc = 0.0;
            for (int t = 0; t < n; t++)
                if (valid[t]) acc += exp(s[t] - mx) * V[(size_t)t * N * D + (size_t)h * D + c];
            o[(size_t)j * D + c] = den > 0.0 ? acc / den : 0.0;
        }
    }
    free(s);
}
