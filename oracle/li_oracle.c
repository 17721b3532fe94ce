/*
 * li_oracle.c -- plain, slow, fp64 CPU oracle of the LatentIndex indexer scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm may load this library.  It shares no code,
 * header, table or helper with the CUDA library; the only thing the two sides
 * share is the seeded input generator (li_inputs), which holds none of the
 * method's arithmetic.
 *
 * Sources (the web pages on LatentIndex; citations name page and equation):
 *   [S]  "LatentIndex: Cross-Layer Sharing with Layer-Specific Selection for
 *        Sparse Attention" (paper summary page), Methodology: eq. (3) key
 *        reconstruction, eq. (6) query-side decoder absorption, eq. (7) exact
 *        dot-product identity, eq. (8) per-layer scoring with TopK selection,
 *        and the "Hierarchical Selection" paragraph.
 *   [E]  "LatentIndex -- Shared indexer cache, per-layer token choice"
 *        (explainer page): native DSA indexer key cache of 132 B per token per
 *        layer (fp8 keys + scale), the 192-value latent, the absorption
 *        identity q.(D c) = (D^T q).c, and HS with an 8,192-token cart.
 *   [S] Methodology, "Shared Latent Cache", eqs. (1)-(2): the latent of a
 *        token is built from the anchor layer's hidden state x as
 *        z^N = P_N^T x, z^R = Q_t P_R^T x, c = [z^R; z^N].
 *   [S] Methodology, "Layer-specific Key Reconstruction", eqs. (3)-(4): a
 *        decoder's RoPE part satisfies R_t D^R = D^R Q_t through complex
 *        linear combinations within each rotary frequency.
 *
 * Notation.  A decoder is stored as D_l with shape r x d (r = latent rank,
 * d = per-layer indexer key width), so the per-layer key of eq. (3) is
 * k_t = D_l^T c_t and the absorbed query of eq. (6) is q~ = D_l q.  The
 * summary page writes the transpose (its D maps d_C -> d_I); the arithmetic is
 * the same.  The bias b of eq. (3) enters only through beta = q^N . b, which
 * is taken here as a direct input (zero when absent).
 *
 * Every function decodes its inputs exactly to fp64 (fp32 and bf16 are exact
 * in fp64; fp8 E4M3 is decoded from the OCP FP8 definition and multiplied by
 * the stored fp32 scale), then evaluates the defining formula in fp64 in the
 * plain order of the equation.  Selection is a full sort of (score desc,
 * index asc); ties therefore go to the lower index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_FP8 = 2, OR_F64 = 3 };

/* OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m/8 * 2^-6; S.1111.111 is NaN; there are no infinities (max 448). */
double or_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expf = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expf == 0xF && mant == 0x7)
        return NAN;
    if (expf == 0)
        mag = ldexp((double)mant / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expf - 7);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double or_bf16_decode(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const void *p, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32: return (double)((const float *)p)[i];
    case OR_BF16: return or_bf16_decode(((const uint16_t *)p)[i]);
    case OR_FP8: return or_e4m3_decode(((const uint8_t *)p)[i]);
    default: return ((const double *)p)[i];
    }
}

/* Decode `rows` rows of `cols` stored values to fp64, multiplying row i by
 * scale[i] when a scale array is given. */
void or_decode_rows(const void *src, int dtype, const float *scale, int64_t rows, int64_t cols,
                    double *dst)
{
    for (int64_t i = 0; i < rows; i++) {
        double s = scale ? (double)scale[i] : 1.0;
        for (int64_t j = 0; j < cols; j++)
            dst[i * cols + j] = s * elem(src, dtype, i * cols + j);
    }
}

/* Eq. (6): q~_{n,l,h} = D_l q_{n,l,h} for every query n (n runs over the B*T
 * queries), layer l < G and head h < H.
 *   q    [N][G][H][d]   (dtype q_t)
 *   D    [G][r][d]      (dtype D_t)
 *   qabs [N][G][H][r]   fp64 out */
void or_absorb(const void *q, int q_t, const void *D, int D_t, int64_t N, int G, int H, int d,
               int r, double *qabs, int nthreads)
{
    #pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t n = 0; n < N; n++) {
        for (int l = 0; l < G; l++) {
            for (int h = 0; h < H; h++) {
                int64_t qrow = ((n * G + l) * H + h) * (int64_t)d;
                int64_t orow = ((n * G + l) * H + h) * (int64_t)r;
                for (int i = 0; i < r; i++) {
                    double acc = 0.0;
                    for (int j = 0; j < d; j++)
                        acc += elem(D, D_t, ((int64_t)l * r + i) * d + j) * elem(q, q_t, qrow + j);
                    qabs[orow + i] = acc;
                }
            }
        }
    }
}

/* Eq. (3) without bias: the per-layer key a decoder reconstructs from the
 * shared latent, k^l_t = D_l^T c_t.
 *   latent [B][L][r] (+ lat_scale [B][L] for fp8), D [G][r][d]
 *   keys   [G][B][L][d] fp64 out */
void or_reconstruct_keys(const void *latent, int lat_t, const float *lat_scale, const void *D,
                         int D_t, int B, int L, int G, int r, int d, double *keys, int nthreads)
{
    int64_t ntok = (int64_t)B * L;
    #pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t n = 0; n < ntok; n++) {
        double s = lat_scale ? (double)lat_scale[n] : 1.0;
        for (int l = 0; l < G; l++) {
            for (int j = 0; j < d; j++) {
                double acc = 0.0;
                for (int i = 0; i < r; i++)
                    acc += elem(D, D_t, ((int64_t)l * r + i) * d + j) * (s * elem(latent, lat_t, n * r + i));
                keys[((int64_t)l * ntok + n) * d + j] = acc;
            }
        }
    }
}

/* Eq. (8): u^l_{n,t} = sum_h w_{n,l,h} * ReLU(q~_{n,l,h} . c_t + beta_{n,l,h})
 * for every query n = b*T + tq, layer l and cached token t in the valid set
 * V_n = { t : t < L and t <= q_pos[tq] } (all of [0, L) when q_pos is NULL);
 * u = -inf outside V_n.
 *   latent [B][L][r] (+ lat_scale [B][L]); qabs [B][T][G][H][r] fp64;
 *   w [B][T][G][H] fp64; beta same shape or NULL; q_pos [T] or NULL
 *   scores [B][T][G][L] fp64 out */
void or_score(const void *latent, int lat_t, const float *lat_scale, const double *qabs,
              const double *w, const double *beta, const int32_t *q_pos, int B, int T, int G,
              int H, int r, int L, double *scores, int nthreads)
{
    int64_t ntok = (int64_t)B * L;
    #pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t n = 0; n < ntok; n++) {
        int b = (int)(n / L);
        int t = (int)(n % L);
        double c[1024];
        double s = lat_scale ? (double)lat_scale[n] : 1.0;
        for (int i = 0; i < r; i++)
            c[i] = s * elem(latent, lat_t, n * r + i);
        for (int tq = 0; tq < T; tq++) {
            int valid = (q_pos == NULL) || (t <= q_pos[tq]);
            int64_t nq = (int64_t)b * T + tq;
            for (int l = 0; l < G; l++) {
                double u = 0.0;
                if (valid) {
                    for (int h = 0; h < H; h++) {
                        int64_t hrow = (nq * G + l) * H + h;
                        double dot = 0.0;
                        for (int i = 0; i < r; i++)
                            dot += qabs[hrow * r + i] * c[i];
                        if (beta)
                            dot += beta[hrow];
                        u += w[hrow] * (dot > 0.0 ? dot : 0.0);
                    }
                } else {
                    u = -INFINITY;
                }
                scores[(nq * G + l) * (int64_t)L + t] = u;
            }
        }
    }
}

typedef struct {
    double v;
    int32_t i;
} or_pair;

/* score descending, then index ascending */
static int or_pair_cmp(const void *a, const void *b)
{
    const or_pair *x = (const or_pair *)a, *y = (const or_pair *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

/* TopK of eq. (8): per row, the indices of the min(k, |V|) largest scores over
 * the valid prefix [0, valid_len[row]) (all L when valid_len is NULL), found by
 * a full sort (score desc, index asc).  idx [rows][k] is written in that
 * order and padded with -1; vals (optional) gets the scores, -inf padded. */
void or_topk(const double *scores, int64_t rows, int L, const int32_t *valid_len, int k,
             int32_t *idx, double *vals, int nthreads)
{
    #pragma omp parallel for num_threads(nthreads) schedule(dynamic)
    for (int64_t row = 0; row < rows; row++) {
        int V = valid_len ? valid_len[row] : L;
        if (V > L) V = L;
        if (V < 0) V = 0;
        or_pair *p = (or_pair *)malloc(sizeof(or_pair) * (size_t)(V > 0 ? V : 1));
        for (int t = 0; t < V; t++) {
            p[t].v = scores[row * (int64_t)L + t];
            p[t].i = t;
        }
        qsort(p, (size_t)V, sizeof(or_pair), or_pair_cmp);
        for (int j = 0; j < k; j++) {
            idx[row * (int64_t)k + j] = j < V ? p[j].i : -1;
            if (vals)
                vals[row * (int64_t)k + j] = j < V ? p[j].v : -INFINITY;
        }
        free(p);
    }
}

/* Hierarchical selection ("Hierarchical Selection" paragraph of the summary
 * page; the 8,192-token cart of the explainer).  For each sequence b:
 *   1. the anchor (layer 0) has scored every valid position; its top-m
 *      positions (same order as TopK) form the candidate set C_b, written to
 *      cand [B][m] (-1 padded when L < m);
 *   2. the anchor's own selection is its top-k, i.e. the first min(k,|C_b|)
 *      entries of that order;
 *   3. every follower l = 1..G-1 rescores only the positions in C_b with its
 *      own scorer and keeps its top-k inside C_b.
 * `scores` holds the per-layer score rows [B][G][L] of eq. (8) (a follower's
 * score of a candidate is the same function value whether or not the other
 * positions were scored).  idx [B][G][k] out, -1 padded. */
void or_hs(const double *scores, int B, int G, int L, int m, int k, int32_t *cand, int32_t *idx,
           int nthreads)
{
    #pragma omp parallel for num_threads(nthreads) schedule(dynamic)
    for (int b = 0; b < B; b++) {
        const double *anchor = scores + ((int64_t)b * G + 0) * L;
        or_pair *p = (or_pair *)malloc(sizeof(or_pair) * (size_t)(L > 0 ? L : 1));
        for (int t = 0; t < L; t++) {
            p[t].v = anchor[t];
            p[t].i = t;
        }
        qsort(p, (size_t)L, sizeof(or_pair), or_pair_cmp);
        int nc = m < L ? m : L;
        for (int j = 0; j < m; j++)
            cand[(int64_t)b * m + j] = j < nc ? p[j].i : -1;
        for (int j = 0; j < k; j++)
            idx[((int64_t)b * G + 0) * k + j] = j < nc ? p[j].i : -1;
        or_pair *f = (or_pair *)malloc(sizeof(or_pair) * (size_t)(nc > 0 ? nc : 1));
        for (int l = 1; l < G; l++) {
            const double *row = scores + ((int64_t)b * G + l) * L;
            for (int j = 0; j < nc; j++) {
                f[j].i = p[j].i;
                f[j].v = row[p[j].i];
            }
            qsort(f, (size_t)nc, sizeof(or_pair), or_pair_cmp);
            for (int j = 0; j < k; j++)
                idx[((int64_t)b * G + l) * k + j] = j < nc ? f[j].i : -1;
        }
        free(f);
        free(p);
    }
}

/* The native DSA lightning indexer of one layer (explainer page: "DSA
 * lightning indexer", "Indexer key cache" of 132 B per token per layer):
 *   I_t = sum_h w_h * ReLU(q_h . k_t)   over the layer's own key cache,
 * which is eq. (8) with G = 1, the latent replaced by the layer's keys and the
 * absorbed query replaced by the raw query (no decoder).
 *   keys [B][L][d] (+ key_scale [B][L]); q [B][H][d] fp64; w [B][H] fp64
 *   scores [B][L] fp64 out */
void or_native_score(const void *keys, int key_t, const float *key_scale, const double *q,
                     const double *w, int B, int H, int d, int L, double *scores, int nthreads)
{
    or_score(keys, key_t, key_scale, q, w, NULL, NULL, B, 1, 1, H, d, L, scores, nthreads);
}

/* Eqs. (1)-(2) of [S]: the shared latent of one new token per sequence.
 *   x   [B][dm]  the anchor layer's hidden state of the token
 *   P   [r][dm]  rows 0 .. rR-1 are P_R^T, rows rR .. r-1 are P_N^T
 *   pos [B]      the token's position t
 *   c   [B][r]   fp64 out: c = [Q_t P_R^T x ; P_N^T x]
 * Q_t is the rotary position encoding: the RoPE branch is read as rR/2
 * complex numbers (c_2i, c_2i+1), and number i is multiplied by
 * exp(i t theta_i) with theta_i = base^(-2i/rR) ("complex linear combinations
 * within each rotary frequency", [S] after eq. (4)). */
void or_append_latent(const void *x, int x_t, const void *P, int P_t, int B, int dm, int r, int rR,
                      double base, const int32_t *pos, double *c, int nthreads)
{
    #pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int b = 0; b < B; b++) {
        double *cb = c + (int64_t)b * r;
        for (int i = 0; i < r; i++) {
            double acc = 0.0;
            for (int j = 0; j < dm; j++)
                acc += elem(P, P_t, (int64_t)i * dm + j) * elem(x, x_t, (int64_t)b * dm + j);
            cb[i] = acc;
        }
        for (int i = 0; i < rR / 2; i++) {
            const double theta = pow(base, -2.0 * i / rR);
            const double ang = (double)pos[b] * theta;
            const double re = cb[2 * i], im = cb[2 * i + 1];
            cb[2 * i] = re * cos(ang) - im * sin(ang);
            cb[2 * i + 1] = re * sin(ang) + im * cos(ang);
        }
    }
}

/* Rotary position encoding applied to the first nR entries of each of n rows
 * of width dim: pair j (v_2j, v_2j+1) of row i is read as a complex number and
 * multiplied by exp(i pos[i] theta_j), theta_j = base^(-2j/nR).  This is R_t
 * of eq. (4) of [S] on the RoPE part of a per-layer key (and the same
 * schedule as Q_t of eq. (1) on the latent's RoPE branch, with nR = rR). */
void or_rope_rotate(double *v, int64_t n, int dim, int nR, double base, const int32_t *pos)
{
    for (int64_t i = 0; i < n; i++) {
        double *row = v + i * dim;
        for (int j = 0; j < nR / 2; j++) {
            const double ang = (double)pos[i] * pow(base, -2.0 * j / nR);
            const double re = row[2 * j], im = row[2 * j + 1];
            row[2 * j] = re * cos(ang) - im * sin(ang);
            row[2 * j + 1] = re * sin(ang) + im * cos(ang);
        }
    }
}

/* The RoPE part of a decoder under the rotary-structure constraint of eq. (4)
 * of [S], R_t D^R = D^R Q_t, "enforced through complex linear combinations
 * within each rotary frequency".  Key pair j (of dR/2; frequency
 * base^(-2j/dR)) and latent pair i (of rR/2; frequency base^(-2i/rR)) are
 * coupled only when the two frequencies are equal, i.e. j * rR == i * dR,
 * and then by the complex number a + ib = (are, aim)[j][i]: the 2 x 2 block
 * [[a, -b], [b, a]], which commutes with every rotation.  Other entries of
 * the coefficient arrays [dR/2][rR/2] are ignored.
 *   DR [dR][rR] fp64 out (key = DR z, the summary page's orientation) */
void or_rotary_decoder(const double *are, const double *aim, int dR, int rR, double *DR)
{
    memset(DR, 0, sizeof(double) * (size_t)dR * (size_t)rR);
    for (int j = 0; j < dR / 2; j++) {
        for (int i = 0; i < rR / 2; i++) {
            if ((int64_t)j * rR != (int64_t)i * dR)
                continue;
            const double a = are[(int64_t)j * (rR / 2) + i], b = aim[(int64_t)j * (rR / 2) + i];
            DR[(int64_t)(2 * j) * rR + 2 * i] = a;
            DR[(int64_t)(2 * j) * rR + 2 * i + 1] = -b;
            DR[(int64_t)(2 * j + 1) * rR + 2 * i] = b;
            DR[(int64_t)(2 * j + 1) * rR + 2 * i + 1] = a;
        }
    }
}

/* Eq. (3) of [S] evaluated the native way, as per-layer indexer keys with
 * their own rotary encoding: for the token of sequence b at position pos[b],
 *   k^R = R_t (D^R_l P_R^T x)        (rotated after decoding)
 *   k^N = D^N_l P_N^T x + b_l
 *   key = [k^R ; k^N]   (d = dR + dN values)
 * which eqs. (1), (4) and (7) say equals the key decoded from the rotated
 * latent, D_l c_t with c_t = [Q_t P_R^T x ; P_N^T x].
 *   x [B][dm] (x_t), P [r][dm] (P_t; rows < rR are P_R^T, the rest P_N^T)
 *   DR [G][dR][rR], DN [G][dN][r - rR], bias [G][dN] or NULL (all fp64)
 *   keys [G][B][dR + dN] fp64 out */
void or_rope_keys(const void *x, int x_t, const void *P, int P_t, int B, int dm, int r, int rR,
                  const double *DR, const double *DN, const double *bias, int G, int dR, int dN,
                  double base, const int32_t *pos, double *keys, int nthreads)
{
    const int d = dR + dN, rN = r - rR;
    #pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int b = 0; b < B; b++) {
        double z[1024];
        for (int i = 0; i < r; i++) {
            double acc = 0.0;
            for (int j = 0; j < dm; j++)
                acc += elem(P, P_t, (int64_t)i * dm + j) * elem(x, x_t, (int64_t)b * dm + j);
            z[i] = acc;                       /* [P_R^T x ; P_N^T x], no rotation yet */
        }
        for (int l = 0; l < G; l++) {
            double *k = keys + ((int64_t)l * B + b) * d;
            for (int j = 0; j < dR; j++) {
                double acc = 0.0;
                for (int i = 0; i < rR; i++)
                    acc += DR[((int64_t)l * dR + j) * rR + i] * z[i];
                k[j] = acc;
            }
            for (int j = 0; j < dN; j++) {
                double acc = bias ? bias[(int64_t)l * dN + j] : 0.0;
                for (int i = 0; i < rN; i++)
                    acc += DN[((int64_t)l * dN + j) * rN + i] * z[rR + i];
                k[dR + j] = acc;
            }
            or_rope_rotate(k, 1, d, dR, base, pos + b);
        }
    }
}
