/*
 * Plain fp64 CPU oracle for causal scaled-dot-product attention, forward and
 * backward.  TEST INFRASTRUCTURE ONLY: the product path never links, loads or
 * calls this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it computes is the *composed* attention of
 *   "xtrain docs/03-autograd-engine.md", section "Attention 用组合，不写 fused kernel"
 *     attn = matmul(softmax(scale(matmul(Q, K^T))), V)
 * with the causal mask of
 *   "xtrain docs/13-flash-attention.md", section "什么是 flash-attention"
 *     (key position j > query position i  ->  logit = -inf)
 * and the logsumexp L = m + log(l) that the same section says the fused forward
 * stores (natural log).
 *
 * The backward goes through the explicit softmax Jacobian-vector product of
 *   "xtrain docs/03-autograd-engine.md", section "各算子 backward 数学", softmax row:
 *     dx[r,c] = y[r,c] * (d[r,c] - sum_c' d[r,c'] * y[r,c'])
 * with the row sum formed directly from the materialised P and dP matrices.  It
 * does NOT use the flash shortcut D_i = dO_i . O_i; that identity is checked
 * against this oracle by the tests instead.
 *
 * Every intermediate is materialised for one head at a time in fp64:
 *   s  = scale * Q K^T           [S,S]   (masked entries = -inf)
 *   P  = row softmax(s)          [S,S]
 *   O  = P V                     [S,hd]
 *   dV = P^T dO                  [S,hd]
 *   dP = dO V^T                  [S,S]
 *   dX = P o (dP - rowsum(P o dP))  (softmax backward)
 *   dS = scale * dX              (scale backward)
 *   dQ = dS K,  dK = dS^T Q      [S,hd]
 * The loops run over every (i, j), masked ones included: exp(-inf) = 0 makes
 * their contribution exactly zero, which keeps the code a literal transcription
 * of the definition.  OpenMP only splits each stage over its output rows.
 *
 * Optional dropout on the attention probabilities: the dropout operator of
 *   "xtrain docs/17-dropout.md" ("Phase T18: Dropout"), section "Key Design
 *   Decisions" (counter-based RNG, inverted scaling, backward with the same mask)
 * inserted between the softmax and the product with V:
 *   Pd = P o C,  C_ij = keep(seed, idx_ij) / (1 - p)     O  = Pd V
 *   dV = Pd^T dO,  dPd = dO V^T,  dP = dPd o C (the dropout node's backward)
 * and then the same softmax and scale backward as above.  idx_ij is the flat
 * index of element (b, i, j) of the [bh, S, S] probability tensor.  The keep
 * decision follows the page: key = seed XOR (idx * 0x9E3779B97F4A7C15),
 * h = splitmix64(key), u = (h >> 40) / 2^24 in fp32, keep = (u >= p).  Here
 * splitmix64(x) is the first output of the SplitMix64 generator started from
 * state x: the state advances by the golden-ratio increment and is then mixed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* s[i][j] = scale * sum_d q[i][d] k[j][d]; -inf where causal and j > i */
static void scores(const double *q, const double *k, long S, long hd, double scale,
                   int causal, double *s)
{
#pragma omp parallel for schedule(dynamic, 8) if (S >= 64)
    for (long i = 0; i < S; ++i) {
        for (long j = 0; j < S; ++j) {
            if (causal && j > i) {
                s[i * S + j] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (long d = 0; d < hd; ++d) acc += q[i * hd + d] * k[j * hd + d];
            s[i * S + j] = scale * acc;
        }
    }
}

/* in place: row i of s becomes softmax(s_i); lse[i] = m_i + log(sum_j exp(s_ij - m_i)) */
static void row_softmax(double *s, long S, double *lse)
{
#pragma omp parallel for schedule(static) if (S >= 64)
    for (long i = 0; i < S; ++i) {
        double *row = s + i * S;
        double m = -INFINITY;
        for (long j = 0; j < S; ++j)
            if (row[j] > m) m = row[j];
        double z = 0.0;
        for (long j = 0; j < S; ++j) {
            row[j] = exp(row[j] - m);
            z += row[j];
        }
        for (long j = 0; j < S; ++j) row[j] /= z;
        lse[i] = m + log(z);
    }
}

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): one step from state x. */
uint64_t xfa_oracle_splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The dropout page's Bernoulli draw for element `index`: 1 = keep, 0 = drop. */
int xfa_oracle_keep(uint64_t seed, uint64_t index, float p)
{
    const uint64_t h = xfa_oracle_splitmix64(seed ^ (index * 0x9E3779B97F4A7C15ull));
    const float u = (float)(h >> 40) / 16777216.0f;
    return u >= p;
}

/* c[i][e] = sum_j a[i][j] b[j][e], a [n][n], b [n][w] */
static void matmul_nn(const double *a, const double *b, long n, long w, double *c)
{
#pragma omp parallel for schedule(static) if (n >= 64)
    for (long i = 0; i < n; ++i) {
        for (long e = 0; e < w; ++e) c[i * w + e] = 0.0;
        for (long j = 0; j < n; ++j) {
            double aij = a[i * n + j];
            for (long e = 0; e < w; ++e) c[i * w + e] += aij * b[j * w + e];
        }
    }
}

/* c[j][e] = sum_i a[i][j] b[i][e], i.e. a^T b; a [n][n], b [n][w] */
static void matmul_tn(const double *a, const double *b, long n, long w, double *c)
{
#pragma omp parallel for schedule(static) if (n >= 64)
    for (long j = 0; j < n; ++j) {
        for (long e = 0; e < w; ++e) c[j * w + e] = 0.0;
        for (long i = 0; i < n; ++i) {
            double aij = a[i * n + j];
            for (long e = 0; e < w; ++e) c[j * w + e] += aij * b[i * w + e];
        }
    }
}

/* c[i][j] = sum_e a[i][e] b[j][e], i.e. a b^T; a, b [n][w], c [n][n] */
static void matmul_nt(const double *a, const double *b, long n, long w, double *c)
{
#pragma omp parallel for schedule(static) if (n >= 64)
    for (long i = 0; i < n; ++i) {
        for (long j = 0; j < n; ++j) {
            double acc = 0.0;
            for (long e = 0; e < w; ++e) acc += a[i * w + e] * b[j * w + e];
            c[i * n + j] = acc;
        }
    }
}

/*
 * One head.  q, k, v, dout: [S][hd] fp64 row-major.  Outputs (caller-owned):
 *   out [S][hd], lse [S]; when dout != NULL also dq, dk, dv [S][hd].
 * C: NULL, or the [S][S] dropout factors applied to P before the product with V.
 * Optional diagnostics (NULL to skip), one value per query row i:
 *   p_rowsum[i]   = sum_j P_ij
 *   pdp_rowsum[i] = sum_j P_ij dP_ij   (the softmax-backward row term)
 *   ds_rowsum[i]  = sum_j dS_ij
 */
static int head_impl(const double *q, const double *k, const double *v, const double *dout, long S, long hd,
                     double scale, int causal, const double *C, double *out, double *lse, double *dq, double *dk,
                     double *dv, double *p_rowsum, double *pdp_rowsum, double *ds_rowsum)
{
    if (!q || !k || !v || !out || !lse || S < 1 || hd < 1) return ORACLE_BAD_ARG;
    if (dout && (!dq || !dk || !dv)) return ORACLE_BAD_ARG;

    double *P = (double *)malloc(sizeof(double) * (size_t)S * (size_t)S);
    if (!P) return ORACLE_NO_MEMORY;
    double *Pd = NULL;   /* P o C when dropout is on */
    if (C) {
        Pd = (double *)malloc(sizeof(double) * (size_t)S * (size_t)S);
        if (!Pd) {
            free(P);
            return ORACLE_NO_MEMORY;
        }
    }

    scores(q, k, S, hd, scale, causal, P);  /* P holds s */
    row_softmax(P, S, lse);                 /* P holds softmax(s) */
    if (C)                                  /* the dropout node's forward */
        for (long e = 0; e < S * S; ++e) Pd[e] = P[e] * C[e];
    matmul_nn(C ? Pd : P, v, S, hd, out);   /* O = P V (or Pd V) */

    if (p_rowsum) {
        for (long i = 0; i < S; ++i) {
            double acc = 0.0;
            for (long j = 0; j < S; ++j) acc += P[i * S + j];
            p_rowsum[i] = acc;
        }
    }

    if (dout) {
        double *dP = (double *)malloc(sizeof(double) * (size_t)S * (size_t)S);
        if (!dP) {
            free(P);
            free(Pd);
            return ORACLE_NO_MEMORY;
        }
        matmul_tn(C ? Pd : P, dout, S, hd, dv);   /* dV = P^T dO (or Pd^T dO) */
        matmul_nt(dout, v, S, hd, dP);            /* dP = dO V^T */
        if (C)                                    /* the dropout node's backward */
            for (long e = 0; e < S * S; ++e) dP[e] *= C[e];

        /* softmax backward, then the scale node's backward, in place in dP */
#pragma omp parallel for schedule(static) if (S >= 64)
        for (long i = 0; i < S; ++i) {
            const double *prow = P + i * S;
            double *drow = dP + i * S;
            double dot = 0.0;
            for (long j = 0; j < S; ++j) dot += drow[j] * prow[j];
            if (pdp_rowsum) pdp_rowsum[i] = dot;
            double dsum = 0.0;
            for (long j = 0; j < S; ++j) {
                drow[j] = scale * (prow[j] * (drow[j] - dot));
                dsum += drow[j];
            }
            if (ds_rowsum) ds_rowsum[i] = dsum;
        }
        matmul_nn(dP, k, S, hd, dq);     /* dQ = dS K   */
        matmul_tn(dP, q, S, hd, dk);     /* dK = dS^T Q */
        free(dP);
    }
    free(P);
    free(Pd);
    return ORACLE_OK;
}

/*
 * causal != 0 applies the mask j > i -> -inf; causal == 0 is plain dense
 * softmax attention (used only by a test that compares against a library
 * routine).  Returns 0, or nonzero on a bad argument / allocation failure.
 */
int xfa_oracle_head(const double *q, const double *k, const double *v, const double *dout,
                    long S, long hd, double scale, int causal,
                    double *out, double *lse, double *dq, double *dk, double *dv,
                    double *p_rowsum, double *pdp_rowsum, double *ds_rowsum)
{
    return head_impl(q, k, v, dout, S, hd, scale, causal, NULL, out, lse, dq, dk, dv, p_rowsum, pdp_rowsum,
                     ds_rowsum);
}

/*
 * The same head with dropout of rate p (0 <= p < 1) on the attention
 * probabilities; element (i, j) of this head has flat index index_base + i*S + j
 * (index_base = b*S*S for head b of a [bh, S, S] probability tensor).
 */
int xfa_oracle_head_dropout(const double *q, const double *k, const double *v, const double *dout,
                            long S, long hd, double scale, int causal, float p, uint64_t seed,
                            uint64_t index_base, double *out, double *lse, double *dq, double *dk,
                            double *dv, double *p_rowsum, double *pdp_rowsum, double *ds_rowsum)
{
    if (!(p >= 0.0f && p < 1.0f) || S < 1) return ORACLE_BAD_ARG;
    double *C = (double *)malloc(sizeof(double) * (size_t)S * (size_t)S);
    if (!C) return ORACLE_NO_MEMORY;
    const double inv_keep = 1.0 / (1.0 - (double)p);
    for (long i = 0; i < S; ++i)
        for (long j = 0; j < S; ++j)
            C[i * S + j] = xfa_oracle_keep(seed, index_base + (uint64_t)(i * S + j), p) ? inv_keep : 0.0;
    const int rc = head_impl(q, k, v, dout, S, hd, scale, causal, C, out, lse, dq, dk, dv, p_rowsum, pdp_rowsum,
                             ds_rowsum);
    free(C);
    return rc;
}

/* number of OpenMP threads the oracle runs with (1 when built without OpenMP) */
int xfa_oracle_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
