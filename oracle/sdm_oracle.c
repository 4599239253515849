/*
 * sdm_oracle.c -- plain CPU oracle for one Sparse Delta Memory (SDM) layer forward.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or call this file. It shares no code with the CUDA path.
 *
 * All arithmetic is fp64. Values are rounded only where the method stores them:
 * projections (q, v) and bank columns, to the storage type (fp32, bf16 RNE, or fp64
 * for the closed-form pins). The steps follow the pages' order:
 *   "Sparse Delta Memory" blog, "How does SDM work?": select slots via product keys,
 *   write with a gated delta rule, read from (possibly different) slots;
 *   "Write & Read": two sub-keys -> outer sum -> top-k; selected columns are first
 *   decayed, then written with the delta rule; the output is a weighted sum of the
 *   retrieved columns (softmax-weighted).
 * Where the pages are silent the frozen readings apply: contiguous query halves,
 * shared sub-key tables, slot id i*n+j, ties by smaller slot id, temperature-1
 * softmax over the kept scores, only selected columns decay.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

/* ---------------------------------------------------------------- storage */

/* bf16 bits -> exact double */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> bf16 bits, round to nearest, ties to even, in one rounding step.
 * bf16 keeps 8 significant bits and fp32's exponent range (normals down to
 * 2^-126, subnormals spaced 2^-133). */
uint16_t orc_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    double ax = fabs(x);
    double r;
    if (ax == 0.0 || isinf(x)) {
        r = x;
    } else if (ax < ldexp(1.0, -126)) {
        r = nearbyint(x * ldexp(1.0, 133)) * ldexp(1.0, -133);
    } else {
        int e;
        double m = frexp(x, &e);               /* x = m * 2^e, 0.5 <= |m| < 1 */
        r = ldexp(nearbyint(ldexp(m, 8)), e - 8);
        if (fabs(r) >= ldexp(1.0, 128))
            r = copysign(INFINITY, x);
    }
    float f = (float)r;                         /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double load(const void* p, int type, size_t i)
{
    switch (type) {
    case ORC_F32: return (double)((const float*)p)[i];
    case ORC_BF16: return bf16_to_double(((const uint16_t*)p)[i]);
    default: return ((const double*)p)[i];
    }
}

static void store(void* p, int type, size_t i, double x)
{
    switch (type) {
    case ORC_F32: ((float*)p)[i] = (float)x; break;   /* C rounds to nearest even */
    case ORC_BF16: ((uint16_t*)p)[i] = orc_bf16_from_double(x); break;
    default: ((double*)p)[i] = x; break;
    }
}

/* round an array of doubles to a storage type (used by tests and wrappers) */
void orc_round_store(const double* in, int64_t count, int type, void* out)
{
    for (int64_t i = 0; i < count; ++i)
        store(out, type, (size_t)i, in[i]);
}

/* --------------------------------------------------------- step P: projections */

/* out[r, c] = stored( sum_k x[r, k] * Wm[k, c] ), x [rows, din], Wm [din, dout].
 * Sum in fp64 with k ascending; rounded once to `type`. */
void orc_project(const void* x, const void* Wm, int type, int64_t rows, int din, int dout,
                 void* out)
{
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)dout);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            for (int c = 0; c < dout; ++c)
                acc[c] = 0.0;
            for (int k = 0; k < din; ++k) {
                double xk = load(x, type, (size_t)r * din + k);
                for (int c = 0; c < dout; ++c)
                    acc[c] += xk * load(Wm, type, (size_t)k * dout + c);
            }
            for (int c = 0; c < dout; ++c)
                store(out, type, (size_t)r * dout + c, acc[c]);
        }
        free(acc);
    }
}

/* ------------------------------------------------------ step A: addressing */

/* Sub-key scores for one query q [dk]: s1[i] = <K1[i], q[0:h]>, s2[j] = <K2[j], q[h:dk]>,
 * h = dk/2, K1, K2 [n, h] row-major. */
void orc_subkey_scores(const void* q, int type, int dk, const void* K1, const void* K2, int n,
                       double* s1, double* s2)
{
    int h = dk / 2;
    for (int i = 0; i < n; ++i) {
        double a = 0.0, b = 0.0;
        for (int c = 0; c < h; ++c) {
            a += load(K1, type, (size_t)i * h + c) * load(q, type, (size_t)c);
            b += load(K2, type, (size_t)i * h + c) * load(q, type, (size_t)(h + c));
        }
        s1[i] = a;
        s2[i] = b;
    }
}

/* a precedes b in the selection order: larger score first, then smaller slot id */
static int precedes(double sa, int32_t ia, double sb, int32_t ib)
{
    return sa > sb || (sa == sb && ia < ib);
}

/* Top-W of the outer sum c[i*n+j] = s1[i] + s2[j] over all n*n slots, by exhaustive
 * scan. Outputs the W slot ids in selection order, their scores, and the gap
 * between the W-th and (W+1)-th score (+inf when n*n == W). */
void orc_topw(const double* s1, const double* s2, int n, int W, int32_t* slot, double* score,
              double* gap)
{
    int keep = W + 1;                 /* keep one extra to measure the boundary gap */
    double* bs = (double*)malloc(sizeof(double) * (size_t)keep);
    int32_t* bi = (int32_t*)malloc(sizeof(int32_t) * (size_t)keep);
    int have = 0;
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < n; ++j) {
            double c = s1[i] + s2[j];
            int32_t id = (int32_t)i * n + j;
            if (have == keep && !precedes(c, id, bs[keep - 1], bi[keep - 1]))
                continue;
            int p = (have < keep) ? have++ : keep - 1;   /* drop the last if full */
            while (p > 0 && precedes(c, id, bs[p - 1], bi[p - 1])) {
                bs[p] = bs[p - 1];
                bi[p] = bi[p - 1];
                --p;
            }
            bs[p] = c;
            bi[p] = id;
        }
    }
    for (int w = 0; w < W; ++w) {
        slot[w] = bi[w];
        score[w] = bs[w];
    }
    *gap = (have > W) ? bs[W - 1] - bs[W] : INFINITY;
    free(bs);
    free(bi);
}

/* Softmax over the W kept scores, temperature 1, max-subtracted. */
void orc_softmax(const double* c, int W, double* w)
{
    double mx = c[0];
    for (int j = 1; j < W; ++j)
        if (c[j] > mx)
            mx = c[j];
    double sum = 0.0;
    for (int j = 0; j < W; ++j) {
        w[j] = exp(c[j] - mx);
        sum += w[j];
    }
    for (int j = 0; j < W; ++j)
        w[j] /= sum;
}

/* Addressing for nq queries q [nq, dk]: slots [nq, W] (selection order), weights
 * [nq, W], scores [nq, W], boundary gap [nq]. */
void orc_address(const void* q, int type, int64_t nq, int dk, const void* K1, const void* K2,
                 int n, int W, int32_t* slots, double* weights, double* scores, double* gaps)
{
#pragma omp parallel
    {
        double* s1 = (double*)malloc(sizeof(double) * (size_t)n);
        double* s2 = (double*)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < nq; ++t) {
            const char* qt = (const char*)q + (size_t)t * dk *
                             (type == ORC_F32 ? 4 : type == ORC_BF16 ? 2 : 8);
            orc_subkey_scores(qt, type, dk, K1, K2, n, s1, s2);
            orc_topw(s1, s2, n, W, slots + t * W, scores + t * W, gaps + t);
            orc_softmax(scores + t * W, W, weights + t * W);
        }
        free(s1);
        free(s2);
    }
}

/* ------------------------------------------- steps W and R: the recurrence */

/* Recurrence of one sequence over T tokens on a subset of R rows of the bank.
 *   M     [N, R]  the selected rows of every slot vector (storage `type`), in place
 *   v     [T, R]  value rows (storage `vtype`), alpha/beta [T]
 *   S, k  [T, W]  write slots and weights;  Rd, r [T, W] read slots and weights
 *   y     [T, R]  output rows (fp64)
 * Per token: decay the selected columns, M' = alpha * M_S; delta rule
 * M_S <- M' + beta * (v - M' k) k^T; store (round) each written column once; then
 * read y = sum_j r_j M[:, Rd_j] from the stored post-write bank.
 * Returns 0, or -1 if a slot id is out of range or repeated within a set. */
int orc_scan(int type, int vtype, int64_t N, int R, int64_t T, int W, void* M, const void* v,
             const double* alpha, const double* beta, const int32_t* S, const double* k,
             const int32_t* Rd, const double* r, double* y)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < W; ++j) {
            int32_t a = S[t * W + j], b = Rd[t * W + j];
            if (a < 0 || a >= N || b < 0 || b >= N)
                return -1;
            for (int l = 0; l < j; ++l)
                if (S[t * W + l] == a || Rd[t * W + l] == b)
                    return -1;
        }
    }
#pragma omp parallel
    {
        double* Mp = (double*)malloc(sizeof(double) * (size_t)W);   /* M' row, per slot */
#pragma omp for schedule(static)
        for (int row = 0; row < R; ++row) {
            for (int64_t t = 0; t < T; ++t) {
                const int32_t* St = S + t * W;
                const double* kt = k + t * W;
                double at = alpha[t], bt = beta[t];
                double vt = load(v, vtype, (size_t)t * R + row);
                /* decay: M' = alpha * M_S ; u' = M' k */
                double up = 0.0;
                for (int j = 0; j < W; ++j) {
                    Mp[j] = at * load(M, type, (size_t)St[j] * R + row);
                    up += Mp[j] * kt[j];
                }
                /* delta rule: M_S <- M' + beta (v - M' k) k^T, stored once */
                for (int j = 0; j < W; ++j)
                    store(M, type, (size_t)St[j] * R + row, Mp[j] + bt * (vt - up) * kt[j]);
                /* read from the post-write bank */
                double acc = 0.0;
                for (int j = 0; j < W; ++j)
                    acc += r[t * W + j] * load(M, type, (size_t)Rd[t * W + j] * R + row);
                y[(size_t)t * R + row] = acc;
            }
        }
        free(Mp);
    }
    return 0;
}

/* Bank initialisation from the learned initial state: banks[b] = M0 for b < B. */
void orc_init_bank(const void* M0, int64_t bytes_per_bank, int B, void* banks)
{
    for (int b = 0; b < B; ++b)
        memcpy((char*)banks + (size_t)b * bytes_per_bank, M0, (size_t)bytes_per_bank);
}
