/*
 * caat_oracle.c -- plain CPU oracle for the partial channel-reduce (PCR) and the
 * row-parallel linear layer of CAAT-Net.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant table with the CUDA path.
 *
 * Source: "Tensor-Parallelism with Partially Synchronized Activations"
 * (Lamprecht, Karnieli, Hanani, Giladi, Soudry; NeurIPS 2025), Introduction,
 * paragraph introducing the partial channel-reduce operation: only a subset S of
 * the hidden-dimension channels is summed across the t tensor-parallel devices;
 * outside S every device keeps its own partial activation.  With S empty the model
 * is an ensemble, with S = all channels it is a vanilla transformer.  The same
 * paragraph requires forward and backward to agree.  The equations and figures of
 * the paper did not survive on the pages, so the arithmetic below is the plainest
 * reading of that prose:
 *
 *   Y_r      = X_r . W_r                (shard r of the K dimension, r = 0..t-1)
 *   Out_r[c] = sum_q Y_q[c]   if c in S (left fold q = 0..t-1)
 *   Out_r[c] = Y_r[c]         otherwise
 *
 * Everything is written as naive loops; floating-point GEMM work accumulates in
 * double.  OpenMP only splits independent output rows across threads.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- threads */

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------ splitmix64 */
/*
 * SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; the 64-bit mixer with Stafford's variant-13
 * constants, as in Java's SplittableRandom).  The state advances by the golden
 * gamma; the output is the mixed state.
 */
static uint64_t sm64_next(uint64_t *state)
{
    uint64_t z;
    *state += 0x9e3779b97f4a7c15ULL;
    z = *state;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

void orc_splitmix64(uint64_t seed, int64_t n, uint64_t *out)
{
    uint64_t st = seed;
    for (int64_t i = 0; i < n; ++i) out[i] = sm64_next(&st);
}

/* ------------------------------------------------------ channel selection */

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * The synchronized set S.  Its size is the fraction p of the h hidden channels
 * (the paper's "partial channel reduce hyperparameter p", p = 0.5 in the 7B run);
 * s = floor(p*h + 1/2), clamped to [0, h].  Which channels are chosen is not
 * stated: layout 0 takes the first s channels, layout 1 takes the first s entries
 * of a Fisher-Yates shuffle of 0..h-1 driven by splitmix64(seed) (i from h-1 down
 * to 1, j = next mod (i+1)), returned sorted.
 * Returns 0 on success, 1 on an invalid argument.
 */
int orc_select_channels(int64_t h, double p, int layout, uint64_t seed,
                        int32_t *idx, int64_t *n_sel)
{
    int64_t s;
    if (h < 0 || !(p >= 0.0 && p <= 1.0) || (layout != 0 && layout != 1) || !idx || !n_sel)
        return 1;
    s = (int64_t)floor(p * (double)h + 0.5);
    if (s < 0) s = 0;
    if (s > h) s = h;
    if (layout == 0) {
        for (int64_t i = 0; i < s; ++i) idx[i] = (int32_t)i;
    } else {
        int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)(h > 0 ? h : 1));
        uint64_t st = seed;
        if (!perm) return 1;
        for (int64_t i = 0; i < h; ++i) perm[i] = (int32_t)i;
        for (int64_t i = h - 1; i >= 1; --i) {
            uint64_t j = sm64_next(&st) % (uint64_t)(i + 1);
            int32_t tmp = perm[i];
            perm[i] = perm[j];
            perm[j] = tmp;
        }
        for (int64_t i = 0; i < s; ++i) idx[i] = perm[i];
        free(perm);
        qsort(idx, (size_t)s, sizeof(int32_t), cmp_i32);
    }
    *n_sel = s;
    return 0;
}

/* Membership of every channel in S, as a 0/1 byte per channel. */
static unsigned char *make_mask(int64_t h, const int32_t *sel, int64_t n_sel)
{
    unsigned char *m = (unsigned char *)calloc((size_t)(h > 0 ? h : 1), 1);
    if (!m) return NULL;
    for (int64_t i = 0; i < n_sel; ++i)
        if (sel[i] >= 0 && sel[i] < h) m[sel[i]] = 1;
    return m;
}

/* ------------------------------------------------------------- bf16 words */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void orc_f32_to_bf16(int64_t n, const float *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}

/* ------------------------------------------------- partial channel-reduce */
/*
 * Y and Out are [t][N][h], dense.  Channels in S get the sum over the t ranks,
 * folded left in rank order; the rest copy the rank's own value.
 * Returns the number of reduced elements (N * |S|), the "communicated" payload.
 */
int64_t orc_pcr_f32(int t, int64_t N, int64_t h, const float *Y,
                    const int32_t *sel, int64_t n_sel, float *Out)
{
    unsigned char *inS = make_mask(h, sel, n_sel);
    int64_t reduced = 0;
    if (!inS) return -1;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < h; ++c) {
            if (inS[c]) {
                float acc = Y[(0 * N + n) * h + c];
                for (int q = 1; q < t; ++q) acc = acc + Y[((int64_t)q * N + n) * h + c];
                for (int r = 0; r < t; ++r) Out[((int64_t)r * N + n) * h + c] = acc;
                reduced += 1;
            } else {
                for (int r = 0; r < t; ++r)
                    Out[((int64_t)r * N + n) * h + c] = Y[((int64_t)r * N + n) * h + c];
            }
        }
    }
    free(inS);
    return reduced;
}

/* bf16 storage: widen exactly, fold in fp32 as above, round once to bf16. */
int64_t orc_pcr_bf16(int t, int64_t N, int64_t h, const uint16_t *Y,
                     const int32_t *sel, int64_t n_sel, uint16_t *Out)
{
    unsigned char *inS = make_mask(h, sel, n_sel);
    int64_t reduced = 0;
    if (!inS) return -1;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < h; ++c) {
            if (inS[c]) {
                float acc = bf16_to_f32(Y[(0 * N + n) * h + c]);
                uint16_t o;
                for (int q = 1; q < t; ++q) acc = acc + bf16_to_f32(Y[((int64_t)q * N + n) * h + c]);
                o = f32_to_bf16(acc);
                for (int r = 0; r < t; ++r) Out[((int64_t)r * N + n) * h + c] = o;
                reduced += 1;
            } else {
                for (int r = 0; r < t; ++r)
                    Out[((int64_t)r * N + n) * h + c] = Y[((int64_t)r * N + n) * h + c];
            }
        }
    }
    free(inS);
    return reduced;
}

/* The same operator in double, used inside the layer oracles below. */
int64_t orc_pcr_f64(int t, int64_t N, int64_t h, const double *Y,
                    const int32_t *sel, int64_t n_sel, double *Out)
{
    unsigned char *inS = make_mask(h, sel, n_sel);
    int64_t reduced = 0;
    if (!inS) return -1;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < h; ++c) {
            if (inS[c]) {
                double acc = Y[(0 * N + n) * h + c];
                for (int q = 1; q < t; ++q) acc = acc + Y[((int64_t)q * N + n) * h + c];
                for (int r = 0; r < t; ++r) Out[((int64_t)r * N + n) * h + c] = acc;
                reduced += 1;
            } else {
                for (int r = 0; r < t; ++r)
                    Out[((int64_t)r * N + n) * h + c] = Y[((int64_t)r * N + n) * h + c];
            }
        }
    }
    free(inS);
    return reduced;
}

/* ------------------------------------------------ row-parallel linear fwd */
/*
 * X is [N][K], W is [K][h] (both dense, row-major, double).  K splits into t
 * equal shards; rank r owns X[:, r*K/t .. (r+1)*K/t) and the matching rows of W
 * (Megatron's row-parallel layer: attention out-projection, MLP down-projection).
 * Y_r = X_r W_r is the rank's partial sum; Out = PCR(Y) with the set S.
 * Out is [t][N][h].  *macs (optional) receives the multiply-adds done.
 * Returns 0, or 1 when K is not divisible by t or memory runs out.
 */
int orc_rowpar_fwd(int t, int64_t N, int64_t K, int64_t h,
                   const double *X, const double *W,
                   const int32_t *sel, int64_t n_sel,
                   double *Out, int64_t *macs)
{
    int64_t kt;
    double *Y;
    if (t < 1 || K % t != 0) return 1;
    kt = K / t;
    Y = (double *)malloc(sizeof(double) * (size_t)((int64_t)t * N * h > 0 ? (int64_t)t * N * h : 1));
    if (!Y) return 1;
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int r = 0; r < t; ++r) {
            double *yrow = Y + ((int64_t)r * N + n) * h;
            for (int64_t c = 0; c < h; ++c) {
                double acc = 0.0;
                for (int64_t k = (int64_t)r * kt; k < (int64_t)(r + 1) * kt; ++k)
                    acc += X[n * K + k] * W[k * h + c];
                yrow[c] = acc;
            }
        }
    }
    if (macs) *macs = N * K * h;
    orc_pcr_f64(t, N, h, Y, sel, n_sel, Out);
    free(Y);
    return 0;
}

/* ----------------------------------------------- row-parallel linear bwd */
/*
 * G is [t][N][h]: the upstream gradient of each rank's output Out_r.
 * mode 0: the gradient is first passed through the same PCR (the operator is
 *         symmetric, so this is the exact gradient of sum_r <G_r, Out_r>);
 * mode 1: each rank uses its own G_r (the reduce is left to the matching
 *         column-parallel layer).
 * dY_r is that per-rank gradient.  dX[:, shard r] = dY_r W_r^T, [N][K];
 * dW[shard r, :] = X_r^T dY_r, [K][h].  Returns 0, or 1 on a bad argument.
 */
int orc_rowpar_bwd(int t, int64_t N, int64_t K, int64_t h,
                   const double *X, const double *W, const double *G,
                   const int32_t *sel, int64_t n_sel, int mode,
                   double *dX, double *dW)
{
    int64_t kt;
    double *dY;
    if (t < 1 || K % t != 0 || (mode != 0 && mode != 1)) return 1;
    kt = K / t;
    dY = (double *)malloc(sizeof(double) * (size_t)((int64_t)t * N * h > 0 ? (int64_t)t * N * h : 1));
    if (!dY) return 1;
    if (mode == 0)
        orc_pcr_f64(t, N, h, G, sel, n_sel, dY);
    else
        memcpy(dY, G, sizeof(double) * (size_t)((int64_t)t * N * h));

    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int r = 0; r < t; ++r) {
            const double *g = dY + ((int64_t)r * N + n) * h;
            for (int64_t k = (int64_t)r * kt; k < (int64_t)(r + 1) * kt; ++k) {
                double acc = 0.0;
                for (int64_t c = 0; c < h; ++c) acc += g[c] * W[k * h + c];
                dX[n * K + k] = acc;
            }
        }
    }

    #pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k) {
        int r = (int)(k / kt);
        for (int64_t c = 0; c < h; ++c) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n)
                acc += X[n * K + k] * dY[((int64_t)r * N + n) * h + c];
            dW[k * h + c] = acc;
        }
    }
    free(dY);
    return 0;
}

/* -------------------------------------------- column-parallel linear layer */
/*
 * The partner of the row-parallel layer inside a transformer block (attention
 * QKV, MLP up-projection).  Rank r multiplies its own input A_r [N][h] (A is
 * [t][N][h]: under partial synchronization the ranks' activations differ) by its
 * column block W1_r = W1[:, r*K/t .. (r+1)*K/t) of W1 [h][K] (row-major, double).
 * Z [N][K] holds rank r's output in column block r.  The forward has no reduce.
 * Returns 0, or 1 when K is not divisible by t.
 */
int orc_colpar_fwd(int t, int64_t N, int64_t h, int64_t K,
                   const double *A, const double *W1, double *Z)
{
    int64_t kt;
    if (t < 1 || K % t != 0) return 1;
    kt = K / t;
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            const int r = (int)(k / kt);
            const double *a = A + ((int64_t)r * N + n) * h;
            double acc = 0.0;
            for (int64_t c = 0; c < h; ++c) acc += a[c] * W1[c * K + k];
            Z[n * K + k] = acc;
        }
    }
    return 0;
}

/*
 * Backward of the column-parallel layer with the partial reduce placed on its
 * input gradient (Megatron's placement; the row-parallel backward then passes
 * each rank's gradient through unreduced).  Reading: the input channels in S are
 * one activation shared by the ranks, so their gradient is the sum of the ranks'
 * contributions; outside S each rank's input is its own.
 *   P_r            = dZ_r W1_r^T     [N][h]  (dZ_r = column block r of dZ [N][K])
 *   dA             = PCR(P) with S   [t][N][h]
 *   dW1[:, block r] = A_r^T dZ_r     [h][K]
 * Returns 0, or 1 on a bad argument.
 */
int orc_colpar_bwd(int t, int64_t N, int64_t h, int64_t K,
                   const double *A, const double *W1, const double *dZ,
                   const int32_t *sel, int64_t n_sel, double *dA, double *dW1)
{
    int64_t kt;
    double *P;
    if (t < 1 || K % t != 0) return 1;
    kt = K / t;
    P = (double *)malloc(sizeof(double) * (size_t)((int64_t)t * N * h > 0 ? (int64_t)t * N * h : 1));
    if (!P) return 1;
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int r = 0; r < t; ++r) {
            double *prow = P + ((int64_t)r * N + n) * h;
            for (int64_t c = 0; c < h; ++c) {
                double acc = 0.0;
                for (int64_t k = (int64_t)r * kt; k < (int64_t)(r + 1) * kt; ++k)
                    acc += dZ[n * K + k] * W1[c * K + k];
                prow[c] = acc;
            }
        }
    }
    orc_pcr_f64(t, N, h, P, sel, n_sel, dA);
    free(P);

    #pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < h; ++c) {
        for (int64_t k = 0; k < K; ++k) {
            const int r = (int)(k / kt);
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n)
                acc += A[((int64_t)r * N + n) * h + c] * dZ[n * K + k];
            dW1[c * K + k] = acc;
        }
    }
    return 0;
}
