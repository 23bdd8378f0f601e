/*
 * CPU oracle for the predictor-guided sparse FFN (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the slow, obviously-correct definition that the CUDA library is
 * checked against.  Only the test suite, the package smoke check and the CPU
 * baseline leg of the benchmark may load it; the product path never does.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Precision: every sum is accumulated in IEEE double, in ascending index order,
 * with no blocking, no reordering and no BLAS.  Weights are widened element by
 * element from their storage type (fp32, IEEE binary16, or Q4_0 blocks).  The
 * one place where floating point decides an integer code -- the Q4_0 quantiser
 * -- takes that decision in binary32, the precision the CUDA quantiser uses.
 *
 * Sources (the method is described in prose only; there is no listing):
 *  - PowerInfer summary page (gptget.net, arXiv 2312.12456), sections
 *    "核心创新" (core innovation) and "方法详解" (method detail): an online
 *    predictor marks the neurons expected to fire, and neuron-aware sparse
 *    operators compute only those neurons; offline profiling finds the hot
 *    neurons.  "关键结果" (key results): ~26% of neurons carry 80% of firings.
 *  - PowerInfer README translation (gittoolsai.com), "常见问题解答" (FAQ) item 2:
 *    supported activations are ReLU, ReGLU and squared ReLU.
 *  - Same README, "量化" (quantization): INT4 weights in the Q4_0 format; a
 *    Q4_0 block is 32 weights sharing one fp16 scale.
 *  Where the pages leave a step open, the reading taken is stated at the
 *  function that implements it.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_F16 1
#define OR_Q4_0 2

#define OR_ACT_RELU 0
#define OR_ACT_RELU2 1

/* One FFN layer plus its predictor, host pointers.  All FFN matrices are
 * neuron-major: row j of w_up / w_gate / w_down belongs to neuron j and holds
 * d_model values.  p1 is [rank][d_model], p2 is [d_ff][rank]. */
typedef struct {
    int64_t d_model, d_ff, rank;
    int32_t gated;      /* 0: fc1 -> act -> fc2.  1: act(gate) * up -> down */
    int32_t act;        /* OR_ACT_RELU or OR_ACT_RELU2 (squared ReLU) */
    int32_t wtype;      /* storage of w_up / w_gate / w_down */
    int32_t ptype;      /* storage of p1 / p2 (OR_F32 or OR_F16) */
    const void *w_up, *w_gate, *w_down;
    const float *b_act;   /* [d_ff] bias of the projection that feeds act(), or NULL */
    const float *b_down;  /* [d_model] or NULL */
    const void *p1, *p2;
    const float *p_bias;  /* [d_ff] or NULL */
    double threshold;
    int64_t dense_prefix; /* neurons [0, dense_prefix) are always active */
} oracle_layer;

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16 -> double, from the format's definition:
 *   sign s (1 bit), exponent e (5 bits, bias 15), fraction f (10 bits)
 *   e == 0       : (-1)^s * 2^-14 * (f / 1024)        (zero / subnormal)
 *   0 < e < 31   : (-1)^s * 2^(e-15) * (1 + f / 1024)
 *   e == 31      : infinity (f == 0) or NaN                                   */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f / 1024.0, -14);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return s ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even, by exhaustive
 * reasoning on the definition: find the two binary16 neighbours of |f| and
 * pick the nearer (the even one on a tie).  Slow and plain on purpose. */
uint16_t oracle_f32_to_f16(float f)
{
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f)) return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00); /* rounds to infinity */
    /* binary16 magnitudes are monotone in their bit pattern 0..0x7bff */
    int lo = 0, hi = 0x7bff;
    while (lo < hi) { /* largest pattern whose value <= a */
        int mid = (lo + hi + 1) / 2;
        if (oracle_f16_to_f64((uint16_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    uint16_t below = (uint16_t)lo;
    double vb = oracle_f16_to_f64(below);
    if (vb == a || below == 0x7bff) return (uint16_t)(sign | below);
    uint16_t above = (uint16_t)(below + 1);
    double va = oracle_f16_to_f64(above);
    double db = a - vb, da = va - a;
    uint16_t pick;
    if (db < da) pick = below;
    else if (da < db) pick = above;
    else pick = (below & 1) ? above : below;
    return (uint16_t)(sign | pick);
}

static double g_f16_table[65536];
static int g_table_ready = 0;

static void ensure_table(void)
{
    if (g_table_ready) return;
    for (int i = 0; i < 65536; ++i) g_f16_table[i] = oracle_f16_to_f64((uint16_t)i);
    g_table_ready = 1;
}

/* ------------------------------------------------------------------------- */
/* Q4_0 storage, split form.  A matrix of `rows` x `cols` (cols % 32 == 0) is
 * cut into blocks of 32 consecutive weights along each row.  Block b of row j
 * stores 16 code bytes and one binary16 scale s.  Element e of a block
 * (0 <= e < 32) has code q = low nibble of byte e for e < 16 and high nibble of
 * byte e-16 for e >= 16; its value is s * (q - 8).  All code bytes come first
 * ([rows][cols/2] bytes, row-major), then all scales ([rows][cols/32] binary16).
 * The pages fix only "32 weights, one fp16 scale"; this arrangement is the
 * reading taken. */
static double q4_0_value(const uint8_t *base, int64_t rows, int64_t cols, int64_t j, int64_t i)
{
    const uint8_t *codes = base;
    const uint16_t *scales = (const uint16_t *)(base + rows * (cols / 2));
    int64_t b = i / 32, e = i % 32;
    uint8_t byte = codes[j * (cols / 2) + b * 16 + (e % 16)];
    int q = (e < 16) ? (byte & 15) : (byte >> 4);
    return g_f16_table[scales[j * (cols / 32) + b]] * (double)(q - 8);
}

/* The quantiser: per block, a = the weight of largest magnitude (first one on
 * ties), scale s = fp16(a / -8), then q = clamp(floor(w / s + 8.5), 0, 15),
 * all in binary32; an all-zero block stores scale +0 and q = 8 everywhere.  The extreme weight
 * maps to q = 0, i.e. exactly a after rounding of s. */
void oracle_q4_0_quantize(const float *src, int64_t rows, int64_t cols, uint8_t *dst)
{
    ensure_table();
    uint8_t *codes = dst;
    uint16_t *scales = (uint16_t *)(dst + rows * (cols / 2));
    for (int64_t j = 0; j < rows; ++j) {
        for (int64_t b = 0; b < cols / 32; ++b) {
            const float *w = src + j * cols + b * 32;
            float amax = w[0];
            for (int e = 1; e < 32; ++e)
                if (fabsf(w[e]) > fabsf(amax)) amax = w[e];
            float s32 = amax / -8.0f;
            uint16_t s16 = s32 == 0.0f ? (uint16_t)0 : oracle_f32_to_f16(s32); /* +0 for an all-zero block */
            float s = (float)g_f16_table[s16];
            uint8_t q[32];
            for (int e = 0; e < 32; ++e) {
                int qi;
                if (s == 0.0f) {
                    qi = 8;
                } else {
                    float t = w[e] / s;
                    t = t + 8.5f;
                    float fl = floorf(t);
                    qi = fl < 0.0f ? 0 : (fl > 15.0f ? 15 : (int)fl);
                }
                q[e] = (uint8_t)qi;
            }
            uint8_t *cb = codes + j * (cols / 2) + b * 16;
            for (int e = 0; e < 16; ++e) cb[e] = (uint8_t)(q[e] | (q[e + 16] << 4));
            scales[j * (cols / 32) + b] = s16;
        }
    }
}

/* Widen element (j, i) of a [rows][cols] matrix stored as `type`. */
static double elem(const void *m, int type, int64_t rows, int64_t cols, int64_t j, int64_t i)
{
    switch (type) {
    case OR_F32: return (double)((const float *)m)[j * cols + i];
    case OR_F16: return g_f16_table[((const uint16_t *)m)[j * cols + i]];
    default: return q4_0_value((const uint8_t *)m, rows, cols, j, i);
    }
}

void oracle_dequantize(const void *m, int32_t type, int64_t rows, int64_t cols, double *out)
{
    ensure_table();
    for (int64_t j = 0; j < rows; ++j)
        for (int64_t i = 0; i < cols; ++i) out[j * cols + i] = elem(m, type, rows, cols, j, i);
}

static double act(int kind, double z)
{
    double r = z > 0.0 ? z : 0.0;
    return kind == OR_ACT_RELU2 ? r * r : r;
}

/* Pre-activation of the projection that feeds act() for neuron j:
 *   fc1 (non-gated) or gate (gated), plus b_act[j].  Ascending i. */
static double pre_act(const oracle_layer *L, const float *x, int64_t j)
{
    const void *w = L->gated ? L->w_gate : L->w_up;
    double s = 0.0;
    for (int64_t i = 0; i < L->d_model; ++i)
        s += elem(w, L->wtype, L->d_ff, L->d_model, j, i) * (double)x[i];
    if (L->b_act) s += (double)L->b_act[j];
    return s;
}

/* Activation of neuron j: act(z_j) non-gated, act(g_j) * u_j gated (ReGLU). */
static double neuron(const oracle_layer *L, const float *x, int64_t j, double *z_out)
{
    double z = pre_act(L, x, j);
    if (z_out) *z_out = z;
    double a = act(L->act, z);
    if (L->gated) {
        double u = 0.0;
        for (int64_t i = 0; i < L->d_model; ++i)
            u += elem(L->w_up, L->wtype, L->d_ff, L->d_model, j, i) * (double)x[i];
        a = a * u;
    }
    return a;
}

/* Sparse FFN over an explicit neuron list (ascending), one token:
 *   y_i = sum_{k} a_{idx_k} * W_down[idx_k, i]   (k ascending)  + b_down_i.
 * The dense FFN is this with idx = 0..d_ff-1.  a_out (optional) receives the
 * activation of each listed neuron, z_out (optional) its pre-activation. */
int oracle_sparse_ffn(const oracle_layer *L, const float *x, const int32_t *idx, int64_t n_idx,
                      double *y, double *a_out, double *z_out)
{
    ensure_table();
    for (int64_t k = 0; k < n_idx; ++k)
        if (idx[k] < 0 || idx[k] >= L->d_ff) return -1;
    for (int64_t i = 0; i < L->d_model; ++i) y[i] = 0.0;
    for (int64_t k = 0; k < n_idx; ++k) {
        int64_t j = idx[k];
        double z;
        double a = neuron(L, x, j, &z);
        if (a_out) a_out[k] = a;
        if (z_out) z_out[k] = z;
        for (int64_t i = 0; i < L->d_model; ++i)
            y[i] += a * elem(L->w_down, L->wtype, L->d_ff, L->d_model, j, i);
    }
    if (L->b_down)
        for (int64_t i = 0; i < L->d_model; ++i) y[i] += (double)L->b_down[i];
    return 0;
}

int oracle_dense_ffn(const oracle_layer *L, const float *x, double *y, double *a_out, double *z_out)
{
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)L->d_ff);
    if (!all) return -2;
    for (int64_t j = 0; j < L->d_ff; ++j) all[j] = (int32_t)j;
    int rc = oracle_sparse_ffn(L, x, all, L->d_ff, y, a_out, z_out);
    free(all);
    return rc;
}

/* True activity: T = { j : pre-activation of the activated projection > 0 }
 * (strict, so z = 0 is inactive; for ReLU and squared ReLU this is exactly the
 * set of neurons whose activation can be non-zero). */
void oracle_true_mask(const oracle_layer *L, const float *x, uint8_t *mask, double *z_out)
{
    ensure_table();
    for (int64_t j = 0; j < L->d_ff; ++j) {
        double z = pre_act(L, x, j);
        if (z_out) z_out[j] = z;
        mask[j] = z > 0.0 ? 1 : 0;
    }
}

/* Low-rank activation predictor (the pages name an "adaptive predictor"
 * without giving its form; the reading taken is d -> r, ReLU, r -> d_ff):
 *   h_k     = max(sum_i P1[k,i] x_i, 0)
 *   logit_j = sum_k P2[j,k] h_k + p_bias_j
 *   mask_j  = logit_j > threshold
 * With an always-on prefix (the pages' split of a layer into hot neurons,
 * found offline and kept on the fast device, and cold ones -- summary page,
 * "方法详解" method detail; here the first dense_prefix neurons of the
 * hot-first order are computed every step): mask_j = 1 for j < dense_prefix,
 * whatever the logit.                                                        */
void oracle_predict(const oracle_layer *L, const float *x, double *h, double *logit, uint8_t *mask)
{
    ensure_table();
    for (int64_t k = 0; k < L->rank; ++k) {
        double s = 0.0;
        for (int64_t i = 0; i < L->d_model; ++i)
            s += elem(L->p1, L->ptype, L->rank, L->d_model, k, i) * (double)x[i];
        h[k] = s > 0.0 ? s : 0.0;
    }
    for (int64_t j = 0; j < L->d_ff; ++j) {
        double s = 0.0;
        for (int64_t k = 0; k < L->rank; ++k)
            s += elem(L->p2, L->ptype, L->d_ff, L->rank, j, k) * h[k];
        if (L->p_bias) s += (double)L->p_bias[j];
        logit[j] = s;
        if (mask) mask[j] = (j < L->dense_prefix || s > L->threshold) ? 1 : 0;
    }
}

/* Active-index compaction: the ascending positions of the non-zero entries of
 * mask; returns their count. */
int64_t oracle_compact(const uint8_t *mask, int64_t n, int32_t *idx)
{
    int64_t c = 0;
    for (int64_t j = 0; j < n; ++j)
        if (mask[j]) idx[c++] = (int32_t)j;
    return c;
}

/* Offline profiling: counts[j] += number of tokens whose pre-activation of the
 * activated projection is > 0.  X is [T][d_model]. */
void oracle_fire_counts(const oracle_layer *L, const float *X, int64_t T, int32_t *counts)
{
    ensure_table();
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < L->d_ff; ++j)
            if (pre_act(L, X + t * L->d_model, j) > 0.0) counts[j] += 1;
}

/* Hot-first order: perm[p] is the neuron placed at storage position p; neurons
 * sorted by firing count, highest first, ties kept in ascending neuron order.
 * Insertion sort: O(n^2) in the worst case, plain on purpose. */
void oracle_hot_first_perm(const int32_t *counts, int64_t n, int32_t *perm)
{
    for (int64_t p = 0; p < n; ++p) {
        int32_t j = (int32_t)p;
        int64_t q = p;
        while (q > 0 && counts[perm[q - 1]] < counts[j]) {
            perm[q] = perm[q - 1];
            --q;
        }
        perm[q] = j;
    }
}

/* Layer-to-layer glue of a stack of FFN layers: v = x + y (residual), then a
 * weightless RMS rescale  out_i = v_i / sqrt(mean_i v_i^2)  (out = 0 when v = 0). */
void oracle_rms_residual(const float *x, const double *y, int64_t d, double *out)
{
    double ss = 0.0;
    for (int64_t i = 0; i < d; ++i) {
        double v = (double)x[i] + y[i];
        ss += v * v;
    }
    double rms = sqrt(ss / (double)d);
    for (int64_t i = 0; i < d; ++i) {
        double v = (double)x[i] + y[i];
        out[i] = rms > 0.0 ? v / rms : 0.0;
    }
}
