/*
 * MXFP4 weight-streaming oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the decode-step
 * weight-streaming path computes. Only the tests, the package's smoke check
 * and the bench's CPU-baseline / reference leg may load it; the product path
 * never does. It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Sources (web pages, cited by title and section):
 *   [Z] "Zyphra Inference Wave 2: accelerating MoE and long-context serving
 *       on MI355X", section "Quantization": MXFP4 is the OCP MX format; each
 *       block of 32 values shares one 8-bit power-of-two scale; each value is
 *       a 4-bit float with magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; 4.25 bits
 *       per value. Same page, section "Kernel Results": the a16w4 fused MoE
 *       (bf16 activations, 4-bit weights) and top-k routed experts.
 *   [A] "megakernel-intro" (AMD ROCm blog), section "3. Low-Precision Data
 *       Types": a shared scale per 32, and decode reads every needed weight
 *       once per pass.
 * Rules the pages leave open (scale = floor(log2 amax) - 2, round to nearest
 * even with saturation, two codes per byte with the even index in the low
 * nibble, gate rows before up rows, softmax over the selected experts) follow
 * the OCP MX reading stated with the workload definitions.
 *
 * Arithmetic: float64 throughout. Every dequantized weight and every
 * product x*w is exact in float64 (8-bit x significand times a 2-bit weight
 * significand times a power of two), so a linear output is the exact dot
 * product up to float64 summation error. Summation runs in k order.
 *
 * Parity pins: every function here is pinned by the not-gpu tests against
 * library routines (CUDA's host-side cuda_fp4.h conversions, torch's E8M0
 * dtype, numpy matmul, Python's exact Fraction sums, scipy softmax/expit),
 * closed forms and brute force. None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* E2M1 magnitudes indexed by the low three bits of a code ([Z] Quantization). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Value of one 4-bit E2M1 code: bit 3 is the sign, bits 0..2 index the
 * magnitude table ([Z] Quantization). */
double oracle_e2m1_value(int code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Value of one E8M0 scale byte: 2^(s-127); the all-ones byte is NaN in the
 * OCP MX encoding and is never produced from finite input. */
double oracle_e8m0_value(int s) {
    if (s == 255) return NAN;
    return ldexp(1.0, s - 127);
}

/* Nearest E2M1 magnitude code for a >= 0. Ties go to the even code (the one
 * whose mantissa bit is 0: round to nearest even). Values above 6, the
 * largest finite magnitude, saturate to 6. */
int oracle_e2m1_round_magnitude(double a) {
    if (a > 6.0) return 7;
    int best = 0;
    double best_d = fabs(a - E2M1_MAG[0]);
    for (int c = 1; c < 8; c++) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Shared scale byte for one block: s = clamp(floor(log2 amax) - 2 + 127,
 * 0, 254), with floor(log2 amax) taken exactly from frexp (amax = m * 2^E,
 * m in [0.5, 1), so floor(log2 amax) = E - 1). An all-zero block gets s = 0. */
int oracle_block_scale(const float* blk) {
    double amax = 0.0;
    for (int i = 0; i < 32; i++) {
        double a = fabs((double)blk[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0) return 0;
    int E;
    (void)frexp(amax, &E);
    int s = (E - 1) - 2 + 127;
    if (s < 0) s = 0;
    if (s > 254) s = 254;
    return s;
}

/* Quantize W[n,k] (float32, row-major, k % 32 == 0) to MXFP4:
 * wq[n, k/2]: byte j of a row holds code(2j) in the low nibble and
 * code(2j+1) in the high nibble; ws[n, k/32]: one E8M0 byte per block.
 * Each value is divided by the block's power of two (exact in float64),
 * rounded to the nearest E2M1 point, and keeps its own sign bit. */
void oracle_quantize(const float* w, int64_t n, int64_t k, uint8_t* wq, uint8_t* ws) {
    const int64_t nb = k / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        for (int64_t b = 0; b < nb; b++) {
            const float* blk = w + r * k + b * 32;
            int s = oracle_block_scale(blk);
            ws[r * nb + b] = (uint8_t)s;
            double inv = ldexp(1.0, 127 - s);
            uint8_t* out = wq + r * (k / 2) + b * 16;
            for (int j = 0; j < 16; j++) {
                int code[2];
                for (int h = 0; h < 2; h++) {
                    float wi = blk[2 * j + h];
                    double v = (double)wi * inv;
                    int mag = oracle_e2m1_round_magnitude(fabs(v));
                    code[h] = (signbit(wi) ? 8 : 0) | mag;
                }
                out[j] = (uint8_t)(code[0] | (code[1] << 4));
            }
        }
    }
}

/* Decoded weight (row r, column c) of a packed matrix with row length k. */
static double dequant_at(const uint8_t* wq, const uint8_t* ws, int64_t k, int64_t r, int64_t c) {
    uint8_t byte = wq[r * (k / 2) + c / 2];
    int code = (c & 1) ? (byte >> 4) : (byte & 15);
    return oracle_e2m1_value(code) * oracle_e8m0_value(ws[r * (k / 32) + c / 32]);
}

/* out[n,k] = dequantized weights in float64. */
void oracle_dequant(const uint8_t* wq, const uint8_t* ws, int64_t n, int64_t k, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++)
        for (int64_t c = 0; c < k; c++) out[r * k + c] = dequant_at(wq, ws, k, r, c);
}

static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Linear layer on the decoded weights ([A] section 3: every weight is read
 * once per pass and applied to every token of the step):
 *   y[t][j] = sum_k x[t,k] * w[row_j, k],  rss[t][j] = sqrt(sum_k (x*w)^2)
 * for the selected rows row_j (rows == NULL selects 0..n-1, then nrows = n).
 * x is bf16 bits [t,k]; y and rss are float64 [t][nrows]. */
void oracle_linear(const uint16_t* x, int64_t t, int64_t k, const uint8_t* wq, const uint8_t* ws,
                   int64_t n, const int64_t* rows, int64_t nrows, double* y, double* rss) {
    (void)n;
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (size_t)k);
#pragma omp for schedule(dynamic, 16)
        for (int64_t j = 0; j < nrows; j++) {
            int64_t r = rows ? rows[j] : j;
            for (int64_t c = 0; c < k; c++) wrow[c] = dequant_at(wq, ws, k, r, c);
            for (int64_t ti = 0; ti < t; ti++) {
                double acc = 0.0, sq = 0.0;
                for (int64_t c = 0; c < k; c++) {
                    double p = bf16_to_double(x[ti * k + c]) * wrow[c];
                    acc += p;
                    sq += p * p;
                }
                y[ti * nrows + j] = acc;
                if (rss) rss[ti * nrows + j] = sqrt(sq);
            }
        }
        free(wrow);
    }
}

/* Router for one token ([Z] Kernel Results / Quantization: each token uses
 * its top-k routed experts): ids = the top_k largest logits in descending
 * order, ties to the smaller expert index; g = softmax over the selected
 * logits, in float64. */
static void route_one(const float* lg, int64_t e, int top_k, int32_t* ids, double* g) {
    for (int j = 0; j < top_k; j++) {
        int best = -1;
        for (int64_t c = 0; c < e; c++) {
            int taken = 0;
            for (int q = 0; q < j; q++)
                if (ids[q] == c) taken = 1;
            if (taken) continue;
            if (best < 0 || lg[c] > lg[best]) best = (int)c;
        }
        ids[j] = best;
    }
    double m = (double)lg[ids[0]];
    double z = 0.0;
    for (int j = 0; j < top_k; j++) {
        g[j] = exp((double)lg[ids[j]] - m);
        z += g[j];
    }
    for (int j = 0; j < top_k; j++) g[j] /= z;
}

void oracle_route(const float* logits, int64_t t, int64_t e, int top_k, int32_t* ids, double* g) {
#pragma omp parallel for schedule(static)
    for (int64_t ti = 0; ti < t; ti++) route_one(logits + ti * e, e, top_k, ids + ti * top_k, g + ti * top_k);
}

/* Grouped top-k MoE on decoded weights, in float64:
 *   for each token t and each selected expert e (weight g):
 *     a = W1_e[0:I] . x_t (gate rows), b = W1_e[I:2I] . x_t (up rows),
 *     h = SiLU(a) * b with SiLU(z) = z / (1 + exp(-z)),
 *     o = W2_e . h
 *   y[t] = sum over the selected experts, in selection order, of g * o.
 * Shared experts ([Z] Quantization: a token uses its top-k routed experts
 * plus the layer's shared experts, e.g. 8 routed and 1 shared of 257): the
 * tables hold n_shared more experts, e .. e + n_shared - 1, which every
 * token applies after its routed ones with weight g = 1 (the pages print no
 * weight for them; 1 is the plain reading of "uses").
 * rss[t][n] = sqrt(sum over (e, j) of (g * h_j * w2_e[n, j])^2).
 * Per-expert pointers (w1q[e], ...) may be NULL for experts no selected
 * token routes to. Tokens and output columns may be subsets (tok / cols
 * NULL selects all); y and rss are [ntok][ncols]. Returns 0, or -1 if a
 * needed expert is missing. */
int oracle_moe(const uint16_t* x, int64_t t, int64_t hidden, const float* logits, int64_t e, int top_k,
               int n_shared, const uint8_t* const* w1q, const uint8_t* const* w1s, const uint8_t* const* w2q,
               const uint8_t* const* w2s, int64_t inter, const int64_t* tok, int64_t ntok,
               const int64_t* cols, int64_t ncols, double* y, double* rss) {
    (void)t;
    int kp = top_k + n_shared; /* pairs per token */
    int64_t npair = ntok * kp;
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)npair);
    double* g = (double*)malloc(sizeof(double) * (size_t)npair);
    double* h = (double*)malloc(sizeof(double) * (size_t)(npair * inter));
    int missing = 0;
    for (int64_t i = 0; i < ntok; i++) {
        int64_t ti = tok ? tok[i] : i;
        route_one(logits + ti * e, e, top_k, ids + i * kp, g + i * kp);
        for (int s = 0; s < n_shared; s++) {
            ids[i * kp + top_k + s] = (int32_t)(e + s);
            g[i * kp + top_k + s] = 1.0;
        }
        for (int j = 0; j < kp; j++) {
            int ex = ids[i * kp + j];
            if (!w1q[ex] || !w1s[ex] || !w2q[ex] || !w2s[ex]) missing = 1;
        }
    }
    if (missing) {
        free(ids);
        free(g);
        free(h);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < npair; p++) {
        int64_t i = p / kp;
        int64_t ti = tok ? tok[i] : i;
        int ex = ids[p];
        const uint16_t* xt = x + ti * hidden;
        for (int64_t r = 0; r < inter; r++) {
            double a = 0.0, b = 0.0;
            for (int64_t c = 0; c < hidden; c++) {
                double xv = bf16_to_double(xt[c]);
                a += xv * dequant_at(w1q[ex], w1s[ex], hidden, r, c);
                b += xv * dequant_at(w1q[ex], w1s[ex], hidden, r + inter, c);
            }
            double silu = a / (1.0 + exp(-a));
            h[p * inter + r] = silu * b;
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t q = 0; q < ntok * ncols; q++) {
        int64_t i = q / ncols;
        int64_t col = cols ? cols[q % ncols] : (q % ncols);
        double acc = 0.0, sq = 0.0;
        for (int j = 0; j < kp; j++) {
            int64_t p = i * kp + j;
            int ex = ids[p];
            double o = 0.0;
            for (int64_t c = 0; c < inter; c++) {
                double term = h[p * inter + c] * dequant_at(w2q[ex], w2s[ex], inter, col, c);
                o += term;
                double gt = g[p] * term;
                sq += gt * gt;
            }
            acc += g[p] * o;
        }
        y[q] = acc;
        if (rss) rss[q] = sqrt(sq);
    }
    free(ids);
    free(g);
    free(h);
    return 0;
}
