/*
 * q4a_oracle.c -- CPU oracle for the row-batched affine-4-bit dequantising
 * matrix-vector product.
 *
 * TEST INFRASTRUCTURE, NOT THE PRODUCT. Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline leg load this file's library. It is plain,
 * single-threaded C computing in IEEE double precision (the quantiser alone
 * works in binary32: those steps decide integer codes, and both sides take
 * them in the same precision). It shares no code,
 * header, table, constant generator or helper with the CUDA library: its own
 * binary16 / bfloat16 decoders, its own nibble extraction, its own loops.
 *
 * Sources (web pages; cited by page and section):
 *   [BATCH_MSL]  "BATCH_MSL" constant page (cherenkov kernels), a Metal kernel
 *                library. Sections used: quantized_rows.metal (fn_q4_rows_h,
 *                fn_q4_2rows_h: the affine-Q4 row dot products),
 *                hyperconnection.metal (fn_group_norm_b, fn_norm_prep_b,
 *                fn_inject_b, fn_qmv_silu_b), experts.metal (fn_topk_softmax_b,
 *                fn_moe_gate_up_b, fn_moe_act_b, fn_moe_down_b),
 *                expert_gemm.metal (fn_expert_qmm) and the prefill helper
 *                fn_qmv_small_b (explicit nibble order and affine form).
 *   [MEMRA]      memra-engine qwen4exp_gpu.rs source page: host reference math
 *                (host_route_softmax_topk with its denominator floor,
 *                f32_to_bf16_rne).
 *
 * What the method computes (restated):
 *   W is [out][in] with 4-bit codes q in 0..15; byte k of a packed row holds
 *   element 2k in its low nibble and element 2k+1 in its high nibble. Every
 *   run of 64 inputs (a group g) has a bfloat16 scale s[o][g] and bias
 *   b[o][g]; the weight is w = s*q + b ([BATCH_MSL] fn_expert_qmm stages
 *   fma(s, code, b)), so that
 *       y[r][o] = sum_g ( s[o][g] * sum_{i in g} q[o][i]*x[r][i]
 *                         + b[o][g] * xsum[r][g] )
 *   ([BATCH_MSL] fn_q4_rows_h accumulates s*sum(q x) + b*xsum per chunk;
 *   fn_qmv_small_b writes the same with the nibble order explicit).
 *   The oracle evaluates the plain definition: it dequantises W explicitly and
 *   forms the dot products in index order, in double precision.
 *
 * Parity pins: every exported function is checked in tests/test_oracle_pins.py
 * against hand-worked examples (tests/golden/), closed forms, invariants and
 * pure-Python brute force on tiny shapes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define Q4O_EXPORT __attribute__((visibility("default")))

/* ---- storage formats ---------------------------------------------------- */

/* IEEE binary16 -> double (exact for every pattern). */
static double half_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);     /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double (the upper half of an fp32 pattern; exact). */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> IEEE binary16, round to nearest, ties to even. */
static uint16_t half_round(double v)
{
    if (isnan(v))
        return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= 65520.0)                              /* max 65504 + half an ulp */
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {                     /* subnormal: m * 2^-24 */
        double m = nearbyint(ldexp(a, 24));        /* 1024 rolls into 0x0400 */
        return sign | (uint16_t)m;
    }
    int e;
    double f = frexp(a, &e);                       /* a = f * 2^e, f in [0.5,1) */
    double r = nearbyint(ldexp(f, 11));            /* 1024 .. 2048 */
    int biased = e - 1 + 15;
    if (r >= 2048.0) {
        r = 1024.0;
        biased += 1;
    }
    if (biased >= 31)
        return sign | 0x7C00;
    return sign | (uint16_t)(biased << 10) | (uint16_t)((int)r - 1024);
}

/* The code of element i of a packed row: low nibble of byte i/2 for even i,
 * high nibble for odd i (the packed layout; [BATCH_MSL] fn_q4_rows_h pairs the
 * low nibbles with the even x stream and the high nibbles with the odd one). */
static int code_at(const uint8_t* row, int64_t i)
{
    uint8_t byte = row[i >> 1];
    return (i & 1) ? (byte >> 4) : (byte & 0x0F);
}

/* ---- exported helpers for the tests ------------------------------------- */

Q4O_EXPORT double q4o_half_value(uint16_t h) { return half_value(h); }
Q4O_EXPORT double q4o_bf16_value(uint16_t b) { return bf16_value(b); }
Q4O_EXPORT uint16_t q4o_half_round(double v) { return half_round(v); }

/* ---- A1: packing -------------------------------------------------------- */

/* codes[rows][in_dim] (one code per byte, masked to 4 bits as the prefill
 * helper fn_qmv_small_b masks each nibble) -> packed[rows][in_dim/2]. */
Q4O_EXPORT void q4o_pack(uint8_t* packed, const uint8_t* codes, int64_t rows, int64_t in_dim)
{
    for (int64_t o = 0; o < rows; o++) {
        for (int64_t k = 0; k < in_dim / 2; k++) {
            int lo = codes[o * in_dim + 2 * k] & 0x0F;
            int hi = codes[o * in_dim + 2 * k + 1] & 0x0F;
            packed[o * (in_dim / 2) + k] = (uint8_t)(lo | (hi << 4));
        }
    }
}

Q4O_EXPORT void q4o_unpack(uint8_t* codes, const uint8_t* packed, int64_t rows, int64_t in_dim)
{
    for (int64_t o = 0; o < rows; o++)
        for (int64_t i = 0; i < in_dim; i++)
            codes[o * in_dim + i] = (uint8_t)code_at(packed + o * (in_dim / 2), i);
}

/* ---- explicit dequantisation -------------------------------------------- */

static void dequant_row(double* w, const uint8_t* prow, const uint16_t* srow,
                        const uint16_t* brow, int64_t in_dim)
{
    for (int64_t i = 0; i < in_dim; i++) {
        double s = bf16_value(srow[i / 64]);
        double b = bf16_value(brow[i / 64]);
        w[i] = s * (double)code_at(prow, i) + b;
    }
}

/* W[rows][in_dim] = s*q + b, in double (exact: a bf16 times a 4-bit integer
 * has at most 12 significant bits). */
Q4O_EXPORT void q4o_dequant(double* w, const uint8_t* packed, const uint16_t* s,
                            const uint16_t* b, int64_t rows, int64_t in_dim)
{
    int64_t groups = in_dim / 64;
    for (int64_t o = 0; o < rows; o++)
        dequant_row(w + o * in_dim, packed + o * (in_dim / 2), s + o * groups,
                    b + o * groups, in_dim);
}

/* ---- A2: per-64-group sums of the fp16 activations ---------------------- */

/* xsum[r][g] = sum_{i in g} x[r][i], in double, index order. The pages keep
 * per-32 sums (fn_norm_prep_b, fn_moe_act_b); one bias covers both halves of
 * a 64-group, so the per-64 sum is the sum of the two. */
Q4O_EXPORT void q4o_xsum(double* xsum, const uint16_t* x, int64_t nb, int64_t in_dim)
{
    int64_t groups = in_dim / 64;
    for (int64_t r = 0; r < nb; r++)
        for (int64_t g = 0; g < groups; g++) {
            double acc = 0.0;
            for (int64_t i = 0; i < 64; i++)
                acc += half_value(x[r * in_dim + g * 64 + i]);
            xsum[r * groups + g] = acc;
        }
}

/* ---- A4: the GEMV, plain definition ------------------------------------- */

/* y[r][o] = sum_i W[o][i] * x[r][i] with W dequantised explicitly, and the
 * per-element acceptance bound 2e-3 * sum_i |W[o][i] x[r][i]| + 1e-5.
 * bound may be NULL. */
Q4O_EXPORT void q4o_gemv(double* y, double* bound, const uint8_t* packed,
                         const uint16_t* s, const uint16_t* b, const uint16_t* x,
                         int64_t nb, int64_t out_dim, int64_t in_dim)
{
    int64_t groups = in_dim / 64;
    double* w = (double*)malloc((size_t)in_dim * sizeof(double));
    double* xv = (double*)malloc((size_t)(nb * in_dim) * sizeof(double));
    for (int64_t i = 0; i < nb * in_dim; i++)
        xv[i] = half_value(x[i]);
    for (int64_t o = 0; o < out_dim; o++) {
        dequant_row(w, packed + o * (in_dim / 2), s + o * groups, b + o * groups, in_dim);
        for (int64_t r = 0; r < nb; r++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < in_dim; i++) {
                double p = w[i] * xv[r * in_dim + i];
                acc += p;
                mag += fabs(p);
            }
            y[r * out_dim + o] = acc;
            if (bound)
                bound[r * out_dim + o] = 2e-3 * mag + 1e-5;
        }
    }
    free(xv);
    free(w);
}

/* The same product in the factored form the kernels use per group:
 * sum_g ( s * sum q x + b * xsum ). Asserted equal to q4o_gemv (up to double
 * rounding) by the pins; not used for parity. */
Q4O_EXPORT void q4o_gemv_factored(double* y, const uint8_t* packed, const uint16_t* s,
                                  const uint16_t* b, const uint16_t* x, int64_t nb,
                                  int64_t out_dim, int64_t in_dim)
{
    int64_t groups = in_dim / 64;
    for (int64_t o = 0; o < out_dim; o++) {
        const uint8_t* prow = packed + o * (in_dim / 2);
        for (int64_t r = 0; r < nb; r++) {
            double acc = 0.0;
            for (int64_t g = 0; g < groups; g++) {
                double qx = 0.0, xs = 0.0;
                for (int64_t i = g * 64; i < g * 64 + 64; i++) {
                    double xv = half_value(x[r * in_dim + i]);
                    qx += (double)code_at(prow, i) * xv;
                    xs += xv;
                }
                acc += bf16_value(s[o * groups + g]) * qx + bf16_value(b[o * groups + g]) * xs;
            }
            y[r * out_dim + o] = acc;
        }
    }
}

/* Selected entries (r_idx[k], o_idx[k]) of the plain-definition product, one
 * dot product each: the full-size parity checks sample outputs this way. */
Q4O_EXPORT void q4o_gemv_entries(double* y, double* bound, const int64_t* r_idx,
                                 const int64_t* o_idx, int64_t n, const uint8_t* packed,
                                 const uint16_t* s, const uint16_t* b, const uint16_t* x,
                                 int64_t in_dim)
{
    int64_t groups = in_dim / 64;
    double* w = (double*)malloc((size_t)in_dim * sizeof(double));
    for (int64_t k = 0; k < n; k++) {
        int64_t o = o_idx[k], r = r_idx[k];
        dequant_row(w, packed + o * (in_dim / 2), s + o * groups, b + o * groups, in_dim);
        double acc = 0.0, mag = 0.0;
        for (int64_t i = 0; i < in_dim; i++) {
            double p = w[i] * half_value(x[r * in_dim + i]);
            acc += p;
            mag += fabs(p);
        }
        y[k] = acc;
        if (bound)
            bound[k] = 2e-3 * mag + 1e-5;
    }
    free(w);
}

/* ---- A6: routed-expert banks -------------------------------------------- */

/* For segment a (expert e = expert_ids[a], slot rows token_offsets[a] ..
 * token_offsets[a+1]-1): y[r] = W_e . x[x_rows ? x_rows[r] : r].
 * The bank holds experts back to back: rows e*out_dim .. (e+1)*out_dim-1.
 * A segment whose expert id is outside [0, n_experts) yields NaN rows
 * (the library's device convention for such a segment). */
Q4O_EXPORT void q4o_gemv_experts(double* y, double* bound, const uint8_t* w_bank,
                                 const uint16_t* s_bank, const uint16_t* b_bank,
                                 const uint16_t* x, const int32_t* x_rows,
                                 const int32_t* expert_ids, const int32_t* token_offsets,
                                 int64_t n_active, int64_t n_experts, int64_t out_dim,
                                 int64_t in_dim)
{
    int64_t groups = in_dim / 64;
    double* w = (double*)malloc((size_t)in_dim * sizeof(double));
    for (int64_t a = 0; a < n_active; a++) {
        int64_t e = expert_ids[a];
        for (int64_t r = token_offsets[a]; r < token_offsets[a + 1]; r++) {
            if (e < 0 || e >= n_experts) {
                for (int64_t o = 0; o < out_dim; o++) {
                    y[r * out_dim + o] = NAN;
                    if (bound)
                        bound[r * out_dim + o] = NAN;
                }
            }
        }
        if (e < 0 || e >= n_experts)
            continue;
        for (int64_t o = 0; o < out_dim; o++) {
            int64_t row = e * out_dim + o;
            dequant_row(w, w_bank + row * (in_dim / 2), s_bank + row * groups,
                        b_bank + row * groups, in_dim);
            for (int64_t r = token_offsets[a]; r < token_offsets[a + 1]; r++) {
                int64_t src = x_rows ? x_rows[r] : r;
                double acc = 0.0, mag = 0.0;
                for (int64_t i = 0; i < in_dim; i++) {
                    double p = w[i] * half_value(x[src * in_dim + i]);
                    acc += p;
                    mag += fabs(p);
                }
                y[r * out_dim + o] = acc;
                if (bound)
                    bound[r * out_dim + o] = 2e-3 * mag + 1e-5;
            }
        }
    }
    free(w);
}

/* ---- A3: RMSNorm prologue ------------------------------------------------ */

/* [BATCH_MSL] fn_group_norm_b with one group per row:
 *   xn[r][i] = x[r][i] * 1/sqrt(mean_i x[r][i]^2 + eps) * (w[i] + shift),
 * evaluated in double and rounded once to binary16 (the fp16 operand the
 * GEMV multiplies). inv_rms (may be NULL) receives the per-row factor. */
Q4O_EXPORT void q4o_rmsnorm_f16(uint16_t* xn, double* inv_rms, const float* x,
                                const uint16_t* w, double eps, double shift,
                                int64_t nb, int64_t n)
{
    for (int64_t r = 0; r < nb; r++) {
        double ss = 0.0;
        for (int64_t i = 0; i < n; i++) {
            double v = (double)x[r * n + i];
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / (double)n + eps);
        if (inv_rms)
            inv_rms[r] = inv;
        for (int64_t i = 0; i < n; i++)
            xn[r * n + i] = half_round((double)x[r * n + i] * inv * (bf16_value(w[i]) + shift));
    }
}

/* ---- A7: SiLU(gate) * up -------------------------------------------------- */

/* [BATCH_MSL] fn_moe_act_b: gate_up[r] = [gate (inter) | up (inter)],
 * h[r][j] = silu(gate[j]) * up[j] with silu(v) = v / (1 + e^-v), in double,
 * rounded once to binary16. */
Q4O_EXPORT void q4o_silu_mul_f16(uint16_t* h, const float* gate_up, int64_t rows, int64_t inter)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < inter; j++) {
            double g = (double)gate_up[r * 2 * inter + j];
            double u = (double)gate_up[r * 2 * inter + inter + j];
            h[r * inter + j] = half_round(g / (1.0 + exp(-g)) * u);
        }
}

/* ---- routing (input generation for the expert workload) ------------------ */

/* [MEMRA] host_route_softmax_topk: softmax over the logits, order experts by
 * probability (descending) then index (ascending), keep top_k, divide by
 * max(sum of the kept probabilities, 6.1035156e-5). [BATCH_MSL]
 * fn_topk_softmax_b breaks ties toward the lower index the same way.
 * Double precision throughout. */
Q4O_EXPORT void q4o_route_topk(int32_t* idx, double* wts, const float* logits,
                               int64_t n_tok, int64_t n_exp, int64_t top_k)
{
    double* p = (double*)malloc((size_t)n_exp * sizeof(double));
    char* taken = (char*)malloc((size_t)n_exp);
    for (int64_t t = 0; t < n_tok; t++) {
        const float* l = logits + t * n_exp;
        double mx = -INFINITY;
        for (int64_t e = 0; e < n_exp; e++)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        double sum = 0.0;
        for (int64_t e = 0; e < n_exp; e++) {
            p[e] = exp((double)l[e] - mx);
            sum += p[e];
        }
        for (int64_t e = 0; e < n_exp; e++) {
            p[e] /= sum;
            taken[e] = 0;
        }
        double chosen = 0.0;
        for (int64_t k = 0; k < top_k; k++) {
            int64_t best = -1;
            for (int64_t e = 0; e < n_exp; e++)
                if (!taken[e] && (best < 0 || p[e] > p[best]))
                    best = e;                      /* strict '>' keeps the lower index on ties */
            taken[best] = 1;
            idx[t * top_k + k] = (int32_t)best;
            wts[t * top_k + k] = p[best];
            chosen += p[best];
        }
        double denom = chosen > 6.1035156e-5 ? chosen : 6.1035156e-5;
        for (int64_t k = 0; k < top_k; k++)
            wts[t * top_k + k] /= denom;
    }
    free(taken);
    free(p);
}

/* ---- MoE combine ---------------------------------------------------------- */

/* [BATCH_MSL] experts.metal, fn_moe_combine_b (part 0 and part 1) and
 * fn_shared_add_rows: the output row of token t is the routing-weighted sum of
 * the expert outputs of its slots, plus, when a shared expert is present, its
 * output scaled by sigmoid(gate_vec . x[t]):
 *     out[t][i] = sum_k w[t][k] * y[slot[t][k]][i]
 *               + sigmoid(sum_j gate[j] * x[t][j]) * y_shared[t][i].
 * Double precision, k in order. bound[t][i] = sum_k |w y| + |g y_shared| and
 * gabs[t] = sum_j |gate[j] x[t][j]| feed the tests' tolerance. A slot id
 * outside [0, n_slots) makes the row NaN (the library's convention). */
Q4O_EXPORT void q4o_moe_combine(double* out, double* bound, double* gabs, const float* y,
                                const int32_t* slot, const float* w, const float* y_shared,
                                const uint16_t* gate, const float* x, int64_t n_tok,
                                int64_t top_k, int64_t n_slots, int64_t hidden)
{
    for (int64_t t = 0; t < n_tok; t++) {
        double g = 0.0, ga = 0.0;
        if (y_shared) {
            double dot = 0.0;
            for (int64_t j = 0; j < hidden; j++) {
                const double term = bf16_value(gate[j]) * (double)x[t * hidden + j];
                dot += term;
                ga += fabs(term);
            }
            g = 1.0 / (1.0 + exp(-dot));
        }
        gabs[t] = ga;
        int bad = 0;
        for (int64_t k = 0; k < top_k; k++)
            if (slot[t * top_k + k] < 0 || slot[t * top_k + k] >= n_slots)
                bad = 1;
        for (int64_t i = 0; i < hidden; i++) {
            double acc = 0.0, a = 0.0;
            if (!bad)
                for (int64_t k = 0; k < top_k; k++) {
                    const double term = (double)w[t * top_k + k] *
                                        (double)y[(int64_t)slot[t * top_k + k] * hidden + i];
                    acc += term;
                    a += fabs(term);
                }
            if (y_shared) {
                const double term = g * (double)y_shared[t * hidden + i];
                acc += term;
                a += fabs(term);
            }
            out[t * hidden + i] = bad ? NAN : acc;
            bound[t * hidden + i] = a;
        }
    }
}

/* ---- GEMV with a SiLU epilogue -------------------------------------------- */

/* [BATCH_MSL] hyperconnection.metal, fn_qmv_silu_b: the Q4 matvec whose outputs go
 * through silu(y / div) (the gated-residual bottleneck):
 *     out[r][o] = v / (1 + e^-v),  v = y[r][o] / div,  y = the plain product above.
 * Double precision; y and its acceptance bound come from q4o_gemv. */
Q4O_EXPORT void q4o_gemv_silu(double* out, double* y, double* bound, const uint8_t* packed,
                              const uint16_t* s, const uint16_t* b, const uint16_t* x, double div,
                              int64_t nb, int64_t out_dim, int64_t in_dim)
{
    q4o_gemv(y, bound, packed, s, b, x, nb, out_dim, in_dim);
    for (int64_t i = 0; i < nb * out_dim; i++) {
        const double v = y[i] / div;
        out[i] = v / (1.0 + exp(-v));
    }
}

/* ---- grouped RMSNorm prologue ----------------------------------------------- */

/* [BATCH_MSL] hyperconnection.metal fn_group_norm_b with `groups` streams per row: the
 * row splits into groups equal segments of width n = in_dim / groups, each normalised
 * with its own mean of squares; the weight is indexed by the position in the whole row:
 *   xn[r][g*n + i] = x[r][g*n + i] / sqrt(mean_i x[r][g*n + i]^2 + eps) * (w[g*n + i] + shift),
 * evaluated in double and rounded once to binary16. inv_rms [nb][groups] may be NULL. */
Q4O_EXPORT void q4o_rmsnorm_groups_f16(uint16_t* xn, double* inv_rms, const float* x,
                                       const uint16_t* w, double eps, double shift,
                                       int64_t nb, int64_t in_dim, int64_t groups)
{
    const int64_t n = in_dim / groups;
    for (int64_t r = 0; r < nb; r++)
        for (int64_t g = 0; g < groups; g++) {
            const float* xs = x + r * in_dim + g * n;
            double ss = 0.0;
            for (int64_t i = 0; i < n; i++)
                ss += (double)xs[i] * (double)xs[i];
            const double inv = 1.0 / sqrt(ss / (double)n + eps);
            if (inv_rms)
                inv_rms[r * groups + g] = inv;
            for (int64_t i = 0; i < n; i++)
                xn[r * in_dim + g * n + i] = half_round((double)xs[i] * inv * (bf16_value(w[g * n + i]) + shift));
        }
}

/* [BATCH_MSL] hyperconnection.metal fn_inject_b, and fn_norm_prep_b with inject = 1. A row
 * holds `groups` hyper-connection streams of n = in_dim / groups inputs each; stream g of row r
 * first receives the layer output scaled by twice a sigmoid of its mixing logit,
 *     x'[r][g n + i] = x[r][g n + i] + out[r][i] * 2 / (1 + e^(-logit[r][g] / groups)),
 * and is then RMS-normalised on its own, exactly as q4o_rmsnorm_groups_f16 does:
 *     xn[r][g n + i] = fp16( x'[r][g n + i] * rsqrt(mean_i x'[r][g n + i]^2 + eps) * (w[g n + i] + shift) ).
 * Every step in double; x_new receives x'. */
Q4O_EXPORT void q4o_inject_rmsnorm_groups_f16(uint16_t* xn, double* x_new, const float* x, const float* out,
                                              const float* logit, const uint16_t* w, double eps, double shift,
                                              int64_t nb, int64_t in_dim, int64_t groups)
{
    const int64_t n = in_dim / groups;
    for (int64_t r = 0; r < nb; r++)
        for (int64_t g = 0; g < groups; g++) {
            const double wgt = 2.0 / (1.0 + exp(-(double)logit[r * groups + g] / (double)groups));
            double* xs = x_new + r * in_dim + g * n;
            double ss = 0.0;
            for (int64_t i = 0; i < n; i++) {
                xs[i] = (double)x[r * in_dim + g * n + i] + (double)out[r * n + i] * wgt;
                ss += xs[i] * xs[i];
            }
            const double inv = 1.0 / sqrt(ss / (double)n + eps);
            for (int64_t i = 0; i < n; i++)
                xn[r * in_dim + g * n + i] = half_round(xs[i] * inv * (bf16_value(w[g * n + i]) + shift));
        }
}

/* ---- derived low-bit codes (2-bit and 3-bit) ------------------------------------ */

/* [BATCH_MSL] quantized_rows.metal fn_q2_rows_h and fn_q3_rows_h. The low-bit codes are
 * derived from the 4-bit ones: q2 = q4 >> 2 with the quad midpoint w = (4 q2 + 1.5) s + b,
 * and q3 = q4 >> 1 with w = (2 q3 + 0.5) s + b. The 2-bit row is a run of 32-code chunks,
 * two little-endian 32-bit words each; byte b of word t of chunk c holds four 2-bit fields
 * (the masked casts of the kernel pair them with the even / odd activation streams):
 *     field 0 (bits 1:0)  element 32c + 2(8t + b)
 *     field 1 (bits 3:2)  element 32c + 2(8t + 4 + b)
 *     field 2 (bits 5:4)  element 32c + 2(8t + b) + 1
 *     field 3 (bits 7:6)  element 32c + 2(8t + 4 + b) + 1
 * A 3-bit code is 2 * upper + lowest: the upper two bits (= q2) in the 2-bit layout, and one
 * 32-bit word per chunk of lowest bits, the bit of the element in field j of byte b of upper
 * word t sitting at bit 4t + j of byte b. The pages interleave the three words of a chunk;
 * this library keeps the lowest-bit words as a plane of their own ([rows][in/32] words). */

/* element index (within its 32-code chunk) of field j, byte b, word t */
static int lowbit_element(int t, int b, int j)
{
    const int even_slot = 8 * t + ((j & 1) ? 4 : 0) + b;   /* index in the even / odd stream */
    return 2 * even_slot + ((j & 2) ? 1 : 0);
}

/* codes[rows][in_dim] (4-bit codes, one per byte) -> the 2-bit packed rows [rows][in_dim/4]. */
Q4O_EXPORT void q4o_lowbit_pack2(uint8_t* w2, const uint8_t* codes, int64_t rows, int64_t in_dim)
{
    for (int64_t o = 0; o < rows; o++)
        for (int64_t c = 0; c < in_dim / 32; c++)
            for (int t = 0; t < 2; t++)
                for (int b = 0; b < 4; b++) {
                    int v = 0;
                    for (int j = 0; j < 4; j++) {
                        const int q4 = codes[o * in_dim + 32 * c + lowbit_element(t, b, j)] & 0x0F;
                        v |= (q4 >> 2) << (2 * j);
                    }
                    w2[o * (in_dim / 4) + 8 * c + 4 * t + b] = (uint8_t)v;
                }
}

/* codes[rows][in_dim] -> the lowest-bit plane of the 3-bit codes [rows][in_dim/8] bytes. */
Q4O_EXPORT void q4o_lowbit_pack3lo(uint8_t* wlo, const uint8_t* codes, int64_t rows, int64_t in_dim)
{
    for (int64_t o = 0; o < rows; o++)
        for (int64_t c = 0; c < in_dim / 32; c++)
            for (int b = 0; b < 4; b++) {
                int v = 0;
                for (int t = 0; t < 2; t++)
                    for (int j = 0; j < 4; j++) {
                        const int q4 = codes[o * in_dim + 32 * c + lowbit_element(t, b, j)] & 0x0F;
                        v |= ((q4 >> 1) & 1) << (4 * t + j);
                    }
                wlo[o * (in_dim / 8) + 4 * c + b] = (uint8_t)v;
            }
}

/* The code of element i of a row, read back from the packed layout: q2 (wlo NULL) or q3. */
static int lowbit_code_at(const uint8_t* w2row, const uint8_t* wlorow, int64_t i)
{
    const int64_t c = i / 32;
    const int e = (int)(i % 32);
    const int odd = e & 1;
    const int slot = e >> 1;                 /* 0..15 in the even / odd stream */
    const int t = slot / 8;
    const int hi4 = (slot % 8) >= 4;
    const int b = slot % 4;
    const int j = (hi4 ? 1 : 0) + (odd ? 2 : 0);
    const int up = (w2row[8 * c + 4 * t + b] >> (2 * j)) & 3;
    if (!wlorow)
        return up;
    const int lo = (wlorow[4 * c + b] >> (4 * t + j)) & 1;
    return 2 * up + lo;
}

/* codes[rows][in_dim] = the derived codes read back from the packed layout. */
Q4O_EXPORT void q4o_lowbit_codes(uint8_t* codes, const uint8_t* w2, const uint8_t* wlo,
                                 int64_t rows, int64_t in_dim)
{
    for (int64_t o = 0; o < rows; o++)
        for (int64_t i = 0; i < in_dim; i++)
            codes[o * in_dim + i] = (uint8_t)lowbit_code_at(w2 + o * (in_dim / 4),
                                                            wlo ? wlo + o * (in_dim / 8) : NULL, i);
}

/* y[r][o] = sum_i w[o][i] x[r][i] with w = (4 q2 + 1.5) s + b (wlo NULL: 2-bit) or
 * w = (2 q3 + 0.5) s + b (3-bit), dequantised explicitly in double; bound as q4o_gemv. */
Q4O_EXPORT void q4o_gemv_lowbit(double* y, double* bound, const uint8_t* w2, const uint8_t* wlo,
                                const uint16_t* s, const uint16_t* b, const uint16_t* x,
                                int64_t nb, int64_t out_dim, int64_t in_dim)
{
    const int64_t groups = in_dim / 64;
    double* w = (double*)malloc((size_t)in_dim * sizeof(double));
    double* xv = (double*)malloc((size_t)(nb * in_dim) * sizeof(double));
    for (int64_t i = 0; i < nb * in_dim; i++)
        xv[i] = half_value(x[i]);
    for (int64_t o = 0; o < out_dim; o++) {
        const uint8_t* w2row = w2 + o * (in_dim / 4);
        const uint8_t* wlorow = wlo ? wlo + o * (in_dim / 8) : NULL;
        for (int64_t i = 0; i < in_dim; i++) {
            const double sv = bf16_value(s[o * groups + i / 64]);
            const double bv = bf16_value(b[o * groups + i / 64]);
            const double q = (double)lowbit_code_at(w2row, wlorow, i);
            w[i] = wlorow ? sv * (2.0 * q + 0.5) + bv : sv * (4.0 * q + 1.5) + bv;
        }
        for (int64_t r = 0; r < nb; r++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < in_dim; i++) {
                const double p = w[i] * xv[r * in_dim + i];
                acc += p;
                mag += fabs(p);
            }
            y[r * out_dim + o] = acc;
            if (bound)
                bound[r * out_dim + o] = 2e-3 * mag + 1e-5;
        }
    }
    free(xv);
    free(w);
}

/* [BATCH_MSL] expert_gemm.metal fn_expert_qmm (prefill: 8/16/32-token tiles of fp32
 * activations) and the routed form of fn_q2_rows_h / fn_q3_rows_h (decode): the low-bit codes
 * of a routed-expert bank. For segment a (expert e = expert_ids[a], slot rows token_offsets[a]
 * .. token_offsets[a+1]-1), y[r][o] = sum_i W_e[o][i] * x[src][i] with src = x_rows ? x_rows[r]
 * : r and the quad or pair midpoint W = s (4 q2 + 1.5) + b (bits 2; wlo_bank NULL) or
 * W = s (2 q3 + 0.5) + b (bits 3), every step in double; x is fp32 (x32) or binary16 (x16),
 * taken as given. An expert id outside [0, n_experts) gives NaN rows; bound as q4o_gemv. */
Q4O_EXPORT void q4o_experts_lowbit(double* y, double* bound, const uint8_t* w2_bank, const uint8_t* wlo_bank,
                                   const uint16_t* s_bank, const uint16_t* b_bank, const float* x32,
                                   const uint16_t* x16, const int32_t* x_rows, const int32_t* expert_ids,
                                   const int32_t* token_offsets, int64_t n_active, int64_t n_experts,
                                   int64_t out_dim, int64_t in_dim)
{
    const int64_t groups = in_dim / 64;
    double* w = (double*)malloc((size_t)in_dim * sizeof(double));
    for (int64_t a = 0; a < n_active; a++) {
        const int64_t e = expert_ids[a];
        if (e < 0 || e >= n_experts) {
            for (int64_t r = token_offsets[a]; r < token_offsets[a + 1]; r++)
                for (int64_t o = 0; o < out_dim; o++) {
                    y[r * out_dim + o] = NAN;
                    if (bound)
                        bound[r * out_dim + o] = NAN;
                }
            continue;
        }
        for (int64_t o = 0; o < out_dim; o++) {
            const int64_t row = e * out_dim + o;
            const uint8_t* w2row = w2_bank + row * (in_dim / 4);
            const uint8_t* wlorow = wlo_bank ? wlo_bank + row * (in_dim / 8) : NULL;
            for (int64_t i = 0; i < in_dim; i++) {
                const double sv = bf16_value(s_bank[row * groups + i / 64]);
                const double bv = bf16_value(b_bank[row * groups + i / 64]);
                const double q = (double)lowbit_code_at(w2row, wlorow, i);
                w[i] = wlorow ? sv * (2.0 * q + 0.5) + bv : sv * (4.0 * q + 1.5) + bv;
            }
            for (int64_t r = token_offsets[a]; r < token_offsets[a + 1]; r++) {
                const int64_t src = x_rows ? x_rows[r] : r;
                double acc = 0.0, mag = 0.0;
                for (int64_t i = 0; i < in_dim; i++) {
                    const double xv = x32 ? (double)x32[src * in_dim + i] : half_value(x16[src * in_dim + i]);
                    const double p = w[i] * xv;
                    acc += p;
                    mag += fabs(p);
                }
                y[r * out_dim + o] = acc;
                if (bound)
                    bound[r * out_dim + o] = 2e-3 * mag + 1e-5;
            }
        }
    }
    free(w);
}

/* ---- prefill helpers ---------------------------------------------------------------- */

/* [BATCH_MSL] fn_qmv_small_b: the projection straight from fp32 activations (few output
 * rows, any number of input rows). y[r][o] = sum_i w[o][i] x[r][i], w = s q + b dequantised
 * explicitly, x the fp32 values as given, in double; bound as q4o_gemv. */
Q4O_EXPORT void q4o_gemv_f32x(double* y, double* bound, const uint8_t* packed, const uint16_t* s,
                              const uint16_t* b, const float* x, int64_t nb, int64_t out_dim, int64_t in_dim)
{
    const int64_t groups = in_dim / 64;
    double* w = (double*)malloc((size_t)in_dim * sizeof(double));
    for (int64_t o = 0; o < out_dim; o++) {
        dequant_row(w, packed + o * (in_dim / 2), s + o * groups, b + o * groups, in_dim);
        for (int64_t r = 0; r < nb; r++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < in_dim; i++) {
                const double p = w[i] * (double)x[r * in_dim + i];
                acc += p;
                mag += fabs(p);
            }
            y[r * out_dim + o] = acc;
            if (bound)
                bound[r * out_dim + o] = 2e-3 * mag + 1e-5;
        }
    }
    free(w);
}

/* binary32 -> bfloat16, round to nearest even (NaN -> a quiet NaN). */
static uint16_t bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof(u));
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return 0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* A 4-bit affine quantiser for float weights. The pages never define one; this is the plain
 * min/max reading, every step in binary32 (the precision that decides the integer codes):
 *   b = bf16(min_g w) (a zero minimum stored as +0),  s = bf16((max_g w - b) / 15) when
 *   max_g w > b, else 0,
 *   q = clamp(rint((w - b) / s), 0, 15) when s > 0, else 0,
 * with b and s their bfloat16 values, rint rounding half to even. Writes the packed codes
 * [rows][in_dim/2] (as q4o_pack), s and b [rows][in_dim/64]. w must be finite. */
Q4O_EXPORT void q4o_quantize(uint8_t* packed, uint16_t* s, uint16_t* b, const float* w,
                             int64_t rows, int64_t in_dim)
{
    const int64_t groups = in_dim / 64;
    uint8_t* codes = (uint8_t*)malloc((size_t)in_dim);
    for (int64_t o = 0; o < rows; o++) {
        for (int64_t g = 0; g < groups; g++) {
            const float* wg = w + o * in_dim + g * 64;
            float mn = wg[0], mx = wg[0];
            for (int i = 1; i < 64; i++) {
                if (wg[i] < mn) mn = wg[i];
                if (wg[i] > mx) mx = wg[i];
            }
            const uint16_t bb = bf16_round(mn == 0.0f ? 0.0f : mn);   /* a zero minimum is +0 */
            const float bf = (float)bf16_value(bb);
            const float range = mx - bf;
            const uint16_t sb = range > 0.0f ? bf16_round(range / 15.0f) : (uint16_t)0;
            const float sf = (float)bf16_value(sb);
            for (int i = 0; i < 64; i++) {
                int q = 0;
                if (sf > 0.0f) {
                    const float t = rintf((wg[i] - bf) / sf);
                    q = t < 0.0f ? 0 : (t > 15.0f ? 15 : (int)t);
                }
                codes[g * 64 + i] = (uint8_t)q;
            }
            s[o * groups + g] = sb;
            b[o * groups + g] = bb;
        }
        q4o_pack(packed + o * (in_dim / 2), codes, 1, in_dim);
    }
    free(codes);
}
