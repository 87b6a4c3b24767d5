/*
 * q4a.h -- C ABI of libq4a.so, the row-batched affine-4-bit dequantising
 * matrix-vector product for NVIDIA GB300 (sm_103a).
 *
 * The operation (restated from three web pages on the subject; citations name
 * the page and the section of it):
 *   W is [out_dim][in_dim] with 4-bit codes q in 0..15, packed two per byte:
 *   byte k of a row holds element 2k in its low nibble and element 2k+1 in its
 *   high nibble. Every run of 64 inputs (group g) of a row has a bfloat16 scale
 *   s[o][g] and bias b[o][g]; the weight is w = s*q + b. For NB activation rows
 *       y[r][o] = sum_g ( s[o][g] * sum_{i in g} q[o][i] * x[r][i]
 *                         + b[o][g] * xsum[r][g] ),   xsum[r][g] = sum_{i in g} x[r][i].
 *   ("BATCH_MSL" constant page, quantized_rows.metal: fn_q4_rows_h and
 *   fn_q4_2rows_h; the prefill helper fn_qmv_small_b states the nibble order
 *   explicitly; expert_gemm.metal stages w = fma(s, code, b).)
 *
 * Conventions shared by every entry point:
 *   - Every buffer pointer is caller-owned DEVICE memory unless the argument
 *     says "host". The library allocates no memory and keeps no per-call state.
 *     It never reads device buffers from the host.
 *   - fp16 buffers hold IEEE binary16 bit patterns, bf16 buffers bfloat16 bit
 *     patterns (both as uint16_t). Matrices are row-major, rows contiguous.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and runs asynchronously; a call returns once its kernels are
 *     launched. Outputs are fully overwritten (never accumulated into).
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and leaves outputs untouched.
 *   - Kernels never trap and never wait without a bound. A kernel that gives up
 *     a bounded wait records it in a device error word; q4a_check_device_error
 *     reports it.
 *   - Results are deterministic: identical inputs give bit-identical outputs
 *     (no floating-point atomics).
 */
#ifndef Q4A_H
#define Q4A_H

#include <stdint.h>

#if defined(__GNUC__)
#define Q4A_API __attribute__((visibility("default")))
#else
#define Q4A_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same underlying type). */
typedef struct CUstream_st* q4a_stream_t;

typedef enum q4a_status {
    Q4A_OK = 0,
    Q4A_ERR_NULL = 1,        /* a required pointer is NULL                          */
    Q4A_ERR_SHAPE = 2,       /* a size or an index table is out of range            */
    Q4A_ERR_ALIGN = 3,       /* a pointer misses the alignment stated below         */
    Q4A_ERR_UNSUPPORTED = 4, /* valid but not supported (device, size limit)        */
    Q4A_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed (see q4a_last_cuda_error) */
    Q4A_ERR_TIMEOUT = 6      /* a kernel gave up a bounded wait (q4a_check_device_error) */
} q4a_status;

/* Upper limits of the host-side schedule. */
#define Q4A_MAX_SEGMENTS 512   /* routed-expert segments per q4a_gemv_experts call */


/* Static string for a status code (never NULL). */
Q4A_API const char* q4a_status_string(q4a_status status);

/* The cudaError_t value behind the most recent Q4A_ERR_CUDA on the calling
 * host thread (0 if none). */
Q4A_API int q4a_last_cuda_error(void);

/*
 * q4a_pack -- A1: pack one-code-per-byte matrices into the 4-bit row layout.
 *   w_packed  out  uint8 [rows][in_dim/2]; byte k of a row = codes[2k] | codes[2k+1] << 4
 *   codes     in   uint8 [rows][in_dim]; each code is masked to its low 4 bits
 *                  (the prefill helper fn_qmv_small_b masks every nibble with 0xF)
 *   Requires rows >= 1, in_dim >= 64, in_dim % 64 == 0, both pointers 16-byte aligned.
 *   ("BATCH_MSL", quantized_rows.metal: low nibbles pair with the even x stream,
 *   high nibbles with the odd one.)
 */
Q4A_API q4a_status q4a_pack(uint8_t* w_packed, const uint8_t* codes, int64_t rows, int64_t in_dim,
                    q4a_stream_t stream);

/*
 * q4a_xsum -- A2: per-64-group sums of fp16 activations, accumulated in fp32.
 *   xsum  out  fp32 [nb][in_dim/64];  xsum[r][g] = sum_{i in g} x[r][i]
 *   x     in   fp16 [nb][in_dim]
 *   Requires nb >= 1, in_dim % 64 == 0, x 16-byte aligned, xsum 4-byte aligned.
 *   (The pages keep per-32 sums: "BATCH_MSL" fn_norm_prep_b and fn_moe_act_b;
 *   one bias covers both halves of a 64-group, so this is their pairwise sum.)
 */
Q4A_API q4a_status q4a_xsum(float* xsum, const uint16_t* x, int nb, int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv -- A4: y = W.x for nb activation rows.
 *   y        out  fp32 [nb][out_dim]
 *   w        in   uint8 [out_dim][in_dim/2], packed as q4a_pack writes it
 *   s, b     in   bf16 [out_dim][in_dim/64] scales and biases
 *   x        in   fp16 [nb][in_dim]
 *   Requires nb >= 1, out_dim >= 1 (any value, odd included), in_dim >= 64,
 *   in_dim % 64 == 0; w and x 16-byte aligned; s and b 2-byte aligned.
 *   Kernel choice: the tensor-core path (weights dequantised into TMEM, tcgen05.mma) takes
 *   nb >= 64, nb >= 9 when out_dim >= 38912 (a 256-row unit for every SM) and nb >= 17 when
 *   out_dim >= 12288 (48 units), provided
 *   in_dim % 512 == 0 and s, b are 16-byte aligned; everything else runs the GEMV kernel
 *   (q4a_gemv_kernel_choice tells which, without launching).
 *   The GEMV kernel keeps a CTA's
 *   K-slice of the activations and of the row block's scales and biases in shared memory:
 *   rows longer than that budget allows, even split across 8 CTAs, return
 *   Q4A_ERR_UNSUPPORTED before any launch. Every in_dim up to 98304 runs at NB 1, up to
 *   65536 at NB <= 4, up to 16384 at NB <= 16 and up to 4096 at any NB (8192, 12288 and
 *   16384 run at any NB too); matrices of a few tiles reach further (short row blocks leave
 *   more room: 131072 inputs at NB 1 on 16 rows).
 *   ("BATCH_MSL", hyperconnection.metal fn_qmv_silu_b over quantized_rows.metal
 *   fn_q4_rows_h; experts.metal fn_moe_down_b for the two-rows-per-pass form.)
 */
Q4A_API q4a_status q4a_gemv(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                    const uint16_t* x, int nb, int64_t out_dim, int64_t in_dim,
                    q4a_stream_t stream);

/*
 * q4a_gemv_gate_up_silu -- the gate and up projections of a gated MLP in one pass, with the
 * activation in the output epilogue ("BATCH_MSL", experts.metal fn_moe_gate_up_b followed by
 * fn_moe_act_b):  h[r][o] = fp16( silu(g) * u ),  g = (W_gate.x)[r][o],  u = (W_up.x)[r][o],
 * silu(v) = v / (1 + e^-v), g and u in fp32, rounded once to binary16.
 *   h      out  fp16 [nb][inter]
 *   w      in   uint8 [2 * inter][in_dim/2]: rows [0, inter) are W_gate, [inter, 2 inter) W_up
 *   s, b   in   bf16 [2 * inter][in_dim/64], same row order
 *   x      in   fp16 [nb][in_dim]
 *   Requires nb in 1..256, inter >= 1 and inter % 16 == 0, in_dim % 64 == 0; w and x 16-byte
 *   aligned, s, b and h 2-byte aligned. Always runs on the GEMV kernel, whose fused row blocks
 *   fetch scales and biases with 2D TMA boxes only: in_dim % 512 != 0, or s / b not 16-byte
 *   aligned, returns Q4A_ERR_UNSUPPORTED.
 */
Q4A_API q4a_status q4a_gemv_gate_up_silu(uint16_t* h, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                                         const uint16_t* x, int nb, int64_t inter, int64_t in_dim,
                                         q4a_stream_t stream);

/*
 * q4a_gemv_rmsnorm_gate_up_silu -- q4a_gemv_gate_up_silu on RMS-normalised activations (the
 * prologue of q4a_gemv_rmsnorm, one normalisation group): a decode layer's whole first half.
 *   x_raw, norm_w, eps, shift as q4a_gemv_rmsnorm; nb in 1..32; everything else as
 *   q4a_gemv_gate_up_silu.
 */
Q4A_API q4a_status q4a_gemv_rmsnorm_gate_up_silu(uint16_t* h, const uint8_t* w, const uint16_t* s,
                                                 const uint16_t* b, const float* x_raw, const uint16_t* norm_w,
                                                 float eps, float shift, int nb, int64_t inter, int64_t in_dim,
                                                 q4a_stream_t stream);

/*
 * q4a_decode_mlp -- one decode layer's gated MLP in one call: RMSNorm, the gate and up
 * projections with the silu(gate)*up epilogue, then the down projection of h; the same result
 * as q4a_gemv_rmsnorm_gate_up_silu followed by q4a_gemv on h ("BATCH_MSL",
 * hyperconnection.metal fn_norm_prep_b / fn_group_norm_b, then experts.metal fn_moe_gate_up_b,
 * fn_moe_act_b and fn_moe_down_b: the dense form of the same chain).
 *   y         out  fp32 [nb][hidden]
 *   h         out  fp16 [nb][inter], h = fp16(silu(W_gate.xn) * (W_up.xn)), the down
 *                  projection's input
 *   w_gu, s_gu, b_gu   in  [2*inter][hidden/2] codes, [2*inter][hidden/64] bf16: gate rows,
 *                  then up rows (as q4a_gemv_gate_up_silu)
 *   x_raw, norm_w, eps, shift   in  as q4a_gemv_rmsnorm (one normalisation group)
 *   w_dn, s_dn, b_dn   in  [hidden][inter/2] codes, [hidden][inter/64] bf16
 *   Two launches, the same kernels as the separate entry points; the second starts under
 *   programmatic dependent launch while the first drains.
 *   Requires 1 <= nb <= 32, hidden % 512 == 0, inter % 64 == 0; w_gu, w_dn, x_raw, norm_w and
 *   h 16-byte aligned; s_gu, b_gu 16-byte aligned; s_dn, b_dn 2-byte aligned. Everything is
 *   planned before anything is launched, so a rejected call launches nothing.
 */
Q4A_API q4a_status q4a_decode_mlp(float* y, uint16_t* h, const uint8_t* w_gu, const uint16_t* s_gu,
                                  const uint16_t* b_gu, const float* x_raw, const uint16_t* norm_w, float eps,
                                  float shift, const uint8_t* w_dn, const uint16_t* s_dn, const uint16_t* b_dn,
                                  int nb, int64_t hidden, int64_t inter, q4a_stream_t stream);

/*
 * q4a_quantize -- a 4-bit affine quantiser for float weights (a prefill helper; the pages define
 * none). Per 64-input group, every step in binary32:
 *     b = bf16(min w),  s = bf16((max w - b) / 15) if max w > b else 0,
 *     q = clamp(rint((w - b) / s), 0, 15) if s > 0 else 0   (b, s their bfloat16 values)
 *   w_packed  out  uint8 [rows][in_dim/2] as q4a_pack writes it
 *   s, b      out  bf16 [rows][in_dim/64]
 *   w         in   fp32 [rows][in_dim], finite values
 *   Requires rows >= 1, in_dim % 64 == 0, w and w_packed 16-byte aligned, s and b 2-byte aligned.
 */
Q4A_API q4a_status q4a_quantize(uint8_t* w_packed, uint16_t* s, uint16_t* b, const float* w, int64_t rows,
                                int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_f32x -- y = W.x straight from fp32 activations, for a few output rows over any number
 * of activation rows ("BATCH_MSL", hyperconnection.metal fn_qmv_small_b: the narrow projections
 * of prefill). Code word wi of a row holds elements 8wi .. 8wi+7, element 8wi + e in nibble e;
 * per word the kernel accumulates s * sum(q x) + b * sum(x) in fp32.
 *   y        out  fp32 [nb][out_dim]
 *   w, s, b  in   as q4a_gemv
 *   x        in   fp32 [nb][in_dim]
 *   Requires nb >= 1, in_dim % 64 == 0, w and x 16-byte aligned. CUDA cores, not tensor cores:
 *   meant for narrow outputs; wide ones belong to q4a_gemv.
 */
Q4A_API q4a_status q4a_gemv_f32x(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b, const float* x,
                                 int nb, int64_t out_dim, int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_lowbit_pack -- derived low-bit codes of a packed 4-bit matrix ("BATCH_MSL",
 * quantized_rows.metal fn_q2_rows_h and fn_q3_rows_h: codes q4 >> 2 and q4 >> 1).
 *   w_up      out  uint8 [rows][in_dim/4]: the 2-bit codes q4 >> 2 (also the upper two bits of
 *                  the 3-bit codes). Per 32-code chunk two little-endian 32-bit words; byte b
 *                  of word t holds in bits 2j+1:2j the code of element 2(8t + 4(j&1) + b) + (j>>1)
 *                  of the chunk (the layout the 2-bit kernel's masked casts read).
 *   w_lo      out  uint8 [rows][in_dim/8] or NULL: the lowest bits of the 3-bit codes,
 *                  (q4 >> 1) & 1, one word per chunk, the bit of the element in field j of byte
 *                  b of word t at bit 4t + j of byte b. (The pages interleave the three words
 *                  of a chunk; this library keeps the lowest-bit words as their own plane.)
 *   w_packed  in   uint8 [rows][in_dim/2], packed as q4a_pack writes it
 *   Requires rows >= 1, in_dim % 64 == 0, every pointer 16-byte aligned. The caller owns all
 *   buffers; nothing is allocated.
 */
Q4A_API q4a_status q4a_lowbit_pack(uint8_t* w_up, uint8_t* w_lo, const uint8_t* w_packed, int64_t rows,
                                   int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_lowbit -- y = W.x with W from derived low-bit codes ("BATCH_MSL", quantized_rows.metal
 * fn_q2_rows_h, fn_q3_rows_h): the quad midpoint w = (4 q2 + 1.5) s + b for bits = 2, and
 * w = (2 q3 + 0.5) s + b with q3 = 2 * upper + lowest for bits = 3.
 *   bits       2 or 3 (else Q4A_ERR_UNSUPPORTED)
 *   w_up, w_lo as q4a_lowbit_pack writes them (w_lo ignored for bits = 2, required for 3)
 *   y, s, b, x, nb, out_dim, in_dim as q4a_gemv; bits = 3 also needs in_dim % 128 == 0.
 *   Any nb >= 1 up to 256 runs on the GEMV kernel (no tensor-core path for low-bit codes).
 */
Q4A_API q4a_status q4a_gemv_lowbit(float* y, int bits, const uint8_t* w_up, const uint8_t* w_lo,
                                   const uint16_t* s, const uint16_t* b, const uint16_t* x, int nb,
                                   int64_t out_dim, int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_silu -- q4a_gemv whose outputs go through silu(y / div) on the way out
 * ("BATCH_MSL", hyperconnection.metal fn_qmv_silu_b: the gated-residual bottleneck):
 *     y[r][o] = v / (1 + e^-v),  v = (W.x)[r][o] / div
 *   div  finite and nonzero (else Q4A_ERR_SHAPE); all other arguments, layouts, kernel
 *   choice and errors as q4a_gemv.
 */
Q4A_API q4a_status q4a_gemv_silu(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                         const uint16_t* x, float div, int nb, int64_t out_dim, int64_t in_dim,
                         q4a_stream_t stream);

/*
 * q4a_gemv_experts -- A6: the GEMV over a routed-expert bank.
 *   y              out   fp32 [n_rows][out_dim]; row r = W_e . x[x_rows ? x_rows[r] : r]
 *                        for the segment a with token_offsets[a] <= r < token_offsets[a+1]
 *                        and e = expert_ids[a]
 *   w_bank         in    uint8 [n_experts*out_dim][in_dim/2], expert e at rows e*out_dim..
 *   s_bank, b_bank in    bf16 [n_experts*out_dim][in_dim/64]
 *   x              in    fp16 [*][in_dim]; with x_rows == NULL it has n_rows rows
 *   x_rows         in    int32 [n_rows] device array or NULL; every entry must be a
 *                        valid row index of x (device contents are not read by the host)
 *   expert_ids     HOST  int32 [n_active]
 *   token_offsets  HOST  int32 [n_active+1], token_offsets[0] == 0, non-decreasing,
 *                        token_offsets[n_active] == n_rows
 *   Requires 1 <= n_active <= Q4A_MAX_SEGMENTS, n_experts >= 1, n_rows >= 1, and the
 *   q4a_gemv shape/alignment rules. A segment whose expert id lies outside
 *   [0, n_experts) produces NaN rows (a loud failure, never an out-of-bounds read).
 *   The expert list and offsets are host arrays because the host publishes the
 *   union of routed experts after the router ("BATCH_MSL", experts.metal: the
 *   grouped-expert section; fn_moe_gate_up_b and fn_moe_down_b run one pass per
 *   unique expert over all of its rows).
 */
Q4A_API q4a_status q4a_gemv_experts(float* y, const uint8_t* w_bank, const uint16_t* s_bank,
                            const uint16_t* b_bank, const uint16_t* x, const int32_t* x_rows,
                            const int32_t* expert_ids, const int32_t* token_offsets,
                            int n_active, int n_experts, int64_t n_rows, int64_t out_dim,
                            int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_experts_gate_up_silu -- q4a_gemv_experts over a bank of fused gate|up experts with
 * the activation in the epilogue ("BATCH_MSL", experts.metal fn_moe_gate_up_b followed by
 * fn_moe_act_b): expert e holds its gate rows at e*2*inter .. e*2*inter+inter-1 and its up
 * rows right after them, and for row r of segment a (expert e = expert_ids[a])
 *     h[r][i] = fp16( silu(g) * u ),  g = (W_e,gate . x_r)[i],  u = (W_e,up . x_r)[i]
 * with x_r = x[x_rows ? x_rows[r] : r]; no fp32 gate|up output exists.
 *   h              out   fp16 [n_rows][inter]
 *   w_bank         in    uint8 [n_experts*2*inter][in_dim/2]
 *   s_bank, b_bank in    bf16 [n_experts*2*inter][in_dim/64], 16-byte aligned
 *   x, x_rows, expert_ids, token_offsets, n_active, n_rows as q4a_gemv_experts.
 *   Requires inter % 16 == 0 and in_dim % 512 == 0 (the fused row blocks fetch the gate and
 *   up scales with 2D TMA boxes); other layouts return Q4A_ERR_UNSUPPORTED. A segment whose
 *   expert id lies outside [0, n_experts) produces NaN rows of h.
 */
Q4A_API q4a_status q4a_gemv_experts_gate_up_silu(uint16_t* h, const uint8_t* w_bank, const uint16_t* s_bank,
                                                 const uint16_t* b_bank, const uint16_t* x, const int32_t* x_rows,
                                                 const int32_t* expert_ids, const int32_t* token_offsets,
                                                 int n_active, int n_experts, int64_t n_rows, int64_t inter,
                                                 int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_experts_lowbit -- q4a_gemv_experts over derived low-bit codes, on binary16 or fp32
 * activations: the routed form of the 2/3-bit products ("BATCH_MSL", quantized_rows.metal
 * fn_q2_rows_h / fn_q3_rows_h for decode rows; expert_gemm.metal fn_expert_qmm, the low-bit
 * routed-expert contraction of prefill over 8/16/32-token tiles of fp32 rows). The weight of
 * code q is the quad midpoint s (4 q + 1.5) + b (bits = 2) or the pair midpoint
 * s (2 q + 0.5) + b (bits = 3, q = 2 * upper + lowest), as q4a_gemv_lowbit.
 *   w_up_bank, w_lo_bank  in  the bank's codes as q4a_lowbit_pack writes them:
 *                  [n_experts*out_dim][in_dim/4] and (bits 3) [n_experts*out_dim][in_dim/8]
 *   x              in  [*][in_dim], binary16 (x_is_f32 = 0) or fp32 (x_is_f32 != 0); fp32 rows are
 *                  rounded to binary16 when staged, as the pages' contraction rounds them to
 *                  half (|x| must stay within the binary16 range)
 *   everything else as q4a_gemv_experts (segments of up to 32 rows run as one tile, longer
 *   ones in 32-row pieces). bits = 3 needs in_dim % 128 == 0; bits other than 2 or 3 return
 *   Q4A_ERR_UNSUPPORTED.
 */
Q4A_API q4a_status q4a_gemv_experts_lowbit(float* y, int bits, const uint8_t* w_up_bank, const uint8_t* w_lo_bank,
                                           const uint16_t* s_bank, const uint16_t* b_bank, const void* x,
                                           int x_is_f32, const int32_t* x_rows, const int32_t* expert_ids,
                                           const int32_t* token_offsets, int n_active, int n_experts,
                                           int64_t n_rows, int64_t out_dim, int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_rmsnorm -- A3 + A4: RMSNorm prologue fused into the GEMV.
 *   x_raw   in  fp32 [nb][in_dim] un-normalised activations
 *   norm_w  in  bf16 [in_dim]
 *   The GEMV input is xn = fp16( x_raw * rsqrt(mean(x_raw^2) + eps) * (norm_w + shift) )
 *   per row (one normalisation group spanning the whole row), then y = W.xn as q4a_gemv.
 *   ("BATCH_MSL", hyperconnection.metal fn_group_norm_b; fn_norm_prep_b hands the
 *   GEMV an fp16 copy plus group sums of the normalised row.)
 *   Requires eps >= 0, x_raw 16-byte aligned, norm_w 16-byte aligned; otherwise as q4a_gemv.
 */
Q4A_API q4a_status q4a_gemv_rmsnorm(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                            const float* x_raw, const uint16_t* norm_w, float eps, float shift,
                            int nb, int64_t out_dim, int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_rmsnorm_grouped -- q4a_gemv_rmsnorm with norm_groups normalisation segments
 * per row ("BATCH_MSL", hyperconnection.metal fn_group_norm_b with groups > 1, the
 * multi-stream form of fn_norm_prep_b): with n = in_dim / norm_groups,
 *     xn[r][g*n + i] = fp16( x_raw[r][g*n + i] * rsqrt(mean_i x_raw[r][g*n + i]^2 + eps)
 *                            * (norm_w[g*n + i] + shift) ),   then y = W.xn.
 *   Requires 1 <= norm_groups <= 8 and in_dim % (64 * norm_groups) == 0; otherwise as
 *   q4a_gemv_rmsnorm (which is this call with norm_groups = 1).
 */
Q4A_API q4a_status q4a_gemv_rmsnorm_grouped(float* y, const uint8_t* w, const uint16_t* s,
                                    const uint16_t* b, const float* x_raw, const uint16_t* norm_w,
                                    float eps, float shift, int norm_groups, int nb, int64_t out_dim,
                                    int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_gemv_inject_rmsnorm_grouped -- q4a_gemv_rmsnorm_grouped whose prologue first injects a
 * layer output into every hyper-connection stream of the row ("BATCH_MSL",
 * hyperconnection.metal fn_inject_b, and fn_norm_prep_b with inject = 1): with
 * n = in_dim / norm_groups, stream g of row r is
 *     x'[r][g*n + i] = x_raw[r][g*n + i] + out[r][i] * 2 / (1 + e^(-logit[r][g] / norm_groups))
 * (fp32, one fused multiply-add), then xn = the grouped RMSNorm of x' and y = W.xn.
 *   y        out  fp32 [nb][out_dim]
 *   x_new    out  fp32 [nb][in_dim]: x', or NULL. It may not overlap x_raw or out (every CTA
 *                 cluster of the GEMV re-reads them; Q4A_ERR_SHAPE otherwise).
 *   x_raw    in   fp32 [nb][in_dim], the hyper-connection streams of each row
 *   out      in   fp32 [nb][n], the layer output injected into every stream
 *   logit    in   fp32 [nb][norm_groups], the per-stream mixing logits
 *   Requires out and x_new 16-byte aligned, logit 4-byte aligned; everything else as
 *   q4a_gemv_rmsnorm_grouped.
 */
Q4A_API q4a_status q4a_gemv_inject_rmsnorm_grouped(float* y, float* x_new, const uint8_t* w, const uint16_t* s,
                                                   const uint16_t* b, const float* x_raw, const float* out,
                                                   const float* logit, const uint16_t* norm_w, float eps,
                                                   float shift, int norm_groups, int nb, int64_t out_dim,
                                                   int64_t in_dim, q4a_stream_t stream);

/*
 * q4a_silu_mul_xsum -- A7: the step between the two routed-expert GEMVs.
 *   h        out  fp16 [rows][inter];  h[r][j] = fp16( silu(gate) * up ),
 *                 silu(v) = v / (1 + e^-v), gate = gate_up[r][j], up = gate_up[r][inter + j]
 *   hsum     out  fp32 [rows][inter/64] group sums of the fp16 h values (may be NULL)
 *   gate_up  in   fp32 [rows][2*inter]
 *   Requires rows >= 1, inter % 64 == 0, gate_up and h 16-byte aligned, hsum 4-byte aligned.
 *   ("BATCH_MSL", experts.metal fn_moe_act_b: sums of the fp16-rounded values.)
 */
Q4A_API q4a_status q4a_silu_mul_xsum(uint16_t* h, float* hsum, const float* gate_up, int64_t rows,
                             int64_t inter, q4a_stream_t stream);

/*
 * q4a_moe_combine -- the step after the routed-expert down projection: each token's
 * output row is the routing-weighted sum of its experts' rows, plus the shared expert's
 * row scaled by a sigmoid gate ("BATCH_MSL", experts.metal fn_moe_combine_b parts 0
 * and 1, fn_scatter_add_rows, fn_shared_add_rows):
 *     out[t][i] = sum_{k < top_k} w[t][k] * y[slot[t][k]][i]
 *               + sigmoid( sum_j gate[j] * x[t][j] ) * y_shared[t][i]   (if y_shared)
 *   out       out  fp32 [n_tok][hidden], fully overwritten
 *   y         in   fp32 [n_slots][hidden] expert output rows (q4a_gemv_experts' y)
 *   slot      in   int32 [n_tok][top_k] device array: row of y for token t's k-th expert
 *   w         in   fp32 [n_tok][top_k] device array: routing weights
 *   y_shared  in   fp32 [n_tok][hidden] shared-expert output, or NULL (no shared term;
 *                  gate and x are then ignored)
 *   gate      in   bf16 [hidden] shared-expert gate vector
 *   x         in   fp32 [n_tok][hidden] the input the gate reads
 *   The k terms are added in k order (deterministic). A slot outside [0, n_slots)
 *   makes that token's row NaN (a loud failure, never an out-of-bounds read).
 *   Requires n_tok >= 1, 1 <= top_k <= 64, hidden % 4 == 0; out, y, y_shared, x
 *   16-byte aligned, slot and w 4-byte aligned, gate 2-byte aligned.
 */
Q4A_API q4a_status q4a_moe_combine(float* out, const float* y, const int32_t* slot, const float* w,
                           int n_tok, int top_k, int64_t n_slots, int64_t hidden,
                           const float* y_shared, const uint16_t* gate, const float* x,
                           q4a_stream_t stream);

/*
 * q4a_gemv_kernel_choice -- which kernel q4a_gemv (and q4a_gemv_silu) would launch for these
 * arguments: 1 for the tensor-core path, 0 for the GEMV kernel (the rule under q4a_gemv).
 * Host-only: it launches nothing, touches no device memory and reads only the addresses of
 * s and b (their alignment). Invalid shapes return 0 (the call itself would reject them).
 */
Q4A_API int q4a_gemv_kernel_choice(const uint16_t* s, const uint16_t* b, int nb, int64_t out_dim, int64_t in_dim);

/*
 * q4a_debug_withhold_stage -- a hook for testing the failure path: the next launch of the
 * GEMV kernel made from this host thread (any q4a_gemv* entry point whose work runs there;
 * not the tensor-core path) never loads weight stage `stage` of each CTA (counted from 0), so
 * its consumer warps give up their bounded wait on it after about a second, finish the launch
 * with garbage outputs, and q4a_check_device_error then reports Q4A_ERR_TIMEOUT. The kernel
 * issues no copy after the give-up and waits for the copies it already issued before it
 * exits. stage = -1 clears a pending request. Returns Q4A_ERR_SHAPE for stage < -1.
 */
Q4A_API q4a_status q4a_debug_withhold_stage(int stage);

/*
 * q4a_check_device_error -- synchronise `stream`, then report and clear the
 * device error word: Q4A_ERR_TIMEOUT if a kernel of this library gave up a
 * bounded wait since the last check (its outputs are then garbage),
 * Q4A_ERR_CUDA if the synchronisation failed, Q4A_OK otherwise.
 */
Q4A_API q4a_status q4a_check_device_error(q4a_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4A_H */
