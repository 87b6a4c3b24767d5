// q4a_api.cu -- the C ABI of libq4a.so: argument validation, segment scheduling and
// dispatch to the kernels. Every check runs on the host before anything is launched.
#include <string.h>

#include <vector>

#include "q4a_internal.h"
#include "q4a_prefill.h"

namespace q4a {

static thread_local int t_last_cuda_error = 0;
static thread_local int t_withhold_stage = -1;

int take_withhold_stage() {
    const int v = t_withhold_stage;
    t_withhold_stage = -1;
    return v;
}

q4a_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return Q4A_ERR_CUDA;
}

q4a_status cuda_fail_drv(CUresult r) {
    t_last_cuda_error = (int)r;
    return Q4A_ERR_CUDA;
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

q4a_status check_matrix_shape(int64_t out_dim, int64_t in_dim) {
    if (out_dim < 1 || in_dim < kGroup || in_dim % kGroup != 0) return Q4A_ERR_SHAPE;
    if (out_dim > (int64_t)1 << 30 || in_dim > (int64_t)1 << 24) return Q4A_ERR_UNSUPPORTED;
    return Q4A_OK;
}

// Split an activation range into segments of at most 32 rows (the widest kernel variant).
void push_segments(std::vector<Segment>& out, int32_t row0, int64_t tok0, int64_t ntok) {
    for (int64_t t = 0; t < ntok; t += 32) {
        Segment s;
        s.row0 = row0;
        s.tok0 = (int32_t)(tok0 + t);
        s.ntok = (int32_t)(ntok - t < 32 ? ntok - t : 32);
        s.pad = 0;
        out.push_back(s);
    }
}

}  // namespace
}  // namespace q4a

using namespace q4a;

extern "C" {

const char* q4a_status_string(q4a_status status) {
    switch (status) {
        case Q4A_OK: return "ok";
        case Q4A_ERR_NULL: return "a required pointer is NULL";
        case Q4A_ERR_SHAPE: return "a size or an index table is out of range";
        case Q4A_ERR_ALIGN: return "a pointer misses its required alignment";
        case Q4A_ERR_UNSUPPORTED: return "valid but unsupported (device or size limit)";
        case Q4A_ERR_CUDA: return "a CUDA call failed";
        case Q4A_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    }
    return "unknown status";
}

int q4a_last_cuda_error(void) { return t_last_cuda_error; }

int q4a_gemv_kernel_choice(const uint16_t* s, const uint16_t* b, int nb, int64_t out_dim, int64_t in_dim) {
    if (!s || !b || nb < 1 || check_matrix_shape(out_dim, in_dim) != Q4A_OK) return 0;
    return dense_tc_eligible(s, b, nb, out_dim, in_dim) ? 1 : 0;
}

q4a_status q4a_debug_withhold_stage(int stage) {
    if (stage < -1) return Q4A_ERR_SHAPE;
    t_withhold_stage = stage;
    return Q4A_OK;
}

q4a_status q4a_pack(uint8_t* w_packed, const uint8_t* codes, int64_t rows, int64_t in_dim,
                    q4a_stream_t stream) {
    if (!w_packed || !codes) return Q4A_ERR_NULL;
    if (rows < 1 || in_dim < kGroup || in_dim % kGroup != 0) return Q4A_ERR_SHAPE;
    if (!aligned(w_packed, 16) || !aligned(codes, 16)) return Q4A_ERR_ALIGN;
    return launch_pack(w_packed, codes, rows, in_dim, (cudaStream_t)stream);
}

q4a_status q4a_lowbit_pack(uint8_t* w_up, uint8_t* w_lo, const uint8_t* w_packed, int64_t rows, int64_t in_dim,
                           q4a_stream_t stream) {
    if (!w_up || !w_packed) return Q4A_ERR_NULL;
    if (rows < 1 || in_dim < kGroup || in_dim % kGroup != 0) return Q4A_ERR_SHAPE;
    if (!aligned(w_packed, 16) || !aligned(w_up, 16) || (w_lo && !aligned(w_lo, 16))) return Q4A_ERR_ALIGN;
    return launch_lowbit_pack(w_up, w_lo, w_packed, rows, in_dim, (cudaStream_t)stream);
}

q4a_status q4a_quantize(uint8_t* w_packed, uint16_t* s, uint16_t* b, const float* w, int64_t rows, int64_t in_dim,
                        q4a_stream_t stream) {
    if (!w_packed || !s || !b || !w) return Q4A_ERR_NULL;
    if (rows < 1 || in_dim < kGroup || in_dim % kGroup != 0) return Q4A_ERR_SHAPE;
    if (!aligned(w_packed, 16) || !aligned(w, 16) || !aligned(s, 2) || !aligned(b, 2)) return Q4A_ERR_ALIGN;
    return launch_quantize(w_packed, s, b, w, rows, in_dim, (cudaStream_t)stream);
}

q4a_status q4a_gemv_f32x(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b, const float* x, int nb,
                         int64_t out_dim, int64_t in_dim, q4a_stream_t stream) {
    if (!y || !w || !s || !b || !x) return Q4A_ERR_NULL;
    if (nb < 1) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(out_dim, in_dim);
    if (st != Q4A_OK) return st;
    if ((int64_t)nb * out_dim > ((int64_t)1 << 36)) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(s, 2) || !aligned(b, 2) || !aligned(y, 4))
        return Q4A_ERR_ALIGN;
    return launch_gemv_f32x(y, w, s, b, x, nb, out_dim, in_dim, (cudaStream_t)stream);
}

q4a_status q4a_xsum(float* xsum, const uint16_t* x, int nb, int64_t in_dim, q4a_stream_t stream) {
    if (!xsum || !x) return Q4A_ERR_NULL;
    if (nb < 1 || in_dim < kGroup || in_dim % kGroup != 0) return Q4A_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(xsum, 4)) return Q4A_ERR_ALIGN;
    return launch_xsum(xsum, x, nb, in_dim, (cudaStream_t)stream);
}

}  // extern "C"

namespace q4a {
namespace {

q4a_status gemv_common(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b, const uint16_t* x,
                       int nb, int64_t out_dim, int64_t in_dim, bool silu, float silu_div, cudaStream_t stream) {
    if (!y || !w || !s || !b || !x) return Q4A_ERR_NULL;
    if (nb < 1) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(out_dim, in_dim);
    if (st != Q4A_OK) return st;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(s, 2) || !aligned(b, 2) || !aligned(y, 4))
        return Q4A_ERR_ALIGN;
    if (dense_tc_eligible(s, b, nb, out_dim, in_dim))
        return launch_dense_tc(w, s, b, x, y, nb, out_dim, in_dim, silu, silu_div, stream);
    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    if ((int)segs.size() > kDenseMaxSeg) return Q4A_ERR_UNSUPPORTED;
    GemvLaunch L = {};
    L.w = w;
    L.tensor_rows = out_dim;
    L.s = s;
    L.b = b;
    L.x = x;
    L.y = y;
    L.out_dim = out_dim;
    L.in_dim = in_dim;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = nb < 32 ? nb : 32;
    L.silu = silu;
    L.silu_div = silu_div;
    return launch_gemv(L, stream);
}

}  // namespace
}  // namespace q4a

extern "C" {

q4a_status q4a_gemv(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                    const uint16_t* x, int nb, int64_t out_dim, int64_t in_dim, q4a_stream_t stream) {
    return gemv_common(y, w, s, b, x, nb, out_dim, in_dim, false, 1.0f, (cudaStream_t)stream);
}

q4a_status q4a_gemv_lowbit(float* y, int bits, const uint8_t* w_up, const uint8_t* w_lo, const uint16_t* s,
                           const uint16_t* b, const uint16_t* x, int nb, int64_t out_dim, int64_t in_dim,
                           q4a_stream_t stream) {
    if (bits != 2 && bits != 3) return Q4A_ERR_UNSUPPORTED;
    if (!y || !w_up || !s || !b || !x || (bits == 3 && !w_lo)) return Q4A_ERR_NULL;
    if (nb < 1) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(out_dim, in_dim);
    if (st != Q4A_OK) return st;
    if (bits == 3 && in_dim % 128 != 0) return Q4A_ERR_SHAPE;   // lowest-bit rows: 16-byte multiples
    if (!aligned(w_up, 16) || (w_lo && !aligned(w_lo, 16)) || !aligned(x, 16) || !aligned(s, 2) ||
        !aligned(b, 2) || !aligned(y, 4))
        return Q4A_ERR_ALIGN;
    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    if ((int)segs.size() > kDenseMaxSeg) return Q4A_ERR_UNSUPPORTED;
    GemvLaunch L = {};
    L.w = w_up;
    L.w_lo = bits == 3 ? w_lo : nullptr;
    L.code_bits = bits;
    L.tensor_rows = out_dim;
    L.s = s;
    L.b = b;
    L.x = x;
    L.y = y;
    L.out_dim = out_dim;
    L.in_dim = in_dim;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = nb < 32 ? nb : 32;
    return launch_gemv(L, (cudaStream_t)stream);
}

q4a_status q4a_gemv_silu(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                         const uint16_t* x, float div, int nb, int64_t out_dim, int64_t in_dim,
                         q4a_stream_t stream) {
    if (!(div == div) || div == 0.0f || !(div - div == 0.0f)) return Q4A_ERR_SHAPE;   // finite, nonzero
    return gemv_common(y, w, s, b, x, nb, out_dim, in_dim, true, div, (cudaStream_t)stream);
}

q4a_status q4a_gemv_rmsnorm_grouped(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                                    const float* x_raw, const uint16_t* norm_w, float eps, float shift,
                                    int norm_groups, int nb, int64_t out_dim, int64_t in_dim,
                                    q4a_stream_t stream) {
    if (!y || !w || !s || !b || !x_raw || !norm_w) return Q4A_ERR_NULL;
    if (nb < 1 || !(eps >= 0.0f) || norm_groups < 1) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(out_dim, in_dim);
    if (st != Q4A_OK) return st;
    if (in_dim % ((int64_t)kGroup * norm_groups) != 0) return Q4A_ERR_SHAPE;
    if (nb > 32 || norm_groups > kMaxNormGroups) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x_raw, 16) || !aligned(norm_w, 16) || !aligned(s, 2) ||
        !aligned(b, 2) || !aligned(y, 4))
        return Q4A_ERR_ALIGN;
    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    GemvLaunch L = {};
    L.w = w;
    L.tensor_rows = out_dim;
    L.s = s;
    L.b = b;
    L.x = x_raw;
    L.norm_w = norm_w;
    L.eps = eps;
    L.shift = shift;
    L.y = y;
    L.out_dim = out_dim;
    L.in_dim = in_dim;
    L.rmsnorm = true;
    L.norm_groups = norm_groups;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = nb;
    return launch_gemv(L, (cudaStream_t)stream);
}

q4a_status q4a_gemv_inject_rmsnorm_grouped(float* y, float* x_new, const uint8_t* w, const uint16_t* s,
                                           const uint16_t* b, const float* x_raw, const float* out,
                                           const float* logit, const uint16_t* norm_w, float eps, float shift,
                                           int norm_groups, int nb, int64_t out_dim, int64_t in_dim,
                                           q4a_stream_t stream) {
    if (!y || !w || !s || !b || !x_raw || !out || !logit || !norm_w) return Q4A_ERR_NULL;
    if (nb < 1 || !(eps >= 0.0f) || norm_groups < 1) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(out_dim, in_dim);
    if (st != Q4A_OK) return st;
    if (in_dim % ((int64_t)kGroup * norm_groups) != 0) return Q4A_ERR_SHAPE;
    if (x_new) {
        // every cluster of the GEMV re-reads x_raw and out: the updated stream may not overlap them
        const uintptr_t xb = reinterpret_cast<uintptr_t>(x_new), xe = xb + (uintptr_t)(nb * in_dim * 4);
        const uintptr_t rb = reinterpret_cast<uintptr_t>(x_raw), re = rb + (uintptr_t)(nb * in_dim * 4);
        const uintptr_t ob = reinterpret_cast<uintptr_t>(out), oe = ob + (uintptr_t)(nb * (in_dim / norm_groups) * 4);
        if ((xb < re && rb < xe) || (xb < oe && ob < xe)) return Q4A_ERR_SHAPE;
    }
    if (nb > 32 || norm_groups > kMaxNormGroups) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x_raw, 16) || !aligned(norm_w, 16) || !aligned(out, 16) || !aligned(logit, 4) ||
        (x_new && !aligned(x_new, 16)) || !aligned(s, 2) || !aligned(b, 2) || !aligned(y, 4))
        return Q4A_ERR_ALIGN;
    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    GemvLaunch L = {};
    L.w = w;
    L.tensor_rows = out_dim;
    L.s = s;
    L.b = b;
    L.x = x_raw;
    L.norm_w = norm_w;
    L.eps = eps;
    L.shift = shift;
    L.y = y;
    L.out_dim = out_dim;
    L.in_dim = in_dim;
    L.rmsnorm = true;
    L.norm_groups = norm_groups;
    L.inj_out = out;
    L.inj_logit = logit;
    L.x_new = x_new;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = nb;
    return launch_gemv(L, (cudaStream_t)stream);
}

q4a_status q4a_gemv_gate_up_silu(uint16_t* h, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                                 const uint16_t* x, int nb, int64_t inter, int64_t in_dim, q4a_stream_t stream) {
    if (!h || !w || !s || !b || !x) return Q4A_ERR_NULL;
    if (nb < 1 || inter < 1 || inter % 16 != 0) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(2 * inter, in_dim);
    if (st != Q4A_OK) return st;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(s, 2) || !aligned(b, 2) || !aligned(h, 2))
        return Q4A_ERR_ALIGN;
    // the fused row blocks fetch the gate and up rows' scales with 2D TMA boxes only
    if (in_dim % 512 != 0 || !aligned(s, 16) || !aligned(b, 16)) return Q4A_ERR_UNSUPPORTED;
    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    if ((int)segs.size() > kDenseMaxSeg) return Q4A_ERR_UNSUPPORTED;
    GemvLaunch L = {};
    L.w = w;
    L.tensor_rows = 2 * inter;
    L.s = s;
    L.b = b;
    L.x = x;
    L.h = h;
    L.fused_gate_up = true;
    L.out_dim = inter;
    L.in_dim = in_dim;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = nb < 32 ? nb : 32;
    return launch_gemv(L, (cudaStream_t)stream);
}

q4a_status q4a_gemv_rmsnorm_gate_up_silu(uint16_t* h, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                                         const float* x_raw, const uint16_t* norm_w, float eps, float shift,
                                         int nb, int64_t inter, int64_t in_dim, q4a_stream_t stream) {
    if (!h || !w || !s || !b || !x_raw || !norm_w) return Q4A_ERR_NULL;
    if (nb < 1 || !(eps >= 0.0f) || inter < 1 || inter % 16 != 0) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(2 * inter, in_dim);
    if (st != Q4A_OK) return st;
    if (nb > 32) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x_raw, 16) || !aligned(norm_w, 16) || !aligned(s, 2) ||
        !aligned(b, 2) || !aligned(h, 2))
        return Q4A_ERR_ALIGN;
    if (in_dim % 512 != 0 || !aligned(s, 16) || !aligned(b, 16)) return Q4A_ERR_UNSUPPORTED;
    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    GemvLaunch L = {};
    L.w = w;
    L.tensor_rows = 2 * inter;
    L.s = s;
    L.b = b;
    L.x = x_raw;
    L.norm_w = norm_w;
    L.eps = eps;
    L.shift = shift;
    L.h = h;
    L.fused_gate_up = true;
    L.out_dim = inter;
    L.in_dim = in_dim;
    L.rmsnorm = true;
    L.norm_groups = 1;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = nb;
    return launch_gemv(L, (cudaStream_t)stream);
}

q4a_status q4a_decode_mlp(float* y, uint16_t* h, const uint8_t* w_gu, const uint16_t* s_gu, const uint16_t* b_gu,
                          const float* x_raw, const uint16_t* norm_w, float eps, float shift, const uint8_t* w_dn,
                          const uint16_t* s_dn, const uint16_t* b_dn, int nb, int64_t hidden, int64_t inter,
                          q4a_stream_t stream) {
    if (!y || !h || !w_gu || !s_gu || !b_gu || !x_raw || !norm_w || !w_dn || !s_dn || !b_dn) return Q4A_ERR_NULL;
    if (nb < 1 || !(eps >= 0.0f) || inter < kGroup || inter % kGroup != 0) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(2 * inter, hidden);
    if (st != Q4A_OK) return st;
    st = check_matrix_shape(hidden, inter);
    if (st != Q4A_OK) return st;
    if (nb > 32) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(w_gu, 16) || !aligned(x_raw, 16) || !aligned(norm_w, 16) || !aligned(s_gu, 2) ||
        !aligned(b_gu, 2) || !aligned(h, 16) || !aligned(w_dn, 16) || !aligned(s_dn, 2) || !aligned(b_dn, 2) ||
        !aligned(y, 4))
        return Q4A_ERR_ALIGN;
    if (hidden % 512 != 0 || !aligned(s_gu, 16) || !aligned(b_gu, 16)) return Q4A_ERR_UNSUPPORTED;

    std::vector<Segment> segs;
    push_segments(segs, 0, 0, nb);
    GemvLaunch gu = {};
    gu.w = w_gu;
    gu.tensor_rows = 2 * inter;
    gu.s = s_gu;
    gu.b = b_gu;
    gu.x = x_raw;
    gu.norm_w = norm_w;
    gu.eps = eps;
    gu.shift = shift;
    gu.h = h;
    gu.fused_gate_up = true;
    gu.out_dim = inter;
    gu.in_dim = hidden;
    gu.rmsnorm = true;
    gu.norm_groups = 1;
    gu.nseg = (int)segs.size();
    gu.seg = segs.data();
    gu.max_ntok = nb;

    GemvLaunch dn = {};
    dn.w = w_dn;
    dn.tensor_rows = hidden;
    dn.s = s_dn;
    dn.b = b_dn;
    dn.x = h;
    dn.y = y;
    dn.out_dim = hidden;
    dn.in_dim = inter;
    dn.nseg = gu.nseg;
    dn.seg = segs.data();
    dn.max_ntok = nb;
    // plan both launches before either is made: a rejected call launches nothing
    gu.plan_only = dn.plan_only = true;
    st = launch_gemv(gu, (cudaStream_t)stream);
    if (st != Q4A_OK) return st;
    st = launch_gemv(dn, (cudaStream_t)stream);
    if (st != Q4A_OK) return st;
    gu.plan_only = dn.plan_only = false;
    st = launch_gemv(gu, (cudaStream_t)stream);
    if (st != Q4A_OK) return st;
    return launch_gemv(dn, (cudaStream_t)stream);
}

q4a_status q4a_gemv_rmsnorm(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                            const float* x_raw, const uint16_t* norm_w, float eps, float shift,
                            int nb, int64_t out_dim, int64_t in_dim, q4a_stream_t stream) {
    return q4a_gemv_rmsnorm_grouped(y, w, s, b, x_raw, norm_w, eps, shift, 1, nb, out_dim, in_dim, stream);
}

}  // extern "C"

namespace q4a {
namespace {

// The routed-expert schedule shared by the 4-bit and the low-bit entry points: host checks of
// the segment table, NaN rows for out-of-range expert ids, one launch over every segment.
// y (fp32 [n_rows][out_dim]) or, with h set, the fused gate|up form: experts of 2 * out_dim rows
// (gate, then up) and h = fp16(silu(gate) * up) [n_rows][out_dim].
q4a_status experts_common(float* y, uint16_t* h, const uint8_t* w_bank, const uint8_t* w_lo_bank, int code_bits,
                          const uint16_t* s_bank, const uint16_t* b_bank, const void* x, bool x_f32,
                          const int32_t* x_rows, const int32_t* expert_ids, const int32_t* token_offsets,
                          int n_active, int n_experts, int64_t n_rows, int64_t out_dim, int64_t in_dim,
                          cudaStream_t stream) {
    const bool fg = h != nullptr;
    const int64_t rows_per_expert = fg ? 2 * out_dim : out_dim;
    if (n_active < 1 || n_active > Q4A_MAX_SEGMENTS || n_experts < 1 || n_rows < 1) return Q4A_ERR_SHAPE;
    if (fg && (out_dim < 16 || out_dim % 16 != 0)) return Q4A_ERR_SHAPE;
    q4a_status st = check_matrix_shape(rows_per_expert, in_dim);
    if (st != Q4A_OK) return st;
    if (code_bits == 3 && in_dim % 128 != 0) return Q4A_ERR_SHAPE;   // lowest-bit rows: 16-byte multiples
    if ((int64_t)n_experts * rows_per_expert > ((int64_t)1 << 31) - 16) return Q4A_ERR_UNSUPPORTED;
    if (n_rows > ((int64_t)1 << 31) - 1) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(w_bank, 16) || (w_lo_bank && !aligned(w_lo_bank, 16)) || !aligned(x, 16) || !aligned(s_bank, 2) ||
        !aligned(b_bank, 2) || (y && !aligned(y, 4)) || (fg && !aligned(h, 16)) || (x_rows && !aligned(x_rows, 4)))
        return Q4A_ERR_ALIGN;
    // the fused row blocks fetch the gate and up rows' scales with 2D TMA boxes only
    if (fg && (in_dim % 512 != 0 || !aligned(s_bank, 16) || !aligned(b_bank, 16))) return Q4A_ERR_UNSUPPORTED;
    if (token_offsets[0] != 0 || token_offsets[n_active] != n_rows) return Q4A_ERR_SHAPE;
    for (int a = 0; a < n_active; ++a)
        if (token_offsets[a + 1] < token_offsets[a]) return Q4A_ERR_SHAPE;

    std::vector<Segment> segs;
    std::vector<int> bad;
    for (int a = 0; a < n_active; ++a) {
        const int64_t n = token_offsets[a + 1] - token_offsets[a];
        if (n == 0) continue;
        const int32_t e = expert_ids[a];
        if (e < 0 || e >= n_experts) {
            bad.push_back(a);
            continue;
        }
        push_segments(segs, (int32_t)((int64_t)e * rows_per_expert), token_offsets[a], n);
    }
    if ((int)segs.size() > Q4A_MAX_SEGMENTS) return Q4A_ERR_UNSUPPORTED;
    int max_ntok = 0;
    for (const Segment& sg : segs) max_ntok = sg.ntok > max_ntok ? sg.ntok : max_ntok;
    GemvLaunch L = {};
    L.w = w_bank;
    L.w_lo = code_bits == 3 ? w_lo_bank : nullptr;
    L.code_bits = code_bits;
    L.tensor_rows = (int64_t)n_experts * rows_per_expert;
    L.s = s_bank;
    L.b = b_bank;
    L.x = x;
    L.x_f32 = x_f32;
    L.x_rows = x_rows;
    L.y = y;
    L.h = h;
    L.fused_gate_up = fg;
    L.out_dim = out_dim;
    L.in_dim = in_dim;
    L.experts = true;
    L.nseg = (int)segs.size();
    L.seg = segs.data();
    L.max_ntok = max_ntok;
    if (!segs.empty()) {   // plan before the first launch: a rejected call launches nothing
        L.plan_only = true;
        st = launch_gemv(L, stream);
        if (st != Q4A_OK) return st;
        L.plan_only = false;
    }
    for (int a : bad) {
        const int64_t r0 = token_offsets[a], nr = token_offsets[a + 1] - token_offsets[a];
        st = fg ? launch_fill_nan_h(h, r0, nr, out_dim, stream) : launch_fill_nan(y, r0, nr, out_dim, stream);
        if (st != Q4A_OK) return st;
    }
    if (segs.empty()) return Q4A_OK;
    return launch_gemv(L, stream);
}

}  // namespace
}  // namespace q4a

extern "C" {

q4a_status q4a_gemv_experts(float* y, const uint8_t* w_bank, const uint16_t* s_bank,
                            const uint16_t* b_bank, const uint16_t* x, const int32_t* x_rows,
                            const int32_t* expert_ids, const int32_t* token_offsets, int n_active,
                            int n_experts, int64_t n_rows, int64_t out_dim, int64_t in_dim,
                            q4a_stream_t stream) {
    if (!y || !w_bank || !s_bank || !b_bank || !x || !expert_ids || !token_offsets) return Q4A_ERR_NULL;
    return experts_common(y, nullptr, w_bank, nullptr, 4, s_bank, b_bank, x, false, x_rows, expert_ids, token_offsets,
                          n_active, n_experts, n_rows, out_dim, in_dim, (cudaStream_t)stream);
}

q4a_status q4a_gemv_experts_gate_up_silu(uint16_t* h, const uint8_t* w_bank, const uint16_t* s_bank,
                                         const uint16_t* b_bank, const uint16_t* x, const int32_t* x_rows,
                                         const int32_t* expert_ids, const int32_t* token_offsets, int n_active,
                                         int n_experts, int64_t n_rows, int64_t inter, int64_t in_dim,
                                         q4a_stream_t stream) {
    if (!h || !w_bank || !s_bank || !b_bank || !x || !expert_ids || !token_offsets) return Q4A_ERR_NULL;
    return experts_common(nullptr, h, w_bank, nullptr, 4, s_bank, b_bank, x, false, x_rows, expert_ids, token_offsets,
                          n_active, n_experts, n_rows, inter, in_dim, (cudaStream_t)stream);
}

q4a_status q4a_gemv_experts_lowbit(float* y, int bits, const uint8_t* w_up_bank, const uint8_t* w_lo_bank,
                                   const uint16_t* s_bank, const uint16_t* b_bank, const void* x, int x_is_f32,
                                   const int32_t* x_rows, const int32_t* expert_ids, const int32_t* token_offsets,
                                   int n_active, int n_experts, int64_t n_rows, int64_t out_dim, int64_t in_dim,
                                   q4a_stream_t stream) {
    if (bits != 2 && bits != 3) return Q4A_ERR_UNSUPPORTED;
    if (!y || !w_up_bank || !s_bank || !b_bank || !x || !expert_ids || !token_offsets || (bits == 3 && !w_lo_bank))
        return Q4A_ERR_NULL;
    return experts_common(y, nullptr, w_up_bank, bits == 3 ? w_lo_bank : nullptr, bits, s_bank, b_bank, x, x_is_f32 != 0,
                          x_rows, expert_ids, token_offsets, n_active, n_experts, n_rows, out_dim, in_dim,
                          (cudaStream_t)stream);
}

q4a_status q4a_silu_mul_xsum(uint16_t* h, float* hsum, const float* gate_up, int64_t rows,
                             int64_t inter, q4a_stream_t stream) {
    if (!h || !gate_up) return Q4A_ERR_NULL;
    if (rows < 1 || inter < kGroup || inter % kGroup != 0) return Q4A_ERR_SHAPE;
    if (!aligned(h, 16) || !aligned(gate_up, 16) || (hsum && !aligned(hsum, 4))) return Q4A_ERR_ALIGN;
    return launch_silu_mul_xsum(h, hsum, gate_up, rows, inter, (cudaStream_t)stream);
}

q4a_status q4a_moe_combine(float* out, const float* y, const int32_t* slot, const float* w, int n_tok,
                           int top_k, int64_t n_slots, int64_t hidden, const float* y_shared,
                           const uint16_t* gate, const float* x, q4a_stream_t stream) {
    if (!out || !y || !slot || !w) return Q4A_ERR_NULL;
    if (y_shared && (!gate || !x)) return Q4A_ERR_NULL;
    if (n_tok < 1 || top_k < 1 || n_slots < 1 || hidden < 4 || hidden % 4 != 0) return Q4A_ERR_SHAPE;
    if (top_k > kCombineMaxK || n_slots > ((int64_t)1 << 31) - 1) return Q4A_ERR_UNSUPPORTED;
    if ((int64_t)n_tok * ((hidden + 1023) / 1024) > ((int64_t)1 << 31) - 1) return Q4A_ERR_UNSUPPORTED;
    if (!aligned(out, 16) || !aligned(y, 16) || !aligned(slot, 4) || !aligned(w, 4) ||
        (y_shared && (!aligned(y_shared, 16) || !aligned(x, 16) || !aligned(gate, 2))))
        return Q4A_ERR_ALIGN;
    return launch_moe_combine(out, y, slot, w, n_tok, top_k, n_slots, hidden, y_shared, y_shared ? gate : nullptr,
                              y_shared ? x : nullptr, (cudaStream_t)stream);
}

q4a_status q4a_check_device_error(q4a_stream_t stream) {
    uint32_t word = 0;
    q4a_status st = read_and_clear_device_error((cudaStream_t)stream, &word);
    if (st != Q4A_OK) return st;
    uint32_t word_tc = 0;
    st = read_and_clear_dense_tc_error(&word_tc);
    if (st != Q4A_OK) return st;
    return (word | word_tc) ? Q4A_ERR_TIMEOUT : Q4A_OK;
}

}  // extern "C"
