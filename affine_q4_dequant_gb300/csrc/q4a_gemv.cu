// q4a_gemv.cu -- the row-batched affine-4-bit dequantising GEMV on sm_103a.
//
// Operation (restated from the "BATCH_MSL" constant page, quantized_rows.metal,
// fn_q4_rows_h / fn_q4_2rows_h): for every output row o and activation row r,
//     y[r][o] = sum_g ( s[o][g] * sum_{i in g} q[o][i] x[r][i] + b[o][g] * xsum[r][g] ).
//
// GB300 design (not the pages' Metal design):
//  * One CTA per SM: 1 producer warp + 8 consumer warps. The producer streams the
//    packed weights with 2D TMA boxes (16 rows x 128 bytes, 128-byte swizzle) and
//    the bf16 scale/bias rows with cp.async into a ring of shared-memory stages
//    guarded by mbarriers (full: TMA bytes + copy arrivals; empty: consumer warps).
//  * A thread-block cluster of C CTAs splits the input dimension K; every CTA of
//    the cluster owns the same output rows and one K-slice. Each CTA stages its
//    K-slice of the activations once, as ready-made mma B fragments plus fp32
//    group sums, and reuses them for all of its rows. Partial sums meet through
//    distributed shared memory; the reduction order is fixed (deterministic).
//  * Consumer warp wg takes group wg of every 8-group stage, for every 16-row tile
//    of the row block (several independent tiles per warp hide the mma and
//    shared-memory latencies). Per 16-row tile and group it runs 4 steps of
//    mma.sync m16n8k16 (f16 in, f32 accumulate) per 8 activation rows: the A
//    operand is the raw codes, pulled out of each 32-bit word by masks into
//    binary16 subnormals (code * 2^-24, exact); the high nibble of a byte lands
//    at 16x and the matching activations are pre-scaled by 1/16. A dot product
//    does not depend on the order of its terms, so every thread feeds the words
//    ldmatrix gives it and the activation fragments carry the same permutation.
//    The per-group result is scaled by s (times 2^24) and b*xsum is added, both
//    in fp32: the tensor cores never see a rounded weight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <stdio.h>
#include <stdlib.h>

#include <string.h>

#include <map>
#include <mutex>
#include <string>
#include <unordered_map>

#include "q4a_device.cuh"
#include "q4a_internal.h"

namespace q4a {
namespace {

// ---- PTX wrappers ----------------------------------------------------------------

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}



__device__ __forceinline__ float half2_sum(uint32_t h2) {
    const __half2 v = *reinterpret_cast<const __half2*>(&h2);
    return __low2float(v) + __high2float(v);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// ---- the job sequence (identical in the producer and the consumers) -------------------

struct Job {
    int seg;      // segment index
    int tile;     // first tile of the block within the segment
    int ntile;    // tiles in this row block (1 .. mt)
};

template <class P>
__device__ __forceinline__ bool next_job(const P& p, int& t, int t_end, Job& j) {
    if (t >= t_end) return false;
    const int seg = t / p.tiles_per_seg;
    const int tile = t - seg * p.tiles_per_seg;
    int n = p.tiles_per_seg - tile;
    if (n > t_end - t) n = t_end - t;
    if (n > p.mt) n = p.mt;
    j.seg = seg;
    j.tile = tile;
    j.ntile = n;
    t += n;
    return true;
}

// This CTA's share of one op: its K-slice (in groups), the stages per row block and its
// cluster's range of schedule units.
struct OpRange {
    int kg0, kg1, gsz, nks, t_begin, t_end;
};

__device__ __forceinline__ OpRange op_range(const GemvOp& o, int crank, int cid, int n_clusters) {
    OpRange r;
    r.kg0 = crank * o.gs;
    r.kg1 = min(o.groups, r.kg0 + o.gs);
    r.gsz = r.kg1 - r.kg0;
    r.nks = (r.gsz + kStageGroups - 1) / kStageGroups;
    r.t_begin = (int)(((int64_t)cid * o.n_tiles) / n_clusters);
    r.t_end = (int)(((int64_t)(cid + 1) * o.n_tiles) / n_clusters);
    return r;
}

// The injection weight of stream g of activation row slot: 2 sigmoid(logit / streams)
// ("BATCH_MSL" hyperconnection.metal fn_inject_b, fn_norm_prep_b with inject = 1).
template <class P>
__device__ __forceinline__ float inject_weight(const P& p, int64_t slot, int g) {
    return 2.0f / (1.0f + expf(-p.inj_logit[slot * p.norm_groups + g] / (float)p.norm_groups));
}

// ---- activation staging -----------------------------------------------------------------

// Writes the CTA's K-slice of the activation rows of one segment as mma B fragments
// (xfrag) and fp32 group sums (xsum). Item (tok, gl, t) covers elements 8t..8t+7 and
// 32+8t..32+8t+7 of group gl for activation row tok; the four t of an item sit in one
// lane quad, which sums its group. Each batch issues all of its global loads before
// any arithmetic, so the staging costs about one memory latency per batch.
//
// Derived low-bit codes (CB = 2 or 3) pair lane quad t with the 16 consecutive inputs
// 16t..16t+15 of a group (the 2-bit word t of the group's 16 bytes holds exactly those), and
// step j with the inputs whose codes sit in bit field j of the word's bytes: the even inputs
// 16t + {0,2,4,6} (j = 0) and 16t + {8,10,12,14} (j = 1), the odd ones after them (j = 2, 3);
// field j is read in place (value 4^j * code), so step j's activations are scaled by 4^-j.
// XF: the activations are fp32 (prefill); staging rounds them to binary16, the operand type of
// the mma, as the pages' prefill contraction does (it rounds its fp32 rows to half).
template <int NT, bool RMS, int CB, bool XF, bool INJ, class P>
__device__ void stage_x_t(const P& p, const Segment& sg, int kg0, int gsz, uint8_t* xfrag,
                          float* xsum_s, const float* inv_s, int ctid, bool write_xnew) {
    static_assert(CB == 4 || !RMS, "the RMSNorm prologue is built for 4-bit codes only");
    static_assert(!(RMS && XF), "the RMSNorm prologue reads fp32 rows itself");
    constexpr int NTOK = NT * 8;
    constexpr int BATCH = RMS ? 2 : 4;
    constexpr int NLD = RMS ? (INJ ? 10 : 6) : (XF ? 4 : 2);   // RMSNorm: x (4), norm weight (2), injected output (4)
    constexpr int NTH = kConsumerWarps * 32;
    const int items = sg.ntok * gsz * 4;
    const int ntm = p.ntok_max;
    const uint32_t scale_odd = 0x2C002C00u;   // half2(1/16, 1/16)
    constexpr bool inj = RMS && INJ;   // injection code only in the kernels built for it
    for (int base = 0; base < items; base += BATCH * NTH) {
        // phase 1: loads
        uint4 ld[BATCH][NLD];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int i = base + k * NTH + ctid;
            const int rest = i >> 2;
            const int gl = rest % gsz;
            const int tok = rest / gsz;
            const bool on = i < items;
#pragma unroll
            for (int q = 0; q < NLD; ++q) ld[k][q] = make_uint4(0, 0, 0, 0);
            if (on) {
                const int slot = sg.tok0 + tok;
                const int64_t src = p.x_rows ? (int64_t)p.x_rows[slot] : (int64_t)slot;
                const int64_t col = (int64_t)(kg0 + gl) * kGroup + (CB == 4 ? 8 : 16) * (i & 3);
                if constexpr (!RMS && XF) {
                    // fp32: the item's two runs of 8 inputs, 16 bytes at a time
                    const float* xr = static_cast<const float*>(p.x) + src * p.in_dim + col;
                    ld[k][0] = ld_nc_16(xr);
                    ld[k][1] = ld_nc_16(xr + 4);
                    ld[k][2] = ld_nc_16(xr + (CB == 4 ? 32 : 8));
                    ld[k][3] = ld_nc_16(xr + (CB == 4 ? 36 : 12));
                } else if constexpr (!RMS) {
                    const __half* xr = static_cast<const __half*>(p.x) + src * p.in_dim + col;
                    ld[k][0] = ld_nc_16(xr);
                    ld[k][1] = ld_nc_16(xr + (CB == 4 ? 32 : 8));
                } else {
                    const float* xr = static_cast<const float*>(p.x) + src * p.in_dim + col;
                    ld[k][0] = ld_nc_16(xr);
                    ld[k][1] = ld_nc_16(xr + 4);
                    ld[k][2] = ld_nc_16(xr + 32);
                    ld[k][3] = ld_nc_16(xr + 36);
                    ld[k][4] = ld_nc_16(p.norm_w + col);
                    ld[k][5] = ld_nc_16(p.norm_w + col + 32);
                    if constexpr (inj) {
                        // the item's 16 inputs lie in one 64-group, hence in one stream
                        const int64_t seg = col / p.norm_width;
                        const float* orow = p.inj_out + src * p.norm_width + (col - seg * p.norm_width);
                        ld[k][6] = ld_nc_16(orow);
                        ld[k][7] = ld_nc_16(orow + 4);
                        ld[k][8] = ld_nc_16(orow + 32);
                        ld[k][9] = ld_nc_16(orow + 36);
                    }
                }
            }
        }
        // phase 2: fragments, sums, stores
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int i = base + k * NTH + ctid;
            const bool live = i < items;
            const int t = i & 3;
            const int rest = i >> 2;
            const int gl = rest % gsz;
            const int tok = rest / gsz;
            uint32_t v[4], u[4];
            if constexpr (!RMS && XF) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint4 f0 = ld[k][2 * half], f1 = ld[k][2 * half + 1];
                    const uint32_t xs[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                    uint32_t* dst = half ? u : v;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        __half2 h = __floats2half2_rn(__uint_as_float(xs[2 * q]), __uint_as_float(xs[2 * q + 1]));
                        dst[q] = *reinterpret_cast<uint32_t*>(&h);
                    }
                }
            } else if constexpr (!RMS) {
                v[0] = ld[k][0].x; v[1] = ld[k][0].y; v[2] = ld[k][0].z; v[3] = ld[k][0].w;
                u[0] = ld[k][1].x; u[1] = ld[k][1].y; u[2] = ld[k][1].z; u[3] = ld[k][1].w;
            } else {
                // the item's 16 inputs lie in one 64-group, hence in one normalisation segment
                const int seg = (int)(((int64_t)(kg0 + gl) * kGroup) / p.norm_width);
                const float inv = live ? inv_s[tok * p.norm_groups + seg] : 0.f;
                const int64_t slot = sg.tok0 + tok;
                const float wgt = inj && live ? inject_weight(p, slot, seg) : 0.f;
                float* xn_row = inj && write_xnew && live ? p.x_new + slot * p.in_dim + (int64_t)(kg0 + gl) * kGroup + 8 * t
                                                   : nullptr;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint4 f0 = ld[k][2 * half], f1 = ld[k][2 * half + 1], wv = ld[k][4 + half];

                    float xs[8] = {__uint_as_float(f0.x), __uint_as_float(f0.y), __uint_as_float(f0.z),
                                   __uint_as_float(f0.w), __uint_as_float(f1.x), __uint_as_float(f1.y),
                                   __uint_as_float(f1.z), __uint_as_float(f1.w)};
                    if constexpr (inj) {
                        const uint4 o0 = ld[k][6 + 2 * half], o1 = ld[k][7 + 2 * half];
                        const uint32_t os[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) xs[e] = fmaf(__uint_as_float(os[e]), wgt, xs[e]);
                        if (xn_row) {
                            *reinterpret_cast<float4*>(xn_row + 32 * half) = make_float4(xs[0], xs[1], xs[2], xs[3]);
                            *reinterpret_cast<float4*>(xn_row + 32 * half + 4) = make_float4(xs[4], xs[5], xs[6], xs[7]);
                        }
                    }
                    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
                    uint32_t* dst = half ? u : v;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float w0 = bf16_to_f32(ww[q] & 0xFFFFu) + p.shift;
                        const float w1 = bf16_to_f32(ww[q] >> 16) + p.shift;
                        __half2 h = __floats2half2_rn(xs[2 * q] * inv * w0, xs[2 * q + 1] * inv * w1);
                        dst[q] = *reinterpret_cast<uint32_t*>(&h);
                    }
                }
            }
            float part = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) part += half2_sum(v[q]) + half2_sum(u[q]);
            if constexpr (CB != 4) {
                // v: inputs 16t + 0..7, u: 16t + 8..15 (pairs). Step j, fragment b0 = k-low
                // (code bytes 0 and 2), b1 = k-high (bytes 1 and 3).
                const uint32_t sc1 = 0x34003400u, sc2 = 0x2C002C00u, sc3 = 0x24002400u;   // 4^-1, 4^-2, 4^-3
                uint32_t bfr[8];
                bfr[0] = __byte_perm(v[0], v[2], 0x5410);                     // j0: x0, x4
                bfr[1] = __byte_perm(v[1], v[3], 0x5410);                     //     x2, x6
                bfr[2] = hmul2_u32(__byte_perm(u[0], u[2], 0x5410), sc1);     // j1: x8, x12
                bfr[3] = hmul2_u32(__byte_perm(u[1], u[3], 0x5410), sc1);     //     x10, x14
                bfr[4] = hmul2_u32(__byte_perm(v[0], v[2], 0x7632), sc2);     // j2: x1, x5
                bfr[5] = hmul2_u32(__byte_perm(v[1], v[3], 0x7632), sc2);     //     x3, x7
                bfr[6] = hmul2_u32(__byte_perm(u[0], u[2], 0x7632), sc3);     // j3: x9, x13
                bfr[7] = hmul2_u32(__byte_perm(u[1], u[3], 0x7632), sc3);     //     x11, x15
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                if (live) {
                    uint8_t* f = xfrag + ((size_t)(gl * 2) * ntm + tok) * 64 + t * 16;
                    *reinterpret_cast<uint4*>(f) = make_uint4(bfr[0], bfr[1], bfr[2], bfr[3]);
                    *reinterpret_cast<uint4*>(f + (size_t)ntm * 64) = make_uint4(bfr[4], bfr[5], bfr[6], bfr[7]);
                    if (t == 0) xsum_s[gl * NTOK + tok] = part * 5.9604644775390625e-08f;
                }
                continue;
            }
            // B fragments for the 4 mma steps: step j pairs element j with j+4 (v: word t,
            // u: word t+4). Odd steps come from the high nibbles (16x) -> scale by 1/16.
            uint32_t b01[4], b23[4];
            b01[0] = __byte_perm(v[0], v[2], 0x5410);
            b01[1] = hmul2_u32(__byte_perm(v[0], v[2], 0x7632), scale_odd);
            b01[2] = __byte_perm(v[1], v[3], 0x5410);
            b01[3] = hmul2_u32(__byte_perm(v[1], v[3], 0x7632), scale_odd);
            b23[0] = __byte_perm(u[0], u[2], 0x5410);
            b23[1] = hmul2_u32(__byte_perm(u[0], u[2], 0x7632), scale_odd);
            b23[2] = __byte_perm(u[1], u[3], 0x5410);
            b23[3] = hmul2_u32(__byte_perm(u[1], u[3], 0x7632), scale_odd);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            if (live) {
                uint8_t* f = xfrag + ((size_t)(gl * 2) * ntm + tok) * 64 + t * 16;
                *reinterpret_cast<uint4*>(f) = make_uint4(b01[0], b23[0], b01[1], b23[1]);
                *reinterpret_cast<uint4*>(f + (size_t)ntm * 64) = make_uint4(b01[2], b23[2], b01[3], b23[3]);
                // kept in units of 2^-24, the scale of the mma partial sums (see the epilogue)
                if (t == 0) xsum_s[gl * NTOK + tok] = part * 5.9604644775390625e-08f;
            }
        }
    }
}

// Staging of one op's activations: the RMSNorm form when the op asks for it (kernels built
// with RMS), the plain fp16 form otherwise.
template <int NT, bool RMS, int CB, bool XF, bool INJ, class P>
__device__ __forceinline__ void stage_x(const P& p, bool rms, const Segment& sg, int kg0, int gsz, uint8_t* xfrag,
                                        float* xsum_s, const float* inv_s, int ctid, bool write_xnew) {
    if constexpr (RMS) {
        if (rms) {
            stage_x_t<NT, true, CB, false, INJ>(p, sg, kg0, gsz, xfrag, xsum_s, inv_s, ctid, write_xnew);
            return;
        }
    }
    stage_x_t<NT, false, CB, XF, false>(p, sg, kg0, gsz, xfrag, xsum_s, inv_s, ctid, false);
}

// B fragments of the bias term sum_g b[o][g] * xsum[r][g], an m16n8k16 contraction over
// groups (bf16 operands): per 16-group block, activation row tok and lane quad t, the
// pairs of groups (2t, 2t+1) and (2t+8, 2t+9) of xsum (already times 2^-24), split into
// a bf16 high part and a bf16 remainder, so that hi + lo carries ~16 bits.
__device__ void stage_xbias(const float* xsum_s, int ntok_seg, int ntok_max, int ntok_stride, int gsz,
                            uint8_t* xbias, int ctid) {
    const int nblk = (gsz + 15) / 16;
    const int items = nblk * ntok_seg * 4;
    for (int i = ctid; i < items; i += kConsumerWarps * 32) {
        const int t = i & 3;
        const int rest = i >> 2;
        const int tok = rest % ntok_seg;
        const int gb = rest / ntok_seg;
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            float v[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int gl = gb * 16 + 2 * t + 8 * pr + e;
                v[e] = gl < gsz ? xsum_s[gl * ntok_stride + tok] : 0.f;
            }
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[0], v[1]);
            const float2 hf = __bfloat1622float2(h);
            const __nv_bfloat162 l = __floats2bfloat162_rn(v[0] - hf.x, v[1] - hf.y);
            hi[pr] = *reinterpret_cast<const uint32_t*>(&h);
            lo[pr] = *reinterpret_cast<const uint32_t*>(&l);
        }
        *reinterpret_cast<uint4*>(xbias + ((size_t)gb * ntok_max + tok) * 64 + t * 16) = make_uint4(hi[0], hi[1], lo[0], lo[1]);
    }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Sum of squares of this CTA's K-slice of every activation row (the RMSNorm prologue), per
// normalisation segment of the row (ssq_s[tok * G + seg]; segments outside the slice get 0).
// Work units are (row, segment, part): with fewer rows than consumer warps every row is split
// into parts so that all warps load at once (one memory round trip at NB 1); each lane keeps
// 16 independent 16-byte loads in flight. The parts' sums meet in `red` in a fixed order.
template <int NT, bool INJ, class P>
__device__ void rms_partial(const P& p, const Segment& sg, int kg0, int gsz, float* ssq_s, float* red, int warp,
                            int lane, int ctid) {
    constexpr int NTOK = NT * 8;
    constexpr int U = 16;
    const int G = p.norm_groups;
    constexpr bool inj = INJ;
    const int ntok = sg.ntok;
    const int parts = ntok >= kConsumerWarps ? 1 : kConsumerWarps / ntok;
    const int units = ntok * G * parts;
    const int64_t k_lo = (int64_t)kg0 * kGroup, k_hi = k_lo + (int64_t)gsz * kGroup;
    for (int u = warp; u < units; u += kConsumerWarps) {
        const int part = u % parts;
        const int seg = (u / parts) % G;
        const int tok = u / parts / G;
        const int64_t s_lo = llmax(k_lo, (int64_t)seg * p.norm_width);
        const int64_t s_hi = llmin(k_hi, (int64_t)(seg + 1) * p.norm_width);
        float acc = 0.f;
        if (s_lo < s_hi) {
            const int64_t slot = sg.tok0 + tok;
            const float4* xr = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + slot * p.in_dim + s_lo);
            // injection: the stream's inputs plus out[slot][i] * weight, i = column - seg * width
            const float4* orow = inj ? reinterpret_cast<const float4*>(p.inj_out + slot * p.norm_width +
                                                                        (s_lo - (int64_t)seg * p.norm_width))
                                     : nullptr;
            const float wgt = inj ? inject_weight(p, slot, seg) : 0.f;
            const int chunks = (int)((s_hi - s_lo) / 4);   // float4 chunks of this segment's part
            const int c_lo = (int)((int64_t)chunks * part / parts), c_hi = (int)((int64_t)chunks * (part + 1) / parts);
            for (int c0 = c_lo; c0 < c_hi; c0 += 32 * U) {
                float4 f[U];
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const int c = c0 + k * 32 + lane;
                    f[k] = c < c_hi ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if constexpr (inj) {
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const int c = c0 + k * 32 + lane;
                        const float4 o = c < c_hi ? __ldg(orow + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                        f[k].x = fmaf(o.x, wgt, f[k].x);
                        f[k].y = fmaf(o.y, wgt, f[k].y);
                        f[k].z = fmaf(o.z, wgt, f[k].z);
                        f[k].w = fmaf(o.w, wgt, f[k].w);
                    }
                }
#pragma unroll
                for (int k = 0; k < U; ++k)
                    acc += f[k].x * f[k].x + f[k].y * f[k].y + f[k].z * f[k].z + f[k].w * f[k].w;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) red[u] = acc;
    }
    consumer_sync();
    for (int e = ctid; e < NTOK * G; e += kConsumerWarps * 32) {
        const int tok = e / G;
        float tot = 0.f;
        if (tok < ntok)
            for (int q = 0; q < parts; ++q) tot += red[e * parts + q];
        ssq_s[e] = tot;
    }
}

// ---- the producer's once-per-row-block paths, out of line ------------------------------
// A launch starts with a cold instruction cache, and a GEMV kernel carries code for several
// scale/bias fetch modes of which one runs: keeping these paths out of line keeps the code a
// launch actually fetches small (the stage loop and the consumers' mma loop stay inline).

// Raw mode: 1D boxes over the contiguous [rows][groups] scales and biases of a row block into
// a raw staging buffer. The first element is rounded down to a 16-byte boundary (TMA rule);
// the consumers' transform skips the difference.
__device__ __noinline__ void raw_issue(const GemvOp& p, const Segment& sgb, int tile, int ntile, uint8_t* dst,
                                      uint32_t raw_elems, uint32_t bar) {
    const int64_t r0 = (int64_t)sgb.row0 + (int64_t)tile * 16;
    const int rv = (int)llmin((int64_t)ntile * 16, p.out_dim - (int64_t)tile * 16);
    const int64_t e0 = r0 * p.groups;
    const int64_t e0a = e0 & ~(int64_t)7;
    const int nbx = (int)((e0 - e0a + (int64_t)rv * p.groups + kRawBox - 1) / kRawBox);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after the last transform's reads
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * nbx * kRawBox * 2));
#pragma unroll 1
    for (int k = 0; k < nbx; ++k) {
        tma_load_1d(smem_addr(dst + k * kRawBox * 2), &p.tmap_s1, (int)(e0a + (int64_t)k * kRawBox), bar);
        tma_load_1d(smem_addr(dst + raw_elems * 2u + k * kRawBox * 2), &p.tmap_b1, (int)(e0a + (int64_t)k * kRawBox),
                    bar);
    }
}

// 2D-TMA mode: one box per 64-group chunk of the K-slice and per part (fused: gate rows, up
// rows), as tall as the row block.
__device__ __noinline__ void sb_tma_issue(const GemvOp& p, uint8_t* sdst, uint32_t bar, int64_t trow0, int kg0,
                                         int gsz, int ntile, int parts, int half_mt) {
    const int nchunk = (gsz + 63) / 64;
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * parts * nchunk * ntile * kTileBytes));
    const int mi = ntile - 1;
#pragma unroll 1
    for (int part = 0; part < parts; ++part) {
        const int64_t prow = trow0 + (part ? p.out_dim : 0);
        const int mbase = part * half_mt;
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
            const uint32_t o = (uint32_t)((c * p.sb_tiles + mbase) * kTileBytes);
            tma_load_2d(smem_addr(sdst + o), &p.tmap_s[mi], kg0 + 64 * c, (int)prow, bar);
            tma_load_2d(smem_addr(sdst + p.sb_pitch + o), &p.tmap_b[mi], kg0 + 64 * c, (int)prow, bar);
        }
    }
}

// Element-copy mode (anything TMA cannot fetch; full K): the producer lanes copy the row
// block's scales and biases into the swizzled layout; groups up to the next 16-group block are
// zeroed for the bias contraction.
__device__ __noinline__ void sb_plain_copy(const GemvOp& p, uint8_t* sdst, int64_t trow0, int rows_valid, int kg0,
                                          int gsz, int lane) {
    const uint8_t* s8 = reinterpret_cast<const uint8_t*>(p.s);
    const uint8_t* b8 = reinterpret_cast<const uint8_t*>(p.b);
    const int64_t srow_bytes = (int64_t)p.groups * 2;
    const int gpad = (gsz + 15) / 16 * 16;
    const int n = 2 * rows_valid * gpad;
#pragma unroll 1
    for (int i = lane; i < n; i += 32) {
        const int k = i % gpad;
        const int rr = i / gpad;
        const int isb = rr >= rows_valid;
        const int r = rr - isb * rows_valid;
        uint16_t v = 0;
        if (k < gsz)
            v = *reinterpret_cast<const uint16_t*>((isb ? b8 : s8) + (trow0 + r) * srow_bytes + (int64_t)(kg0 + k) * 2);
        const uint32_t o = (uint32_t)(((k >> 6) * p.sb_tiles * 16 + r) * 128) +
                           ((uint32_t)(((k >> 3) & 7) ^ (r & 7)) << 4) + 2u * (k & 7);
        *reinterpret_cast<uint16_t*>(sdst + (size_t)isb * p.sb_pitch + o) = v;
    }
}

// Before the CTA exits, lane 0 waits for every copy it issued and no consumer waited for
// (after an abort): the last `S` ring stages (bit k of st_bits: stage it - 1 - k), the last
// `nsb` scale/bias fetches and the raw buffers' latest fills.
template <int kRawBufs>
__device__ __noinline__ void drain_copies(const uint64_t* full_b, int S, int it, uint32_t st_bits, const uint64_t* sbfull_b,
                                         int nsb, int blk, uint32_t sb_bits, const uint64_t* rawfull_b,
                                         int raw_rb0, int raw_rb1, int raw_rb2) {
    int slot = (it - 1) % S, round = (it - 1) / S;
#pragma unroll 1
    for (int k = 0; k < S && k < it; ++k) {
        if ((st_bits >> k) & 1u) mbar_drain(smem_addr(full_b + slot), (uint32_t)round & 1u);
        if (--slot < 0) {
            slot = S - 1;
            --round;
        }
    }
#pragma unroll 1
    for (int k = 0; k < nsb && k < blk; ++k)
        if ((sb_bits >> k) & 1u) {
            const int q = blk - 1 - k;
            mbar_drain(smem_addr(sbfull_b + q % nsb), (uint32_t)(q / nsb) & 1u);
        }
    if (raw_rb0 >= 0) mbar_drain(smem_addr(rawfull_b), ((uint32_t)raw_rb0 / (uint32_t)kRawBufs) & 1u);
    if (raw_rb1 >= 0) mbar_drain(smem_addr(rawfull_b + 1), ((uint32_t)raw_rb1 / (uint32_t)kRawBufs) & 1u);
    if (kRawBufs > 2 && raw_rb2 >= 0) mbar_drain(smem_addr(rawfull_b + 2), ((uint32_t)raw_rb2 / (uint32_t)kRawBufs) & 1u);
}

// Raw mode, consumer side: rearrange a row block's raw [rows][groups] scales and biases into
// the swizzled [64-group chunk][row][128 B] layout, one thread per (scales | biases, row,
// 8-group granule), one 16-byte store each; groups up to the next 16-group block are zeros for
// the bias contraction.
__device__ __noinline__ void raw_rearrange(const GemvOp& p, const uint16_t* rs_, uint32_t raw_elems, uint8_t* sdst,
                                          int64_t e0, int gsz, int rv, int ctid) {
    const int off = (int)(e0 - (e0 & ~(int64_t)7));
    const int ngr = (gsz + 15) / 16 * 2;                 // 8-group granules, padded
    const int items = 2 * rv * ngr;
#pragma unroll 1
    for (int it2 = ctid; it2 < items; it2 += kConsumerWarps * 32) {
        const int isb = it2 >= rv * ngr;
        const int rest = it2 - isb * rv * ngr;
        const int r = rest / ngr;
        const int u = rest - r * ngr;
        const uint16_t* src = rs_ + (size_t)isb * raw_elems + off + r * gsz;
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k0 = 8 * u + 2 * e;
            const uint32_t lo = k0 < gsz ? (uint32_t)src[k0] : 0u;
            const uint32_t hi = k0 + 1 < gsz ? (uint32_t)src[k0 + 1] : 0u;
            pk[e] = lo | (hi << 16);
        }
        const uint32_t o = (uint32_t)((((u >> 3) * p.sb_tiles * 16) + r) * 128) + ((uint32_t)((u & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(sdst + (size_t)isb * p.sb_pitch + o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
}

// ---- the kernel --------------------------------------------------------------------------

// CB: code bits. 4: packed nibbles. 2: derived 2-bit codes q4 >> 2, w = (4 q + 1.5) s + b.
// 3: derived 3-bit codes q4 >> 1 = 2 * (2-bit upper part) + lowest bit, w = (2 q + 0.5) s + b.
// FG: fused gate|up. The matrix holds the gate rows [0, out_dim) and then the up rows; a
// "tile" of the schedule is a unit of 16 gate rows and the 16 up rows with the same index,
// kept in shared-memory tiles u and MT/2 + u of the row block, and the epilogue writes
// h = fp16(silu(gate) * up) instead of y ("BATCH_MSL" experts.metal fn_moe_act_b).
// MTT: tiles per row block (0: the default for NT). Rows that a short row block lacks still
// cost their mma work (the tile loop is unrolled for a fixed tile count), so launches whose
// clusters get only a few tiles use a kernel built for that many.
// RAWD (raw scale mode, 4-bit routed experts): the consumers read each row block's scales and
// biases straight from the raw staging buffer ([rows][groups] bf16, as TMA copied it) instead of
// first rearranging them into the swizzled layout; a buffer is handed back after the row
// block's bias term.
template <int NT, bool RMS, int MAXSEG, int CB = 4, bool FG = false, int MTT = 0, bool XF = false, bool INJ = false,
          bool RAWD = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ GemvParams<MAXSEG> pp) {
    constexpr int NTOK = NT * 8;
    constexpr int MT = MTT ? MTT : tiles_per_block(NT);  // tiles per row block
    constexpr int TPW = MT;                  // tiles per consumer warp: all of the row block
    static_assert(MT >= 1 && MT <= kNumMaps, "row blocks of at most kNumMaps tiles: one tensor map per height");
    static_assert(!RAWD || (CB == 4 && !FG && !RMS), "direct raw reads: plain 4-bit products");
    constexpr int kRawBufs = raw_bufs(RAWD);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemLayout& L = pp.lay;
    uint8_t* ring = smem + L.ring;
    uint8_t* xfrag = smem + L.xfrag;
    float* xsum_s = reinterpret_cast<float*>(smem + L.xsum);
    uint8_t* sbuf = smem + L.sb;                              // [2][s rows | b rows]
    float* wpart = reinterpret_cast<float*>(smem + L.wpart);
    float* cpart = reinterpret_cast<float*>(smem + L.cpart);
    float* ssq_s = reinterpret_cast<float*>(smem + L.ssq);   // [NTOK] sum of squares, [NTOK] inv
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    const int S = pp.stages;
    uint64_t* full_b = bars;              // [S]  TMA bytes of a stage landed
    uint64_t* empty_b = bars + S;         // [S]  every consumer warp is done with a stage
    uint64_t* sbfull_b = bars + 2 * S;    // [2]  a row block's scales/biases landed
    uint64_t* sbempty_b = bars + 2 * S + 2;  // [2] every consumer warp is done with them
    uint64_t* rawfull_b = bars + 2 * S + 4;  // [kRawBufs] raw mode: a row block's raw scales/biases landed
    uint64_t* rawempty_b = rawfull_b + kRawBufs;   // [kRawBufs] raw mode: the consumers are done with them
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(rawempty_b + kRawBufs);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int C = pp.cluster;
    const int crank = C > 1 ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / C;

    grid_dep_launch();
    if (warp == kConsumerWarps && lane < 3 * kNumMaps) {
        // fetch the tensor-map descriptors in parallel before their first use
        const GemvOp& p = pp.op;
        const CUtensorMap* m = lane < kNumMaps ? &p.tmap_w[lane]
                               : lane < 2 * kNumMaps ? &p.tmap_s[lane - kNumMaps] : &p.tmap_b[lane - 2 * kNumMaps];
        if (lane < kNumMaps || p.sb_mode == kSbTma)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
        if (p.sb_mode == kSbRaw && lane < 2) prefetch_tensormap(lane ? &p.tmap_b1 : &p.tmap_s1);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(full_b + s), 1);
            mbar_init(smem_addr(empty_b + s), kConsumerWarps);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(smem_addr(sbfull_b + q), 1);
            mbar_init(smem_addr(sbempty_b + q), kConsumerWarps);
        }
        for (int q = 0; q < kRawBufs; ++q) {
            mbar_init(smem_addr(rawfull_b + q), 1);
            mbar_init(smem_addr(rawempty_b + q), RAWD ? kConsumerWarps : 1);
        }
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ======================= producer warp =======================
        // Under programmatic dependent launch this CTA may start while the previous kernel of
        // the stream still runs, and that kernel may have written the weights (a pack or a
        // quantiser, or any kernel of the caller's): the weight loads wait for it to complete.
        grid_dep_wait();
        int it = 0, blk = 0;
        int rs = 0;             // ring slot and its phase
        uint32_t rph = 0;
        bool pending = false;   // an un-waited cluster-barrier arrival
        // Lane 0's record of the copies it issued (bit 0: the latest), drained before the CTA
        // exits: after an abort the consumers no longer wait for them. Once the abort flag is
        // set no new copy is issued; the control flow (and every cluster barrier) stays as is.
        uint32_t st_bits = 0, sb_bits = 0;
        static_assert(kRawBufs <= 3, "one register per raw buffer below");
        int raw_rb0 = -1, raw_rb1 = -1, raw_rb2 = -1;   // raw mode: the row block each buffer received
        uint8_t* raw = smem + L.raw;   // raw mode: [kRawBufs buffers][scales | biases][raw_elems] bf16
        const GemvOp& p = pp.op;
        const bool fg = FG && p.fg;
        const OpRange R0 = op_range(p, crank, cid, pp.n_clusters);
        const int kg0 = R0.kg0, kg1 = R0.kg1, gsz = R0.gsz, nks = R0.nks, t_end = R0.t_end;
        if (RMS && p.rms && C > 1) {   // matches the consumers' norm exchange
            cluster_arrive();
            pending = true;
        }
        auto raw_issue_to = [&](const Job& jb, int buf, int rb) {
            if (lane != 0 || *abort_flag) return;
            if constexpr (kRawBufs == 2) {
                if (buf) raw_rb1 = rb; else raw_rb0 = rb;
            } else {
                if (buf == 0) raw_rb0 = rb;
                else if (buf == 1) raw_rb1 = rb;
                else raw_rb2 = rb;
            }
            raw_issue(p, pp.seg[jb.seg], jb.tile, jb.ntile, raw + (size_t)buf * 2u * L.raw_elems * 2u, L.raw_elems,
                      smem_addr(rawfull_b + buf));
        };
        int t = R0.t_begin;
        Job j;
        if (p.sb_mode == kSbRaw) {
            int t2 = t;
            Job j0;
            if (next_job(p, t2, t_end, j0)) raw_issue_to(j0, 0, 0);
            __syncwarp();
        }
        while (next_job(p, t, t_end, j)) {
            const Segment& sg = pp.seg[j.seg];
            const int64_t lrow0 = (int64_t)j.tile * 16;                 // row within the segment
            const int rows_valid = (int)llmin((int64_t)j.ntile * 16, p.out_dim - lrow0);
            const int64_t trow0 = (int64_t)sg.row0 + lrow0;              // row within the tensor
            // -- scales and biases of the whole row block, full rows of the K-slice --
            {
                const int nsb = (int)L.n_sb;
                const int q = blk % nsb;
                // (raw mode: the consumers write the rearranged scales themselves)
                if (blk >= nsb && p.sb_mode != kSbRaw)
                    mbar_wait(smem_addr(sbempty_b + q), (uint32_t)(blk / nsb - 1) & 1u, abort_flag);
                uint8_t* sdst = sbuf + (size_t)q * L.sb_buf;
                const uint32_t bar = smem_addr(sbfull_b + q);
                if (p.sb_mode == kSbTma) {
                    if (lane == 0) sb_bits <<= 1;
                    if (lane == 0 && !*abort_flag) {
                        sb_bits |= 1u;
                        sb_tma_issue(p, sdst, bar, trow0, kg0, gsz, j.ntile, fg ? 2 : 1, MT / 2);
                    }
                } else if (p.sb_mode == kSbRaw) {
                    // the next row block's raw scales/biases, into the buffer the consumers
                    // released kRawBufs - 1 row blocks ago
                    int t2 = t;
                    Job jn;
                    if (next_job(p, t2, t_end, jn)) {
                        if constexpr (kRawBufs == 2) {
                            const int nbuf = (blk + 1) & 1;
                            if (blk + 1 >= 2)
                                mbar_wait(smem_addr(rawempty_b + nbuf), (uint32_t)((blk + 1) / 2 - 1) & 1u, abort_flag);
                            raw_issue_to(jn, nbuf, blk + 1);
                        } else {
                            const uint32_t nb1 = (uint32_t)blk + 1u;
                            const int nbuf = (int)(nb1 % (uint32_t)kRawBufs);
                            if (nb1 >= (uint32_t)kRawBufs)
                                mbar_wait(smem_addr(rawempty_b + nbuf), (nb1 / (uint32_t)kRawBufs - 1u) & 1u, abort_flag);
                            raw_issue_to(jn, nbuf, blk + 1);
                        }
                    }
                } else {
                    sb_plain_copy(p, sdst, trow0, rows_valid, kg0, gsz, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar);
                }
                __syncwarp();
            }
            // -- the packed weights, one stage per 8 groups --
            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = rs;
                const uint32_t ph = rph;
                if (++rs == S) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (it >= S) mbar_wait(smem_addr(empty_b + s), ph ^ 1u, abort_flag);
                const uint32_t full = smem_addr(full_b + s);
                uint8_t* st = ring + (size_t)s * L.stage_bytes;
                const int g0 = kg0 + ks * kStageGroups;
                const int ng = min(kStageGroups, kg1 - g0);
                // box columns of 128 bytes: 4 groups of nibbles, 8 groups of 2-bit codes
                const int nbox = CB == 4 ? (ng + 3) / 4 : 1;
                if (lane == 0) st_bits <<= 1;
                if (lane == 0 && !*abort_flag && it != p.withhold_stage) {
                    st_bits |= 1u;
                    // One box per box column as tall as the row block: the TMA engine pays per
                    // box (small boxes cap the stream well below HBM), so few large boxes.
                    mbar_arrive_expect_tx(full, (uint32_t)((fg ? 2 : 1) * j.ntile *
                                                           (nbox * kTileBytes + (CB == 3 ? kLoTileBytes : 0))));
                    const int mi = j.ntile - 1;
                    for (int part = 0; part < (fg ? 2 : 1); ++part) {   // fused: gate rows, up rows
                        const int64_t prow = trow0 + (part ? p.out_dim : 0);
                        const int mbase = part * (MT / 2);
                        for (int c = 0; c < nbox; ++c)
                            tma_load_2d(smem_addr(st + (c * MT + mbase) * kTileBytes), &p.tmap_w[mi],
                                        CB == 4 ? (g0 + 4 * c) * 32 : g0 * 16, (int)prow, full);
                        if constexpr (CB == 3)   // lowest bits: 8 bytes per group and row
                            tma_load_2d(smem_addr(st + MT * kTileBytes + mbase * kLoTileBytes), &p.tmap_lo[mi], g0 * 8,
                                        (int)prow, full);
                    }
                }
                __syncwarp();
            }
            if (C > 1) {
                if (pending) cluster_wait();
                cluster_arrive();
                pending = true;
            }
            ++blk;
        }
        if (lane == 0)
            drain_copies<kRawBufs>(full_b, S, it, st_bits, sbfull_b, (int)L.n_sb, blk, sb_bits, rawfull_b, raw_rb0,
                                   raw_rb1, raw_rb2);
        __syncwarp();
        if (pending) cluster_wait();
    } else {
        // ======================= consumer warps =======================
        const int ctid = threadIdx.x;       // 0 .. 32 * kConsumerWarps - 1
        const int wg = warp;                // group slot = group index within each stage
        const int g = lane >> 2;
        const int tq = lane & 3;
        grid_dep_wait();   // activations, the row map and y may belong to the previous kernel
        float acc[TPW][NT][4];
        uint8_t* xbias = smem + L.xbias;
        int rs = 0;            // ring slot and its phase
        uint32_t rph = 0;
        int blk = 0;
        const GemvOp& p = pp.op;
        const bool fg = FG && p.fg;
        const bool rms = RMS && p.rms;
        const OpRange R0 = op_range(p, crank, cid, pp.n_clusters);
        const int kg0 = R0.kg0, gsz = R0.gsz, nks = R0.nks, t_end = R0.t_end;

        if (rms) {
            // Sum of squares of this CTA's K-slice per activation row, exchanged across the
            // cluster so every CTA normalises with the full-row statistics.
            rms_partial<NT, INJ>(p, pp.seg[0], kg0, gsz, ssq_s, wpart, warp, lane, ctid);
            if (C > 1) {
                cluster_arrive();
                cluster_wait();
            } else {
                consumer_sync();
            }
            const int ng = NTOK * p.norm_groups;
            for (int e = ctid; e < ng; e += kConsumerWarps * 32) {
                float tot = 0.f;
                for (int c = 0; c < C; ++c)
                    tot += C > 1 ? ld_peer_f32(map_peer(smem_addr(ssq_s + e), c)) : ssq_s[e];
                ssq_s[NTOK * kMaxNormGroups + e] = rsqrtf(tot / (float)p.norm_width + p.eps);
            }
            consumer_sync();
        }

        // Per-warp constants (32-bit shared addresses; per-tile steps are immediates).
        // ldmatrix: rows 0-7 / 8-15 of a tile, 16-byte granules 2*(wg&3) and 2*(wg&3)+1 of
        // its box column; 128-byte swizzle granule ^= row & 7.
        const uint32_t lrow = (uint32_t)((lane & 7) + ((lane >> 3) & 1) * 8);
        // 4-bit: lanes 16-31 address the group's second granule; low-bit: the next tile
        const uint32_t lgran = CB == 4 ? (uint32_t)(wg & 3) * 2 + (uint32_t)(lane >> 4) : (uint32_t)wg;
        const uint32_t ldsm_base = smem_addr(ring) + lrow * 128 + ((lgran ^ (lrow & 7)) << 4) +
                                   (CB == 4 ? (uint32_t)(((wg >> 2) * MT) * kTileBytes)
                                            : (uint32_t)(lane >> 4) * (uint32_t)kTileBytes);
        // 3-bit: this lane's lowest-bit word (chunk tq/2 of group wg, row g), shifted so that
        // the bits of its half (word tq & 1 of the upper codes) sit at bits j of each byte
        const uint32_t lo_base = smem_addr(ring) + (uint32_t)(MT * kTileBytes) + (uint32_t)g * 64u +
                                 (uint32_t)wg * 8u + (uint32_t)(tq >> 1) * 4u;
        const uint32_t lo_shift = 4u * (uint32_t)(tq & 1);
        // B fragments of group gl, row tok: xfrag + ((gl*2 + jp)*ntok_max + tok)*64 + tq*16
        const uint32_t xf_jp = (uint32_t)p.ntok_max * 64u;
        const uint32_t xf_base = smem_addr(xfrag) + (uint32_t)wg * 2u * xf_jp + (uint32_t)g * 64u + (uint32_t)tq * 16u;
        const uint32_t xf_stage = (uint32_t)kStageGroups * 2u * xf_jp;
        // scales: [chunk][row][128 B]; this lane's rows g (and g+8) of the warp's first tile
        const uint32_t s_lane = (uint32_t)(g * 128) + 2u * (uint32_t)wg;
        int staged_seg = -1;
        int t = R0.t_begin;
        Job j;
        while (next_job(p, t, t_end, j)) {
            const Segment& sg = pp.seg[j.seg];
            if (j.seg != staged_seg) {
                stage_x<NT, RMS, CB, XF, INJ>(p, rms, sg, kg0, gsz, xfrag, xsum_s, ssq_s + NTOK * kMaxNormGroups, ctid,
                                     rms && cid == 0 && p.x_new != nullptr);
                consumer_sync();
                stage_xbias(xsum_s, sg.ntok, p.ntok_max, NTOK, gsz, xbias, ctid);
                consumer_sync();
                staged_seg = j.seg;
            }
            const int ntok = sg.ntok;
#pragma unroll
            for (int mi = 0; mi < TPW; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[mi][nt][k] = 0.f;

            const int q = blk % (int)L.n_sb;
            const int rbuf = kRawBufs == 2 ? (blk & 1) : (int)((uint32_t)blk % (uint32_t)kRawBufs);
            // RAWD: this lane's scale of (row g, group wg) of the row block's first tile in the raw
            // buffer, and the buffer's biases
            uint32_t raw_sl = 0, raw_b = 0;
            int raw_off = 0;
            if (p.sb_mode == kSbRaw) {
                mbar_wait(smem_addr(rawfull_b + rbuf),
                          (kRawBufs == 2 ? (uint32_t)(blk >> 1) : (uint32_t)blk / (uint32_t)kRawBufs) & 1u, abort_flag);
                const uint16_t* rs_ = reinterpret_cast<const uint16_t*>(smem + L.raw + (size_t)rbuf * 2u * L.raw_elems * 2u);
                const int64_t e0 = ((int64_t)sg.row0 + (int64_t)j.tile * 16) * p.groups;
                raw_off = (int)(e0 - (e0 & ~(int64_t)7));
                if constexpr (RAWD) {
                    raw_b = smem_addr(rs_) + L.raw_elems * 2u;
                    raw_sl = smem_addr(rs_) + 2u * (uint32_t)(raw_off + g * gsz + wg);
                } else {
                    // Rearrange the row block's raw scales and biases (every warp of the previous
                    // row block has passed its epilogue barrier, so the buffer is free).
                    const int rv = (int)llmin((int64_t)j.ntile * 16, p.out_dim - (int64_t)j.tile * 16);
                    raw_rearrange(p, rs_, L.raw_elems, sbuf + (size_t)q * L.sb_buf, e0, gsz, rv, ctid);
                    consumer_sync();
                    if (ctid == 0) mbar_arrive(smem_addr(rawempty_b + rbuf));
                }
            } else {
                mbar_wait(smem_addr(sbfull_b + q), (uint32_t)(blk / (int)L.n_sb) & 1u, abort_flag);
            }
            const uint8_t* sbs = sbuf + (size_t)q * L.sb_buf;         // scales
            const uint8_t* sbb = sbs + p.sb_pitch;                    // biases
            const uint32_t s_blk = smem_addr(sbs) + s_lane;
            bool tok_ok[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) tok_ok[nt] = nt * 8 + g < ntok;
            for (int ks = 0; ks < nks; ++ks) {
                mbar_wait(smem_addr(full_b + rs), rph, abort_flag);
                if (wg < min(kStageGroups, gsz - ks * kStageGroups)) {
                    // Slots beyond the row block read stale stage data and are never stored.
                    // 4-bit: w[mi][0..3] = rows g, g+8 of granule 0, then of granule 1 (8 nibbles each).
                    // Low-bit: w[mi][0], w[mi][1] = rows g, g+8 (16 codes each), two tiles per ldmatrix.
                    uint32_t w[TPW][CB == 4 ? 4 : 2];
                    const uint32_t st = ldsm_base + (uint32_t)rs * L.stage_bytes;
                    if constexpr (CB == 4) {
#pragma unroll
                        for (int mi = 0; mi < TPW; ++mi)
                            ldsm_x4(st + (uint32_t)(mi * kTileBytes), w[mi][0], w[mi][1], w[mi][2], w[mi][3]);
                    } else {
#pragma unroll
                        for (int mi = 0; mi < TPW; mi += 2)
                            ldsm_x4(st + (uint32_t)(mi * kTileBytes), w[mi][0], w[mi][1], w[mi + 1][0], w[mi + 1][1]);
                    }
                    uint32_t lw[TPW][2];   // 3-bit: the lowest-bit words of rows g, g+8
                    if constexpr (CB == 3) {
                        const uint32_t lb = lo_base + (uint32_t)rs * L.stage_bytes;
#pragma unroll
                        for (int mi = 0; mi < TPW; ++mi) {
                            lw[mi][0] = lds_u32(lb + (uint32_t)(mi * kLoTileBytes)) >> lo_shift;
                            lw[mi][1] = lds_u32(lb + (uint32_t)(mi * kLoTileBytes + 8 * 64)) >> lo_shift;
                        }
                    }
                    uint32_t bf[NT][8];
                    const uint32_t xf = xf_base + (uint32_t)ks * xf_stage;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        // activation row nt*8 + g of the segment; rows beyond it multiply zeros
                        uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
                        if (tok_ok[nt]) {
                            q0 = lds_v4(xf + (uint32_t)(nt * 512));
                            q1 = lds_v4(xf + xf_jp + (uint32_t)(nt * 512));
                        }
                        bf[nt][0] = q0.x; bf[nt][1] = q0.y; bf[nt][2] = q0.z; bf[nt][3] = q0.w;
                        bf[nt][4] = q1.x; bf[nt][5] = q1.y; bf[nt][6] = q1.z; bf[nt][7] = q1.w;
                    }
                    // group gl = 8ks + wg: chunk ks/8, granule (ks & 7) ^ g, element wg
                    // (RAWD: row-major [rows][gsz] from the row block's first element)
                    const uint32_t sa = RAWD ? raw_sl + (uint32_t)(16 * ks)
                                             : s_blk + (uint32_t)((ks >> 3) * p.sb_tiles * kTileBytes) +
                                                   ((uint32_t)((ks & 7) ^ g) << 4);
#pragma unroll
                    for (int mi = 0; mi < TPW; ++mi) {
                        // The mma partial sums are sum(q x) * 2^-24; s multiplies them as is and
                        // the result is multiplied by 2^24 once at the end (no scale overflows).
                        // Low-bit codes: the steps compute sum(q x) / (4 or 2); the scale restores it.
                        constexpr float kq = CB == 4 ? 1.0f : (CB == 2 ? 4.0f : 2.0f);
                        float s0, s1;
                        if constexpr (RAWD) {   // next tile: 16 rows on; row + 8: 8 rows on
                            s0 = kq * bf16_to_f32(lds_u16(sa + (uint32_t)(mi * 32 * gsz)));
                            s1 = kq * bf16_to_f32(lds_u16(sa + (uint32_t)(mi * 32 * gsz + 16 * gsz)));
                        } else {
                            s0 = kq * bf16_to_f32(lds_u16(sa + (uint32_t)(mi * kTileBytes)));
                            s1 = kq * bf16_to_f32(lds_u16(sa + (uint32_t)(mi * kTileBytes + 1024)));
                        }
                        // h[a][jj]: mma step jj's A register a (a0/a2: row g, a1/a3: row g+8)
                        uint32_t h[4][4];
                        if constexpr (CB == 4) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint32_t v8 = w[mi][k] >> 8;
                                h[k][0] = w[mi][k] & 0x000F000Fu;
                                h[k][1] = w[mi][k] & 0x00F000F0u;
                                h[k][2] = v8 & 0x000F000Fu;
                                h[k][3] = v8 & 0x00F000F0u;
                            }
                        } else if constexpr (CB == 2) {
                            // field jj of bytes 0, 2 (k-low) and of bytes 1, 3 (k-high), in place
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const uint32_t v8 = w[mi][r] >> 8;
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj) {
                                    h[r][jj] = w[mi][r] & (0x00030003u << (2 * jj));
                                    h[2 + r][jj] = v8 & (0x00030003u << (2 * jj));
                                }
                            }
                        } else {
                            // code = 2 * upper + lowest, assembled in bits 2jj .. 2jj+2 of each half:
                            // the upper field moved up one bit, the lowest bit (bit jj of the byte
                            // once the lane's word half is shifted down) moved to bit 2jj
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const uint32_t u1 = w[mi][r] << 1, u7 = w[mi][r] >> 7;
                                const uint32_t l = lw[mi][r];
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj) {
                                    const uint32_t mu = 0x00060006u << (2 * jj), ml = 0x00010001u << (2 * jj);
                                    h[r][jj] = (u1 & mu) | ((l << jj) & ml);
                                    h[2 + r][jj] = (u7 & mu) | ((l >> (8 - jj)) & ml);
                                }
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                mma_f16(d, h[0][jj], h[1][jj], h[2][jj], h[3][jj], bf[nt][2 * jj],
                                        bf[nt][2 * jj + 1]);
                            float* a = acc[mi][nt];
                            a[0] = fmaf(s0, d[0], a[0]);
                            a[1] = fmaf(s0, d[1], a[1]);
                            a[2] = fmaf(s1, d[2], a[2]);
                            a[3] = fmaf(s1, d[3], a[3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(empty_b + rs));
                if (++rs == S) {
                    rs = 0;
                    rph ^= 1u;
                }
            }

            // ---- bias term: sum_g b[o][g] * xsum[r][g], once per row block ----
            // bf16 mma over 16-group blocks; A (biases) comes straight from the swizzled smem
            // rows through ldmatrix, B is the hi/lo split group sums.
            {
                const int nblk = (gsz + 15) / 16;
                for (int gb = kGroupSlots - 1 - wg; gb < nblk; gb += kGroupSlots) {   // last warps first
                    uint32_t bx[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        uint4 v = make_uint4(0, 0, 0, 0);
                        if (tok_ok[nt])
                            v = lds_v4(smem_addr(xbias) + (uint32_t)((gb * p.ntok_max + nt * 8 + g) * 64 + tq * 16));
                        bx[nt][0] = v.x; bx[nt][1] = v.y; bx[nt][2] = v.z; bx[nt][3] = v.w;
                    }
                    // groups 16gb..16gb+15 = granules 2*(gb&3), +1 of 64-group chunk gb>>2
                    const uint32_t gran = (uint32_t)(gb & 3) * 2 + (uint32_t)(lane >> 4);
                    const uint32_t boff = smem_addr(sbb) + (uint32_t)((gb >> 2) * p.sb_tiles * kTileBytes) + lrow * 128 +
                                          ((gran ^ (lrow & 7)) << 4);
#pragma unroll
                    for (int mi = 0; mi < TPW; ++mi) {
                        uint32_t a0, a1, a2, a3;
                        if constexpr (RAWD) {
                            // A fragment of m16n8k16: rows g, g + 8 x groups 16gb + 2tq (+1), + 8 (+9)
                            auto bpair = [&](int row, int gl) -> uint32_t {
                                const uint32_t e = raw_b + 2u * (uint32_t)(raw_off + (mi * 16 + row) * gsz + gl);
                                const uint32_t lo = gl < gsz ? lds_u16(e) : 0u;
                                const uint32_t hi = gl + 1 < gsz ? lds_u16(e + 2u) : 0u;
                                return lo | (hi << 16);
                            };
                            const int gl0 = gb * 16 + 2 * tq;
                            a0 = bpair(g, gl0);
                            a1 = bpair(g + 8, gl0);
                            a2 = bpair(g, gl0 + 8);
                            a3 = bpair(g + 8, gl0 + 8);
                        } else {
                            ldsm_x4(boff + (uint32_t)(mi * kTileBytes), a0, a1, a2, a3);
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_bf16(acc[mi][nt], a0, a1, a2, a3, bx[nt][0], bx[nt][1]);
                            mma_bf16(acc[mi][nt], a0, a1, a2, a3, bx[nt][2], bx[nt][3]);
                        }
                        if constexpr (CB != 4) {
                            // the reconstruction offset: + (1.5 or 0.5) * sum_g s[o][g] * xsum[r][g]
                            constexpr float koff = CB == 2 ? 1.5f : 0.5f;
                            ldsm_x4(boff - p.sb_pitch + (uint32_t)(mi * kTileBytes), a0, a1, a2, a3);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                float d2[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_bf16(d2, a0, a1, a2, a3, bx[nt][0], bx[nt][1]);
                                mma_bf16(d2, a0, a1, a2, a3, bx[nt][2], bx[nt][3]);
#pragma unroll
                                for (int e = 0; e < 4; ++e) acc[mi][nt][e] = fmaf(koff, d2[e], acc[mi][nt][e]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(sbempty_b + q));
            if constexpr (RAWD) {
                if (lane == 0) mbar_arrive(smem_addr(rawempty_b + rbuf));   // the raw buffer is free
            }

            // ---- end of the row block: reduce over group slots, then over the cluster ----
            const int R = j.ntile * 16;
#pragma unroll
            for (int mi = 0; mi < TPW; ++mi) {
                const int m = mi;
                if ((fg ? m % (MT / 2) : m) >= j.ntile) continue;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float* w0 = wpart + ((size_t)wg * (16 * MT) + m * 16 + g) * NTOK + nt * 8 + 2 * tq;
                    *reinterpret_cast<float2*>(w0) = make_float2(acc[mi][nt][0], acc[mi][nt][1]);
                    *reinterpret_cast<float2*>(w0 + 8 * NTOK) = make_float2(acc[mi][nt][2], acc[mi][nt][3]);
                }
            }
            consumer_sync();
            float* cp = cpart + (size_t)(blk & 1) * (16 * MT) * NTOK;
            // fused: the gate rows [0, R) and the up rows [8 MT, 8 MT + R) of the row block
            for (int e0 = ctid; e0 < (fg ? 2 : 1) * R * NTOK; e0 += kConsumerWarps * 32) {
                const int e = (fg && e0 >= R * NTOK) ? e0 - R * NTOK + 8 * MT * NTOK : e0;
                const size_t stride = (size_t)(16 * MT) * NTOK;
                float v = wpart[e];
#pragma unroll
                for (int qq = 1; qq < kGroupSlots; ++qq) v += wpart[e + qq * stride];
                cp[e] = v;
            }
            if (C > 1) {
                cluster_arrive();
                cluster_wait();
            } else {
                consumer_sync();
            }
            const int64_t lrow0 = (int64_t)j.tile * 16;
            const int rows_valid = (int)llmin((int64_t)R, p.out_dim - lrow0);
            const int rc = (R + C - 1) / C;
            const int ra = crank * rc;
            const int rb = min(R, ra + rc);
            const int nr = rb - ra;
            if (nr > 0) {
                const uint32_t cp_addr = smem_addr(cp);
                for (int e = ctid; e < nr * sg.ntok; e += kConsumerWarps * 32) {
                    const int tok = e / nr;
                    const int row = ra + (e - tok * nr);
                    if (row >= rows_valid) continue;
                    float v;
                    if (C > 1) {
                        const uint32_t off = (uint32_t)((row * NTOK + tok) * 4);
                        v = 0.f;
                        for (int c = 0; c < C; ++c) v += ld_peer_f32(map_peer(cp_addr + off, (uint32_t)c));
                    } else {
                        v = cp[row * NTOK + tok];
                    }
                    if (fg) {
                        float u;
                        if (C > 1) {
                            const uint32_t off = (uint32_t)(((8 * MT + row) * NTOK + tok) * 4);
                            u = 0.f;
                            for (int c = 0; c < C; ++c) u += ld_peer_f32(map_peer(cp_addr + off, (uint32_t)c));
                        } else {
                            u = cp[(8 * MT + row) * NTOK + tok];
                        }
                        const float gt = v * 16777216.0f;
                        const float hv = gt / (1.0f + expf(-gt)) * (u * 16777216.0f);
                        p.h[(int64_t)(sg.tok0 + tok) * p.out_dim + lrow0 + row] = __half_as_ushort(__float2half_rn(hv));
                        continue;
                    }
                    float out = v * 16777216.0f;
                    if (p.post_silu) {   // silu(y / div): the gated-residual bottleneck epilogue
                        const float t = out / p.post_div;
                        out = t / (1.0f + expf(-t));
                    }
                    p.y[(int64_t)(sg.tok0 + tok) * p.out_dim + lrow0 + row] = out;
                }
            }
            ++blk;
        }
    }
    if (C > 1) {
        // No CTA leaves while a peer may still read its shared memory.
        cluster_arrive();
        cluster_wait();
    }
}

template <int MAXSEG>
struct KernelSet;

}  // namespace

// ---- host side ---------------------------------------------------------------------------

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

// Encoded tensor maps, keyed by every argument of the encode call: a map is a pure function of
// them, and a decode step calls the same products with the same buffers over and over, so the
// host-side encode (several per launch) runs once per buffer instead of once per call.
CUresult encode_tiled_cached(CUtensorMap* out, CUtensorMapDataType dtype, cuuint32_t rank, void* ptr,
                             const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                             const cuuint32_t* estr, CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                             CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob) {
    struct Key {
        uint64_t v[20];
    } key;
    memset(&key, 0, sizeof(key));
    key.v[0] = (uint64_t)dtype | ((uint64_t)rank << 8) | ((uint64_t)il << 16) | ((uint64_t)sw << 24) |
               ((uint64_t)l2 << 32) | ((uint64_t)oob << 40);
    key.v[1] = reinterpret_cast<uint64_t>(ptr);
    for (cuuint32_t i = 0; i < rank && i < 5; ++i) {
        key.v[2 + i] = dims[i];
        key.v[7 + i] = i + 1 < rank ? strides[i] : 0;
        key.v[12 + i] = ((uint64_t)box[i] << 32) | estr[i];
    }
    const std::string k(reinterpret_cast<const char*>(&key), sizeof(key));
    static std::mutex mu;
    static std::unordered_map<std::string, CUtensorMap> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(k);
        if (it != cache.end()) {
            *out = it->second;
            return CUDA_SUCCESS;
        }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    const CUresult r = enc(out, dtype, rank, ptr, dims, strides, box, estr, il, sw, l2, oob);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() >= 16384) cache.clear();   // a bound for callers that churn buffers
        cache.emplace(k, *out);
    }
    return r;
}

namespace {

struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
    bool ok = false;
};

// The current device's SM count and shared-memory limit; a failing query is recorded for
// q4a_last_cuda_error (the caller returns Q4A_ERR_CUDA).
DeviceInfo device_info() {
    int dev = 0;
    DeviceInfo d;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_fail(e);
        return d;
    }
    static DeviceInfo cache[64];
    if (dev < 64 && cache[dev].ok) return cache[dev];
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        cuda_fail(e);
        return d;
    }
    d.ok = d.sm_count > 0;
    if (dev < 64) cache[dev] = d;
    return d;
}

// Per-device caches of the function attribute and of the cluster occupancy, filled on
// first use so that later calls (including under stream capture) make no queries.
struct OccKey {
    const void* fn;
    int dev, cluster;
    uint32_t smem;
    bool operator<(const OccKey& o) const {
        if (fn != o.fn) return fn < o.fn;
        if (dev != o.dev) return dev < o.dev;
        if (cluster != o.cluster) return cluster < o.cluster;
        return smem < o.smem;
    }
};

std::mutex g_cache_mu;
std::map<OccKey, int> g_occ_cache;
std::map<std::pair<const void*, int>, uint32_t> g_smem_set;

template <int NT, bool RMS, int MAXSEG, int CB = 4, bool FG = false, int MTT = 0, bool XF = false, bool INJ = false,
          bool RAWD = false>
int occupancy_clusters(int cluster, uint32_t smem_bytes) {
    auto kern = gemv_kernel<NT, RMS, MAXSEG, CB, FG, MTT, XF, INJ, RAWD>;
    const void* fn = reinterpret_cast<const void*>(kern);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const DeviceInfo di = device_info();
    std::lock_guard<std::mutex> lock(g_cache_mu);
    uint32_t& set = g_smem_set[{fn, dev}];
    if (set < (uint32_t)di.max_smem_optin) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        set = (uint32_t)di.max_smem_optin;
    }
    const OccKey key{fn, dev, cluster, smem_bytes};
    auto it = g_occ_cache.find(key);
    if (it == g_occ_cache.end()) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3((unsigned)(di.sm_count / cluster * cluster), 1, 1);
        int occ = 0;
        if (cudaOccupancyMaxActiveClusters(&occ, kern, &cfg) != cudaSuccess || occ <= 0) {
            cudaGetLastError();
            occ = di.sm_count / cluster;
        }
        it = g_occ_cache.emplace(key, occ).first;
    }
    return it->second;
}

template <int MAXSEG>
int cluster_capacity_t(int nt, bool rms, int cluster, uint32_t smem_bytes, int cb) {
    if constexpr (MAXSEG == kDenseMaxSeg) {
        if (cb == 2) {
            if (nt == 1) return occupancy_clusters<1, false, MAXSEG, 2>(cluster, smem_bytes);
            if (nt == 2) return occupancy_clusters<2, false, MAXSEG, 2>(cluster, smem_bytes);
            return occupancy_clusters<4, false, MAXSEG, 2>(cluster, smem_bytes);
        }
        if (cb == 3) {
            if (nt == 1) return occupancy_clusters<1, false, MAXSEG, 3>(cluster, smem_bytes);
            if (nt == 2) return occupancy_clusters<2, false, MAXSEG, 3>(cluster, smem_bytes);
            return occupancy_clusters<4, false, MAXSEG, 3>(cluster, smem_bytes);
        }
        if (rms) {
            if (nt == 1) return occupancy_clusters<1, true, MAXSEG>(cluster, smem_bytes);
            if (nt == 2) return occupancy_clusters<2, true, MAXSEG>(cluster, smem_bytes);
            return occupancy_clusters<4, true, MAXSEG>(cluster, smem_bytes);
        }
    }
    if (nt == 1) return occupancy_clusters<1, false, MAXSEG>(cluster, smem_bytes);
    if (nt == 2) return occupancy_clusters<2, false, MAXSEG>(cluster, smem_bytes);
    return occupancy_clusters<4, false, MAXSEG>(cluster, smem_bytes);
}

int cluster_capacity(int nt, bool rms, bool experts, int cluster, uint32_t smem_bytes, int cb, bool fg) {
    if (fg) {
        if (rms) {
            if (nt == 1) return occupancy_clusters<1, true, kDenseMaxSeg, 4, true>(cluster, smem_bytes);
            if (nt == 2) return occupancy_clusters<2, true, kDenseMaxSeg, 4, true>(cluster, smem_bytes);
            return occupancy_clusters<4, true, kDenseMaxSeg, 4, true>(cluster, smem_bytes);
        }
        if (nt == 1) return occupancy_clusters<1, false, kDenseMaxSeg, 4, true>(cluster, smem_bytes);
        if (nt == 2) return occupancy_clusters<2, false, kDenseMaxSeg, 4, true>(cluster, smem_bytes);
        return occupancy_clusters<4, false, kDenseMaxSeg, 4, true>(cluster, smem_bytes);
    }
    return experts ? cluster_capacity_t<Q4A_MAX_SEGMENTS>(nt, rms, cluster, smem_bytes, 4)
                   : cluster_capacity_t<kDenseMaxSeg>(nt, rms, cluster, smem_bytes, cb);
}

template <int NT, bool RMS, int MAXSEG, int CB = 4, bool FG = false, int MTT = 0, bool XF = false, bool INJ = false,
          bool RAWD = false>
q4a_status launch_variant(GemvParams<MAXSEG>& prm, uint32_t smem_bytes, cudaStream_t stream) {
    auto kern = gemv_kernel<NT, RMS, MAXSEG, CB, FG, MTT, XF, INJ, RAWD>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)prm.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = occupancy_clusters<NT, RMS, MAXSEG, CB, FG, MTT, XF, INJ, RAWD>(prm.cluster, smem_bytes);
    if (max_clusters <= 0) return Q4A_ERR_CUDA;
    prm.n_clusters = max_clusters < prm.op.n_tiles ? max_clusters : prm.op.n_tiles;
    cfg.gridDim = dim3((unsigned)(prm.n_clusters * prm.cluster), 1, 1);
    cfg.numAttrs = 2;
    static const bool debug = getenv("Q4A_DEBUG") != nullptr;
    if (debug)
        fprintf(stderr,
                "q4a gemv: nt=%d rms=%d segs=%d out=%lld in=%lld cluster=%d gs=%d mt=%d stages=%d "
                "clusters=%d (max %d) tiles=%d smem=%u sb_mode=%d\n",
                NT, (int)RMS, prm.nseg, (long long)prm.op.out_dim, (long long)prm.op.in_dim, prm.cluster, prm.op.gs,
                prm.op.mt, prm.stages, prm.n_clusters, max_clusters, prm.op.n_tiles, smem_bytes, prm.op.sb_mode);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
    if (e != cudaSuccess) return cuda_fail(e);
    return Q4A_OK;
}

// One op of a launch from its description: the tensor maps of its codes (and 3-bit lowest
// bits), of its scales and biases in the chosen fetch mode, and its shape and schedule.
struct OpMapKey {
    const void* w;
    const void* w_lo;
    const void* s;
    const void* b;
    int64_t rows, in_dim;
    int32_t cb, sb_mode;
    bool operator==(const OpMapKey& k) const { return memcmp(this, &k, sizeof(*this)) == 0; }
};
struct OpMapKeyHash {
    size_t operator()(const OpMapKey& k) const {
        const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
        uint64_t h = 1469598103934665603ull;   // FNV-1a over the key's bytes
        for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ p[i]) * 1099511628211ull;
        return (size_t)h;
    }
};
struct OpMaps {
    CUtensorMap w[kNumMaps], lo[kNumMaps], s[kNumMaps], b[kNumMaps], s1, b1;
};
std::mutex g_opmap_mu;
std::unordered_map<OpMapKey, OpMaps, OpMapKeyHash> g_opmaps;

// Every tensor map an op may use: codes (and the 3-bit lowest bits) for each row-block height,
// and the scales and biases in the chosen fetch mode.
q4a_status encode_op_maps(GemvOp& o, const GemvLaunch& L, int sb_mode) {
    auto enc = encode_tiled_cached;
    const int cb = L.code_bits;
    const int G = (int)(L.in_dim / kGroup);
    // packed codes: in_dim/2 bytes per row (nibbles) or in_dim/4 (2-bit codes; the 3-bit
    // codes' upper two bits); the 3-bit lowest-bit plane: in_dim/8 bytes per row
    const int64_t wrow = cb == 4 ? L.in_dim / 2 : L.in_dim / 4;
    const cuuint64_t dims[2] = {(cuuint64_t)wrow, (cuuint64_t)L.tensor_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)wrow};
    const cuuint32_t estr[2] = {1u, 1u};
    for (int i = 0; i < kNumMaps; ++i) {
        const cuuint32_t box[2] = {(cuuint32_t)kBoxBytes, (cuuint32_t)(16 * (i + 1))};
        CUresult r = enc(&o.tmap_w[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(L.w), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
        if (cb == 3) {
            const cuuint64_t ldims[2] = {(cuuint64_t)(L.in_dim / 8), (cuuint64_t)L.tensor_rows};
            const cuuint64_t lstrides[1] = {(cuuint64_t)(L.in_dim / 8)};
            const cuuint32_t lbox[2] = {64u, (cuuint32_t)(16 * (i + 1))};
            r = enc(&o.tmap_lo[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(L.w_lo), ldims, lstrides,
                    lbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
        }
    }
    if (sb_mode == kSbTma) {
        const cuuint64_t sdims[2] = {(cuuint64_t)G, (cuuint64_t)L.tensor_rows};
        const cuuint64_t sstrides[1] = {(cuuint64_t)G * 2};
        for (int i = 0; i < kNumMaps; ++i) {
            const cuuint32_t box[2] = {64u, (cuuint32_t)(16 * (i + 1))};
            for (int k = 0; k < 2; ++k) {
                CUresult r = enc(k ? &o.tmap_b[i] : &o.tmap_s[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                 const_cast<uint16_t*>(k ? L.b : L.s), sdims, sstrides, box, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
            }
        }
    }
    if (sb_mode == kSbRaw) {
        const cuuint64_t rdims[1] = {(cuuint64_t)(L.tensor_rows * G)};
        const cuuint64_t rstrides[1] = {0};
        const cuuint32_t rbox[1] = {(cuuint32_t)kRawBox};
        for (int k = 0; k < 2; ++k) {
            CUresult r = enc(k ? &o.tmap_b1 : &o.tmap_s1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 1,
                             const_cast<uint16_t*>(k ? L.b : L.s), rdims, rstrides, rbox, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
        }
    }
    return Q4A_OK;
}

q4a_status fill_op(GemvOp& o, const GemvLaunch& L, int gs, int mt_units, int sb_mode, int sb_tiles, uint32_t sb_pitch) {
    if (!encode_fn()) return Q4A_ERR_UNSUPPORTED;
    // The tensor maps of this matrix and fetch mode, encoded once and reused: a call's host
    // time is otherwise dominated by looking up ~18 maps one at a time.
    OpMapKey key;
    memset(&key, 0, sizeof(key));
    key.w = L.w;
    key.w_lo = L.w_lo;
    key.s = L.s;
    key.b = L.b;
    key.rows = L.tensor_rows;
    key.in_dim = L.in_dim;
    key.cb = L.code_bits;
    key.sb_mode = sb_mode;
    bool cached = false;
    {
        std::lock_guard<std::mutex> lock(g_opmap_mu);
        auto it = g_opmaps.find(key);
        if (it != g_opmaps.end()) {
            const OpMaps& m = it->second;
            memcpy(o.tmap_w, m.w, sizeof(m.w));
            memcpy(o.tmap_lo, m.lo, sizeof(m.lo));
            memcpy(o.tmap_s, m.s, sizeof(m.s));
            memcpy(o.tmap_b, m.b, sizeof(m.b));
            o.tmap_s1 = m.s1;
            o.tmap_b1 = m.b1;
            cached = true;
        }
    }
    if (!cached) {
        const q4a_status st = encode_op_maps(o, L, sb_mode);
        if (st != Q4A_OK) return st;
        OpMaps m;
        memcpy(m.w, o.tmap_w, sizeof(m.w));
        memcpy(m.lo, o.tmap_lo, sizeof(m.lo));
        memcpy(m.s, o.tmap_s, sizeof(m.s));
        memcpy(m.b, o.tmap_b, sizeof(m.b));
        m.s1 = o.tmap_s1;
        m.b1 = o.tmap_b1;
        std::lock_guard<std::mutex> lock(g_opmap_mu);
        if (g_opmaps.size() >= 4096) g_opmaps.clear();   // a bound for callers that churn buffers
        g_opmaps.emplace(key, m);
    }
    const int G = (int)(L.in_dim / kGroup);
    o.s = L.s;
    o.b = L.b;
    o.x = L.x;
    o.x_rows = L.x_rows;
    o.norm_w = L.norm_w;
    o.inj_out = L.inj_out;
    o.inj_logit = L.inj_logit;
    o.x_new = L.inj_out ? L.x_new : nullptr;
    o.y = L.y;
    o.h = L.h;
    o.eps = L.eps;
    o.shift = L.shift;
    o.norm_groups = L.norm_groups > 0 ? L.norm_groups : 1;
    o.norm_width = L.in_dim / o.norm_groups;
    o.post_silu = L.silu ? 1 : 0;
    o.post_div = L.silu ? L.silu_div : 1.0f;
    o.out_dim = L.out_dim;
    o.in_dim = L.in_dim;
    o.groups = G;
    o.gs = gs;
    o.tiles_per_seg = (int)((L.out_dim + 15) / 16);
    o.n_tiles = o.tiles_per_seg * L.nseg;
    o.mt = mt_units;
    o.ntok_max = L.max_ntok;
    o.sb_mode = sb_mode;
    o.sb_tiles = sb_tiles;
    o.sb_pitch = sb_pitch;
    o.rms = L.rmsnorm ? 1 : 0;
    o.fg = L.fused_gate_up ? 1 : 0;
    o.withhold_stage = L.withhold_stage;
    return Q4A_OK;
}

template <int MAXSEG>
q4a_status launch_gemv_t(const GemvLaunch& L, cudaStream_t stream) {
    static_assert(sizeof(GemvParams<MAXSEG>) < 32000, "kernel parameter block too large");
    const DeviceInfo di = device_info();
    if (!di.ok) return Q4A_ERR_CUDA;
    if (!encode_fn()) return Q4A_ERR_UNSUPPORTED;
    if (L.nseg > MAXSEG) return Q4A_ERR_SHAPE;

    const int nt = L.max_ntok <= 8 ? 1 : (L.max_ntok <= 16 ? 2 : 4);
    int mt = tiles_per_block(nt);
    const int cb = L.code_bits;
    if (cb != 4 && (L.rmsnorm || (cb != 2 && cb != 3))) return Q4A_ERR_UNSUPPORTED;
    if (L.x_f32 && (!L.experts || cb == 4 || L.rmsnorm)) return Q4A_ERR_UNSUPPORTED;
    if (L.inj_out && (!L.rmsnorm || L.fused_gate_up || cb != 4 || MAXSEG != kDenseMaxSeg)) return Q4A_ERR_UNSUPPORTED;
    const bool fg = L.fused_gate_up;
    if (fg && (cb != 4 || L.silu || L.x_f32 || L.out_dim % 16 != 0 || !L.h || (L.experts && L.rmsnorm)))
        return Q4A_ERR_UNSUPPORTED;
    // schedule units per row block: tiles, or (fused) gate|up tile pairs
    int mt_units = fg ? mt / 2 : mt;
    const int G = (int)(L.in_dim / kGroup);
    // 4-bit routed experts in raw scale mode read the raw buffers directly (no rearrangement)
    const bool rawd = MAXSEG != kDenseMaxSeg && cb == 4 && !fg && !L.rmsnorm && !L.x_f32;

    // Cluster size (K split). Candidates are powers of two whose K-slice leaves room for a
    // ring of at least 3 stages (a deeper ring matters less than avoiding the split: each
    // split row block pays a cluster-wide barrier and a DSMEM reduction). Among them: the smallest that gives every cluster >= 3 row
    // tiles (a row block worth a few TMA boxes) while its co-resident clusters still cover
    // >= 90% of the SMs (clusters must fit inside a GPC, which can strand SMs).
    const int ntm = L.max_ntok;
    auto slice = [&](int c) {
        int g = (G + c - 1) / c;
        if (c > 1) g = (g + 7) / 8 * 8;         // slices start on a stage boundary
        return g;
    };
    const int64_t n_tiles = (int64_t)((L.out_dim + 15) / 16) * L.nseg;
    const int64_t tile_work = fg ? 2 * n_tiles : n_tiles;   // 16-row tiles to stream (fused: 2 per unit)
    const bool al16 = (reinterpret_cast<uintptr_t>(L.s) % 16 == 0) && (reinterpret_cast<uintptr_t>(L.b) % 16 == 0);
    // Scales/biases of a full-K row block: 2D TMA when rows are 16-byte multiples, else 1D
    // TMA of the contiguous block when it fits the raw staging budget, else element copies.
    int sbm_full = kSbPlain;
    if (G % 8 == 0 && al16)
        sbm_full = kSbTma;
    else if (al16 && L.tensor_rows * G < ((int64_t)1 << 31) - kRawBox &&
             (uint64_t)(16 * mt) * (uint64_t)G + 7u <= kRawBudget)
        sbm_full = kSbRaw;
    auto sbmode = [&](int c) { return c == 1 ? sbm_full : kSbTma; };
    // Row-block height with c-CTA clusters: plain dense products whose clusters get at most 2 or
    // 4 tiles run the kernel built for row blocks of that height (the default height would spend
    // mma work on absent rows). Decided per candidate c, so that the shared-memory fit of c is
    // judged with the row blocks c would run.
    const bool short_ok = MAXSEG == kDenseMaxSeg && !fg && !L.rmsnorm && cb == 4 && nt <= 2;
    const int mt_default = mt;
    auto mt_for = [&](int c) {
        if (!short_ok) return mt_default;
        const int64_t clusters = di.sm_count / c;
        const int64_t per = (n_tiles + clusters - 1) / clusters;
        return per <= 2 ? 2 : (per <= 4 ? 4 : mt_default);
    };
    auto sbufs = [&](int c) {
        const int64_t clusters = di.sm_count / c;
        const int units = fg ? mt_for(c) / 2 : mt_for(c);
        return (n_tiles + clusters - 1) / clusters <= units && L.nseg == 1 ? 1 : 2;
    };
    auto fits = [&](int c, int stages) {
        const int g = slice(c);
        if (c > 1 && sbm_full != kSbTma) return false;
        if (c > 1 && (int64_t)g * (c - 1) >= G) return false;
        if (xfrag_bytes(g, ntm) > (uint32_t)kXFragBudget) return false;
        return (int)(smem_layout(nt, mt_for(c), stages, g, ntm, sbmode(c), sbufs(c), cb, 0, rawd).total + 1024) <=
               di.max_smem_optin;
    };
    int C = 0;
    for (int c = 1; c <= 8; c *= 2) {
        if (!fits(c, 3)) continue;
        if (C == 0) C = c;                       // smallest that fits at all
        const int q = cluster_capacity(nt, L.rmsnorm, L.experts, c,
                                       smem_layout(nt, mt_for(c), 3, slice(c), ntm, sbmode(c), sbufs(c), cb, 0, rawd).total +
                                           1024,
                                       cb, fg);
        if (q <= 0) continue;
        if (tile_work >= 3 * (int64_t)q && 10 * (int64_t)q * c >= 9 * (int64_t)di.sm_count) {
            C = c;
            break;
        }
        if (c == C && tile_work >= 3 * (int64_t)q) break;
    }
    if (C == 0) return Q4A_ERR_UNSUPPORTED;
    const int gs = slice(C);
    if (mt_for(C) < mt) {
        mt = mt_for(C);
        mt_units = mt;
    }
    int stages = 8;
    while (stages > 2 && !fits(C, stages)) --stages;
    if (!fits(C, stages)) return Q4A_ERR_UNSUPPORTED;
    const SmemLayout lay = smem_layout(nt, mt, stages, gs, ntm, sbmode(C), sbufs(C), cb, 0, rawd);
    if (L.plan_only) return Q4A_OK;

    static thread_local GemvParams<MAXSEG> prm;   // large: keep it off the stack
    memset(&prm, 0, sizeof(prm));
    GemvLaunch Lw = L;
    Lw.withhold_stage = take_withhold_stage();
    q4a_status st = fill_op(prm.op, Lw, gs, mt_units, sbmode(C), mt, lay.sb_pitch);
    if (st != Q4A_OK) return st;
    prm.cluster = C;
    prm.nseg = L.nseg;
    prm.stages = stages;
    prm.lay = lay;
    for (int i = 0; i < L.nseg; ++i) prm.seg[i] = L.seg[i];

    const uint32_t smem_bytes = lay.total + 1024;
    if constexpr (MAXSEG == kDenseMaxSeg) {
        if (fg) {
            if (L.rmsnorm) {
                if (nt == 1) return launch_variant<1, true, MAXSEG, 4, true>(prm, smem_bytes, stream);
                if (nt == 2) return launch_variant<2, true, MAXSEG, 4, true>(prm, smem_bytes, stream);
                return launch_variant<4, true, MAXSEG, 4, true>(prm, smem_bytes, stream);
            }
            if (nt == 1) return launch_variant<1, false, MAXSEG, 4, true>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 4, true>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 4, true>(prm, smem_bytes, stream);
        }
        if (cb == 2) {
            if (nt == 1) return launch_variant<1, false, MAXSEG, 2>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 2>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 2>(prm, smem_bytes, stream);
        }
        if (cb == 3) {
            if (nt == 1) return launch_variant<1, false, MAXSEG, 3>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 3>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 3>(prm, smem_bytes, stream);
        }
        if (L.rmsnorm && L.inj_out) {   // the injection prologue: its own kernels
            if (nt == 1) return launch_variant<1, true, MAXSEG, 4, false, 0, false, true>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, true, MAXSEG, 4, false, 0, false, true>(prm, smem_bytes, stream);
            return launch_variant<4, true, MAXSEG, 4, false, 0, false, true>(prm, smem_bytes, stream);
        }
        if (L.rmsnorm) {
            if (nt == 1) return launch_variant<1, true, MAXSEG>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, true, MAXSEG>(prm, smem_bytes, stream);
            return launch_variant<4, true, MAXSEG>(prm, smem_bytes, stream);
        }
    }
    if constexpr (MAXSEG != kDenseMaxSeg) {
        if (rawd && sbmode(C) == kSbRaw) {   // short rows: scales and biases read in place
            if (nt == 1) return launch_variant<1, false, MAXSEG, 4, false, 0, false, false, true>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 4, false, 0, false, false, true>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 4, false, 0, false, false, true>(prm, smem_bytes, stream);
        }
        if (fg) {   // routed experts' fused gate|up with the activation in the epilogue
            if (nt == 1) return launch_variant<1, false, MAXSEG, 4, true>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 4, true>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 4, true>(prm, smem_bytes, stream);
        }
        // routed low-bit experts, binary16 or fp32 activations
        if (cb == 2 && !L.x_f32) {
            if (nt == 1) return launch_variant<1, false, MAXSEG, 2>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 2>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 2>(prm, smem_bytes, stream);
        }
        if (cb == 3 && !L.x_f32) {
            if (nt == 1) return launch_variant<1, false, MAXSEG, 3>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 3>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 3>(prm, smem_bytes, stream);
        }
        if (cb == 2) {
            if (nt == 1) return launch_variant<1, false, MAXSEG, 2, false, 0, true>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 2, false, 0, true>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 2, false, 0, true>(prm, smem_bytes, stream);
        }
        if (cb == 3) {
            if (nt == 1) return launch_variant<1, false, MAXSEG, 3, false, 0, true>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, false, MAXSEG, 3, false, 0, true>(prm, smem_bytes, stream);
            return launch_variant<4, false, MAXSEG, 3, false, 0, true>(prm, smem_bytes, stream);
        }
    }
    if constexpr (MAXSEG == kDenseMaxSeg) {
        if (nt == 1 && mt == 2) return launch_variant<1, false, MAXSEG, 4, false, 2>(prm, smem_bytes, stream);
        if (nt == 1 && mt == 4) return launch_variant<1, false, MAXSEG, 4, false, 4>(prm, smem_bytes, stream);
        if (nt == 2 && mt == 2) return launch_variant<2, false, MAXSEG, 4, false, 2>(prm, smem_bytes, stream);
    }
    if (nt == 1) return launch_variant<1, false, MAXSEG>(prm, smem_bytes, stream);
    if (nt == 2) return launch_variant<2, false, MAXSEG>(prm, smem_bytes, stream);
    return launch_variant<4, false, MAXSEG>(prm, smem_bytes, stream);
}

}  // namespace

q4a_status launch_gemv(const GemvLaunch& L, cudaStream_t stream) {
    if (L.experts) return launch_gemv_t<Q4A_MAX_SEGMENTS>(L, stream);
    return launch_gemv_t<kDenseMaxSeg>(L, stream);
}

q4a_status read_and_clear_device_error(cudaStream_t stream, uint32_t* word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t v = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *word = v;
    return Q4A_OK;
}

}  // namespace q4a
