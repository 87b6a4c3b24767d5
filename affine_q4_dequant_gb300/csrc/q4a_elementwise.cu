// q4a_elementwise.cu -- the bandwidth-bound helpers around the GEMV:
//   q4a_pack           (A1) codes -> 4-bit rows
//   q4a_xsum           (A2) per-64-group sums of fp16 activations
//   q4a_silu_mul_xsum  (A7) h = fp16(silu(gate) * up) plus group sums of h
//   q4a_moe_combine    routing-weighted sum of expert rows plus the gated shared expert
//   a NaN fill for routed-expert segments with an out-of-range expert id,
//   q4a_quantize       a 4-bit min/max quantiser for float weights (prefill helper)
//   q4a_gemv_f32x      the projection straight from fp32 activations (prefill helper).
// The elementwise ones are grid-stride kernels over 16-byte vectors, sized to a multiple
// of the SM count, with no shared memory and no waits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4a_internal.h"
#include "q4a_prefill.h"

namespace q4a {
namespace {

// Programmatic dependent launch (see the GEMV kernel): wait for the previous kernel of
// the stream before touching any global data, and let the next one start early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_nc_16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Byte k of the output = code[2k] | code[2k+1] << 4: every output 16-byte vector
// packs 32 consecutive codes (two input vectors). Codes are masked to 4 bits.
// It lets dependent kernels launch only after its last store, behind a device-scope fence;
// the GEMV kernels still read weights only after griddepcontrol.wait (the previous kernel
// complete and its memory visible).
__global__ void pack_kernel(uint4* __restrict__ out, const uint4* __restrict__ in, int64_t n_out_vec) {
    grid_dep_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_out_vec;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 a = ld_nc_16(in + 2 * i);
        const uint4 c = ld_nc_16(in + 2 * i + 1);
        const uint32_t src[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        uint32_t dst[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // two input words (8 codes) -> one output word
            const uint32_t lo = src[2 * k] & 0x0F0F0F0Fu;       // codes 0..3, one per byte
            const uint32_t hi = src[2 * k + 1] & 0x0F0F0F0Fu;   // codes 4..7
            // bytes (c0,c1,c2,c3) -> (c0 | c1<<4, c2 | c3<<4) in the low half word
            const uint32_t plo = (lo | (lo >> 4)) & 0x00FF00FFu;      // (c0|c1<<4) at byte 0, (c2|c3<<4) at byte 2
            const uint32_t phi = (hi | (hi >> 4)) & 0x00FF00FFu;
            dst[k] = __byte_perm(plo, phi, 0x6420);
        }
        out[i] = make_uint4(dst[0], dst[1], dst[2], dst[3]);
    }
    __threadfence();
    grid_dep_launch();
}

// Derived low-bit codes, one thread per 32-code chunk: 16 bytes of nibbles in, the chunk's
// two words of 2-bit codes q4 >> 2 out, and (when wlo is set) its word of lowest bits of the
// 3-bit codes q4 >> 1. Byte b of word t holds in bit field j the code of element
// 2 * (8t + 4 * (j & 1) + b) + (j >> 1); the lowest bit of that element is bit 4t + j of
// byte b of the lowest-bit word.
__global__ void lowbit_pack_kernel(uint2* __restrict__ w2, uint32_t* __restrict__ wlo,
                                   const uint4* __restrict__ in, int64_t n_chunks) {
    grid_dep_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_chunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 a = ld_nc_16(in + i);
        const uint32_t src[4] = {a.x, a.y, a.z, a.w};   // byte k: element 2k (low), 2k + 1 (high)
        uint32_t up[2] = {0u, 0u}, lo = 0u;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int e = 2 * (8 * t + 4 * (j & 1) + b) + (j >> 1);
                    const uint32_t q = (src[e >> 3] >> (8 * ((e >> 1) & 3) + 4 * (e & 1))) & 15u;
                    up[t] |= (q >> 2) << (8 * b + 2 * j);
                    lo |= ((q >> 1) & 1u) << (8 * b + 4 * t + j);
                }
        w2[i] = make_uint2(up[0], up[1]);
        if (wlo) wlo[i] = lo;
    }
    __threadfence();
    grid_dep_launch();
}

// Min/max quantiser, every step in binary32 (it decides the integer codes):
// b = bf16(min), s = bf16((max - b) / 15) when max > b, else 0, and
// q = clamp(rint((w - b) / s), 0, 15) (0 when s = 0), with b and s their bfloat16 values.
// Four lanes per 64-input group: lane j loads float4 number 4k + j of the group (k = 0..3), so
// the four lanes of a group read 64 contiguous bytes per load; the group's min and max meet
// over two xor shuffles, and each lane writes the two packed bytes of each of its vectors.
__global__ void quantize_kernel(uint8_t* __restrict__ packed, uint16_t* __restrict__ s_out,
                                uint16_t* __restrict__ b_out, const float4* __restrict__ w, int64_t n_groups) {
    grid_dep_wait();
    const int j = threadIdx.x & 3;
    const int64_t n_threads = n_groups * 4;
    // warp-uniform trip count (the shuffles take every lane); lanes past the end load zeros
    for (int64_t ti = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; ti - (threadIdx.x & 31) < n_threads;
         ti += (int64_t)gridDim.x * blockDim.x) {
        const int64_t gi = ti >> 2;
        const bool live = gi < n_groups;
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = live ? w[gi * 16 + 4 * k + j] : make_float4(0.f, 0.f, 0.f, 0.f);
        float mn = v[0].x, mx = v[0].x;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mn = fminf(fminf(fminf(fminf(mn, v[k].x), v[k].y), v[k].z), v[k].w);
            mx = fmaxf(fmaxf(fmaxf(fmaxf(mx, v[k].x), v[k].y), v[k].z), v[k].w);
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
        // a zero minimum is stored as +0 (min/max leave the sign of a zero undefined)
        const __nv_bfloat16 bb = __float2bfloat16_rn(mn == 0.0f ? 0.0f : mn);
        const float bf = __bfloat162float(bb);
        const float range = __fsub_rn(mx, bf);
        const __nv_bfloat16 sb = range > 0.0f ? __float2bfloat16_rn(__fdiv_rn(range, 15.0f)) : __float2bfloat16_rn(0.0f);
        const float sf = __bfloat162float(sb);
        if (!live) continue;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float e[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            uint32_t q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                q[t] = 0u;
                if (sf > 0.0f) {
                    const float r = rintf(__fdiv_rn(__fsub_rn(e[t], bf), sf));
                    q[t] = r < 0.0f ? 0u : (r > 15.0f ? 15u : (uint32_t)r);
                }
            }
            // elements 4(4k + j) .. +3: bytes 2(4k + j) and 2(4k + j) + 1 of the group's 32
            const uint16_t two = (uint16_t)(q[0] | (q[1] << 4) | (q[2] << 8) | (q[3] << 12));
            *reinterpret_cast<uint16_t*>(packed + gi * 32 + 2 * (4 * k + j)) = two;
        }
        if (j == 0) {
            s_out[gi] = __bfloat16_as_ushort(sb);
            b_out[gi] = __bfloat16_as_ushort(bb);
        }
    }
    __threadfence();
    grid_dep_launch();
}

// y = W x from fp32 activations, for a few output rows over any number of activation rows:
// one warp per (output row, block of up to 4 activation rows). Lane l takes the 32-bit code
// words l, l + 32, ... of the row (word wi holds elements 8wi .. 8wi+7, element 8wi + e in
// nibble e); per word and activation row sum(q x) and sum(x) in fp32, then
// acc += s * sum(q x) + b * sum(x) with the word's group scale and bias; a fixed xor-shuffle
// tree sums the lanes.
__global__ void gemv_f32x_kernel(float* __restrict__ y, const uint32_t* __restrict__ w,
                                 const uint16_t* __restrict__ s, const uint16_t* __restrict__ b,
                                 const float* __restrict__ x, int64_t nb, int64_t out_dim, int64_t in_dim) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t n_tb = (nb + 3) / 4;
    const int64_t n_items = out_dim * n_tb;
    const int64_t words = in_dim / 8;
    const int64_t groups = in_dim / 64;
    for (int64_t item = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; item < n_items;
         item += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t o = item / n_tb;
        const int64_t r0 = (item - o * n_tb) * 4;
        const int nr = (int)(nb - r0 < 4 ? nb - r0 : 4);
        const uint32_t* wr = w + o * words;
        const uint16_t* sr = s + o * groups;
        const uint16_t* br = b + o * groups;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int64_t wi = lane; wi < words; wi += 32) {
            const uint32_t wd = __ldg(wr + wi);
            const float sv = __bfloat162float(__ushort_as_bfloat16(__ldg(sr + (wi >> 3))));
            const float bv = __bfloat162float(__ushort_as_bfloat16(__ldg(br + (wi >> 3))));
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (t < nr) {
                    const float4* xr = reinterpret_cast<const float4*>(x + (r0 + t) * in_dim + wi * 8);
                    const float4 x0 = __ldg(xr), x1 = __ldg(xr + 1);
                    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    float qd = 0.f, xs = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        qd = fmaf((float)((wd >> (4 * e)) & 15u), xv[e], qd);
                        xs += xv[e];
                    }
                    acc[t] = fmaf(sv, qd, fmaf(bv, xs, acc[t]));
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
        }
        if (lane < nr) {
            float v = acc[0];
#pragma unroll
            for (int t = 1; t < 4; ++t) v = lane == t ? acc[t] : v;
            y[(r0 + lane) * out_dim + o] = v;
        }
    }
    __threadfence();
    grid_dep_launch();
}

// One thread per (row, group): 8 vectors of 8 halves summed in fp32 in index order.
__global__ void xsum_kernel(float* __restrict__ xsum, const __half* __restrict__ x, int64_t n_groups_total) {
    grid_dep_wait();
    grid_dep_launch();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_groups_total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const __half* p = x + i * kGroup;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = ld_nc_16(p + 8 * k);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __half2 h = *reinterpret_cast<const __half2*>(&w[q]);
                acc += __low2float(h);
                acc += __high2float(h);
            }
        }
        xsum[i] = acc;
    }
}

// One thread per 8 outputs; 8 consecutive lanes cover one 64-group and sum it with
// shuffles (the sum of the fp16-rounded values, as the activation step hands them on).
__global__ void silu_mul_kernel(uint16_t* __restrict__ h, float* __restrict__ hsum,
                                const float* __restrict__ gate_up, int64_t rows, int64_t inter) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t per_row = inter / 8;
    const int64_t total = rows * per_row;
    for (int64_t base = blockIdx.x * (int64_t)blockDim.x; base < total; base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const bool live = i < total;
        float part = 0.f;
        if (live) {
            const int64_t r = i / per_row;
            const int64_t j = (i - r * per_row) * 8;
            const float* gp = gate_up + r * 2 * inter + j;
            const float4 g0 = *reinterpret_cast<const float4*>(gp);
            const float4 g1 = *reinterpret_cast<const float4*>(gp + 4);
            const float4 u0 = *reinterpret_cast<const float4*>(gp + inter);
            const float4 u1 = *reinterpret_cast<const float4*>(gp + inter + 4);
            const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            uint32_t out[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a = gv[2 * k] / (1.0f + expf(-gv[2 * k])) * uv[2 * k];
                const float c = gv[2 * k + 1] / (1.0f + expf(-gv[2 * k + 1])) * uv[2 * k + 1];
                const __half2 hv = __floats2half2_rn(a, c);
                out[k] = *reinterpret_cast<const uint32_t*>(&hv);
                part += __low2float(hv) + __high2float(hv);
            }
            *reinterpret_cast<uint4*>(h + r * inter + j) = make_uint4(out[0], out[1], out[2], out[3]);
        }
        // lanes 8k..8k+7 hold one 64-group (inter % 64 == 0 and 32 % 8 == 0)
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        if (live && hsum && (threadIdx.x & 7) == 0) hsum[i / 8] = part;
    }
}

__global__ void fill_nan_kernel(uint32_t* __restrict__ y, int64_t n, uint32_t pattern) {
    grid_dep_wait();
    grid_dep_launch();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        y[i] = pattern;
}

// Routed-expert combine ("BATCH_MSL" page, experts.metal fn_moe_combine_b and
// fn_shared_add_rows):
//     out[t][i] = sum_k w[t][k] * y[slot[t][k]][i]  (+ sigmoid(gate . x[t]) * y_shared[t][i]).
// One CTA per (token, kCombineChunk outputs), 4 outputs per thread. The k terms are added
// in k order and the gate dot reduces in a fixed tree, so the result is deterministic; like
// the pages, every CTA of a token recomputes the gate dot. A slot outside [0, n_slots)
// makes the token's row NaN.
constexpr int kCombineThreads = 256;
constexpr int kCombineChunk = 4 * kCombineThreads;

__global__ void __launch_bounds__(kCombineThreads)
    moe_combine_kernel(float* __restrict__ out, const float* __restrict__ y, const int32_t* __restrict__ slot,
                       const float* __restrict__ w, int top_k, int64_t n_slots, int64_t hidden, int nchunk,
                       const float* __restrict__ y_shared, const uint16_t* __restrict__ gate,
                       const float* __restrict__ x) {
    __shared__ int32_t s_slot[kCombineMaxK];
    __shared__ float s_w[kCombineMaxK];
    __shared__ float s_red[kCombineThreads / 32];
    __shared__ int s_bad;
    grid_dep_wait();
    const int64_t t = blockIdx.x / nchunk;
    const int c = (int)(blockIdx.x % nchunk);
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if ((int)threadIdx.x < top_k) {
        const int32_t sl = slot[t * top_k + threadIdx.x];
        s_slot[threadIdx.x] = sl;
        s_w[threadIdx.x] = w[t * top_k + threadIdx.x];
        if (sl < 0 || (int64_t)sl >= n_slots) atomicOr(&s_bad, 1);
    }
    if (y_shared) {
        const float* xr = x + t * hidden;
        float part = 0.f;
        for (int64_t j = threadIdx.x; j < hidden; j += kCombineThreads)
            part = fmaf(__uint_as_float((uint32_t)gate[j] << 16), xr[j], part);
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = part;
    }
    __syncthreads();
    float g = 0.f;
    if (y_shared) {
        float dot = 0.f;
        for (int i = 0; i < kCombineThreads / 32; ++i) dot += s_red[i];
        g = 1.f / (1.f + expf(-dot));
    }
    const int64_t i0 = (int64_t)c * kCombineChunk + 4 * (int64_t)threadIdx.x;
    if (i0 < hidden) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s_bad) {
            const float nan = __int_as_float(0x7fc00000);
            acc = make_float4(nan, nan, nan, nan);
        } else {
            for (int k = 0; k < top_k; ++k) {
                const float4 v = *reinterpret_cast<const float4*>(y + (int64_t)s_slot[k] * hidden + i0);
                const float wk = s_w[k];
                acc.x = fmaf(wk, v.x, acc.x);
                acc.y = fmaf(wk, v.y, acc.y);
                acc.z = fmaf(wk, v.z, acc.z);
                acc.w = fmaf(wk, v.w, acc.w);
            }
            if (y_shared) {
                const float4 v = *reinterpret_cast<const float4*>(y_shared + t * hidden + i0);
                acc.x = fmaf(g, v.x, acc.x);
                acc.y = fmaf(g, v.y, acc.y);
                acc.z = fmaf(g, v.z, acc.z);
                acc.w = fmaf(g, v.w, acc.w);
            }
        }
        *reinterpret_cast<float4*>(out + t * hidden + i0) = acc;
    }
    grid_dep_launch();
}

template <typename... KArgs, typename... Args>
q4a_status launch_pdl(void (*kern)(KArgs...), int grid, int block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    return e == cudaSuccess ? Q4A_OK : cuda_fail(e);
}

int grid_for(int64_t work, int threads) {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

q4a_status launch_pack(uint8_t* w_packed, const uint8_t* codes, int64_t rows, int64_t in_dim,
                       cudaStream_t stream) {
    const int64_t n_out_vec = rows * in_dim / 32;
    return launch_pdl(pack_kernel, grid_for(n_out_vec, 256), 256, stream, reinterpret_cast<uint4*>(w_packed),
                      reinterpret_cast<const uint4*>(codes), n_out_vec);
}

q4a_status launch_lowbit_pack(uint8_t* w_up, uint8_t* w_lo, const uint8_t* w_packed, int64_t rows,
                              int64_t in_dim, cudaStream_t stream) {
    const int64_t n = rows * in_dim / 32;
    return launch_pdl(lowbit_pack_kernel, grid_for(n, 256), 256, stream, reinterpret_cast<uint2*>(w_up),
                      reinterpret_cast<uint32_t*>(w_lo), reinterpret_cast<const uint4*>(w_packed), n);
}

q4a_status launch_quantize(uint8_t* w_packed, uint16_t* s, uint16_t* b, const float* w, int64_t rows,
                           int64_t in_dim, cudaStream_t stream) {
    const int64_t n = rows * (in_dim / kGroup);
    return launch_pdl(quantize_kernel, grid_for(4 * n, 256), 256, stream, w_packed, s, b,
                      reinterpret_cast<const float4*>(w), n);
}

q4a_status launch_gemv_f32x(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b, const float* x,
                            int64_t nb, int64_t out_dim, int64_t in_dim, cudaStream_t stream) {
    const int64_t warps = out_dim * ((nb + 3) / 4);
    return launch_pdl(gemv_f32x_kernel, grid_for(warps * 32, 256), 256, stream, y,
                      reinterpret_cast<const uint32_t*>(w), s, b, x, nb, out_dim, in_dim);
}

q4a_status launch_xsum(float* xsum, const uint16_t* x, int64_t nb, int64_t in_dim, cudaStream_t stream) {
    const int64_t n = nb * in_dim / kGroup;
    return launch_pdl(xsum_kernel, grid_for(n, 256), 256, stream, xsum, reinterpret_cast<const __half*>(x), n);
}

q4a_status launch_silu_mul_xsum(uint16_t* h, float* hsum, const float* gate_up, int64_t rows,
                                int64_t inter, cudaStream_t stream) {
    const int64_t n = rows * inter / 8;
    return launch_pdl(silu_mul_kernel, grid_for(n, 256), 256, stream, h, hsum, gate_up, rows, inter);
}

q4a_status launch_moe_combine(float* out, const float* y, const int32_t* slot, const float* w, int n_tok,
                              int top_k, int64_t n_slots, int64_t hidden, const float* y_shared,
                              const uint16_t* gate, const float* x, cudaStream_t stream) {
    const int nchunk = (int)((hidden + kCombineChunk - 1) / kCombineChunk);
    return launch_pdl(moe_combine_kernel, n_tok * nchunk, kCombineThreads, stream, out, y, slot, w, top_k,
                      n_slots, hidden, nchunk, y_shared, gate, x);
}

q4a_status launch_fill_nan(float* y, int64_t row0, int64_t nrows, int64_t out_dim, cudaStream_t stream) {
    const int64_t n = nrows * out_dim;
    return launch_pdl(fill_nan_kernel, grid_for(n, 256), 256, stream, reinterpret_cast<uint32_t*>(y + row0 * out_dim), n,
                      0x7fc00000u);
}

q4a_status launch_fill_nan_h(uint16_t* h, int64_t row0, int64_t nrows, int64_t inter, cudaStream_t stream) {
    const int64_t n = nrows * inter / 2;   // inter is even: pairs of binary16 NaNs
    return launch_pdl(fill_nan_kernel, grid_for(n, 256), 256, stream, reinterpret_cast<uint32_t*>(h + row0 * inter), n,
                      0x7e007e00u);
}

}  // namespace q4a
