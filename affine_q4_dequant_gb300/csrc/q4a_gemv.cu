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
//  * Consumer warp (wr, wg) takes group slots {wg, wg+4} of every 8-group stage
//    for the tiles of row half wr. Per 16-row tile and group it runs 4 steps of
//    mma.sync m16n8k16 (f16 in, f32 accumulate) per 8 activation rows: the A
//    operand is the raw codes, pulled out of each 32-bit word by masks into
//    binary16 subnormals (code * 2^-24, exact); the high nibble of a byte lands
//    at 16x and the matching activations are pre-scaled by 1/16. A dot product
//    does not depend on the order of its terms, so every thread feeds the words
//    ldmatrix gives it and the activation fragments carry the same permutation.
//    The per-group result is scaled by s (times 2^24) and b*xsum is added, both
//    in fp32: the tensor cores never see a rounded weight.
#include <cuda_fp16.h>

#include <map>
#include <mutex>

#include "q4a_internal.h"

namespace q4a {

__device__ uint32_t g_device_error;

namespace {

// ---- PTX wrappers ----------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: after kWaitLimitNs the thread records the failure in the device
// error word and in the CTA's abort flag, then carries on. Control flow never
// depends on shared-memory data, so a give-up can only produce garbage values,
// never a hang, a skipped barrier or an out-of-range address.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 31) == 0) {
            if (*abort_flag) return;
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(&g_device_error, 1u);
                *abort_flag = 1u;
                return;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
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

__device__ __forceinline__ uint4 ld_nc_16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

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

// ---- activation staging -----------------------------------------------------------------

// Writes the CTA's K-slice of the activation rows of one segment as mma B fragments
// (xfrag) and fp32 group sums (xsum). Item (tok, gl, t) covers elements 8t..8t+7 and
// 32+8t..32+8t+7 of group gl for activation row tok; the four t of an item sit in one
// lane quad, which sums its group.
template <int NT, bool RMS, class P>
__device__ void stage_x(const P& p, const Segment& sg, int kg0, int gsz, uint8_t* xfrag,
                        float* xsum_s, const float* inv_s, int ctid) {
    constexpr int NTOK = NT * 8;
    const int items = NTOK * gsz * 4;
    const uint32_t scale_odd = 0x2C002C00u;   // half2(1/16, 1/16)
    for (int base = 0; base < items; base += kConsumerWarps * 32) {
        const int i = base + ctid;
        const bool live = i < items;
        const int t = i & 3;
        const int rest = i >> 2;
        const int gl = live ? rest % gsz : 0;
        const int tok = live ? rest / gsz : 0;
        uint32_t v[4] = {0, 0, 0, 0}, u[4] = {0, 0, 0, 0};
        float part = 0.f;
        if (live && tok < sg.ntok) {
            const int slot = sg.tok0 + tok;
            const int64_t src = p.x_rows ? (int64_t)p.x_rows[slot] : (int64_t)slot;
            const int64_t col = (int64_t)(kg0 + gl) * kGroup + 8 * t;
            if constexpr (!RMS) {
                const __half* xr = static_cast<const __half*>(p.x) + src * p.in_dim + col;
                const uint4 a = ld_nc_16(xr);
                const uint4 c = ld_nc_16(xr + 32);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                u[0] = c.x; u[1] = c.y; u[2] = c.z; u[3] = c.w;
            } else {
                const float* xr = static_cast<const float*>(p.x) + src * p.in_dim + col;
                const float inv = inv_s[tok];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const float4 f0 = *reinterpret_cast<const float4*>(xr + 32 * half);
                    const float4 f1 = *reinterpret_cast<const float4*>(xr + 32 * half + 4);
                    const uint4 wv = ld_nc_16(p.norm_w + col + 32 * half);
                    const float xs[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
                    uint32_t* dst = half ? u : v;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float w0 = bf16_to_f32(ww[k] & 0xFFFFu) + p.shift;
                        const float w1 = bf16_to_f32(ww[k] >> 16) + p.shift;
                        __half2 h = __floats2half2_rn(xs[2 * k] * inv * w0, xs[2 * k + 1] * inv * w1);
                        dst[k] = *reinterpret_cast<uint32_t*>(&h);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) part += half2_sum(v[k]) + half2_sum(u[k]);
        }
        // B fragments for the 4 mma steps: step j pairs element j with j+4 (v: words t,
        // u: words t+4). Odd steps come from the high nibbles (16x) -> scale by 1/16.
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
            const int nt = tok >> 3;
            const int lane = ((tok & 7) << 2) | t;
            uint8_t* f = xfrag + ((size_t)(gl * NT + nt) * 2) * 512 + lane * 16;
            *reinterpret_cast<uint4*>(f) = make_uint4(b01[0], b23[0], b01[1], b23[1]);
            *reinterpret_cast<uint4*>(f + 512) = make_uint4(b01[2], b23[2], b01[3], b23[3]);
            if (t == 0) xsum_s[gl * NTOK + tok] = part;
        }
    }
}

// ---- the kernel --------------------------------------------------------------------------

template <int NT, bool RMS, int MAXSEG>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ GemvParams<MAXSEG> p) {
    constexpr int NTOK = NT * 8;
    constexpr int TPW = (NT <= 2) ? 4 : 2;   // tiles per consumer warp (row half)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemLayout& L = p.lay;
    uint8_t* ring = smem + L.ring;
    uint8_t* xfrag = smem + L.xfrag;
    float* xsum_s = reinterpret_cast<float*>(smem + L.xsum);
    float* wpart = reinterpret_cast<float*>(smem + L.wpart);
    float* cpart = reinterpret_cast<float*>(smem + L.cpart);
    float* ssq_s = reinterpret_cast<float*>(smem + L.ssq);   // [NTOK] sum of squares, [NTOK] inv
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 2 * p.stages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int C = p.cluster;
    const int crank = (int)cluster_rank();
    const int cid = blockIdx.x / C;

    // This CTA's K-slice (in groups) and its stage count per row block.
    const int kg0 = crank * p.gs;
    const int kg1 = min(p.groups, kg0 + p.gs);
    const int gsz = kg1 - kg0;
    const int nks = (gsz + kStageGroups - 1) / kStageGroups;

    // This cluster's tile range.
    const int t_begin = (int)(((int64_t)cid * p.n_tiles) / p.n_clusters);
    const int t_end = (int)(((int64_t)(cid + 1) * p.n_tiles) / p.n_clusters);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(bars + s), 33);                   // TMA arrive + 32 copy arrivals
            mbar_init(smem_addr(bars + S + s), kConsumerWarps);   // one arrival per consumer warp
        }
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ======================= producer warp =======================
        const uint8_t* s8 = reinterpret_cast<const uint8_t*>(p.s);
        const uint8_t* b8 = reinterpret_cast<const uint8_t*>(p.b);
        const int64_t srow_bytes = (int64_t)p.groups * 2;
        int it = 0;
        bool pending = false;   // an un-waited cluster-barrier arrival
        if (RMS) {              // matches the consumers' norm exchange
            cluster_arrive();
            pending = true;
        }
        int t = t_begin;
        Job j;
        while (next_job(p, t, t_end, j)) {
            const Segment& sg = p.seg[j.seg];
            const int64_t lrow0 = (int64_t)j.tile * 16;                 // row within the segment
            const int rows_valid = (int)llmin((int64_t)j.ntile * 16, p.out_dim - lrow0);
            const int64_t trow0 = (int64_t)sg.row0 + lrow0;              // row within the tensor
            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                if (it >= S) mbar_wait(smem_addr(bars + S + s), ph ^ 1u, abort_flag);
                const uint32_t full = smem_addr(bars + s);
                uint8_t* st = ring + (size_t)s * L.stage_bytes;
                const int g0 = kg0 + ks * kStageGroups;
                const int ng = min(kStageGroups, kg1 - g0);
                const int nbox = (ng + 3) / 4;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full, (uint32_t)(j.ntile * nbox * kBoxBytesTotal));
                    for (int m = 0; m < j.ntile; ++m)
                        for (int c = 0; c < nbox; ++c)
                            tma_load_2d(smem_addr(st + (m * 2 + c) * kBoxBytesTotal), &p.tmap_w,
                                        (g0 + 4 * c) * 32, (int)(trow0 + 16 * m), full);
                }
                uint8_t* sdst = st + L.stage_w_bytes;                 // s: [rows][16 B]
                uint8_t* bdst = sdst + (size_t)16 * 16 * p.mt;        // b: [rows][16 B]
                if (p.sb_mode == kSb16) {
                    for (int i = lane; i < 2 * rows_valid; i += 32) {
                        const int r = i >> 1;
                        const bool isb = i & 1;
                        const uint8_t* src = (isb ? b8 : s8) + (trow0 + r) * srow_bytes + (int64_t)g0 * 2;
                        cp_async_16(smem_addr((isb ? bdst : sdst) + r * 16), src);
                    }
                    cp_async_arrive_noinc(full);
                } else if (p.sb_mode == kSb4) {
                    const int per_row = (ng + 1) >> 1;                // 4-byte granules per row
                    for (int i = lane; i < 2 * rows_valid * per_row; i += 32) {
                        const int k = i % per_row;
                        const int rr = i / per_row;
                        const int r = rr >> 1;
                        const bool isb = rr & 1;
                        const uint8_t* src =
                            (isb ? b8 : s8) + (trow0 + r) * srow_bytes + (int64_t)g0 * 2 + 4 * k;
                        cp_async_4(smem_addr((isb ? bdst : sdst) + r * 16 + 4 * k), src);
                    }
                    cp_async_arrive_noinc(full);
                } else {
                    for (int i = lane; i < 2 * rows_valid * ng; i += 32) {
                        const int k = i % ng;
                        const int rr = i / ng;
                        const int r = rr >> 1;
                        const bool isb = rr & 1;
                        const uint16_t v = *reinterpret_cast<const uint16_t*>(
                            (isb ? b8 : s8) + (trow0 + r) * srow_bytes + (int64_t)(g0 + k) * 2);
                        *reinterpret_cast<uint16_t*>((isb ? bdst : sdst) + r * 16 + 2 * k) = v;
                    }
                    mbar_arrive(full);
                }
            }
            if (pending) cluster_wait();
            cluster_arrive();
            pending = true;
        }
        if (pending) cluster_wait();
    } else {
        // ======================= consumer warps =======================
        const int ctid = threadIdx.x;       // 0 .. 255
        const int wr = warp >> 2;           // row half
        const int wg = warp & 3;            // group slot
        const int g = lane >> 2;
        const int tq = lane & 3;

        if (RMS) {
            // Sum of squares of this CTA's K-slice per activation row, exchanged across the
            // cluster so every CTA normalises with the full-row statistics.
            const Segment& sg = p.seg[0];
            for (int tok = warp; tok < NTOK; tok += kConsumerWarps) {
                float acc = 0.f;
                if (tok < sg.ntok) {
                    const float* xr = static_cast<const float*>(p.x) +
                                      (int64_t)(sg.tok0 + tok) * p.in_dim + (int64_t)kg0 * kGroup;
                    for (int i = lane * 4; i < gsz * kGroup; i += 128) {
                        const float4 f = *reinterpret_cast<const float4*>(xr + i);
                        acc += f.x * f.x + f.y * f.y + f.z * f.z + f.w * f.w;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) ssq_s[tok] = acc;
            }
            cluster_arrive();
            cluster_wait();
            if (ctid < NTOK) {
                float tot = 0.f;
                for (int c = 0; c < C; ++c) tot += ld_peer_f32(map_peer(smem_addr(ssq_s + ctid), c));
                ssq_s[NTOK + ctid] = rsqrtf(tot / (float)p.in_dim + p.eps);
            }
            consumer_sync();
        }

        float acc[TPW][NT][4];
        int staged_seg = -1;
        int it = 0;
        int blk = 0;
        int t = t_begin;
        Job j;
        while (next_job(p, t, t_end, j)) {
            const Segment& sg = p.seg[j.seg];
            if (j.seg != staged_seg) {
                stage_x<NT, RMS>(p, sg, kg0, gsz, xfrag, xsum_s, ssq_s + NTOK, ctid);
                consumer_sync();
                staged_seg = j.seg;
            }
#pragma unroll
            for (int mi = 0; mi < TPW; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[mi][nt][k] = 0.f;

            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                mbar_wait(smem_addr(bars + s), ph, abort_flag);
                const uint8_t* st = ring + (size_t)s * L.stage_bytes;
                const uint8_t* sst = st + L.stage_w_bytes;
                const uint8_t* bst = sst + (size_t)16 * 16 * p.mt;
                const int ng = min(kStageGroups, gsz - ks * kStageGroups);
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    const int gg = wg + 4 * gi;                 // group within the stage
                    if (gg >= ng) continue;
                    const int gl = ks * kStageGroups + gg;       // group within the K-slice
                    uint32_t bf[NT][8];
                    float2 xs[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint8_t* f = xfrag + ((size_t)(gl * NT + nt) * 2) * 512 + lane * 16;
                        const uint4 q0 = *reinterpret_cast<const uint4*>(f);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(f + 512);
                        bf[nt][0] = q0.x; bf[nt][1] = q0.y; bf[nt][2] = q0.z; bf[nt][3] = q0.w;
                        bf[nt][4] = q1.x; bf[nt][5] = q1.y; bf[nt][6] = q1.z; bf[nt][7] = q1.w;
                        xs[nt] = *reinterpret_cast<const float2*>(xsum_s + gl * NTOK + nt * 8 + 2 * tq);
                    }
                    const uint32_t gran0 = (uint32_t)(gg & 3) * 2;
#pragma unroll
                    for (int mi = 0; mi < TPW; ++mi) {
                        const int m = wr * TPW + mi;
                        if (m >= j.ntile) continue;
                        // ldmatrix x4: rows 0-7 / 8-15 of the tile, 16-byte granules gran0 and
                        // gran0+1 of the box (128-byte swizzle: granule ^= row & 7).
                        const uint32_t box = smem_addr(st + (m * 2 + (gg >> 2)) * kBoxBytesTotal);
                        const uint32_t row = (uint32_t)((lane & 7) + ((lane >> 3) & 1) * 8);
                        const uint32_t gran = gran0 + (uint32_t)(lane >> 4);
                        uint32_t w[4];
                        ldsm_x4(box + row * 128 + ((gran ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
                        // scale and bias of rows g and g+8 for this group
                        const int r0 = m * 16 + g;
                        const float s0 = bf16_to_f32(*reinterpret_cast<const uint16_t*>(sst + r0 * 16 + 2 * gg)) * 16777216.0f;
                        const float s1 = bf16_to_f32(*reinterpret_cast<const uint16_t*>(sst + (r0 + 8) * 16 + 2 * gg)) * 16777216.0f;
                        const float bb0 = bf16_to_f32(*reinterpret_cast<const uint16_t*>(bst + r0 * 16 + 2 * gg));
                        const float bb1 = bf16_to_f32(*reinterpret_cast<const uint16_t*>(bst + (r0 + 8) * 16 + 2 * gg));
                        uint32_t h[4][4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t v8 = w[k] >> 8;
                            h[k][0] = w[k] & 0x000F000Fu;
                            h[k][1] = w[k] & 0x00F000F0u;
                            h[k][2] = v8 & 0x000F000Fu;
                            h[k][3] = v8 & 0x00F000F0u;
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                mma_f16(d, h[0][jj], h[1][jj], h[2][jj], h[3][jj], bf[nt][2 * jj],
                                        bf[nt][2 * jj + 1]);
                            float* a = acc[mi][nt];
                            a[0] = fmaf(s0, d[0], fmaf(bb0, xs[nt].x, a[0]));
                            a[1] = fmaf(s0, d[1], fmaf(bb0, xs[nt].y, a[1]));
                            a[2] = fmaf(s1, d[2], fmaf(bb1, xs[nt].x, a[2]));
                            a[3] = fmaf(s1, d[3], fmaf(bb1, xs[nt].y, a[3]));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(bars + S + s));
            }

            // ---- end of the row block: reduce over group slots, then over the cluster ----
            const int R = j.ntile * 16;
#pragma unroll
            for (int mi = 0; mi < TPW; ++mi) {
                const int m = wr * TPW + mi;
                if (m >= j.ntile) continue;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float* w0 = wpart + ((size_t)wg * (16 * p.mt) + m * 16 + g) * NTOK + nt * 8 + 2 * tq;
                    *reinterpret_cast<float2*>(w0) = make_float2(acc[mi][nt][0], acc[mi][nt][1]);
                    *reinterpret_cast<float2*>(w0 + 8 * NTOK) = make_float2(acc[mi][nt][2], acc[mi][nt][3]);
                }
            }
            consumer_sync();
            float* cp = cpart + (size_t)(blk & 1) * (16 * p.mt) * NTOK;
            for (int e = ctid; e < R * NTOK; e += kConsumerWarps * 32) {
                const size_t stride = (size_t)(16 * p.mt) * NTOK;
                cp[e] = ((wpart[e] + wpart[e + stride]) + wpart[e + 2 * stride]) + wpart[e + 3 * stride];
            }
            cluster_arrive();
            cluster_wait();
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
                    const uint32_t off = (uint32_t)((row * NTOK + tok) * 4);
                    float v = 0.f;
                    for (int c = 0; c < C; ++c) v += ld_peer_f32(map_peer(cp_addr + off, (uint32_t)c));
                    p.y[(int64_t)(sg.tok0 + tok) * p.out_dim + lrow0 + row] = v;
                }
            }
            ++blk;
        }
    }
    // No CTA leaves while a peer may still read its shared memory.
    cluster_arrive();
    cluster_wait();
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

struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
    bool ok = false;
};

DeviceInfo device_info() {
    int dev = 0;
    DeviceInfo d;
    if (cudaGetDevice(&dev) != cudaSuccess) return d;
    static DeviceInfo cache[64];
    if (dev < 64 && cache[dev].ok) return cache[dev];
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
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

template <int NT, bool RMS, int MAXSEG>
q4a_status launch_variant(GemvParams<MAXSEG>& prm, uint32_t smem_bytes, cudaStream_t stream) {
    auto kern = gemv_kernel<NT, RMS, MAXSEG>;
    const void* fn = reinterpret_cast<const void*>(kern);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const DeviceInfo di = device_info();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)prm.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = di.sm_count / prm.cluster;
    {
        std::lock_guard<std::mutex> lock(g_cache_mu);
        uint32_t& set = g_smem_set[{fn, dev}];
        if (set < (uint32_t)di.max_smem_optin) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
            if (e != cudaSuccess) return cuda_fail(e);
            set = (uint32_t)di.max_smem_optin;
        }
        const OccKey key{fn, dev, prm.cluster, smem_bytes};
        auto it = g_occ_cache.find(key);
        if (it == g_occ_cache.end()) {
            // How many clusters fit at once (GPC granularity can strand SMs for C > 1).
            cfg.gridDim = dim3((unsigned)(max_clusters * prm.cluster), 1, 1);
            int occ = 0;
            if (cudaOccupancyMaxActiveClusters(&occ, kern, &cfg) != cudaSuccess || occ <= 0) {
                cudaGetLastError();
                occ = max_clusters;
            }
            it = g_occ_cache.emplace(key, occ).first;
        }
        max_clusters = it->second;
    }
    prm.n_clusters = max_clusters < prm.n_tiles ? max_clusters : prm.n_tiles;
    cfg.gridDim = dim3((unsigned)(prm.n_clusters * prm.cluster), 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, prm);
    if (e != cudaSuccess) return cuda_fail(e);
    return Q4A_OK;
}

template <int MAXSEG>
q4a_status launch_gemv_t(const GemvLaunch& L, cudaStream_t stream) {
    static_assert(sizeof(GemvParams<MAXSEG>) < 32000, "kernel parameter block too large");
    const DeviceInfo di = device_info();
    if (!di.ok) return Q4A_ERR_CUDA;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return Q4A_ERR_UNSUPPORTED;
    if (L.nseg > MAXSEG) return Q4A_ERR_SHAPE;

    const int nt = L.max_ntok <= 8 ? 1 : (L.max_ntok <= 16 ? 2 : 4);
    const int mt = nt <= 2 ? 8 : 4;
    const int G = (int)(L.in_dim / kGroup);

    // Cluster size: the smallest power of two whose K-slice of activation fragments fits.
    int C = 1;
    while (C < 8 && ((G + C - 1) / C) * nt * 1024 > kXFragBudget) C *= 2;
    int gs = (G + C - 1) / C;
    if (C > 1) gs = (gs + 3) / 4 * 4;           // slices start on a TMA box boundary
    while (C > 1 && (int64_t)gs * (C - 1) >= G) { C /= 2; gs = (G + C - 1) / C; if (C > 1) gs = (gs + 3) / 4 * 4; }
    if ((int64_t)gs * nt * 1024 > kXFragBudget) return Q4A_ERR_UNSUPPORTED;

    int stages = 4;
    SmemLayout lay = smem_layout(nt, mt, stages, gs);
    while (stages > 2 && (int)(lay.total + 1024) > di.max_smem_optin) lay = smem_layout(nt, mt, --stages, gs);
    if ((int)(lay.total + 1024) > di.max_smem_optin) return Q4A_ERR_UNSUPPORTED;

    static thread_local GemvParams<MAXSEG> prm;   // large: keep it off the stack
    memset(&prm, 0, sizeof(prm));
    const cuuint64_t dims[2] = {(cuuint64_t)(L.in_dim / 2), (cuuint64_t)L.tensor_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(L.in_dim / 2)};
    const cuuint32_t box[2] = {(cuuint32_t)kBoxBytes, 16u};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(&prm.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(L.w), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail_drv(r);

    prm.s = L.s;
    prm.b = L.b;
    prm.x = L.x;
    prm.x_rows = L.x_rows;
    prm.norm_w = L.norm_w;
    prm.y = L.y;
    prm.eps = L.eps;
    prm.shift = L.shift;
    prm.out_dim = L.out_dim;
    prm.in_dim = L.in_dim;
    prm.groups = G;
    prm.gs = gs;
    prm.cluster = C;
    prm.tiles_per_seg = (int)((L.out_dim + 15) / 16);
    prm.nseg = L.nseg;
    prm.n_tiles = prm.tiles_per_seg * L.nseg;
    prm.mt = mt;
    prm.stages = stages;
    const bool al16 = (reinterpret_cast<uintptr_t>(L.s) % 16 == 0) && (reinterpret_cast<uintptr_t>(L.b) % 16 == 0);
    const bool al4 = (reinterpret_cast<uintptr_t>(L.s) % 4 == 0) && (reinterpret_cast<uintptr_t>(L.b) % 4 == 0);
    if (G % 8 == 0 && gs % 8 == 0 && al16)
        prm.sb_mode = kSb16;
    else if (G % 2 == 0 && al4)
        prm.sb_mode = kSb4;
    else
        prm.sb_mode = kSb2;
    prm.lay = lay;
    for (int i = 0; i < L.nseg; ++i) prm.seg[i] = L.seg[i];

    const uint32_t smem_bytes = lay.total + 1024;
    if constexpr (MAXSEG == kDenseMaxSeg) {
        if (L.rmsnorm) {
            if (nt == 1) return launch_variant<1, true, MAXSEG>(prm, smem_bytes, stream);
            if (nt == 2) return launch_variant<2, true, MAXSEG>(prm, smem_bytes, stream);
            return launch_variant<4, true, MAXSEG>(prm, smem_bytes, stream);
        }
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
