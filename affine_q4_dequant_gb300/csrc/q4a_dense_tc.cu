// q4a_dense_tc.cu -- the dense path of q4a_gemv for wide activation batches (NB >= 64).
//
// Operation: the same y as the GEMV kernel (the "BATCH_MSL" constant page,
// quantized_rows.metal, fn_q4_rows_h; dequantisation w = s*q + b as in expert_gemm.metal),
//     y[r][o] = sum_i w[o][i] x[r][i],   w[o][i] = s[o][i/64] * q[o][i] + b[o][i/64].
// At NB >= 64 this is a real contraction (2*NB flops per 0.5625 bytes of weights), so the
// weights are dequantised once per call into binary16 and multiplied on the 5th-generation
// tensor cores: tcgen05.mma kind::f16, A (the weights) in TMEM, B (x) in shared memory,
// fp32 accumulators in TMEM.
//
// Precision: every row o gets a power-of-two factor 2^-e_o that puts its largest possible
// weight, max_g (15|s| + |b|), in [2^-6, 2^-5). The operand holds w' = fp16(w * 2^-e_o),
// computed from exact binary16 operands with one fused multiply-add: the masked code bits are
// the binary16 subnormal q * 2^-24 (16 q * 2^-24 for a high nibble) and the scale operand is
// s' * 2^24 (s' * 2^20), below 2^16 for this range. So |w' 2^e_o - w| <= 2^-11 |w| for every
// weight that is not 2^9 below its row's largest, and at most 2^-20 of the largest otherwise
// (binary16 subnormal spacing); the accumulation is fp32 and the epilogue multiplies by 2^e_o
// (exact).
//
// Why A lives in TMEM: a 128 x N x 16 MMA costs the tensor core about 55 cycles for N <= 64
// and 64 cycles at N = 128, while staging A through shared memory (written by the
// dequantising threads, read by the MMA) adds 64 KB of shared-memory traffic per 64-input
// group of a 256-row unit -- more than the 128 bytes/cycle the SM's shared memory moves in
// that time. tcgen05.st writes the dequantised rows straight into TMEM, so shared memory
// only carries the packed codes and the x tiles.
//
// CTA (480 threads, one per SM, persistent over work units of 256 weight rows = two MMA
// tiles of 128 rows that share every x tile):
//   warp 0       TMA producer of the packed codes (128 bytes x 128 rows per box, 4 groups)
//                into a code ring; it waits only for that ring.
//   warp 1       allocates TMEM; one thread issues the MMAs: per group, per tile,
//                4 x (M 128, N NB, K 16) with A from TMEM; a stage holds two groups, so one
//                barrier handshake covers 16 MMAs; commits free the A stage and the x stage,
//                and signal the accumulator after a unit's last group.
//   warps 2..5   epilogue, one TMEM lane quarter each: exponents of the next unit's rows
//                (ahead of time), then tcgen05.ld of the accumulators, * 2^e, y stores.
//   warps 6..13  dequantisation, one weight row per thread (warp w owns TMEM lane quarter
//                w % 4 of tile (w - 6) / 4): codes from the code ring, scale and bias from
//                global memory, 64 binary16 weights per group into a TMEM A stage.
//   warp 14      TMA producer of the x tile of every group (64 inputs x NB rows).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>

#include "q4a_device.cuh"
#include "q4a_internal.h"

namespace q4a {
namespace {

constexpr int kTcM = 128;                   // rows of one MMA tile (one TMEM lane per row)
constexpr int kTcUm = 2;                    // MMA tiles per work unit
constexpr int kTcUnitRows = kTcM * kTcUm;   // 256
constexpr int kTcChunkGroups = 4;           // groups per code stage: 128 bytes of each row
constexpr int kTcTileBytes = kTcM * 128;    // one 128-row tile of 128-byte rows: 16 KB
constexpr int kTcACols = 32;                // TMEM columns of one tile's group: 64 fp16
constexpr int kTcSG = 2;                    // groups per operand stage (one handshake per 128 inputs)
constexpr int kTcAStages = 2;               // A stages in TMEM: [stage][tile][group][32 columns]
constexpr int kTcWarpProducer = 0;
constexpr int kTcWarpMma = 1;
constexpr int kTcWarpEpi0 = 2;
constexpr int kTcEpiWarps = 4;
constexpr int kTcWarpDq0 = kTcWarpEpi0 + kTcEpiWarps;
constexpr int kTcDqSplit = 1;               // dequantisation threads per weight row (column parts)
constexpr int kTcDqCols = kTcACols / kTcDqSplit;             // TMEM columns per thread and group
constexpr int kTcDqWarps = 4 * kTcUm * kTcDqSplit;
constexpr int kTcWarpX = kTcWarpDq0 + kTcDqWarps;          // x-tile producer
constexpr int kTcThreads = (kTcWarpX + 1) * 32;
constexpr int kTcMaxN = 128;                // activation rows per launch (MMA N, TMEM budget)
constexpr int kTcYCols = 16;                // accumulator columns per TMEM load (tcgen05.ld 32x32b.x16)
// y store boxes: 128 weight rows x YC activation rows fp32, two alternating; YC = 16, or 32 with one
// accumulator set (N > 64), where the MMA waits for the epilogue to drain: half the box handoffs
__host__ __device__ constexpr uint32_t tc_ybox_bytes(int yc) { return (uint32_t)kTcM * (uint32_t)yc * 4u; }
constexpr int kTcEpiBarrier = 1;            // named barrier of the epilogue warps
static_assert(kTcDqWarps * 32 == kTcUnitRows * kTcDqSplit, "kTcDqSplit dequantisation threads per unit row");
static_assert(kTcDqSplit == 1 || kTcDqSplit == 2, "16-byte code chunks (32 weights, 16 TMEM columns) per thread");
static_assert(kTcEpiWarps * 32 == kTcM, "one epilogue thread per TMEM lane");

struct TcLayout {
    uint32_t code;        // code ring: cs stages of kTcUm tiles
    uint32_t code_stage;
    uint32_t xr;          // x ring: xs stages of [kTcSG groups][n_pad rows][128 bytes]
    uint32_t x_stage;
    uint32_t ybuf;        // 2 y store boxes [yc][kTcM] fp32
    uint32_t exps;        // [2][kTcUnitRows] fp32 2^-e of the rows of the next two units
    uint32_t bars;
    uint32_t tmem_slot;
    uint32_t abort;
    uint32_t total;
    int32_t cs, xs;
};

__host__ __device__ inline TcLayout tc_layout(int n_pad, int cs, int xs, int yc) {
    TcLayout L;
    L.cs = cs;
    L.xs = xs;
    L.code = 0;
    L.code_stage = (uint32_t)kTcUm * kTcTileBytes;
    L.xr = L.code + (uint32_t)cs * L.code_stage;
    L.x_stage = (uint32_t)kTcSG * n_pad * 128u;             // n_pad % 16 == 0: 2 KB multiples
    L.ybuf = L.xr + (uint32_t)xs * L.x_stage;
    L.exps = L.ybuf + 2u * tc_ybox_bytes(yc);
    L.bars = L.exps + 2u * kTcUnitRows * 4u;
    // code_full[cs] code_empty[cs] x_full[xs] x_empty[xs] a_full[A] a_empty[A]
    // acc_full[2] acc_empty[2] exp_full[2] exp_empty[2] exp_first
    L.tmem_slot = L.bars + (uint32_t)(2 * cs + 2 * xs + 2 * kTcAStages + 9) * 8u;
    L.abort = L.tmem_slot + 4u;
    L.total = L.abort + 4u;
    return L;
}

struct TcParams {
    CUtensorMap tmap_w;   // uint8 [out_dim][in_dim/2], box 128 bytes x 128 rows, 128B swizzle
    CUtensorMap tmap_x;   // fp16 [nb][in_dim], box 64 x n_pad, 128B swizzle
    CUtensorMap tmap_y;   // fp32 [nb][out_dim], box kTcM x YC, no swizzle (when y_tma)
    const uint16_t* s;    // bf16 [out_dim][groups]
    const uint16_t* b;
    float* y;             // fp32 [nb][out_dim]
    int64_t out_dim;
    int32_t groups;
    int32_t nb;           // activation rows of this launch, 1 .. kTcMaxN
    int32_t n_pad;        // nb rounded up to 16: the MMA N
    int32_t n_units;      // ceil(out_dim / 256)
    int32_t acc_bufs;     // TMEM accumulator sets: 2 lets one unit's epilogue overlap the next
    uint32_t a_col0;      // first TMEM column of the A stages (after the accumulators)
    uint32_t tmem_cols;
    uint32_t idesc;       // tcgen05 instruction descriptor (f16 x f16 -> f32, M 128, N n_pad)
    float silu_div;       // output epilogue silu(y / silu_div) when silu
    int32_t silu;
    int32_t y_tma;        // y leaves through shared memory and TMA stores (else one store per value)
    TcLayout lay;
};

// ---- tcgen05 wrappers --------------------------------------------------------------------

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_alloc(uint32_t slot_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand of 128-byte rows, 128-byte swizzle,
// 8-row groups 1024 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// D (TMEM) += A (TMEM, 128 lanes x 8 columns of fp16 pairs) * B (shared memory descriptor).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 TMEM lanes (this warp's quarter) x N columns from N registers per thread (asynchronous:
// tc_wait_st orders it before the MMA that reads it).
template <int N>
__device__ __forceinline__ void tc_st(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N == 16 || N == 32, "x16 or x32");
    if constexpr (N == 16) {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
            "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
            : "memory");
    } else {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
            "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
            "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
            "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
            "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
            : "memory");
    }
}

// Keeps N registers live up to this point (the sources of an issued tcgen05.st).
template <int N>
__device__ __forceinline__ void keep_live(const uint32_t (&r)[N]) {
#pragma unroll
    for (int i = 0; i < N; i += 8)
        asm volatile("" ::"r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]),
                     "r"(r[i + 6]), "r"(r[i + 7]));
}

// Completion of this thread's earlier tcgen05.st: once per operand stage, before the MMA warp
// is told the stage is ready (a wait after every store would serialise the dequantisation of
// a stage's groups on the store latency).
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// One thread of the (converged) warp returns true.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(pred)::"memory");
    return pred != 0;
}

// Arrives on the mbarrier once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 TMEM lanes (this warp's quarter) x 16 fp32 columns: thread i gets lane base+i. The load
// is asynchronous; tc_ld16_wait completes it and names the registers, so the compiler cannot
// move a use of them above the wait.
__device__ __forceinline__ void tc_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_ld16_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Shared -> global tensor store of one box; completion is tracked per bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most one of this thread's bulk stores may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// All of this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kTcEpiBarrier), "n"(kTcEpiWarps * 32) : "memory");
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 ld_nc_8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Byte k of a packed word holds elements 2k (low nibble) and 2k+1 (high nibble). Returns
// (w[2k], w[2k+1]) as binary16: the byte is copied into both halves and masked to the low
// nibble (half 0) and the high nibble (half 1); as bit patterns the halves are the binary16
// subnormals q * 2^-24 and 16 q * 2^-24 (exact), and one fused multiply-add (subnormal
// operands are not flushed) applies (s' 2^24, s' 2^20) and (b', b').
template <int K>
__device__ __forceinline__ uint32_t dequant_pair(uint32_t word, __half2 sc, __half2 bi) {
    uint32_t t;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(word), "n"(0x4040 | (K << 8) | K));
    t &= 0x00F0000Fu;
    return h2_bits(__hfma2(bits_h2(t), sc, bi));
}

// 2^-e for a row whose largest weight magnitude is at most m: e = floor(log2 m) + 6, so
// m * 2^-e lies in [2^-6, 2^-5); e is clamped to [-126, 126] (2^-e and 2^e stay normal fp32;
// rows whose weights reach 2^121 are out of range and come out non-finite).
__device__ __forceinline__ int row_exponent(float m) {
    if (!(m > 0.f) || !(m <= 3.0e38f)) return 0;
    const int E = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
    int e = E + 6;
    return e < -126 ? -126 : (e > 126 ? 126 : e);
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// max over 8 groups of 15|s| + |b| (bf16 values, exact in fp32)
__device__ __forceinline__ float bound8(uint4 sv, uint4 bv) {
    const uint32_t ss[4] = {sv.x, sv.y, sv.z, sv.w};
    const uint32_t bb[4] = {bv.x, bv.y, bv.z, bv.w};
    float m = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float s0 = fabsf(bf16_to_f32(ss[h] & 0xFFFFu)), s1 = fabsf(bf16_to_f32(ss[h] >> 16));
        const float b0 = fabsf(bf16_to_f32(bb[h] & 0xFFFFu)), b1 = fabsf(bf16_to_f32(bb[h] >> 16));
        m = fmaxf(m, fmaxf(fmaf(15.f, s0, b0), fmaf(15.f, s1, b1)));
    }
    return m;
}

// Row weight bound max_g (15|s[o][g]| + |b[o][g]|) of row row0 + lane, 0 beyond out_dim. The
// warp reads its 32 rows together, 4 rows of 64 groups (4 x 128 bytes) per load instruction
// (one row per thread would touch 32 cache lines per instruction); 8 lanes share a row and
// reduce with shuffles. All 32 lanes must call it.
__device__ __forceinline__ float warp_row_bound(const uint16_t* s, const uint16_t* b, int64_t row0, int64_t out_dim,
                                                int G, int lane) {
    const int sub = lane >> 3, part = lane & 7;
    float mp[8];
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) mp[pp] = 0.f;
    for (int k0 = 0; k0 < G; k0 += 64) {
        const int g = k0 + part * 8;
        uint4 sv[8], bv[8];
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) {
            const int64_t row = row0 + pp * 4 + sub;
            const bool on = g < G && row < out_dim;
            sv[pp] = on ? ld_nc_16(s + row * G + g) : make_uint4(0, 0, 0, 0);
            bv[pp] = on ? ld_nc_16(b + row * G + g) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) mp[pp] = fmaxf(mp[pp], bound8(sv[pp], bv[pp]));
    }
    float own = 0.f;
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
        float m = mp[pp];
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        const float got = __shfl_sync(0xffffffffu, m, (lane & 3) << 3);   // row 4 pp + (lane & 3)
        if ((lane >> 2) == pp) own = got;
    }
    return own;
}

template <int YC>
__global__ void __launch_bounds__(kTcThreads, 1) dense_tc_kernel(const __grid_constant__ TcParams p) {
    static_assert(YC % kTcYCols == 0, "y boxes of whole TMEM loads");
    constexpr int NL = YC / kTcYCols;   // TMEM loads per y box
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcLayout& L = p.lay;
    const int CS = L.cs, XS = L.xs;
    constexpr int AS = kTcAStages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* code_full = bars;
    uint64_t* code_empty = code_full + CS;
    uint64_t* x_full = code_empty + CS;
    uint64_t* x_empty = x_full + XS;
    uint64_t* a_full = x_empty + XS;
    uint64_t* a_empty = a_full + AS;
    uint64_t* acc_full = a_empty + AS;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* exp_full = acc_empty + 2;
    uint64_t* exp_empty = exp_full + 2;
    uint64_t* exp_first = exp_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L.abort);
    float* exps = reinterpret_cast<float*>(smem + L.exps);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.groups;
    const int nchunks = (G + kTcChunkGroups - 1) / kTcChunkGroups;

    grid_dep_launch();
    if (warp == kTcWarpProducer && lane == 0) prefetch_tensormap(&p.tmap_w);
    if (warp == kTcWarpX && lane == 0) prefetch_tensormap(&p.tmap_x);
    if (threadIdx.x == 0) {
        for (int i = 0; i < CS; ++i) {
            mbar_init(smem_addr(code_full + i), 1);
            mbar_init(smem_addr(code_empty + i), kTcDqWarps);
        }
        for (int i = 0; i < XS; ++i) {
            mbar_init(smem_addr(x_full + i), 1);
            mbar_init(smem_addr(x_empty + i), 1);
        }
        for (int i = 0; i < AS; ++i) {
            mbar_init(smem_addr(a_full + i), kTcDqWarps);
            mbar_init(smem_addr(a_empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(acc_full + i), 1);
            mbar_init(smem_addr(acc_empty + i), kTcEpiWarps);
            mbar_init(smem_addr(exp_full + i), kTcEpiWarps);
            mbar_init(smem_addr(exp_empty + i), kTcDqWarps);
        }
        mbar_init(smem_addr(exp_first), kTcDqWarps);
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcWarpMma) tc_alloc(smem_addr(tmem_slot), p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTcWarpProducer) {
        // ======================= TMA producer: codes =======================
        if (lane == 0) {
            grid_dep_wait();   // the codes may be written by the previous kernel of the stream
            int ci = 0;
            for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x) {
                const int64_t row0 = (int64_t)unit * kTcUnitRows;
                const int tiles = (int)llmin((int64_t)kTcUm, (p.out_dim - row0 + kTcM - 1) / kTcM);
                for (int c = 0; c < nchunks; ++c, ++ci) {
                    const int s = ci % CS;
                    if (ci >= CS) mbar_wait(smem_addr(code_empty + s), (uint32_t)(ci / CS - 1) & 1u, abort_flag);
                    const uint32_t full = smem_addr(code_full + s);
                    mbar_arrive_expect_tx(full, (uint32_t)(tiles * kTcTileBytes));
                    for (int u = 0; u < tiles; ++u)
                        tma_load_2d(smem_addr(smem + L.code + s * L.code_stage + u * kTcTileBytes), &p.tmap_w,
                                    c * 128, (int)(row0 + u * kTcM), full);
                }
            }
        }
        __syncwarp();
    } else if (warp == kTcWarpX) {
        // ======================= TMA producer: x tiles =======================
        if (lane == 0) {
            grid_dep_wait();   // x may be written by the previous kernel of the stream
            int xi = 0;
            for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x) {
                for (int g = 0; g < G; g += kTcSG, ++xi) {
                    const int sx = xi % XS;
                    if (xi >= XS) mbar_wait(smem_addr(x_empty + sx), (uint32_t)(xi / XS - 1) & 1u, abort_flag);
                    const uint32_t xf = smem_addr(x_full + sx);
                    mbar_arrive_expect_tx(xf, L.x_stage);
                    for (int gi = 0; gi < kTcSG; ++gi)
                        tma_load_2d(smem_addr(smem + L.xr + sx * L.x_stage + gi * p.n_pad * 128), &p.tmap_x,
                                    (g + gi) * 64, 0, xf);
                }
            }
        }
        __syncwarp();
    } else if (warp == kTcWarpMma) {
        // ======================= MMA issuer =======================
        // The whole warp runs the loop (so the stage addresses are warp-uniform values) and
        // one elected thread issues the MMAs and commits.
        int gi = 0, li = 0;
        for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x, ++li) {
            const int buf = li % p.acc_bufs;
            if (li >= p.acc_bufs)
                mbar_wait(smem_addr(acc_empty + buf), (uint32_t)(li / p.acc_bufs - 1) & 1u, abort_flag);
            __syncwarp();
            tc_fence_after();
            const uint32_t d0 = tmem + (uint32_t)(buf * kTcUm * p.n_pad);
            for (int g = 0; g < G; g += kTcSG, ++gi) {
                const int sx = gi % XS, sa = gi % AS;
                mbar_wait(smem_addr(x_full + sx), (uint32_t)(gi / XS) & 1u, abort_flag);
                mbar_wait(smem_addr(a_full + sa), (uint32_t)(gi / AS) & 1u, abort_flag);
                __syncwarp();
                tc_fence_after();
                const uint32_t xs0 = smem_addr(smem + L.xr + sx * L.x_stage);
                const uint32_t a0 = tmem + p.a_col0 + (uint32_t)(sa * kTcUm * kTcSG * kTcACols);
                if (elect_one()) {
#pragma unroll
                    for (int gg = 0; gg < kTcSG; ++gg) {
                        const uint64_t bd = smem_desc(xs0 + (uint32_t)(gg * p.n_pad * 128));
#pragma unroll
                        for (int u = 0; u < kTcUm; ++u)
#pragma unroll
                            for (int k = 0; k < 4; ++k)   // K 16 per MMA: 8 TMEM columns of A, 32 bytes of x
                                tc_mma_ts(d0 + (uint32_t)(u * p.n_pad),
                                          a0 + (uint32_t)((u * kTcSG + gg) * kTcACols + 8 * k), bd + 2u * k, p.idesc,
                                          (uint32_t)(g + gg + k));
                    }
                    tc_commit(smem_addr(x_empty + sx));
                    tc_commit(smem_addr(a_empty + sa));
                }
            }
            __syncwarp();
            if (elect_one()) tc_commit(smem_addr(acc_full + buf));
            __syncwarp();
        }
    } else if (warp < kTcWarpDq0) {
        // ======================= epilogue =======================
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
        const int rl = quarter * 32 + lane;           // row within each 128-row tile
        const bool elected = warp == kTcWarpEpi0 && lane == 0;   // issues the y stores
        const uint32_t ybuf = smem_addr(smem + L.ybuf);
        int ych = 0;                                  // y boxes stored so far (buffer = ych & 1)
        if (elected && p.y_tma) prefetch_tensormap(&p.tmap_y);
        float esc_next[kTcUm];
        auto exponents = [&](int unit, int slot) {
#pragma unroll
            for (int u = 0; u < kTcUm; ++u) {
                const int64_t row = (int64_t)unit * kTcUnitRows + u * kTcM + rl;
                const float m = warp_row_bound(p.s, p.b, row - lane, p.out_dim, G, lane);
                int e = 0;
                float dq = 0.f;                       // rows beyond out_dim dequantise to 0
                if (row < p.out_dim) {
                    e = row_exponent(m);
                    dq = pow2f(-e);
                }
                esc_next[u] = pow2f(e);
                exps[slot * kTcUnitRows + u * kTcM + rl] = dq;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(exp_full + slot));
        };
        // Row factors: the dequantisation threads compute their first unit's themselves (one row
        // each, into slot 0, signalled on exp_first); this warp group computes every later
        // unit's one unit ahead, unit j (j >= 1) into slot j % 2 as that slot's write
        // k = (j - 1) / 2.
        grid_dep_wait();   // scales, biases and y may belong to the previous kernel of the stream
        int li = 0;
        for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x, ++li) {
            float esc[kTcUm];
            if (li == 0) {
                mbar_wait(smem_addr(exp_first), 0u, abort_flag);
#pragma unroll
                for (int u = 0; u < kTcUm; ++u) {
                    const float dqv = exps[u * kTcM + rl];   // 2^-e, or 0 beyond out_dim
                    esc[u] = dqv > 0.f ? 1.0f / dqv : 1.0f;  // exact: a power of two
                }
            } else {
#pragma unroll
                for (int u = 0; u < kTcUm; ++u) esc[u] = esc_next[u];
            }
            const int nxt = unit + gridDim.x;
            if (nxt < p.n_units) {
                const int j = li + 1, slot = j & 1, k = (j - 1) >> 1;
                if (k >= 1) mbar_wait(smem_addr(exp_empty + slot), (uint32_t)(k - 1) & 1u, abort_flag);
                exponents(nxt, slot);
            }
            const int buf = li % p.acc_bufs;
            mbar_wait(smem_addr(acc_full + buf), (uint32_t)(li / p.acc_bufs) & 1u, abort_flag);
            tc_fence_after();
            // The accumulators leave YC columns at a time in a rolled loop: the epilogue runs once
            // per unit, so its code is cold each time, and a short loop body fetches far fewer
            // instruction lines than an unrolled sweep. The next YC columns' TMEM loads are in
            // flight while the current ones are stored. With y_tma, each YC columns go to one of
            // two shared-memory boxes [YC][128] and leave with one tensor store (the box's rows
            // beyond out_dim and columns beyond nb are clipped by the tensor map): a store
            // instruction per value and activation row costs far more issue time than its bytes.
            const int nh = p.n_pad / YC;
#pragma unroll 1
            for (int u = 0; u < kTcUm; ++u) {
                const int64_t row0 = (int64_t)unit * kTcUnitRows + u * kTcM;
                const int64_t row = row0 + rl;
                const float eu = u == 0 ? esc[0] : esc[1];
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((buf * kTcUm + u) * p.n_pad);
                uint32_t r[NL][kTcYCols];
#pragma unroll
                for (int l = 0; l < NL; ++l) tc_ld16_issue(taddr + (uint32_t)(l * kTcYCols), r[l]);
#pragma unroll
                for (int l = 0; l < NL; ++l) tc_ld16_wait(r[l]);
#pragma unroll 1
                for (int h = 0; h < nh; ++h) {
                    uint32_t rn[NL][kTcYCols];   // the next box's columns (the last ones again at the end)
                    const uint32_t tn = taddr + (uint32_t)(min(h + 1, nh - 1) * YC);
#pragma unroll
                    for (int l = 0; l < NL; ++l) tc_ld16_issue(tn + (uint32_t)(l * kTcYCols), rn[l]);
                    const int c0 = h * YC;
                    float o[YC];
#pragma unroll
                    for (int l = 0; l < NL; ++l)
#pragma unroll
                        for (int j = 0; j < kTcYCols; ++j) o[l * kTcYCols + j] = __uint_as_float(r[l][j]) * eu;
                    if (p.silu) {
#pragma unroll
                        for (int j = 0; j < YC; ++j) {
                            const float t = o[j] / p.silu_div;
                            o[j] = t / (1.0f + expf(-t));
                        }
                    }
                    if (p.y_tma) {
                        if (elected) bulk_wait_read_1();   // the store that last read this box is done with it
                        epi_sync();
                        const uint32_t yb = ybuf + (uint32_t)(ych & 1) * tc_ybox_bytes(YC);
#pragma unroll
                        for (int j = 0; j < YC; ++j) sts_f32(yb + (uint32_t)(j * kTcM + rl) * 4u, o[j]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        epi_sync();
                        if (elected && row0 < p.out_dim) tma_store_2d(&p.tmap_y, yb, (int)row0, c0);
                        ++ych;
                    } else if (row < p.out_dim) {
#pragma unroll
                        for (int j = 0; j < YC; ++j)
                            if (c0 + j < p.nb) p.y[(int64_t)(c0 + j) * p.out_dim + row] = o[j];
                    }
#pragma unroll
                    for (int l = 0; l < NL; ++l) tc_ld16_wait(rn[l]);
#pragma unroll
                    for (int l = 0; l < NL; ++l)
#pragma unroll
                        for (int j = 0; j < kTcYCols; ++j) r[l][j] = rn[l][j];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(acc_empty + buf));
        }
        if (elected && p.y_tma) bulk_wait_all();   // no CTA exits while its y stores read shared memory
    } else if (warp < kTcWarpX) {
        // ======================= dequantisation =======================
        const int quarter = warp & 3;                     // TMEM lanes this warp may write
        const int dw = warp - kTcWarpDq0;
        const int u = (dw >> 2) % kTcUm;                  // tile
        const int hc = dw / (4 * kTcUm);                  // column part of every group
        const int rl = quarter * 32 + lane;               // row within the tile = TMEM lane
        const int r = u * kTcM + rl;                      // row within the unit
        const uint32_t rsw = (uint32_t)rl & 7u;
        const uint32_t code_base = smem_addr(smem + L.code) + (uint32_t)(u * kTcTileBytes) + (uint32_t)rl * 128u;
        const uint32_t a_lane = tmem + ((uint32_t)(quarter * 32) << 16) + p.a_col0 +
                                (uint32_t)(u * kTcSG * kTcACols + hc * kTcDqCols);
        constexpr int kChunks = kTcDqCols / 16;           // 16-byte code chunks per thread and group
        grid_dep_wait();   // scales and biases may be written by the previous kernel of the stream
        int ci = 0, gi = 0, li = 0;
        // scale and bias words of the next chunk (across units: the next unit's first chunk is
        // loaded during this unit's last one)
        uint2 s_nx = make_uint2(0, 0), b_nx = make_uint2(0, 0);
        if ((int)blockIdx.x < p.n_units) {
            const int64_t row = (int64_t)blockIdx.x * kTcUnitRows + r;
            if (row < p.out_dim) {
                s_nx = ld_nc_8(p.s + row * G);
                b_nx = ld_nc_8(p.b + row * G);
            }
        }
        for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x, ++li) {
            const int slot = li & 1;
            const int64_t row = (int64_t)unit * kTcUnitRows + r;
            const bool valid = row < p.out_dim;
            const uint16_t* srow = p.s + (valid ? row : 0) * G;
            const uint16_t* brow = p.b + (valid ? row : 0) * G;
            float dq;
            if (li == 0) {
                // the first unit's row factor: computed here, not waited for
                const float m = warp_row_bound(p.s, p.b, row - lane, p.out_dim, G, lane);
                dq = valid ? pow2f(-row_exponent(m)) : 0.f;
                exps[r] = dq;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(exp_first));
            } else {
                const int k = (li - 1) >> 1;
                mbar_wait(smem_addr(exp_full + slot), (uint32_t)k & 1u, abort_flag);
                dq = exps[slot * kTcUnitRows + r];
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(exp_empty + slot));
            }
            const int64_t nrow = (int64_t)(unit + gridDim.x) * kTcUnitRows + r;
            const bool nvalid = unit + (int)gridDim.x < p.n_units && nrow < p.out_dim;
            for (int c = 0; c < nchunks; ++c, ++ci) {
                const uint2 s_cur = s_nx, b_cur = b_nx;
                if (c + 1 < nchunks) {
                    if (valid) {
                        s_nx = ld_nc_8(srow + (c + 1) * kTcChunkGroups);
                        b_nx = ld_nc_8(brow + (c + 1) * kTcChunkGroups);
                    }
                } else {
                    s_nx = nvalid ? ld_nc_8(p.s + nrow * G) : make_uint2(0, 0);
                    b_nx = nvalid ? ld_nc_8(p.b + nrow * G) : make_uint2(0, 0);
                }
                const int cs_ = ci % CS;
                mbar_wait(smem_addr(code_full + cs_), (uint32_t)(ci / CS) & 1u, abort_flag);
                const uint32_t cb = code_base + (uint32_t)cs_ * L.code_stage;
                // Groups alternate between two register sets: a tcgen05.st reads its source
                // registers after it issues, so the next group's unpack must not overwrite them.
                uint32_t hb[2][kTcDqCols];
#pragma unroll
                for (int k = 0; k < kTcChunkGroups; ++k) {   // G % 8 == 0: every chunk is full
                    const int sa = gi % AS;
                    const int gg = k % kTcSG;           // group within the operand stage
                    const uint32_t sp = k < 2 ? s_cur.x : s_cur.y;
                    const uint32_t bp = k < 2 ? b_cur.x : b_cur.y;
                    const float sf = bf16_to_f32((k & 1) ? (sp >> 16) : (sp & 0xFFFFu)) * dq;
                    const float bfv = bf16_to_f32((k & 1) ? (bp >> 16) : (bp & 0xFFFFu)) * dq;
                    const __half2 sc = __floats2half2_rn(sf * 16777216.0f, sf * 1048576.0f);   // 2^24, 2^20
                    const __half2 bi = __floats2half2_rn(bfv, bfv);
                    uint32_t words[4 * kChunks];
#pragma unroll
                    for (int v = 0; v < kChunks; ++v) {
                        const uint4 q = lds_v4(cb + ((((uint32_t)(2 * k + hc * kChunks + v)) ^ rsw) << 4));
                        words[4 * v] = q.x;
                        words[4 * v + 1] = q.y;
                        words[4 * v + 2] = q.z;
                        words[4 * v + 3] = q.w;
                    }
                    uint32_t (&h)[kTcDqCols] = hb[k & 1];
#pragma unroll
                    for (int w8 = 0; w8 < 4 * kChunks; ++w8) {
                        h[4 * w8 + 0] = dequant_pair<0>(words[w8], sc, bi);
                        h[4 * w8 + 1] = dequant_pair<1>(words[w8], sc, bi);
                        h[4 * w8 + 2] = dequant_pair<2>(words[w8], sc, bi);
                        h[4 * w8 + 3] = dequant_pair<3>(words[w8], sc, bi);
                    }
                    if (gg == 0) {
                        if (gi >= AS) mbar_wait(smem_addr(a_empty + sa), (uint32_t)(gi / AS - 1) & 1u, abort_flag);
                        tc_fence_after();
                    }
                    tc_st<kTcDqCols>(a_lane + (uint32_t)((sa * kTcUm * kTcSG + gg) * kTcACols), h);
                    if (k > 0) keep_live<kTcDqCols>(hb[(k + 1) & 1]);
                    if (gg == kTcSG - 1) {
                        tc_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_addr(a_full + sa));
                        ++gi;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(code_empty + cs_));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcWarpMma) tc_dealloc(tmem, p.tmem_cols);
}

// ---- host side ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tc_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct TcDevice {
    int sm_count = 0;
    int max_smem = 0;
    bool attr_set = false;
};

std::mutex g_tc_mu;
std::map<int, TcDevice> g_tc_dev;

// Layout choice: the deepest code ring that fits (its depth is the HBM prefetch distance),
// then the x ring. The smem request never drops below half an SM, so two CTAs never share
// one SM's TMEM (the allocation can then never wait).
bool tc_pick_layout(int n_pad, int yc, int max_smem, TcLayout& out, uint32_t& smem_bytes) {
    static const int order[6][2] = {{4, 8}, {4, 6}, {4, 4}, {3, 4}, {3, 3}, {2, 3}};
    for (int i = 0; i < 6; ++i) {
        const TcLayout L = tc_layout(n_pad, order[i][0], order[i][1], yc);
        const uint32_t need = L.total + 1024u;
        if ((int)need <= max_smem) {
            out = L;
            smem_bytes = need < (uint32_t)max_smem / 2u + 4096u ? (uint32_t)max_smem / 2u + 4096u : need;
            return true;
        }
    }
    return false;
}

q4a_status launch_chunk(const TcDevice& dev, const uint8_t* w, const uint16_t* s, const uint16_t* b,
                        const uint16_t* x, float* y, int nb, int64_t out_dim, int64_t in_dim, bool silu,
                        float silu_div, cudaStream_t stream) {
    EncodeTiledFn enc = tc_encode_fn();
    if (!enc) return Q4A_ERR_UNSUPPORTED;
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    const cuuint32_t estr[2] = {1u, 1u};
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(in_dim / 2), (cuuint64_t)out_dim};
        const cuuint64_t strides[1] = {(cuuint64_t)(in_dim / 2)};
        const cuuint32_t box[2] = {128u, (cuuint32_t)kTcM};
        CUresult r = encode_tiled_cached(&prm.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
    }
    const int n_pad = (nb + 15) / 16 * 16;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)in_dim, (cuuint64_t)nb};
        const cuuint64_t strides[1] = {(cuuint64_t)in_dim * 2};
        const cuuint32_t box[2] = {64u, (cuuint32_t)n_pad};
        CUresult r = encode_tiled_cached(&prm.tmap_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
    }
    // TMEM (512 columns): accumulators [acc_bufs][kTcUm][n_pad], then the A stages
    // [kTcAStages][kTcUm][kTcSG][32]
    const int a_cols = kTcAStages * kTcUm * kTcSG * kTcACols;
    prm.acc_bufs = 2 * kTcUm * n_pad + a_cols <= 512 ? 2 : 1;
    if (prm.acc_bufs * kTcUm * n_pad + a_cols > 512) return Q4A_ERR_UNSUPPORTED;
    // y box width: 32 columns where one accumulator set makes the MMA wait for each unit's drain
    const int yc = prm.acc_bufs == 1 && n_pad % 32 == 0 ? 32 : 16;
    // y through tensor stores: rows 16-byte aligned (out_dim % 4 == 0, y 16-byte aligned), and at
    // least one full box of rows so the box never exceeds the tensor.
    prm.y_tma = (out_dim % 4 == 0 && out_dim >= kTcM && reinterpret_cast<uintptr_t>(y) % 16 == 0) ? 1 : 0;
    if (prm.y_tma) {
        const cuuint64_t dims[2] = {(cuuint64_t)out_dim, (cuuint64_t)nb};
        const cuuint64_t strides[1] = {(cuuint64_t)out_dim * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kTcM, (cuuint32_t)yc};
        CUresult r = encode_tiled_cached(&prm.tmap_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, dims, strides, box, estr,
                                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
    }
    uint32_t smem_bytes = 0;
    if (!tc_pick_layout(n_pad, yc, dev.max_smem, prm.lay, smem_bytes)) return Q4A_ERR_UNSUPPORTED;
    prm.s = s;
    prm.b = b;
    prm.y = y;
    prm.out_dim = out_dim;
    prm.groups = (int32_t)(in_dim / kGroup);
    prm.nb = nb;
    prm.n_pad = n_pad;
    prm.silu = silu ? 1 : 0;
    prm.silu_div = silu ? silu_div : 1.0f;
    prm.n_units = (int32_t)((out_dim + kTcUnitRows - 1) / kTcUnitRows);
    prm.a_col0 = (uint32_t)(prm.acc_bufs * kTcUm * n_pad);
    uint32_t cols = 32;
    while (cols < prm.a_col0 + (uint32_t)a_cols) cols *= 2;
    prm.tmem_cols = cols;
    prm.idesc = (1u << 4)                          // D: fp32
                | (0u << 7) | (0u << 10)           // A, B: fp16
                | (0u << 15) | (0u << 16)          // both K-major
                | ((uint32_t)(n_pad >> 3) << 17)   // N
                | ((uint32_t)(kTcM >> 4) << 24);   // M
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(prm.n_units < dev.sm_count ? prm.n_units : dev.sm_count), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static const bool debug = getenv("Q4A_DEBUG") != nullptr;
    if (debug)
        fprintf(stderr, "q4a dense_tc: out=%lld in=%lld nb=%d n_pad=%d units=%d grid=%u cs=%d xs=%d acc_bufs=%d "
                "tmem_cols=%u smem=%u y_box=%d\n", (long long)out_dim, (long long)in_dim, nb, n_pad, prm.n_units,
                cfg.gridDim.x, prm.lay.cs, prm.lay.xs, prm.acc_bufs, prm.tmem_cols, smem_bytes, yc);
    const cudaError_t e = yc == 32 ? cudaLaunchKernelEx(&cfg, dense_tc_kernel<32>, prm)
                                   : cudaLaunchKernelEx(&cfg, dense_tc_kernel<16>, prm);
    if (e != cudaSuccess) return cuda_fail(e);
    return Q4A_OK;
}

}  // namespace

bool dense_tc_eligible(const uint16_t* s, const uint16_t* b, int nb, int64_t out_dim, int64_t in_dim) {
    // From NB 64; from NB 9 on matrices tall enough to give every SM a 256-row unit (4096 x
    // 151936 LM head: 87 us at NB 9..16 against 97..106 us on the GEMV kernel at NB 9..12, which
    // keeps NB 8 at 78 us); from NB 17 on matrices of 48 units or more (4096 -> 12288: 24 us at
    // NB 24..32 against 33..38 us, while NB 16 takes 19 us on the GEMV kernel and 23 us here).
    // Shorter matrices have too few units to fill the GPU (12288 -> 4096, 16 units: 66..79 us
    // at NB 16..63 against 18..76 us).
    const bool wide = nb >= kDenseTcMinRows || (nb >= kDenseTcTallMinRows && out_dim >= (int64_t)kDenseTcTallRows) ||
                      (nb >= kDenseTcMidMinRows && out_dim >= (int64_t)kDenseTcMidRows);
    return wide && (in_dim / kGroup) % 8 == 0 && reinterpret_cast<uintptr_t>(s) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(b) % 16 == 0;
}

q4a_status launch_dense_tc(const uint8_t* w, const uint16_t* s, const uint16_t* b, const uint16_t* x, float* y,
                           int nb, int64_t out_dim, int64_t in_dim, bool silu, float silu_div,
                           cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    TcDevice d;
    {
        std::lock_guard<std::mutex> lock(g_tc_mu);
        TcDevice& c = g_tc_dev[dev];
        if (!c.attr_set) {
            cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, dev);
            cudaDeviceGetAttribute(&c.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            e = cudaFuncSetAttribute(dense_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, c.max_smem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(dense_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, c.max_smem);
            if (e != cudaSuccess) return cuda_fail(e);
            c.attr_set = c.sm_count > 0;
        }
        d = c;
    }
    if (!d.attr_set) return Q4A_ERR_CUDA;
    for (int t0 = 0; t0 < nb; t0 += kTcMaxN) {
        const int n = nb - t0 < kTcMaxN ? nb - t0 : kTcMaxN;
        const q4a_status st = launch_chunk(d, w, s, b, x + (int64_t)t0 * in_dim, y + (int64_t)t0 * out_dim, n,
                                           out_dim, in_dim, silu, silu_div, stream);
        if (st != Q4A_OK) return st;
    }
    return Q4A_OK;
}

q4a_status read_and_clear_dense_tc_error(uint32_t* word) {
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *word = v;
    return Q4A_OK;
}

}  // namespace q4a
