// q4a_internal.h -- declarations shared by the translation units of libq4a.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q4a.h"

namespace q4a {

// ---- fixed geometry of the GEMV kernels ---------------------------------------
constexpr int kGroup = 64;              // inputs per scale/bias group
constexpr int kStageGroups = 8;         // groups per pipeline stage (512 inputs)
constexpr int kBoxBytes = 128;          // TMA box width in bytes (4 groups), 128B swizzle
constexpr int kBoxBytesTotal = 16 * kBoxBytes;  // one box: 16 rows x 128 bytes
constexpr int kConsumerWarps = 8;       // 2 row halves x 4 group slots
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kDenseMaxSeg = 8;         // token chunks of one dense call
constexpr int kXFragBudget = 64 * 1024; // staged activation fragments per CTA
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits give up after ~1 s

// s/b copy modes of the producer warp
enum SbMode : int { kSb16 = 0, kSb4 = 1, kSb2 = 2 };

struct Segment {
    int32_t row0;   // first row of this segment's matrix in the (bank) tensor
    int32_t tok0;   // first activation slot (row of y, index into x_rows)
    int32_t ntok;   // activation rows of the segment (1 .. 8*NT)
    int32_t pad;
};

// Shared-memory carve-up, identical on host and device.
struct SmemLayout {
    uint32_t stage_bytes, stage_w_bytes, ring, xfrag, xsum, wpart, cpart, ssq, bars, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int nt, int mt, int stages, int gs) {
    SmemLayout L;
    const uint32_t ntok = 8u * nt, rows = 16u * mt;
    L.stage_w_bytes = (uint32_t)mt * 2u * kBoxBytesTotal;
    L.stage_bytes = L.stage_w_bytes + rows * 32u;          // + s and b, 16 bytes per row each
    L.ring = 0;                                             // relative to a 1024-aligned base
    L.xfrag = L.ring + (uint32_t)stages * L.stage_bytes;
    L.xsum = L.xfrag + (uint32_t)gs * nt * 1024u;
    L.wpart = align_up(L.xsum + (uint32_t)gs * ntok * 4u, 16);
    L.cpart = L.wpart + 4u * rows * ntok * 4u;
    L.ssq = L.cpart + 2u * rows * ntok * 4u;
    L.bars = align_up(L.ssq + 2u * ntok * 4u, 8);
    L.total = L.bars + 2u * (uint32_t)stages * 8u + 16u;
    return L;
}

template <int MAXSEG>
struct GemvParams {
    CUtensorMap tmap_w;       // 2D uint8: dim0 = in_dim/2 bytes, dim1 = tensor rows
    const uint16_t* s;        // bf16 [rows][G]
    const uint16_t* b;
    const void* x;            // fp16 [*][in_dim] (or fp32 x_raw for the RMSNorm variant)
    const int32_t* x_rows;    // may be null
    const uint16_t* norm_w;   // bf16 [in_dim] (RMSNorm variant)
    float* y;                 // fp32 [slots][out_dim]
    float eps, shift;
    int64_t out_dim;          // rows per segment matrix
    int64_t in_dim;
    int32_t groups;           // in_dim / 64
    int32_t gs;               // groups per CTA K-slice
    int32_t cluster;          // CTAs per cluster (K split)
    int32_t n_clusters;
    int32_t tiles_per_seg;    // ceil(out_dim / 16)
    int32_t n_tiles;          // nseg * tiles_per_seg
    int32_t nseg;
    int32_t mt;               // tiles per row block
    int32_t stages;           // ring depth
    int32_t sb_mode;
    SmemLayout lay;
    Segment seg[MAXSEG];
};

// Launch description assembled by the API layer.
struct GemvLaunch {
    const uint8_t* w;
    int64_t tensor_rows;      // rows of the whole (bank) tensor
    const uint16_t* s;
    const uint16_t* b;
    const void* x;
    const int32_t* x_rows;
    const uint16_t* norm_w;
    float* y;
    float eps, shift;
    int64_t out_dim, in_dim;
    bool rmsnorm;
    bool experts;
    int nseg;
    const Segment* seg;
    int max_ntok;
};

q4a_status launch_gemv(const GemvLaunch& L, cudaStream_t stream);
q4a_status launch_pack(uint8_t* w_packed, const uint8_t* codes, int64_t rows, int64_t in_dim,
                       cudaStream_t stream);
q4a_status launch_xsum(float* xsum, const uint16_t* x, int64_t nb, int64_t in_dim,
                       cudaStream_t stream);
q4a_status launch_silu_mul_xsum(uint16_t* h, float* hsum, const float* gate_up, int64_t rows,
                                int64_t inter, cudaStream_t stream);
q4a_status launch_fill_nan(float* y, int64_t row0, int64_t nrows, int64_t out_dim,
                           cudaStream_t stream);
q4a_status read_and_clear_device_error(cudaStream_t stream, uint32_t* word);

// Records a CUDA error for q4a_last_cuda_error and returns Q4A_ERR_CUDA.
q4a_status cuda_fail(cudaError_t e);
q4a_status cuda_fail_drv(CUresult r);

}  // namespace q4a
