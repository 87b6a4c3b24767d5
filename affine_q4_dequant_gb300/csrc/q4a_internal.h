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
constexpr int kTileBytes = 16 * kBoxBytes;      // one 16-row tile of one box column: 2 KB
constexpr int kNumMaps = 6;                     // box heights 16, 32, ..., 96 rows: one box per
                                                // box column of a row block (at most 6 tiles)
constexpr int kGroupSlots = kStageGroups; // one consumer warp per group of a stage
constexpr int kConsumerWarps = kGroupSlots;       // each owns every tile of the row block
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kDenseMaxSeg = 8;         // token chunks of one dense call
constexpr int kXFragBudget = 128 * 1024; // staged activation fragments per CTA
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits give up after ~1 s
constexpr uint32_t kSuspendHintNs = 20000;        // per try_wait sleep bound
constexpr int kDenseTcMinRows = 64;   // q4a_gemv batches this wide take the tensor-core path,
constexpr int kDenseTcTallRows = 152 * 256;   // from kDenseTcTallMinRows rows on matrices this tall
constexpr int kDenseTcTallMinRows = 9;        // (a 256-row unit for every SM),
constexpr int kDenseTcMidRows = 48 * 256;     // and from kDenseTcMidMinRows rows on matrices this tall
constexpr int kDenseTcMidMinRows = 17;        // (where the GEMV kernel needs 4 activation tiles)
constexpr int kCombineMaxK = 64;      // q4a_moe_combine: experts per token
constexpr int kMaxNormGroups = 8;     // q4a_gemv_rmsnorm_grouped: normalisation segments per row
// raw scale mode: row blocks of raw scales/biases in flight (3 where the consumers read them in
// place for a whole row block, 2 where they rearrange them first)
__host__ __device__ constexpr int raw_bufs(bool raw_direct) { return raw_direct ? 3 : 2; }

// How the producer fetches a row block's scales and biases into shared memory. Both modes
// write the same layout: [64-group chunk][row][128 bytes], 16-byte granule u of row r
// stored at granule u ^ (r & 7) (the TMA 128-byte swizzle).
//   kSbTma   2D TMA boxes of 64 groups x rows (groups % 8 == 0, 16-byte aligned bases)
//   kSbRaw   the row block's [rows][groups] scales (and biases) are contiguous: 1D TMA boxes
//            of 256 elements fetch them, one row block ahead, into a raw staging buffer,
//            and the consumer warps rearrange them in shared memory (16-byte aligned bases,
//            any group count up to a staging budget; full K only)
//   kSbPlain producer lanes copy element by element (anything else; full K only)
enum SbMode : int { kSbTma = 0, kSbRaw = 1, kSbPlain = 2 };
constexpr int kRawBox = 256;                 // elements per 1D box of the raw mode
constexpr uint32_t kRawBudget = 4096;        // raw staging elements per array and buffer

struct Segment {
    int32_t row0;   // first row of this segment's matrix in the (bank) tensor
    int32_t tok0;   // first activation slot (row of y, index into x_rows)
    int32_t ntok;   // activation rows of the segment (1 .. 8*NT)
    int32_t pad;
};

// Shared-memory carve-up, identical on host and device.
struct SmemLayout {
    uint32_t stage_bytes;   // one ring stage of packed codes: 4-bit: mt tiles x 2 box columns
                            // x 2 KB; 2-bit: one box column; 3-bit: one box column (upper
                            // two bits), then mt x 1 KB of lowest-bit words ([tile][row][64 B])
    uint32_t ring, xfrag, xsum, xbias, sb, sb_pitch, sb_buf, n_sb, wpart, cpart, ssq, raw, raw_elems, bars, total;
    // raw, raw_elems: the raw mode's staging buffers [2 buffers][scales | biases][raw_elems] bf16
    // sb_pitch: bytes of one row block's scales (the biases follow); sb_buf: both
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Row tiles (16 rows) per row block. Every consumer warp holds accumulators for all of
// them: 4 * nt * mt fp32 per lane (24 / 32 / 32 at nt = 1 / 2 / 4).
__host__ __device__ constexpr int tiles_per_block(int nt) { return nt == 1 ? 6 : (nt == 2 ? 4 : 2); }

// Staged activation fragments: [group][step pair][activation row][lane quad] x 16 bytes,
// i.e. 128 bytes per (group, row) -- the size of the fp16 activations themselves.
__host__ __device__ inline uint32_t xfrag_bytes(int gs, int ntok_max) { return (uint32_t)gs * ntok_max * 128u; }

// Row pitch of the staged scale/bias rows: at least the K-slice's groups, padded so that
// its 32-bit word count is 4 mod 8 -- the 8 rows a warp reads at once then fall in 8
// different banks.
// Bytes of one row block's scales (or biases): swizzled 64-group chunks.
__host__ __device__ inline uint32_t sb_bytes(int /*sb_mode*/, int gs, int rows) {
    return (uint32_t)((gs + 63) / 64) * rows * 128u;
}

// Bytes of the lowest-bit words of one 16-row tile in a ring stage (3-bit codes): 8 groups x
// 8 bytes per row.
constexpr uint32_t kLoTileBytes = 16u * 64u;

__host__ __device__ inline SmemLayout smem_layout(int nt, int mt, int stages, int gs, int ntok_max,
                                                  int sb_mode, int sb_bufs, int code_bits = 4,
                                                  uint32_t sb_pitch_bytes = 0, bool raw_direct = false) {
    SmemLayout L;
    const uint32_t ntok = 8u * nt, rows = 16u * mt;
    L.stage_bytes = (uint32_t)mt * (code_bits == 4 ? 2u : 1u) * kTileBytes +   // [box column][rows][128 B]
                    (code_bits == 3 ? (uint32_t)mt * kLoTileBytes : 0u);
    L.ring = 0;                                             // relative to a 1024-aligned base
    L.xfrag = L.ring + (uint32_t)stages * L.stage_bytes;
    L.xsum = L.xfrag + align_up(xfrag_bytes(gs, ntok_max), 16);
    L.sb_pitch = sb_pitch_bytes ? sb_pitch_bytes : sb_bytes(sb_mode, gs, rows);   // scales, then biases
    // raw_direct (raw mode only): the consumers read the raw buffers, no swizzled scale/bias buffers
    raw_direct = raw_direct && sb_mode == kSbRaw;
    L.sb_buf = raw_direct ? 0u : 2u * L.sb_pitch;
    L.xbias = align_up(L.xsum + (uint32_t)gs * ntok * 4u, 16);   // bf16 hi/lo group sums
    L.sb = align_up(L.xbias + (uint32_t)((gs + 15) / 16) * ntok_max * 64u, 1024);
    L.n_sb = (uint32_t)sb_bufs;                             // 2 when a CTA has several row blocks
    L.wpart = L.sb + L.n_sb * L.sb_buf;
    L.cpart = L.wpart + (uint32_t)kGroupSlots * rows * ntok * 4u;
    L.ssq = L.cpart + 2u * rows * ntok * 4u;
    L.raw = align_up(L.ssq + 2u * ntok * (uint32_t)kMaxNormGroups * 4u, 128);   // sums, then factors
    // a row block's elements plus up to 7 in front (the box start is rounded down to 16 bytes)
    L.raw_elems = sb_mode == kSbRaw ? align_up(rows * (uint32_t)gs + 7u, (uint32_t)kRawBox) : 0u;
    const uint32_t nrb = (uint32_t)raw_bufs(raw_direct);
    L.bars = align_up(L.raw + nrb * 2u * L.raw_elems * 2u, 8);
    // full[stages] empty[stages] sbfull[2] sbempty[2] rawfull[nrb] rawempty[nrb], then the abort flag
    L.total = L.bars + (2u * (uint32_t)stages + 4u + 2u * nrb) * 8u + 16u;
    return L;
}

// The product a launch computes: its weights, input, output and schedule.
struct GemvOp {
    CUtensorMap tmap_w[kNumMaps];  // 2D uint8: dim0 = in_dim/2 bytes, dim1 = tensor rows;
                                   // box 128 bytes x 16 (i + 1) rows, 128-byte swizzle
    CUtensorMap tmap_s[kNumMaps];  // 2D bf16 scales/biases: dim0 = groups, dim1 = rows;
    CUtensorMap tmap_b[kNumMaps];  // box 64 groups x 16 (i + 1) rows, 128-byte swizzle
    CUtensorMap tmap_s1;           // raw mode: 1D bf16 views of s and b (rows * groups
    CUtensorMap tmap_b1;           // elements), box kRawBox elements
    CUtensorMap tmap_lo[kNumMaps]; // 3-bit codes: lowest-bit plane, dim0 = in_dim/8 bytes,
                                   // box 64 bytes x 16 (i + 1) rows, no swizzle
    const uint16_t* s;        // bf16 [rows][G]
    const uint16_t* b;
    const void* x;            // fp16 [*][in_dim] (or fp32 x_raw for the RMSNorm variant)
    const int32_t* x_rows;    // may be null
    const uint16_t* norm_w;   // bf16 [in_dim] (RMSNorm variant)
    const float* inj_out;     // RMSNorm variant, injection: fp32 [slots][norm_width] added to every
    const float* inj_logit;   // stream g of a row with weight 2 sigmoid(logit[slot][g] / norm_groups)
    float* x_new;             // fp32 [slots][in_dim]: the injected stream (written by cluster 0), or null
    float* y;                 // fp32 [slots][out_dim]
    uint16_t* h;              // fused gate|up: fp16 silu(gate) * up [slots][out_dim]
    float eps, shift;
    float post_div;           // output epilogue silu(y / post_div) when post_silu
    int32_t post_silu;
    int32_t norm_groups;      // RMSNorm variant: segments per row, each normalised on its own
    int64_t norm_width;       // in_dim / norm_groups
    int64_t out_dim;          // rows per segment matrix
    int64_t in_dim;
    int32_t groups;           // in_dim / 64
    int32_t gs;               // groups per CTA K-slice
    int32_t tiles_per_seg;    // ceil(out_dim / 16)
    int32_t n_tiles;          // nseg * tiles_per_seg
    int32_t mt;               // schedule units per row block (fused gate|up: pairs of tiles)
    int32_t ntok_max;         // activation rows of the widest segment (<= 8 * NT)
    int32_t sb_mode;
    int32_t sb_tiles;         // 16-row tiles per 64-group chunk of a row block's staged scales
    uint32_t sb_pitch;        // bytes from a row block's staged scales to its biases
    int32_t rms;              // RMSNorm prologue: x is fp32 x_raw (kernels built with RMS)
    int32_t fg;               // fused gate|up epilogue into h (kernels built with FG)
    int32_t withhold_stage;   // failure-path testing: weight stage (per CTA) never loaded, -1 none
};

template <int MAXSEG>
struct GemvParams {
    GemvOp op;
    int32_t cluster;          // CTAs per cluster (K split)
    int32_t n_clusters;
    int32_t nseg;
    int32_t stages;           // ring depth
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
    bool silu;                // output epilogue y -> silu(y / silu_div)
    float silu_div;
    int norm_groups;          // RMSNorm variant: normalisation segments per row (>= 1)
    const float* inj_out = nullptr;   // RMSNorm variant: hyper-connection injection (see GemvParams)
    const float* inj_logit = nullptr;
    float* x_new = nullptr;
    bool fused_gate_up = false;   // w holds gate rows [0, out_dim) then up rows [out_dim, 2 out_dim);
    uint16_t* h = nullptr;        // the output is h = fp16(silu(gate) * up) [slots][out_dim]
    bool x_f32 = false;       // the activations are fp32 (rounded to binary16 when staged)
    int code_bits = 4;        // 4 (w: packed nibbles), 2 or 3 (w: 2-bit codes [rows][in/4],
    const uint8_t* w_lo = nullptr;  // w_lo: the 3-bit codes' lowest-bit plane [rows][in/8])
    bool experts;
    int nseg;
    const Segment* seg;
    int max_ntok;
    bool plan_only = false;               // validate and plan, launch nothing
    int withhold_stage = -1;              // see GemvOp
};

q4a_status launch_gemv(const GemvLaunch& L, cudaStream_t stream);
q4a_status launch_pack(uint8_t* w_packed, const uint8_t* codes, int64_t rows, int64_t in_dim,
                       cudaStream_t stream);
q4a_status launch_xsum(float* xsum, const uint16_t* x, int64_t nb, int64_t in_dim,
                       cudaStream_t stream);
q4a_status launch_lowbit_pack(uint8_t* w_up, uint8_t* w_lo, const uint8_t* w_packed, int64_t rows,
                              int64_t in_dim, cudaStream_t stream);
q4a_status launch_silu_mul_xsum(uint16_t* h, float* hsum, const float* gate_up, int64_t rows,
                                int64_t inter, cudaStream_t stream);
q4a_status launch_fill_nan(float* y, int64_t row0, int64_t nrows, int64_t out_dim,
                           cudaStream_t stream);
q4a_status launch_fill_nan_h(uint16_t* h, int64_t row0, int64_t nrows, int64_t inter, cudaStream_t stream);
q4a_status launch_moe_combine(float* out, const float* y, const int32_t* slot, const float* w, int n_tok,
                              int top_k, int64_t n_slots, int64_t hidden, const float* y_shared,
                              const uint16_t* gate, const float* x, cudaStream_t stream);
q4a_status read_and_clear_device_error(cudaStream_t stream, uint32_t* word);

// Dense path for wide batches (q4a_dense_tc.cu): dequantise to binary16 tiles, tcgen05.mma.
// Eligible when in_dim % 512 == 0, s and b are 16-byte aligned, and nb >= kDenseTcMinRows (or
// nb >= kDenseTcTallMinRows with out_dim >= kDenseTcTallRows).
bool dense_tc_eligible(const uint16_t* s, const uint16_t* b, int nb, int64_t out_dim, int64_t in_dim);
q4a_status launch_dense_tc(const uint8_t* w, const uint16_t* s, const uint16_t* b, const uint16_t* x, float* y,
                           int nb, int64_t out_dim, int64_t in_dim, bool silu, float silu_div,
                           cudaStream_t stream);
q4a_status read_and_clear_dense_tc_error(uint32_t* word);   // after a stream synchronisation

// cuTensorMapEncodeTiled with a cache keyed by every argument (q4a_gemv.cu).
CUresult encode_tiled_cached(CUtensorMap* out, CUtensorMapDataType dtype, cuuint32_t rank, void* ptr,
                             const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                             const cuuint32_t* estr, CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                             CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob);

// The stage q4a_debug_withhold_stage asked the next GEMV-kernel launch of this host thread to
// withhold (-1: none); reading it clears it.
int take_withhold_stage();

// Records a CUDA error for q4a_last_cuda_error and returns Q4A_ERR_CUDA.
q4a_status cuda_fail(cudaError_t e);
q4a_status cuda_fail_drv(CUresult r);

}  // namespace q4a
