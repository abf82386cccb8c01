// internal.h -- declarations shared by the host API and the kernel translation
// units of libgemm_nt.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "out_store.cuh"

namespace gnt {

// Work distribution of the tcgen05 kernel.
constexpr int kModeTiles = 0;     // whole tiles, round-robin over CTAs
constexpr int kModeStreamK = 1;   // even share of (tile, k-block) iterations per CTA
constexpr int kModeRowSplit = 2;  // even share of rows per CTA (<= 128 each), all of K

// Device status word bits (OR-ed by kernels, read and cleared by gemm_nt_check).
constexpr uint32_t kStatusTimeout = 1u;

// Parameters of the tcgen05 kernel.  "X" is the operand on the MMA's M side
// (128 rows per tile), "Y" the operand on its N side (BN rows per tile).
// Without swapping X = A and Y = B and Out[x][y]; with swapping (small M)
// X = B, Y = A and the tile is written transposed, Out[y][x].
struct TcParams {
    void* out;            // fp32, fp16 or bf16 elements (out_type)
    int out_type;         // kOutF32, kOutF16 or kOutBF16
    uint32_t idesc_bits;  // instruction-descriptor bits ORed into every MMA: A/B element
                          // type (0: fp16) and the A (bit 15) / B (bit 16) MN-major flags
    int x_mn;             // 1: X is MN-major (tiles of 64 rows x 64 K per TMA box)
    int y_mn;             // 1: Y is MN-major
    int64_t ldo;
    int64_t stride_o;
    int rows_x;
    int rows_y;
    int batch;
    int tiles_x;
    int tiles_y;
    int num_kb;           // k-blocks of 64 per tile (K tail zero-filled by TMA)
    int tiles_per_batch;  // tiles_x * tiles_y
    int num_tiles;        // batch * tiles_per_batch
    int group_x;          // grouped raster: x-tiles per group
    int mode;             // kModeTiles, kModeStreamK or kModeRowSplit
    long long total_iters;  // num_tiles * num_kb
    int x_bmul;           // 1 if X's tensor map has a batch dimension, 0 if shared
    int y_bmul;
    int vec4;             // Out base and ldo allow 4-element vector stores
    int x_box_bytes;      // bytes of one X box (its height x 128 B; at most 16 KB)
    // 0, or the width (6 or 4 bits) of packed A/B elements: their loads spread 16
    // packed elements over each 16-byte chunk of shared memory but credit the
    // stage barrier with the packed global bytes, width / 8 of the shared ones
    int ab_packed_bits;
    // Stream-K on the pair kernel: tiles [sk_first, num_tiles) are cut into
    // even k-block ranges, one per pair.  Each partial piece leaves its slice in
    // ws; per-(tile, CTA, epilogue warp) counters in ws_flags pick the warp that
    // arrives last, which sums the slices in k order and stores Out.
    int sk_first;           // = num_tiles when stream-K is off
    long long sk_iters;     // (num_tiles - sk_first) * num_kb
    int sk_pairs;           // pairs [0, sk_pairs) share the stream-K iterations
    float* ws;              // [pairs][2 slots][2 CTAs][8 warps][4 chunks][32 cols][32 rows] fp32
    uint32_t* ws_flags;     // [stream-K tiles][2 CTAs][8 warps], zero between launches
    uint32_t* status;     // device status word
    unsigned long long wait_limit;  // bounded-wait limit, SM clock cycles
    int fault;            // test hook: 0 none, 1 drop a producer stage, 2 skip a release
    // Block-scaled 8-bit inputs (kind 2 of tc05_launch): the scale atoms of X
    // and Y, 512 bytes per (128-row block, 128-element K block), row block-major
    // (atom (r, k) at offset (r * num_kb + k) * 512), one set per batch.
    const uint8_t* sf_x;
    const uint8_t* sf_y;
    long long sf_x_bstride;  // bytes between batches (0: shared)
    long long sf_y_bstride;
    int sf_box_kg;           // CTA-pair kernel: K block groups per scale box (<= 8, <= the tensor's)
    int sf_box_rb;           // CTA-pair kernel: row blocks per B scale box (1 or 2)
};

struct MmaParams {
    const void* A;  // 2-byte elements (fp16, bf16) or 1-byte ones (E4M3, E5M2)
    const void* B;
    void* out;
    int out_type;
    int M, N, K, batch;
    int64_t lda, ldb, ldo;
    int64_t stride_a, stride_b, stride_o;
    int vec_a;  // A's rows start on 8-element boundaries (vector loads of 8 elements)
    int vec_b;
    int a_mn;   // 1: A is MN-major, A(i, k) at A[k*lda + i]
    int b_mn;   // 1: B is MN-major, B(j, k) at B[k*ldb + j]
};

// tcgen05 kernel family.  bn in {64, 128, 256}; swap selects the transposed
// epilogue; kind 0: 16-bit inputs, 1: 8-bit inputs, 2: 8-bit inputs with block
// scales (bn 64 or 128, 128-row X tiles).  Returns the launch status.
cudaError_t tc05_configure(int bn, bool swap);  // one-time per device
// The same kernel with other instruction shapes: tm = 64 rows on the plain
// M = 64 MMA (bn 64, 128, 256), or ws: the weight-stationary MMA with tm = 64
// (bn 128, 256) or 32 (bn 256).  Kinds 0 and 1 (no block scales); X = A.
cudaError_t tc05_small_configure();  // one-time per device
cudaError_t tc05_small_launch(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int bn, int tm,
                              bool ws, int grid, int kind, cudaStream_t stream);
cudaError_t tc05_launch(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int bn,
                        bool swap, int grid, int kind, cudaStream_t stream);

// Block scales: plain (rows, ceil(K/32)) E8M0 bytes, row pitch ld, batch
// stride `stride` -> the atom layout of TcParams::sf_x (missing rows and K
// blocks filled with 127, a scale of one).
cudaError_t mx_pack_launch(const uint8_t* plain, int64_t ld, int64_t stride, uint8_t* packed, int64_t rows,
                           int64_t K, int64_t batch, cudaStream_t stream);

// CTA-pair tcgen05 kernel: 256 x 256 tiles on clusters of two CTAs.
// tc05_pair_configure reports how many pairs can be resident at once.
cudaError_t tc05_pair_configure(int* max_pairs);  // one-time per device
// Workspace bytes the pair kernel's stream-K pieces need for `pairs` pairs.
constexpr size_t kPairSliceBytes = 128 * 256 * 4;
constexpr size_t pair_workspace_bytes(int pairs)
{
    return static_cast<size_t>(pairs) * 4 * kPairSliceBytes + static_cast<size_t>(pairs) * 2 * 8 * 4;
}
// pbn: tile columns per pair, 256, 224 or 192 (B tensor maps use boxes of pbn/2
// rows).  direct: epilogue without shared-memory staging and a 7-stage ring;
// needs Out rows 32-byte aligned and no split (p.sk_pairs == 0).
cudaError_t tc05_pair_launch(const CUtensorMap& tma, const CUtensorMap& tmb, const TcParams& p, int pairs, int pbn,
                             bool direct, int kind, cudaStream_t stream, const CUtensorMap* tmsa = nullptr,
                             const CUtensorMap* tmsb = nullptr);

// in_type: the A/B element type, a gemm_dtype_t value (fp16, bf16, E4M3, E5M2).
cudaError_t mmasync_launch(const MmaParams& p, int in_type, cudaStream_t stream);
cudaError_t probe_launch(const uint16_t* A, const uint16_t* B, uint32_t* ar, uint32_t* br, float* dr,
                         cudaStream_t stream);

// Scratch of the pair kernel's split (stream-K) path in memory that the caller
// of run_pair_no_alloc owns: `slices` holds the slices of up to `slice_pairs`
// launched pairs (4 * kPairSliceBytes each), `counters` the counters of up to
// `counter_tiles` split tiles (16 words each).
struct PairScratch {
    float* slices;
    int slice_pairs;
    uint32_t* counters;
    int counter_tiles;
};
// Fills in the current device's fixed scratch; returns a gemm_status_t value.
typedef int (*PairScratchFn)(PairScratch* out);

// The CTA-pair kernel without any allocation.  Host-side argument errors are
// returned before any CUDA call; `scratch` is called only for valid, non-empty
// arguments.  Plans the call exactly like the automatic path does for the
// CTA-pair kernel (the same planner); returns GEMM_ERR_SCRATCH_TOO_SMALL if that
// plan needs more than the scratch holds.
int run_pair_no_alloc(const void* A, const void* B, float* Out, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldo, int64_t strideA, int64_t strideB, int64_t strideO, int64_t batch,
                      PairScratchFn scratch, cudaStream_t stream);

}  // namespace gnt
