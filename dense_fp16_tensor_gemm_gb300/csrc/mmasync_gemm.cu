// mmasync_gemm.cu -- ldmatrix + mma.sync m16n8k16 kernel for Out = A @ B.T on
// any layout (unaligned bases, odd leading dimensions, tiny or ragged shapes),
// and the one-warp fragment probe.
//
// "Warp Matrix Instructions" ("From Shared Memory to a Matrix Product") computes
// one 16x8 output tile with a single warp: the operands are staged in shared
// memory, ldmatrix.x4 loads A (16x16) as four 8x8 matrices in the order
// (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15),
// ldmatrix.x2 loads B (8x16) as (k 0-7), (k 8-15), and one mma.sync m16n8k16
// (row.col, f32 accumulators, C = 0) leaves dr[r] for lane l at
// Out[l/4 + 8*(r/2), 2*(l%4) + r%2].  "Other Fragment Shapes and Transfers" adds
// that a longer K is several issues accumulating into the previous D.
// "copy -> ldstmatrix" ("Algorithm" steps 3-4) gives the shared-memory rule:
// each lane supplies the address of one 16-byte row, so row strides are
// multiples of 8 fp16.
//
// This kernel tiles that warp product: a CTA of 4 warps owns a 64x64 output
// tile, each warp a 32x32 sub-tile (2 x 4 m16n8 tiles), and K advances 32 at a
// time through shared memory with 80-byte row pitch (16-byte aligned rows,
// conflict-free ldmatrix).  Out-of-range rows and the K tail are zero-filled
// while staging, and stores are masked.
//
// 8-bit float operands (E4M3, E5M2) are widened to fp16 while staging (exact)
// and multiplied on the same fp16 MMA.
//
// An MN-major operand (A stored as (K, M), B as (K, N)) is staged as it lies,
// 32 K-rows of 64 elements with a 144-byte pitch, i.e. a column-major shared
// tile of the operand; "copy -> ldstmatrix" ("Algorithm" step 3) reads such a
// tile with the .trans form of ldmatrix, whose lane t receives elements
// (2(t%4), t/4) and (2(t%4)+1, t/4) of each 8x8 block: with K on the block's
// rows that is exactly the fragment the row-major tile gives.
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace gnt {

namespace {

constexpr int MBM = 64, MBN = 64, MBK = 32, MPAD = 8;
constexpr int MPITCH = MBK + MPAD;  // 40 fp16 = 80 bytes
constexpr int MNPITCH = 64 + 8;     // MN-major tile: 72 fp16 = 144 bytes per K-row
constexpr int MThreads = 128;
constexpr int kTileElems = MBM * MPITCH;  // >= MBK * MNPITCH
static_assert(MBK * MNPITCH <= kTileElems, "MN-major tile fits the slot");

// Element types of A and B (gemm_dtype_t values).  The 16-bit types are staged
// as they are; the 8-bit floats are widened to fp16 while staging, which is
// exact (every E4M3 and E5M2 value is an fp16 value), and multiplied on the
// fp16 MMA.
constexpr int kInF16 = 0, kInBF16 = 1, kInE4M3 = 3, kInE5M2 = 4;

template <int IN>
struct Elem {
    using T = uint16_t;
    static __device__ __forceinline__ uint16_t get(const T* g) { return *g; }
    static __device__ __forceinline__ uint4 get8(const T* g) { return *reinterpret_cast<const uint4*>(g); }
};

template <int IN>
struct Elem8 {
    using T = uint8_t;
    static __device__ __forceinline__ uint16_t get(const T* g)
    {
        return __nv_cvt_fp8_to_halfraw(*g, IN == kInE5M2 ? __NV_E5M2 : __NV_E4M3).x;
    }
    static __device__ __forceinline__ uint4 get8(const T* g)
    {
        const uint2 raw = *reinterpret_cast<const uint2*>(g);
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t word = e < 2 ? raw.x : raw.y;
            const int sh = (e & 1) * 16;
            const uint16_t lo = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((word >> sh) & 0xff),
                                                        IN == kInE5M2 ? __NV_E5M2 : __NV_E4M3).x;
            const uint16_t hi = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((word >> (sh + 8)) & 0xff),
                                                        IN == kInE5M2 ? __NV_E5M2 : __NV_E4M3).x;
            w[e] = lo | (static_cast<uint32_t>(hi) << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <>
struct Elem<kInE4M3> : Elem8<kInE4M3> {};
template <>
struct Elem<kInE5M2> : Elem8<kInE5M2> {};

// Stage one (rows x 32) operand tile into shared memory as fp16 (or bf16),
// zero-filling everything outside rows < nrows and k < K.
template <int IN>
__device__ __forceinline__ void stage_tile(uint16_t* sdst, const void* src_v, int64_t ld, int row0, int nrows,
                                           int k0, int K, bool vec)
{
    using E = Elem<IN>;
    const typename E::T* src = static_cast<const typename E::T*>(src_v);
    const int tid = threadIdx.x;
    if (vec) {
        // 64 rows x 4 chunks of 8 fp16 = 256 chunks, two per thread.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = tid + i * MThreads;
            const int r = c >> 2;
            const int kc = (c & 3) * 8;
            const int row = row0 + r;
            const int k = k0 + kc;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row < nrows) {
                const typename E::T* g = src + static_cast<int64_t>(row) * ld + k;
                if (k + 8 <= K) {
                    v = E::get8(g);
                } else if (k < K) {
                    uint16_t tmp[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        tmp[e] = (k + e < K) ? E::get(g + e) : uint16_t(0);
                    v = make_uint4(tmp[0] | (uint32_t(tmp[1]) << 16), tmp[2] | (uint32_t(tmp[3]) << 16),
                                   tmp[4] | (uint32_t(tmp[5]) << 16), tmp[6] | (uint32_t(tmp[7]) << 16));
                }
            }
            *reinterpret_cast<uint4*>(sdst + r * MPITCH + kc) = v;
        }
    } else {
        // Element-wise, consecutive threads on consecutive k.
#pragma unroll 4
        for (int i = 0; i < (64 * MBK) / MThreads; ++i) {
            const int e = tid + i * MThreads;
            const int r = e / MBK;
            const int kk = e % MBK;
            const int row = row0 + r;
            const int k = k0 + kk;
            uint16_t v = 0;
            if (row < nrows && k < K)
                v = E::get(src + static_cast<int64_t>(row) * ld + k);
            sdst[r * MPITCH + kk] = v;
        }
    }
}

// Stage one MN-major operand tile, rows [mn0, mn0 + 64) x k in [k0, k0 + 32),
// from src (element (r, k) at src[k*ld + r]) into sdst[kk][r - mn0], zero
// outside r < nmn and k < K.
template <int IN>
__device__ __forceinline__ void stage_tile_mn(uint16_t* sdst, const void* src_v, int64_t ld, int mn0, int nmn,
                                              int k0, int K, bool vec)
{
    using E = Elem<IN>;
    const typename E::T* src = static_cast<const typename E::T*>(src_v);
    const int tid = threadIdx.x;
    if (vec) {
        // 32 K-rows x 8 chunks of 8 elements, two chunks per thread.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = tid + i * MThreads;
            const int kk = c >> 3;
            const int rc = (c & 7) * 8;
            const int k = k0 + kk;
            const int r = mn0 + rc;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k < K) {
                const typename E::T* g = src + static_cast<int64_t>(k) * ld + r;
                if (r + 8 <= nmn) {
                    v = E::get8(g);
                } else if (r < nmn) {
                    uint16_t tmp[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        tmp[e] = (r + e < nmn) ? E::get(g + e) : uint16_t(0);
                    v = make_uint4(tmp[0] | (uint32_t(tmp[1]) << 16), tmp[2] | (uint32_t(tmp[3]) << 16),
                                   tmp[4] | (uint32_t(tmp[5]) << 16), tmp[6] | (uint32_t(tmp[7]) << 16));
                }
            }
            *reinterpret_cast<uint4*>(sdst + kk * MNPITCH + rc) = v;
        }
    } else {
        // Element-wise, consecutive threads on consecutive rows of the operand.
#pragma unroll 4
        for (int i = 0; i < (MBK * 64) / MThreads; ++i) {
            const int e = tid + i * MThreads;
            const int kk = e >> 6;
            const int rr = e & 63;
            const int k = k0 + kk;
            const int r = mn0 + rr;
            uint16_t v = 0;
            if (r < nmn && k < K)
                v = E::get(src + static_cast<int64_t>(k) * ld + r);
            sdst[kk * MNPITCH + rr] = v;
        }
    }
}

// Out rows [row0, ...) of one 64x64 CTA tile through the D-fragment map.
template <int OT>
__device__ __forceinline__ void store_tile(const MmaParams& p, int b, int m0, int n0, int wm, int wn, int lane,
                                           const float (&acc)[2][4][4])
{
    using S = OutStore<OT>;
    typename S::T* Ob = static_cast<typename S::T*>(p.out) + static_cast<int64_t>(b) * p.stride_o;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = m0 + wm * 32 + mi * 16 + (lane >> 2) + 8 * (r >> 1);
                const int col = n0 + wn * 32 + nb * 8 + 2 * (lane & 3) + (r & 1);
                if (row < p.M && col < p.N)
                    S::st1(Ob + static_cast<int64_t>(row) * p.ldo + col, acc[mi][nb][r]);
            }
}

template <int IN>
__global__ void __launch_bounds__(MThreads) mmasync_gemm_kernel(const MmaParams p)
{
    __shared__ __align__(16) uint16_t As[kTileElems];
    __shared__ __align__(16) uint16_t Bs[kTileElems];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wm = warp >> 1, wn = warp & 1;
    const int m0 = blockIdx.y * MBM, n0 = blockIdx.x * MBN;

    for (int b = blockIdx.z; b < p.batch; b += gridDim.z) {
        using ET = typename Elem<IN>::T;
        const ET* Ab = static_cast<const ET*>(p.A) + static_cast<int64_t>(b) * p.stride_a;
        const ET* Bb = static_cast<const ET*>(p.B) + static_cast<int64_t>(b) * p.stride_b;
        float acc[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    acc[i][j][r] = 0.f;

        for (int k0 = 0; k0 < p.K; k0 += MBK) {
            __syncthreads();  // previous tile fully consumed
            if (p.a_mn)
                stage_tile_mn<IN>(As, Ab, p.lda, m0, p.M, k0, p.K, p.vec_a);
            else
                stage_tile<IN>(As, Ab, p.lda, m0, p.M, k0, p.K, p.vec_a);
            if (p.b_mn)
                stage_tile_mn<IN>(Bs, Bb, p.ldb, n0, p.N, k0, p.K, p.vec_b);
            else
                stage_tile<IN>(Bs, Bb, p.ldb, n0, p.N, k0, p.K, p.vec_b);
            __syncthreads();
#pragma unroll
            for (int ks = 0; ks < MBK; ks += 16) {
                // Lane l addresses row l%8 of 8x8 block q = l/8.
                const int q = lane >> 3, r8 = lane & 7;
                uint32_t af[2][4];
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                    if (p.a_mn) {
                        // block q: rows m + 8(q%2), k + 8(q/2); K runs down the shared tile
                        const int krow = ks + (q >> 1) * 8 + r8;
                        const int col = wm * 32 + mi * 16 + (q & 1) * 8;
                        ldmatrix_x4_trans(smem_u32(As + krow * MNPITCH + col), af[mi][0], af[mi][1], af[mi][2],
                                          af[mi][3]);
                    } else {
                        const int row = wm * 32 + mi * 16 + (lane & 15);
                        const int col = ks + (lane >> 4) * 8;
                        ldmatrix_x4(smem_u32(As + row * MPITCH + col), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
                    }
                }
                uint32_t bfr[4][2];
#pragma unroll
                for (int nj = 0; nj < 2; ++nj) {
                    if (p.b_mn) {
                        // block q: k + 8(q%2), n + 8(q/2)
                        const int krow = ks + (q & 1) * 8 + r8;
                        const int col = wn * 32 + nj * 16 + (q >> 1) * 8;
                        ldmatrix_x4_trans(smem_u32(Bs + krow * MNPITCH + col), bfr[2 * nj][0], bfr[2 * nj][1],
                                          bfr[2 * nj + 1][0], bfr[2 * nj + 1][1]);
                    } else {
                        // lanes 0-7: n 0-7 @k, 8-15: n 0-7 @k+8, 16-23: n 8-15 @k, 24-31: n 8-15 @k+8
                        const int row = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
                        const int col = ks + ((lane >> 3) & 1) * 8;
                        ldmatrix_x4(smem_u32(Bs + row * MPITCH + col), bfr[2 * nj][0], bfr[2 * nj][1],
                                    bfr[2 * nj + 1][0], bfr[2 * nj + 1][1]);
                    }
                }
#pragma unroll
                for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb)
                        if (IN == kInBF16)
                            mma_m16n8k16_bf16(acc[mi][nb], af[mi], bfr[nb][0], bfr[nb][1], acc[mi][nb]);
                        else
                            mma_m16n8k16(acc[mi][nb], af[mi], bfr[nb][0], bfr[nb][1], acc[mi][nb]);
            }
        }

        if (p.out_type == kOutF16)
            store_tile<kOutF16>(p, b, m0, n0, wm, wn, lane, acc);
        else if (p.out_type == kOutBF16)
            store_tile<kOutBF16>(p, b, m0, n0, wm, wn, lane, acc);
        else
            store_tile<kOutF32>(p, b, m0, n0, wm, wn, lane, acc);
    }
}

// One warp, the warp example verbatim in structure: lanes copy elements
// lane + 32q of A and B into shared memory, ldmatrix.x4 / .x2, one MMA with
// C = 0, and the raw registers are written out lane-major.
__global__ void __launch_bounds__(32) probe_kernel(const uint16_t* A, const uint16_t* B, uint32_t* ar_out,
                                                    uint32_t* br_out, float* dr_out)
{
    __shared__ __align__(16) uint16_t a[16 * 16];
    __shared__ __align__(16) uint16_t b[8 * 16];
    const int lane = threadIdx.x;
    for (int q = 0; q < 8; ++q)
        a[lane + 32 * q] = A[lane + 32 * q];
    for (int q = 0; q < 4; ++q)
        b[lane + 32 * q] = B[lane + 32 * q];
    __syncthreads();
    uint32_t ar[4], br[2];
    ldmatrix_x4(smem_u32(a + (lane & 15) * 16 + (lane >> 4) * 8), ar[0], ar[1], ar[2], ar[3]);
    ldmatrix_x2(smem_u32(b + (lane & 7) * 16 + ((lane >> 3) & 1) * 8), br[0], br[1]);
    float dr[4];
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    mma_m16n8k16(dr, ar, br[0], br[1], zero);
    for (int r = 0; r < 4; ++r) {
        ar_out[lane * 4 + r] = ar[r];
        dr_out[lane * 4 + r] = dr[r];
    }
    for (int r = 0; r < 2; ++r)
        br_out[lane * 2 + r] = br[r];
}

}  // namespace

cudaError_t mmasync_launch(const MmaParams& p, int in_type, cudaStream_t stream)
{
    dim3 grid((p.N + MBN - 1) / MBN, (p.M + MBM - 1) / MBM, p.batch < 65535 ? p.batch : 65535);
    if (grid.y > 65535)
        return cudaErrorInvalidConfiguration;
    switch (in_type) {
    case kInF16: mmasync_gemm_kernel<kInF16><<<grid, MThreads, 0, stream>>>(p); break;
    case kInBF16: mmasync_gemm_kernel<kInBF16><<<grid, MThreads, 0, stream>>>(p); break;
    case kInE4M3: mmasync_gemm_kernel<kInE4M3><<<grid, MThreads, 0, stream>>>(p); break;
    case kInE5M2: mmasync_gemm_kernel<kInE5M2><<<grid, MThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t probe_launch(const uint16_t* A, const uint16_t* B, uint32_t* ar, uint32_t* br, float* dr,
                         cudaStream_t stream)
{
    probe_kernel<<<1, 32, 0, stream>>>(A, B, ar, br, dr);
    return cudaGetLastError();
}

}  // namespace gnt
