// tc05_common.cuh -- pieces shared by the tcgen05 kernels (one CTA per tile,
// and CTA pairs): work decomposition, bounded mbarrier waits and the epilogue
// that moves one finished TMEM accumulator to Out.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace gnt {
namespace tc {

constexpr int BM = 128;  // MMA rows per CTA (TMEM lanes)
constexpr int BK = 64;   // K per stage: 64 fp16 = one 128-byte swizzle row

// One operand tile of ROWS rows x BK into a stage slot.  K-major: one box
// {BK, ROWS} at (k, row).  MN-major: ROWS/64 boxes {64 rows, BK} at (row + 64j,
// k), 8 KB apart (the chunks sw128_mnmajor_desc expects).  Either way the slot
// receives ROWS x 128 bytes.  PAIR: the completion is signalled on the
// leader CTA's barrier (bar is a cluster address).  Only tiles of whole
// 64-row chunks can be MN-major (the host never sets mn for others).
template <int ROWS, bool PAIR = false>
__device__ __forceinline__ void load_operand(uint32_t slot, const CUtensorMap* map, uint32_t bar, bool mn, int k,
                                             int row, int b)
{
    if (ROWS % 64 == 0 && mn) {
#pragma unroll
        for (int j = 0; j < ROWS / 64; ++j) {
            if (PAIR)
                tma_load_3d_pair(slot + j * kMnChunkBytes, map, bar, row + 64 * j, k, b);
            else
                tma_load_3d(slot + j * kMnChunkBytes, map, bar, row + 64 * j, k, b);
        }
    } else {
        if (PAIR)
            tma_load_3d_pair(slot, map, bar, k, row, b);
        else
            tma_load_3d(slot, map, bar, k, row, b);
    }
}

// The same tile, fetched into L2 only.
template <int ROWS>
__device__ __forceinline__ void prefetch_operand(const CUtensorMap* map, bool mn, int k, int row, int b)
{
    if (ROWS % 64 == 0 && mn) {
#pragma unroll
        for (int j = 0; j < ROWS / 64; ++j)
            tma_prefetch_l2_3d(map, row + 64 * j, k, b);
    } else {
        tma_prefetch_l2_3d(map, k, row, b);
    }
}

// Tile index -> (batch, x tile, y tile).  Within a batch, tiles are taken in
// groups of group_x x-tiles, column by column, so CTAs running at the same time
// share X rows and Y rows in L2.
__device__ __forceinline__ void decode_tile(const TcParams& p, int tile, int& b, int& tx, int& ty)
{
    b = tile / p.tiles_per_batch;
    const int t = tile - b * p.tiles_per_batch;
    const int span = p.group_x * p.tiles_y;
    const int g = t / span;
    const int first_x = g * p.group_x;
    const int rem_x = p.tiles_x - first_x;
    const int gx = rem_x < p.group_x ? rem_x : p.group_x;
    const int r = t - g * span;
    tx = first_x + r % gx;
    ty = r / gx;
}

// One piece of work: output rows [x0, xend) x columns [y0, y0 + BN) of batch b,
// k-blocks [kb0, kb1).  `partial` when the k range is not the whole of K.
struct Seg {
    int b, x0, xend, y0, kb0, kb1;
    bool partial;
    int sk_t;  // stream-K tile index (from sk_first), -1 outside stream-K
    int slot;  // workspace slot of a stream-K piece: 0 first of the CTA's range, 1 last
};

// Walks this CTA's share of the work.
//   kModeTiles     whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...
//   kModeStreamK   the contiguous range of (tile, k-block) iterations
//                  [total*c/G, total*(c+1)/G), cut at tile borders
//   kModeRowSplit  one piece per CTA: rows [rows_x*c/G, rows_x*(c+1)/G) (at
//                  most 128) over all of K; the 128-row operand box starts at
//                  the first row, so neighbouring boxes overlap and only the
//                  CTA's own rows are stored
template <int BN, int TM = BM>
struct WorkIter {
    long long it, end;
    int tile, step, mode;
    const TcParams& p;

    __device__ explicit WorkIter(const TcParams& prm) : p(prm)
    {
        mode = p.mode;
        if (mode == kModeStreamK) {
            it = p.total_iters * blockIdx.x / gridDim.x;
            end = p.total_iters * (blockIdx.x + 1) / gridDim.x;
        } else {
            tile = blockIdx.x;
            step = gridDim.x;
        }
    }

    __device__ bool next(Seg& s)
    {
        int t, tx, ty;
        s.sk_t = -1;
        s.slot = 0;
        if (mode == kModeRowSplit) {
            if (tile >= static_cast<int>(gridDim.x))
                return false;
            const long long rx = p.rows_x;
            s.b = 0;
            s.x0 = static_cast<int>(rx * tile / gridDim.x);
            s.xend = static_cast<int>(rx * (tile + 1) / gridDim.x);
            s.y0 = 0;
            s.kb0 = 0;
            s.kb1 = p.num_kb;
            s.partial = false;
            tile += step;
            return true;
        }
        if (mode == kModeStreamK) {
            if (it >= end)
                return false;
            t = static_cast<int>(it / p.num_kb);
            s.kb0 = static_cast<int>(it - static_cast<long long>(t) * p.num_kb);
            const long long k1 = s.kb0 + (end - it);
            s.kb1 = k1 < p.num_kb ? static_cast<int>(k1) : p.num_kb;
            it += s.kb1 - s.kb0;
        } else {
            if (tile >= p.num_tiles)
                return false;
            t = tile;
            s.kb0 = 0;
            s.kb1 = p.num_kb;
            tile += step;
        }
        decode_tile(p, t, s.b, tx, ty);
        s.x0 = tx * TM;
        s.xend = s.x0 + TM < p.rows_x ? s.x0 + TM : p.rows_x;
        s.y0 = ty * BN;
        s.partial = s.kb0 != 0 || s.kb1 != p.num_kb;
        return true;
    }
};

// The slow path of wait_bounded, kept out of line so the issue loops that call
// it stay short: sleep in try_wait until the phase completes, giving up when
// another thread has raised the abort flag or after `limit` cycles.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                       unsigned long long limit)
{
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 1000000u))
            return true;
        if (*abort_flag)
            return false;
        if (static_cast<unsigned long long>(clock64() - t0) > limit)
            return false;
    }
}

// Bounded wait.  Returns false if the limit passed or another role aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                             unsigned long long limit)
{
    return mbar_try_wait(bar, parity) || wait_slow(bar, parity, abort_flag, limit);
}

__device__ __forceinline__ void raise_timeout(const TcParams& p, volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicOr(p.status, kStatusTimeout);
}


// Stores one 32x32 chunk of the accumulator held row-per-thread (lane i has
// row x_row0 + i, columns col0..col0+31 in v[]): transpose through shared
// memory (16-byte slots XOR-swizzled by row) so the global stores are
// row-contiguous across the warp.  Rows beyond nx and columns beyond rows_y
// are not stored; `atomic` adds into (fp32) Out instead of storing.  obase
// points at element 0 of this batch's Out.
template <int OT>
__device__ __forceinline__ void store_rows_chunk(const TcParams& p, typename OutStore<OT>::T* obase, int x_row0,
                                                 int nx, int col0, const float (&v)[32], int lane, float* stage_buf,
                                                 bool atomic)
{
    using S = OutStore<OT>;
    float4* sb4 = reinterpret_cast<float4*>(stage_buf);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        sb4[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    if (p.vec4 && !atomic) {
        // 8 lanes per 32-column row segment, 4 rows per instruction
        const int ch = lane & 7, rsub = lane >> 3;
        const int ncol = p.rows_y - (col0 + ch * 4);
        typename S::T* dst = obase + static_cast<int64_t>(x_row0 + rsub) * p.ldo + col0 + ch * 4;
        const int64_t step = 4 * p.ldo;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = i * 4 + rsub;
            const float4 w = sb4[rr * 8 + (ch ^ (rr & 7))];
            if (rr < nx) {
                if (ncol >= 4) {
                    S::st4(dst, w);
                } else {
                    if (ncol > 0) S::st1(dst, w.x);
                    if (ncol > 1) S::st1(dst + 1, w.y);
                    if (ncol > 2) S::st1(dst + 2, w.z);
                }
            }
            dst += step;
        }
    } else if (col0 + lane < p.rows_y) {
        // one column per lane, 32 rows
        typename S::T* dst = obase + static_cast<int64_t>(x_row0) * p.ldo + col0 + lane;
        const float* src = stage_buf + (lane & 3);
        const int g = lane >> 2;
        if (atomic) {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                const float w = src[rr * 32 + ((g ^ (rr & 7)) << 2)];
                if (rr < nx) S::add1(dst, w);
                dst += p.ldo;
            }
        } else {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                const float w = src[rr * 32 + ((g ^ (rr & 7)) << 2)];
                if (rr < nx) S::st1(dst, w);
                dst += p.ldo;
            }
        }
    }
    __syncwarp();
}

// fp32 Out rows that are not 16-byte aligned.  A 32-column row segment
// stored one float per lane would cover two 128-byte lines; here every store
// instruction writes one aligned line of one row instead.  Row rr's columns
// start sr floats into a line, and the staging area keeps the row rotated by
// sr: chunk column i at word (i + sr) mod 32.  So word l holds the line's
// column l, from this chunk (l >= sr) or, for l < sr, from the previous
// chunk's last sr columns, which stay in words 0 .. sr-1 until this chunk's
// line is stored: the chunk's first 32 - sr columns go in before the line
// stores, its last sr columns after them.  The last chunk's tail is stored
// after the loop.  No bank conflicts when ldo is odd (the rows' rotations then
// differ).  Only columns in [y0 + c_begin, min(y0 + c_end, rows_y)) and rows
// below nx are stored, so the result is that of epilogue_store.
__device__ __forceinline__ void epilogue_store_lines(const TcParams& p, uint32_t tbase, float* obase, int x_row0,
                                                     int nx, int y0, int c_begin, int c_end, int lane,
                                                     float* stage_buf)
{
    const int cb = y0 + c_begin;
    const int ce = min(y0 + c_end, p.rows_y);
    float* const row0 = obase + static_cast<int64_t>(x_row0) * p.ldo + cb;  // element (x_row0, cb)
    const uint32_t s0 = (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row0)) >> 2) & 31u;
    const uint32_t sstep = static_cast<uint32_t>(p.ldo) & 31u;
    const int s_own = static_cast<int>((s0 + static_cast<uint32_t>(lane) * sstep) & 31u);  // sr of this lane's row
    float* const wrot = stage_buf + lane * 32 + s_own;  // chunk column i goes to wrot[i] or wrot[i - 32]
    const float* const rcol = stage_buf + lane;
    int c = c_begin;
#pragma unroll 1
    for (; c < c_end; c += 32) {
        if (nx <= 0 || y0 + c >= p.rows_y)
            break;  // warp-uniform
        uint32_t r[32];
        tmem_ld32_wait(tbase + static_cast<uint32_t>(c), r);
        // Opaque copies of the loop-invariant row pointer and rotation, so that
        // the 32 row pointers and rotations are formed here in every chunk
        // rather than hoisted out of the loop into registers.
        uint32_t sr;
        uint64_t dst_bits;
        asm volatile("mov.b32 %0, %1;" : "=r"(sr) : "r"(s0));
        asm volatile("mov.b64 %0, %1;" : "=l"(dst_bits) : "l"(reinterpret_cast<uint64_t>(row0)));
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < 32 - s_own)
                wrot[i] = __uint_as_float(r[i]);
        __syncwarp();
        const int gl = (y0 + c) - cb + lane;  // this lane's column, from cb, if its row started on a line
        float* dst = reinterpret_cast<float*>(dst_bits);
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            const int g = gl - static_cast<int>(sr);
            if (rr < nx && g >= 0 && g < ce - cb)
                __stcs(dst + g, rcol[rr * 32]);
            dst += p.ldo;
            sr = (sr + sstep) & 31u;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i >= 32 - s_own)
                wrot[i - 32] = __uint_as_float(r[i]);
    }
    __syncwarp();
    if (c > c_begin) {
        // the last chunk's columns [y0 + c - sr, y0 + c), in words 0 .. sr-1
        const int gl = (y0 + c) - cb + lane;
        float* dst = row0;
        uint32_t sr = s0;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            const int g = gl - static_cast<int>(sr);
            if (rr < nx && static_cast<uint32_t>(lane) < sr && g < ce - cb)
                __stcs(dst + g, rcol[rr * 32]);
            dst += p.ldo;
            sr = (sr + sstep) & 31u;
        }
    }
    __syncwarp();  // the staging area is rewritten by the next call
}

// One epilogue warp's share of a finished accumulator: TMEM lane quadrant q
// (tile rows s.x0 + 32q .. +31) and accumulator columns [c_begin, c_end),
// where `tacc` is the TMEM address of the accumulator's first column.  Other
// accumulator layouts (64-row and weight-stationary MMAs) give the quadrant's
// first tile row (row_off >= 0), its number of rows (row_cap) and the tile
// column of its TMEM column 0 (col_off).
// Rows >= s.xend and columns >= rows_y are not stored; `stage_buf` is this
// warp's 32x32 fp32 staging area (unused when SWAP).  Partial segments (a
// k range short of all of K) add into (fp32) Out with atomics.
template <bool SWAP, int OT>
__device__ __forceinline__ void epilogue_store(const TcParams& p, const Seg& s, uint32_t tacc, int q,
                                               int c_begin, int c_end, int lane, float* stage_buf,
                                               int row_off = -1, int row_cap = 32, int col_off = 0)
{
    using S = OutStore<OT>;
    const bool partial = s.partial;
    const uint32_t tbase = tacc + (static_cast<uint32_t>(q * 32) << 16);
    typename S::T* obase = static_cast<typename S::T*>(p.out) + static_cast<int64_t>(s.b) * p.stride_o;
    const int x_row0 = s.x0 + (row_off < 0 ? q * 32 : row_off);
    int nx = s.xend - x_row0;  // valid rows of this quadrant
    if (nx > row_cap)
        nx = row_cap;
    const int y0 = s.y0 + col_off;
    if constexpr (!SWAP && OT == kOutF32) {
        if (!partial && !p.vec4) {
            epilogue_store_lines(p, tbase, obase, x_row0, nx, y0, c_begin, c_end, lane, stage_buf);
            return;
        }
    }
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
        if (nx <= 0 || y0 + c >= p.rows_y)
            break;  // warp-uniform: nothing of this chunk is inside Out
        uint32_t r[32];
        tmem_ld32_wait(tbase + static_cast<uint32_t>(c), r);
        if (SWAP) {
            // Thread <-> x (consecutive Out columns): each j is one
            // coalesced row segment across the warp.
            const int ny = p.rows_y - (y0 + c);
            if (lane < nx) {
                typename S::T* dst = obase + static_cast<int64_t>(y0 + c) * p.ldo + (x_row0 + lane);
                if (partial) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j < ny) S::add1(dst, __uint_as_float(r[j]));
                        dst += p.ldo;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j < ny) S::st1(dst, __uint_as_float(r[j]));
                        dst += p.ldo;
                    }
                }
            }
        } else {
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k)
                v[k] = __uint_as_float(r[k]);
            store_rows_chunk<OT>(p, obase, x_row0, nx, y0 + c, v, lane, stage_buf, partial);
        }
    }
}

// Direct epilogue for Out rows whose starts are aligned to 8 elements (ldo a
// multiple of 8, base aligned to 8 elements): no shared-memory staging.  TMEM
// is read with the 16x256b shape, which hands each quad of lanes 8
// consecutive columns of one row, so each pair store of a warp writes whole
// 8-element row segments (32 bytes of fp32).  Same coverage and masking as
// epilogue_store.
template <int OT>
__device__ __forceinline__ void epilogue_store_direct(const TcParams& p, const Seg& s, uint32_t tacc, int q,
                                                      int c_begin, int c_end, int lane)
{
    using S = OutStore<OT>;
    typename S::T* obase = static_cast<typename S::T*>(p.out) + static_cast<int64_t>(s.b) * p.stride_o;
    const int x_row0 = s.x0 + q * 32;
    const int nx = s.xend - x_row0;
    const int rsub = lane >> 2;
    const int csub = 2 * (lane & 3);
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
        if (nx <= 0 || s.y0 + c >= p.rows_y)
            break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h * 16 >= nx)
                break;
            uint32_t r[16];
            tmem_ld16x256_x4_wait(tacc + (static_cast<uint32_t>(q * 32 + h * 16) << 16) + static_cast<uint32_t>(c), r);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int row = h * 16 + half * 8 + rsub;  // within the quadrant
                if (row < nx) {
                    typename S::T* dst = obase + static_cast<int64_t>(x_row0 + row) * p.ldo + s.y0 + c + csub;
                    const int ncol = p.rows_y - (s.y0 + c + csub);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float v0 = __uint_as_float(r[4 * j + 2 * half]);
                        const float v1 = __uint_as_float(r[4 * j + 2 * half + 1]);
                        if (ncol - 8 * j >= 2)
                            S::st2(dst + 8 * j, v0, v1);
                        else if (ncol - 8 * j == 1)
                            S::st1(dst + 8 * j, v0);
                    }
                }
            }
        }
    }
}

// The direct epilogue in two halves, for a kernel with a single accumulator:
// the warp first loads its whole share (NCH 32-column chunks from c_begin of
// its lane quadrant, 16x256b as above) into registers, so the caller can free
// the accumulator for the next tile's MMAs before any store is issued, then
// stores from those registers with the same coverage and masking.
template <int NCH>
__device__ __forceinline__ void epilogue_load_direct(uint32_t tacc, int q, int c_begin, uint32_t (&v)[2 * NCH][16])
{
#pragma unroll
    for (int ci = 0; ci < NCH; ++ci)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            tmem_ld16x256_x4_wait(tacc + (static_cast<uint32_t>(q * 32 + h * 16) << 16) +
                                      static_cast<uint32_t>(c_begin + 32 * ci),
                                  v[2 * ci + h]);
}

template <int OT, int NCH>
__device__ __forceinline__ void epilogue_store_direct_regs(const TcParams& p, const Seg& s, int q, int c_begin,
                                                           int lane, const uint32_t (&v)[2 * NCH][16])
{
    using S = OutStore<OT>;
    typename S::T* obase = static_cast<typename S::T*>(p.out) + static_cast<int64_t>(s.b) * p.stride_o;
    const int x_row0 = s.x0 + q * 32;
    const int nx = s.xend - x_row0;
    const int rsub = lane >> 2;
    const int csub = 2 * (lane & 3);
#pragma unroll
    for (int ci = 0; ci < NCH; ++ci) {
        const int c = c_begin + 32 * ci;
        if (nx > 0 && s.y0 + c < p.rows_y) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int row = h * 16 + half * 8 + rsub;  // within the quadrant
                    if (row < nx) {
                        typename S::T* dst = obase + static_cast<int64_t>(x_row0 + row) * p.ldo + s.y0 + c + csub;
                        const int ncol = p.rows_y - (s.y0 + c + csub);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float v0 = __uint_as_float(v[2 * ci + h][4 * j + 2 * half]);
                            const float v1 = __uint_as_float(v[2 * ci + h][4 * j + 2 * half + 1]);
                            if (ncol - 8 * j >= 2)
                                S::st2(dst + 8 * j, v0, v1);
                            else if (ncol - 8 * j == 1)
                                S::st1(dst + 8 * j, v0);
                        }
                    }
                }
            }
        }
    }
}

}  // namespace tc
}  // namespace gnt
