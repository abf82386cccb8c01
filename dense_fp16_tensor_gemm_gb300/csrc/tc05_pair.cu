// tc05_pair.cu -- tcgen05 kernel on CTA pairs (cta_group::2) for Out = A @ B.T.
//
// "Blackwell Tensor Cores" names CTA-pair operation among the MMA forms beyond
// its single-CTA example.  Here a cluster of two CTAs on two SMs owns a
// 256 x 256 output tile: CTA r stages rows [128r, 128r+128) of the tile's A
// panel and rows [128r, 128r+128) of its B panel (half of B) in its own shared
// memory; the leader CTA (rank 0) issues tcgen05.mma.cta_group::2 with shape
// 256x256x16, which reads both CTAs' operands and leaves rows [128r, 128r+128)
// of the fp32 accumulator in CTA r's TMEM.  Compared with one CTA per 128x256
// tile, each SM moves 32 KB per k-block from L2 instead of 48 KB for the same
// MMA work.
//
// Roles per CTA (352 threads): warp 0 producer, warp 1 TMEM allocation (both
// CTAs) and MMA issue (leader only), warps 2-9 epilogue, warp 10 the scale
// copier of block-scaled kernels (others launch it too and it exits at once).
// The kernels are compiled for up to 384 threads: under that bound ptxas
// spills nothing (under 320 the staged-epilogue instances spilled, and their
// 16 x 3001 x 2047 x 1000 product ran 190 us, against 183 us now).
// Synchronisation:
//   full[s]    in the leader: its producer posts the byte count of both CTAs'
//              loads; both CTAs' TMA loads complete on it
//   empty[s]   in each CTA: the leader's MMA commit arrives on both (multicast)
//   tfull[b]   in each CTA: the leader's commit after a tile's last MMA
//   tempty[b]  in the leader: one arrival per epilogue warp of both CTAs
// Every wait is bounded as in the single-CTA kernel.
#include <algorithm>

#include "ptx_mx.cuh"
#include "tc05_common.cuh"

namespace gnt {

namespace {

using namespace tc;

constexpr int kPairThreads = 320;
constexpr int A_BYTES = BM * BK * 2;           // this CTA's 128 rows of A
constexpr int TMEM_COLS = 512;                 // two accumulators (and, block-scaled, the scale slots)
constexpr int BAR_BYTES = 256;
constexpr int kTemptyArrivals = 2 * 8;         // one per epilogue warp, both CTAs

// PBN: tile columns (rows of B) per pair; each CTA stages PBN/2 rows of B.
// Narrower tiles than 256 let the host fit the number of tiles to a whole
// number of rounds over the pairs.  DIRECT: the epilogue stores straight from
// TMEM-loaded registers (Out rows 32-byte aligned), which frees the 32 KB of
// staging for a seventh pipeline stage.
// KIND: 0 16-bit inputs, 1 8-bit, 2 8-bit block-scaled (PBN = 192, or 256
// with a single accumulator).  Block-scaled, each CTA needs the scale atoms of
// its 128 rows of A and those of all of the tile's B rows (each half of the
// pair MMA reads B's scales from its own CTA's TMEM; a 192-row window starts 0
// or 64 rows into a 128-row block, a 256-row one on a block, and either spans
// exactly two atoms).  They come through a ring of two scale stages, each
// holding the atoms of kScaleKb consecutive k-blocks (A: 4 KB in one box, B:
// 8 KB in one box): per-k-block 512-byte bulk copies of the atoms beside the
// data loads slowed the stream down by a third.  (256-wide tiles take B's
// atoms differently, see below.)  TMEM holds the accumulators PBN columns apart
// (one at 256 wide) and, after them, 16 scale columns per data stage (A atom,
// then the B atoms), filled by tcgen05.cp before the stage's MMAs.
constexpr int kSfAtomsB = 2;
constexpr int kScaleKb = 8;
constexpr int kScaleStages = 2;

// Block-scaled 256-wide tiles (SINGLE) keep one accumulator: two 256-column
// ones would leave TMEM no room for the scale slots.  Their epilogue warps
// load their whole share of it into registers and free it at once, then
// store, so the next tile's MMAs wait only for the TMEM reads.
// Their B scales do not go through the scale ring: each data stage carries
// the k-block's two B atoms four times over (4 KB, one TMA box of a map whose
// copy dimension has stride 0), so that one non-replicating .128x256b copy
// fills every lane quadrant.  Two replicating .32x128b.warpx4 copies per
// k-block, beside A's, held the tensor pipe to about 80 % of its rate.  The
// copier warp still issues the copies: issued by the MMA thread before each
// k-block's MMAs, they made the 8192^3 product 28 % slower.
template <int PBN, bool DIRECT, int KIND = 0>
struct PairCfg {
    static constexpr bool MX = KIND == 2;
    static constexpr bool SINGLE = MX && PBN == 256;
    static constexpr int STAGES = SINGLE ? 6 : (DIRECT ? 7 : 6);
    static constexpr int B_BYTES = (PBN / 2) * BK * 2;  // this CTA's half of B
    static constexpr int DATA_BYTES = A_BYTES + B_BYTES;
    static constexpr int SFB_REP_BYTES = SINGLE ? kSfAtomsB * 4 * 512 : 0;  // per data stage
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFB_REP_BYTES;
    // one scale stage: A's atoms, then (not SINGLE) B's
    static constexpr int SC_STAGE_BYTES = (1 + (SINGLE ? 0 : kSfAtomsB)) * kScaleKb * 512;
    static constexpr int SC_BYTES = MX ? kScaleStages * SC_STAGE_BYTES : 0;
    static constexpr int ACC_STRIDE = MX ? PBN : 256;
    static constexpr int SF_COL = SINGLE ? PBN : 2 * PBN;
    static constexpr int SF_COLS = 16;
    static constexpr int EPI_BYTES = DIRECT ? 0 : 8 * 32 * 32 * 4;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + SC_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr uint32_t IDESC = idesc_f16_f32(2 * BM, PBN);
    // epilogue warps 2-5 store columns [0, SPLIT), warps 6-9 [SPLIT, PBN)
    static constexpr int SPLIT = ((PBN / 32 + 1) / 2) * 32;
    static_assert(PBN % 32 == 0 && PBN <= 256 && PBN >= 128, "tile width");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert((3 * STAGES + 6 + 2 * kScaleStages) * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(B_BYTES % 1024 == 0, "stage slots keep the 1024-byte swizzle alignment");
    static_assert(!MX || SF_COL + SF_COLS * STAGES <= TMEM_COLS, "scale slots fit in TMEM");
    static_assert(!MX || PBN == 192 || (PBN == 256 && DIRECT),
                  "block-scaled tiles: 192 wide, or 256 wide with the direct epilogue (two B atoms per stage)");
};

// Pair tiles (256 rows x PBN columns): tiles [0, sk_first) whole and round-robin
// over the pairs; then, for stream-K, pair q < S takes the k-block iterations
// [I*q/S, I*(q+1)/S) of the remaining tiles (I = sk_iters, S = sk_pairs), cut
// at tile borders.
template <int PBN>
struct PairIter {
    int tile, step, rank, pair;
    long long it, it0, end;
    bool in_sk;
    const TcParams& p;

    __device__ PairIter(const TcParams& prm, int r) : rank(r), p(prm)
    {
        pair = blockIdx.x >> 1;
        step = gridDim.x >> 1;
        tile = pair;
        in_sk = false;
        if (pair < p.sk_pairs) {
            it0 = it = p.sk_iters * pair / p.sk_pairs;
            end = p.sk_iters * (pair + 1) / p.sk_pairs;
        } else {
            it0 = it = end = 0;
        }
    }

    __device__ bool next(Seg& s)
    {
        int t;
        if (!in_sk && tile < p.sk_first) {
            t = tile;
            tile += step;
            s.kb0 = 0;
            s.kb1 = p.num_kb;
            s.partial = false;
            s.sk_t = -1;
            s.slot = 0;
        } else {
            in_sk = true;
            if (it >= end)
                return false;
            const int tl = static_cast<int>(it / p.num_kb);
            s.kb0 = static_cast<int>(it - static_cast<long long>(tl) * p.num_kb);
            const long long k1 = s.kb0 + (end - it);
            s.kb1 = k1 < p.num_kb ? static_cast<int>(k1) : p.num_kb;
            s.slot = it == it0 ? 0 : 1;
            it += s.kb1 - s.kb0;
            t = p.sk_first + tl;
            s.partial = s.kb0 != 0 || s.kb1 != p.num_kb;
            s.sk_t = tl;
        }
        int tx, ty;
        decode_tile(p, t, s.b, tx, ty);
        s.x0 = tx * 2 * BM + rank * BM;
        s.xend = s.x0 + BM < p.rows_x ? s.x0 + BM : p.rows_x;
        s.y0 = ty * PBN;
        return true;
    }
};

// Workspace slice of one epilogue warp's portion of a stream-K piece (pair q,
// slot, CTA rank, warp ew): 4 chunks of 32 columns x 32 rows, column-major in
// each chunk, so that lane l's value of column k sits at k*32 + l and every
// store or load of one column is a single 128-byte line.
__device__ __forceinline__ float* sk_portion(const TcParams& p, int q, int slot, int rank, int ew)
{
    return p.ws + ((((static_cast<size_t>(q) * 2 + slot) * 2 + rank) * 8 + ew) * 4) * (32 * 32);
}

// Workspace slot of pair q's piece of stream-K tile t: 0 if t is the first tile
// of q's k range, else 1 (only the first and the last piece of a range can be
// partial).
__device__ __forceinline__ int sk_slot(const TcParams& p, int t, int q)
{
    const int first_tile = static_cast<int>((p.sk_iters * q / p.sk_pairs) / p.num_kb);
    return t == first_tile ? 0 : 1;
}

// Stream-K piece of one epilogue warp (its TMEM quadrant q, columns
// [c_begin, c_end)): store the slice to the workspace, release TMEM, count the
// arrival, and if this warp's portion of the tile is now complete in every
// piece, sum the pieces in k order and store Out.  Nothing here waits on other
// CTAs, so no co-residency is assumed; the sum order, and with it every bit of
// Out, does not depend on which piece arrives last.
template <int OT>
__device__ __forceinline__ void sk_epilogue(const TcParams& p, const Seg& s, uint32_t tacc, int q, int ew,
                                            int c_begin, int c_end, int lane, int rank, float* stage_buf,
                                            uint32_t tempty_leader)
{
    const int S = p.sk_pairs;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const uint32_t tbase = tacc + (static_cast<uint32_t>(q * 32) << 16);
    float* mine = sk_portion(p, pair, s.slot, rank, ew) + lane;
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
        uint32_t r[32];
        tmem_ld32_wait(tbase + static_cast<uint32_t>(c), r);
        float* dst = mine + ((c - c_begin) >> 5) * (32 * 32);
#pragma unroll
        for (int k = 0; k < 32; ++k)
            __stcg(dst + k * 32, __uint_as_float(r[k]));
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0)
        mbar_arrive_cluster(tempty_leader);  // TMEM is free for the next tile
    __threadfence();
    __syncwarp();
    uint32_t* counter = p.ws_flags + (static_cast<size_t>(s.sk_t) * 2 + rank) * 8 + ew;
    uint32_t old = 0;
    if (lane == 0)
        old = atomicAdd(counter, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    // the pairs whose ranges cover this tile: p_first .. p_last
    const long long I = p.sk_iters;
    const long long a = static_cast<long long>(s.sk_t) * p.num_kb, b = a + p.num_kb;
    const int p_first = static_cast<int>(((a + 1) * S - 1) / I);
    const int p_last = static_cast<int>((b * S - 1) / I);
    const int n = p_last - p_first + 1;
    if (static_cast<int>(old) != n - 1)
        return;
    __threadfence();
    if (lane == 0)
        *counter = 0;  // ready for the next launch
    typename OutStore<OT>::T* obase = static_cast<typename OutStore<OT>::T*>(p.out) + static_cast<int64_t>(s.b) * p.stride_o;
    const int x_row0 = s.x0 + q * 32;
    const int nx = s.xend - x_row0;
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
        if (nx <= 0 || s.y0 + c >= p.rows_y)
            break;
        const int chunk = (c - c_begin) >> 5;
        // acc = ((slice_0 + slice_1) + slice_2) + ...: two slices per round trip
        float acc[32];
#pragma unroll 1
        for (int j = 0; j < n; j += 2) {
            const float* src0 = sk_portion(p, p_first + j, sk_slot(p, s.sk_t, p_first + j), rank, ew) +
                                chunk * (32 * 32) + lane;
            const bool two = j + 1 < n;
            const float* src1 = two ? sk_portion(p, p_first + j + 1, sk_slot(p, s.sk_t, p_first + j + 1), rank, ew) +
                                          chunk * (32 * 32) + lane
                                    : src0;
            float v0[32], v1[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                v0[k] = __ldcg(src0 + k * 32);
                v1[k] = __ldcg(src1 + k * 32);
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float t = j == 0 ? v0[k] : acc[k] + v0[k];
                acc[k] = two ? t + v1[k] : t;
            }
        }
        store_rows_chunk<OT>(p, obase, x_row0, nx, s.y0 + c, acc, lane, stage_buf, false);
    }
}

// F8: 8-bit A and B (kind::f8f6f4, 128 elements of K per 128-byte stage row).
// Block-scaled kernels give warp 10 the copy of the scale atoms into TMEM.
template <int PBN, bool DIRECT, int KIND>
__global__ void __launch_bounds__(kPairThreads + 64, 1)
    tc05_pair_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                     const __grid_constant__ CUtensorMap tmsa, const __grid_constant__ CUtensorMap tmsb,
                     const TcParams p)
{
    using C = PairCfg<PBN, DIRECT, KIND>;
    constexpr bool F8 = KIND != 0;
    constexpr bool MX = C::MX;
    constexpr int kStages = C::STAGES;
    constexpr int KE = F8 ? 2 * BK : BK;  // elements of K per stage
    constexpr int kAccStride = C::ACC_STRIDE;
    constexpr int B_BYTES = C::B_BYTES;
    constexpr int STAGE_BYTES = C::STAGE_BYTES;
    constexpr int EPI_BYTES = C::EPI_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* as = smem;
    uint8_t* bs = smem + kStages * A_BYTES;
    // block-scaled 256-wide: data stage s's B atoms, four times over, at
    // sfb_rep + s * SFB_REP_BYTES as [row block h][copy q][512-byte atom]
    uint8_t* sfb_rep = smem + kStages * C::DATA_BYTES;
    // block-scaled: scale stage t holds A's atoms [t][k], then (192-wide) B's [t][rb][k]
    uint8_t* sfs = smem + kStages * STAGE_BYTES;
    float* epi = reinterpret_cast<float*>(sfs + C::SC_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sfs + C::SC_BYTES + EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = bars + 2 * kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint64_t* sc_full = drain + 2;  // leader: both CTAs' scale bytes of scale stage t
    uint64_t* sc_empty = sc_full + kScaleStages;  // each CTA: the copies that read stage t are done
    uint64_t* sf_ready = sc_empty + kScaleStages;  // leader: data stage s's scales are in TMEM
    uint64_t* cdrain = sf_ready + kStages;         // leader: the copier's last copies are done

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), kTemptyArrivals);
        }
        mbar_init(smem_u32(drain), 1);
        for (int t = 0; t < kScaleStages; ++t) {
            mbar_init(smem_u32(&sc_full[t]), 1);
            mbar_init(smem_u32(&sc_empty[t]), 1);
        }
        for (int st = 0; st < kStages; ++st)
            mbar_init(smem_u32(&sf_ready[st]), 1);
        mbar_init(smem_u32(cdrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tma);
        tma_prefetch_map(&tmb);
        if (MX) {
            tma_prefetch_map(&tmsa);
            tma_prefetch_map(&tmsb);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair<TMEM_COLS>(smem_u32(tmem_slot));
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        // warm L2 with this CTA's first ring of tiles while earlier grids finish
        PairIter<PBN> w0(p, static_cast<int>(rank));
        Seg s0;
        if (w0.next(s0)) {
            const int n = s0.kb1 - s0.kb0 < kStages ? s0.kb1 - s0.kb0 : kStages;
            const int yb = s0.y0 + static_cast<int>(rank) * (PBN / 2);
            for (int i = 0; i < n; ++i) {
                prefetch_operand<BM>(&tma, p.x_mn, (s0.kb0 + i) * KE, s0.x0, s0.b * p.x_bmul);
                prefetch_operand<PBN / 2>(&tmb, p.y_mn, (s0.kb0 + i) * KE, yb, s0.b * p.y_bmul);
            }
        }
    }
    pdl_wait();  // global memory only after the preceding grids are done

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;
            // both CTAs' loads of a stage, as credited (packed elements: global
            // bytes), with (256-wide block-scaled) the replicated B atoms
            const uint32_t data_tx = 2 * C::DATA_BYTES * (p.ab_packed_bits ? p.ab_packed_bits : 8) / 8 +
                                     (C::SINGLE ? 2u * 4u * 512u * static_cast<uint32_t>(p.sf_box_rb) : 0u);
            int sst = 0;  // scale stage ring
            uint32_t sphase = 0, sc_filled = 0, sc_parity = 0;
            bool first = true, ok = true;
            PairIter<PBN> w(p, static_cast<int>(rank));
            Seg s;
            while (ok && w.next(s)) {
                const int yb = s.y0 + static_cast<int>(rank) * (PBN / 2);
                // first scale row block of the tile's A rows and of its B rows
                const int rbx = MX ? static_cast<int>((s.b * p.sf_x_bstride) / (512LL * p.num_kb)) + s.x0 / BM : 0;
                const int rby = MX ? static_cast<int>((s.b * p.sf_y_bstride) / (512LL * p.num_kb)) + s.y0 / BM : 0;
                for (int kb = s.kb0; kb < s.kb1; ++kb) {
                    if (MX && (kb == s.kb0 || kb % kScaleKb == 0)) {
                        // the next scale stage: atoms of k-blocks [kb - kb % 8, +8)
                        if (!wait_bounded(smem_u32(&sc_empty[sst]), sphase ^ 1, abort_flag, p.wait_limit)) {
                            raise_timeout(p, abort_flag);
                            ok = false;
                            break;
                        }
                        const uint32_t sb_local = smem_u32(&sc_full[sst]);
                        if (leader) {
                            // both CTAs' boxes: A's p.sf_box_kg atoms, (192-wide) B's p.sf_box_rb times as many
                            mbar_arrive_expect_tx(sb_local, 2 * 512 * p.sf_box_kg * (1 + (C::SINGLE ? 0 : p.sf_box_rb)));
                            sc_filled |= 1u << sst;
                            sc_parity = (sc_parity & ~(1u << sst)) | (sphase << sst);
                        }
                        const uint32_t sb_leader = mapa_shared(sb_local, 0);
                        const uint32_t sd = smem_u32(sfs + sst * C::SC_STAGE_BYTES);
                        const int kg0 = kb - kb % kScaleKb;
                        tma_load_4d_pair(sd, &tmsa, sb_leader, 0, 0, kg0, rbx);
                        if (!C::SINGLE)
                            tma_load_4d_pair(sd + kScaleKb * 512, &tmsb, sb_leader, 0, 0, kg0, rby);
                        if (++sst == kScaleStages) {
                            sst = 0;
                            sphase ^= 1;
                        }
                    }
                    if (!wait_bounded(smem_u32(&empty[stage]), phase ^ 1, abort_flag, p.wait_limit)) {
                        raise_timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    const bool drop = p.fault == 1 && blockIdx.x == 0 && first;
                    first = false;
                    if (!drop) {
                        const uint32_t fb_local = smem_u32(&full[stage]);
                        const uint32_t fb_leader = mapa_shared(fb_local, 0);
                        if (leader) {
                            mbar_arrive_expect_tx(fb_local, data_tx);
                            filled |= 1u << stage;
                            fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                        }
                        load_operand<BM, true>(smem_u32(as + stage * A_BYTES), &tma, fb_leader, p.x_mn, kb * KE,
                                               s.x0, s.b * p.x_bmul);
                        load_operand<PBN / 2, true>(smem_u32(bs + stage * B_BYTES), &tmb, fb_leader, p.y_mn,
                                                    kb * KE, yb, s.b * p.y_bmul);
                        if constexpr (C::SINGLE)
                            tma_load_5d_pair(smem_u32(sfb_rep + stage * C::SFB_REP_BYTES), &tmsb, fb_leader, 0, 0, 0,
                                             kb, rby);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // The leader's full barriers count both CTAs' bytes: waiting for the
            // last fills lets every load of the pair land before either exits.
            for (int st = 0; st < kScaleStages; ++st) {
                if (sc_filled & (1u << st)) {
                    const uint32_t par = (sc_parity >> st) & 1u;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(smem_u32(&sc_full[st]), par) &&
                           static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
                    }
                }
            }
            for (int st = 0; st < kStages; ++st) {
                if (filled & (1u << st)) {
                    const uint32_t par = (fill_parity >> st) & 1u;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(smem_u32(&full[st]), par) &&
                           static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && leader) {
            // The tensor core accepts about one MMA beyond the one it is
            // executing, and an MMA issue blocks until accepted, so whatever this
            // thread does between one k-block's last MMA and the next k-block's
            // first must fit in one MMA's time (~128 cycles at N = 256).  The
            // loop therefore steps stage addresses and descriptor words by
            // additions, and leaves the line only when a wait has to sleep.
            const uint32_t idesc = (MX ? idesc_mx(2 * BM, PBN) : C::IDESC) | p.idesc_bits;
            const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
            const DescWords da = desc_words(smem_u32(as), p.x_mn != 0);
            const DescWords db = desc_words(smem_u32(bs), p.y_mn != 0);
            uint32_t fa = full0, ea = empty0, alo = da.lo, blo = db.lo;
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool skip_release = p.fault == 2 && blockIdx.x == 0;  // test hook: lose one stage release
            bool ok = true;
            PairIter<PBN> w(p, 0);
            Seg s;
            while (ok && w.next(s)) {
                const int buf = C::SINGLE ? 0 : (local & 1);
                const uint32_t use = static_cast<uint32_t>(C::SINGLE ? local : (local >> 1));
                if (!wait_bounded(smem_u32(&tempty[buf]), (use & 1) ^ 1, abort_flag, p.wait_limit)) {
                    raise_timeout(p, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kAccStride);
                const uint32_t y_sf_off = static_cast<uint32_t>((s.y0 % BM) / 32);
                for (int kb = s.kb0; kb < s.kb1; ++kb) {
                    if (!wait_bounded(fa, phase, abort_flag, p.wait_limit)) {
                        raise_timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if constexpr (MX) {
                        // the copier has put this stage's scales into its TMEM slot
                        if (!wait_bounded(smem_u32(&sf_ready[stage]), phase, abort_flag, p.wait_limit)) {
                            raise_timeout(p, abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sft = tmem_base + static_cast<uint32_t>(C::SF_COL + C::SF_COLS * stage);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            tc_mma_pair_mx(d_tmem, alo + k * da.kstep, da.hi, blo + k * db.kstep, db.hi,
                                           idesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4),
                                           sft, sft + 4 + y_sf_off, (k > 0 || kb != s.kb0) ? 1u : 0u);
                    } else {
                        tc_mma_pair_w<F8>(d_tmem, alo, da.hi, blo, db.hi, idesc, kb != s.kb0);
#pragma unroll
                        for (int k = 1; k < BK / 16; ++k)
                            tc_mma_pair_w<F8>(d_tmem, alo + k * da.kstep, da.hi, blo + k * db.kstep, db.hi, idesc,
                                              1u);
                    }
                    if (!skip_release)
                        tc_commit_pair_mc(ea, 0x3);
                    skip_release = false;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                        fa = full0;
                        ea = empty0;
                        alo = da.lo;
                        blo = db.lo;
                    } else {
                        fa += 8;
                        ea += 8;
                        alo += A_BYTES >> 4;
                        blo += B_BYTES >> 4;
                    }
                }
                if (!ok)
                    break;
                tc_commit_pair_mc(smem_u32(&tfull[buf]), 0x3);
                ++local;
            }
            tc_commit_pair(smem_u32(drain));
            const long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(drain), 0) &&
                   static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
            }
        }
    } else if (warp >= 10) {
        // ------------------------------------------------------------ scale copier (leader, block-scaled)
        // Copies each data stage's scale atoms from the scale ring into the
        // stage's TMEM slot (tcgen05.cp.cta_group::2: each CTA's atoms into its
        // own TMEM) and signals sf_ready[stage] when the copies are done, so the
        // MMA thread issues nothing but MMAs.  The slot is rewritten only after
        // the stage's new data has landed, which follows the release of its
        // previous MMAs.
        if (MX && lane == 0 && leader) {
            const uint32_t sf_smem0 = smem_u32(sfs);
            int stage = 0, sst = 0;
            uint32_t phase = 0, sphase = 0, sc_cur = 0;
            bool issued = false;
            PairIter<PBN> w(p, 0);
            Seg s;
            bool ok = true;
            while (ok && w.next(s)) {
                for (int kb = s.kb0; kb < s.kb1; ++kb) {
                    if (!wait_bounded(smem_u32(&full[stage]), phase, abort_flag, p.wait_limit)) {
                        raise_timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    if (kb == s.kb0 || kb % kScaleKb == 0) {
                        if (!wait_bounded(smem_u32(&sc_full[sst]), sphase, abort_flag, p.wait_limit)) {
                            raise_timeout(p, abort_flag);
                            ok = false;
                            break;
                        }
                        sc_cur = sf_smem0 + static_cast<uint32_t>(sst * C::SC_STAGE_BYTES);
                    }
                    tc_fence_after();
                    const uint32_t sft = tmem_base + static_cast<uint32_t>(C::SF_COL + C::SF_COLS * stage);
                    const uint32_t j = static_cast<uint32_t>(kb % kScaleKb);
                    tc_cp_atom_pair(sft, atom_desc(sc_cur + j * 512));
                    if constexpr (C::SINGLE) {
                        // both B atoms from the data stage, each four times over: one copy
                        tc_cp_rows32_pair(sft + 4, rows32_desc(smem_u32(sfb_rep + stage * C::SFB_REP_BYTES), 4 * 512));
                    } else {
                        // B's box: row block a, K block group j at (a * box_kg + j); a B
                        // row block past the tensor (box of one) holds only rows past N
#pragma unroll
                        for (int a = 0; a < kSfAtomsB; ++a)
                            tc_cp_atom_pair(sft + 4 + 4 * a,
                                            atom_desc(sc_cur + (kScaleKb + a * p.sf_box_kg + j) * 512));
                    }
                    tc_commit_pair(smem_u32(&sf_ready[stage]));
                    issued = true;
                    if (kb % kScaleKb == kScaleKb - 1 || kb == s.kb1 - 1) {
                        // the scale stage's last copies: release it in both CTAs
                        tc_commit_pair_mc(smem_u32(&sc_empty[sst]), 0x3);
                        if (++sst == kScaleStages) {
                            sst = 0;
                            sphase ^= 1;
                        }
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (issued) {
                // no copy may still be running when TMEM is released
                tc_commit_pair(smem_u32(cdrain));
                const long long t0 = clock64();
                while (!mbar_try_wait(smem_u32(cdrain), 0) &&
                       static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int ew = warp - 2;
        const int q = warp & 3;
        const int c_begin = (ew >> 2) ? C::SPLIT : 0;
        const int c_end = (ew >> 2) ? PBN : C::SPLIT;
        float* stage_buf = epi + ew * 32 * 32;
        int local = 0;
        PairIter<PBN> w(p, static_cast<int>(rank));
        Seg s;
        while (w.next(s)) {
            const int buf = C::SINGLE ? 0 : (local & 1);
            const uint32_t use = static_cast<uint32_t>(C::SINGLE ? local : (local >> 1));
            if (!wait_bounded(smem_u32(&tfull[buf]), use & 1, abort_flag, p.wait_limit)) {
                raise_timeout(p, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[buf]), 0);
            const uint32_t tacc = tmem_base + static_cast<uint32_t>(buf * kAccStride);
            if constexpr (C::SINGLE) {
                // the warp's 128 columns into registers, the accumulator freed, then the stores
                uint32_t v[2 * (PBN / 2 / 32)][16];
                epilogue_load_direct<PBN / 2 / 32>(tacc, q, c_begin, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(tempty_leader);
                if (p.out_type == kOutF16)
                    epilogue_store_direct_regs<kOutF16, PBN / 2 / 32>(p, s, q, c_begin, lane, v);
                else if (p.out_type == kOutBF16)
                    epilogue_store_direct_regs<kOutBF16, PBN / 2 / 32>(p, s, q, c_begin, lane, v);
                else
                    epilogue_store_direct_regs<kOutF32, PBN / 2 / 32>(p, s, q, c_begin, lane, v);
            } else if (!DIRECT && s.partial) {
                // the host splits only products with fp32 Out
                sk_epilogue<kOutF32>(p, s, tacc, q, ew, c_begin, c_end, lane, static_cast<int>(rank), stage_buf,
                                     tempty_leader);
            } else {
                if (DIRECT) {
                    if (p.out_type == kOutF16)
                        epilogue_store_direct<kOutF16>(p, s, tacc, q, c_begin, c_end, lane);
                    else if (p.out_type == kOutBF16)
                        epilogue_store_direct<kOutBF16>(p, s, tacc, q, c_begin, c_end, lane);
                    else
                        epilogue_store_direct<kOutF32>(p, s, tacc, q, c_begin, c_end, lane);
                } else {
                    if (p.out_type == kOutF16)
                        epilogue_store<false, kOutF16>(p, s, tacc, q, c_begin, c_end, lane, stage_buf);
                    else if (p.out_type == kOutBF16)
                        epilogue_store<false, kOutBF16>(p, s, tacc, q, c_begin, c_end, lane, stage_buf);
                    else
                        epilogue_store<false, kOutF32>(p, s, tacc, q, c_begin, c_end, lane, stage_buf);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(tempty_leader);
            }
            ++local;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair<TMEM_COLS>(tmem_base);
    }
}

cudaLaunchConfig_t pair_config(int grid, int smem, cudaStream_t stream, cudaLaunchAttribute* attr, int threads)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

template <int PBN, bool DIRECT, int KIND>
cudaError_t configure_kind(int* max_pairs)
{
    using C = PairCfg<PBN, DIRECT, KIND>;
    cudaError_t e = cudaFuncSetAttribute(tc05_pair_kernel<PBN, DIRECT, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(2, C::SMEM, nullptr, attr, kPairThreads + 32);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, tc05_pair_kernel<PBN, DIRECT, KIND>, &cfg);
    if (e != cudaSuccess)
        return e;
    *max_pairs = std::min(*max_pairs, n);
    return cudaSuccess;
}

template <int PBN, bool DIRECT>
cudaError_t configure_one(int* max_pairs)
{
    cudaError_t e = configure_kind<PBN, DIRECT, 0>(max_pairs);
    return e == cudaSuccess ? configure_kind<PBN, DIRECT, 1>(max_pairs) : e;
}

template <int PBN, bool DIRECT, int KIND>
cudaError_t launch_kind(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmsa,
                        const CUtensorMap& tmsb, const TcParams& p, int pairs, cudaStream_t stream)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(2 * pairs, PairCfg<PBN, DIRECT, KIND>::SMEM, stream, attr,
                                         kPairThreads + 32);
    return cudaLaunchKernelEx(&cfg, tc05_pair_kernel<PBN, DIRECT, KIND>, tma, tmb, tmsa, tmsb, p);
}

template <int PBN, bool DIRECT>
cudaError_t launch_one(const CUtensorMap& tma, const CUtensorMap& tmb, const TcParams& p, int pairs, int kind,
                       cudaStream_t stream)
{
    // the scale maps are not read unless kind is 2
    if (kind == 1)
        return launch_kind<PBN, DIRECT, 1>(tma, tmb, tma, tmb, p, pairs, stream);
    return launch_kind<PBN, DIRECT, 0>(tma, tmb, tma, tmb, p, pairs, stream);
}

}  // namespace

cudaError_t tc05_pair_configure(int* max_pairs)
{
    int n = 1 << 30;
    cudaError_t e = configure_one<256, false>(&n);
    if (e == cudaSuccess) e = configure_one<224, false>(&n);
    if (e == cudaSuccess) e = configure_one<192, false>(&n);
    if (e == cudaSuccess) e = configure_one<256, true>(&n);
    if (e == cudaSuccess) e = configure_one<224, true>(&n);
    if (e == cudaSuccess) e = configure_one<192, true>(&n);
    if (e == cudaSuccess) e = configure_kind<192, true, 2>(&n);
    if (e == cudaSuccess) e = configure_kind<256, true, 2>(&n);
    if (e == cudaSuccess) e = configure_kind<192, false, 2>(&n);
    if (e != cudaSuccess)
        return e;
    *max_pairs = n;
    return cudaSuccess;
}

cudaError_t tc05_pair_launch(const CUtensorMap& tma, const CUtensorMap& tmb, const TcParams& p, int pairs, int pbn,
                             bool direct, int kind, cudaStream_t stream, const CUtensorMap* tmsa,
                             const CUtensorMap* tmsb)
{
    if (kind == 2) {
        // block-scaled: two 192-wide accumulators, or one 256-wide (direct
        // epilogue only), leave TMEM room for the scale slots
        if ((pbn != 192 && pbn != 256) || (pbn == 256 && !direct) || !tmsa || !tmsb)
            return cudaErrorInvalidValue;
        if (pbn == 256)
            return launch_kind<256, true, 2>(tma, tmb, *tmsa, *tmsb, p, pairs, stream);
        if (direct)
            return launch_kind<192, true, 2>(tma, tmb, *tmsa, *tmsb, p, pairs, stream);
        return launch_kind<192, false, 2>(tma, tmb, *tmsa, *tmsb, p, pairs, stream);
    }
    if (direct) {
        switch (pbn) {
        case 256: return launch_one<256, true>(tma, tmb, p, pairs, kind, stream);
        case 224: return launch_one<224, true>(tma, tmb, p, pairs, kind, stream);
        case 192: return launch_one<192, true>(tma, tmb, p, pairs, kind, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (pbn) {
    case 256: return launch_one<256, false>(tma, tmb, p, pairs, kind, stream);
    case 224: return launch_one<224, false>(tma, tmb, p, pairs, kind, stream);
    case 192: return launch_one<192, false>(tma, tmb, p, pairs, kind, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gnt
