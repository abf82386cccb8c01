// tc05_kernel.cuh -- persistent, warp-specialised tcgen05 kernel for Out = A @ B.T
// (16-, 8-, 6- or 4-bit inputs, fp32 accumulation in Tensor Memory, fp32, fp16
// or bf16 output).
//
// The single-CTA example of "Blackwell Tensor Cores" ("The Accumulator's
// Lifetime") allocates TMEM with warp 0, stages A/B in 128-byte-swizzled shared
// memory (swizzle mode 3, 1024-byte period), lets one thread issue four
// tcgen05.mma kind::f16 of shape 128x64x16 (accumulate off for the first K
// slice), commits them to an mbarrier, waits for phase 0, fences, reads the
// accumulator with tcgen05.ld 32x32b (warp w <-> TMEM lanes 32w..32w+31, one row
// per thread) and releases TMEM after a final barrier.  This kernel keeps those
// steps and turns them into a pipeline that streams K and loops over tiles:
//
//   warp 0      TMA producer: one thread waits for a free stage, posts the
//               expected byte count and issues two 3-D tensor loads (X and Y
//               tiles, 64 fp16 of K each, 128-byte swizzle) into the stage ring.
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one thread
//               issues 4 MMAs 128xBNx16 per stage, committing each stage back to
//               the producer and each finished tile to the epilogue.
//   warps 2-9   epilogue, two warpgroups: TMEM -> registers (32x32b.x32) ->
//               global, overlapped with the next tile's MMAs through the
//               second accumulator.  Each warp owns one TMEM lane quadrant
//               (32 rows) and half of the tile's columns.
//
// Every mbarrier wait is bounded (wait_limit cycles); on expiry the kernel sets
// the device status word and an abort flag, all roles leave their loops, loads
// still in flight are waited for, TMEM is freed and the kernel returns.
#pragma once
#include "ptx_mx.cuh"
#include "tc05_common.cuh"

namespace gnt {

namespace {

using namespace tc;

constexpr int kThreads = 320;  // producer warp, MMA warp, 8 epilogue warps
// block-scaled kernels add warp 10, which copies the scale atoms into TMEM
constexpr int threads_of(int kind) { return kind == 2 ? kThreads + 32 : kThreads; }

// XR: rows of X staged per stage.  128 normally; 112 for the row split of the
// swapped path (shares of at most 112 rows), which packs 10 stages instead of
// 9.  The MMA still reads 128 rows: rows XR..127 come from the next slot and
// only feed accumulator rows that are never stored.
// KIND: 0 16-bit inputs (kind::f16), 1 8-bit inputs (kind::f8f6f4), 2 8-bit
// inputs with block scales (kind::mxf8f6f4).  Block-scaled, the scale atoms
// (512 bytes per 128 rows and 128 elements of K) come through a ring of two
// scale stages of their own, each holding the atoms of kScaleKb consecutive
// k-blocks of X and of Y -- contiguous in the packed layout, so two bulk
// copies per 8 k-blocks instead of two per k-block.  TMEM holds, after the two
// accumulators, 8 columns of scales per data stage (X atom, then Y atom), which
// warp 10 fills with tcgen05.cp once the stage's data has landed (which follows
// the release of the stage's previous MMAs) and signals per data stage, so
// the MMA thread issues nothing but MMAs.
constexpr int kKind16 = 0, kKind8 = 1, kKindMx = 2;
constexpr int kScaleKb = 8;      // k-blocks of scale atoms per scale stage
constexpr int kScaleStages = 2;

constexpr int pow2_at_least(int v)
{
    int r = 32;
    while (r < v)
        r *= 2;
    return r;
}

// TM, WS: other instruction shapes (non-swapped, unscaled only).  TM = 64 with
// WS false issues the plain M = 64 MMA, whose accumulator rows 16q..16q+15
// sit in TMEM lanes 32q..32q+15, all BN columns.  WS true issues the
// weight-stationary form (tcgen05.mma.ws) with M = TM: its accumulator is
// spread over all 128 lanes in BN*TM/128 columns -- for TM = 64 lane quadrants
// 0-1 hold rows 0..63 of columns [0, BN/2) and quadrants 2-3 the same rows of
// [BN/2, BN); for TM = 32 quadrant q holds rows 0..31 of columns
// [q*BN/4, (q+1)*BN/4).  X tiles are TM rows (XR = TM).
template <int BN, bool SWAP, int XR = 128, int KIND = kKind16, int TM = 128, bool WS = false>
struct Cfg {
    static constexpr int X_BYTES = XR * BK * 2;
    static constexpr int Y_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = X_BYTES + Y_BYTES;
    // block-scaled: scale stage t holds X's atoms [t][j], then Y's, j < kScaleKb
    static constexpr int SC_STAGE_BYTES = 2 * kScaleKb * 512;
    static constexpr int SC_BYTES = KIND == kKindMx ? kScaleStages * SC_STAGE_BYTES : 0;
    static constexpr int EPI_BYTES = SWAP ? 0 : 8 * 32 * 32 * 4;  // per-warp 32x32 fp32 staging
    static constexpr int BAR_BYTES = 384;
    static constexpr int BASE_STAGES =
        TM < 128 ? 8 : (BN >= 256 ? 4 : (BN >= 128 ? 6 : (SWAP ? (XR <= 112 ? 10 : 9) : 8)));
    static constexpr int FIT_STAGES = (232448 - 1024 - SC_BYTES - EPI_BYTES - BAR_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = BASE_STAGES < FIT_STAGES ? BASE_STAGES : FIT_STAGES;
    static constexpr int ACC_COLS = WS ? BN * TM / 128 : BN;  // TMEM columns of one accumulator
    static constexpr int SF_COL = 2 * ACC_COLS;               // first TMEM column of the scale slots
    static constexpr int TMEM_COLS = pow2_at_least(2 * ACC_COLS + (KIND == kKindMx ? 8 * STAGES : 0));
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + SC_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr uint32_t IDESC = idesc_f16_f32(TM, BN);
    static_assert(TM == 128 || (!SWAP && KIND != kKindMx && XR == TM), "small tiles: plain operands, X = A");
    static_assert(WS ? (TM == 32 || TM == 64 || TM == 128) && (BN == 64 || BN == 128 || BN == 256)
                     : (TM == 64 || TM == 128), "instruction shapes");
    static_assert(ACC_COLS % 64 == 0, "each epilogue warp takes whole 32-column chunks");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert((3 * STAGES + 5 + 2 * kScaleStages + 1) * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(X_BYTES % 1024 == 0, "stage slots keep the 1024-byte swizzle alignment");
    static_assert(TMEM_COLS <= 512, "Tensor Memory columns");
};

// 8-bit A and B (KIND 1, 2): a stage slot holds 128 elements of K in the same
// 128 bytes per row.
template <int BN, bool SWAP, int XR, int KIND, int TM = 128, bool WS = false>
__global__ void __launch_bounds__(threads_of(KIND), 1)
    tc05_gemm_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                     const TcParams p)
{
    using C = Cfg<BN, SWAP, XR, KIND, TM, WS>;
    constexpr bool F8 = KIND != kKind16;
    constexpr bool MX = KIND == kKindMx;
    constexpr int STAGES = C::STAGES;
    constexpr int KE = F8 ? 2 * BK : BK;  // elements of K per stage

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* xs = smem;
    uint8_t* ys = smem + STAGES * C::X_BYTES;
    uint8_t* sfs = ys + STAGES * C::Y_BYTES;  // MX: the scale stages
    float* epi = reinterpret_cast<float*>(sfs + C::SC_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sfs + C::SC_BYTES + C::EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint64_t* sc_full = drain + 2;                 // MX: scale stage t has landed
    uint64_t* sc_empty = sc_full + kScaleStages;   // MX: the copies that read scale stage t are done
    uint64_t* sf_ready = sc_empty + kScaleStages;  // MX: data stage s's scales are in TMEM
    uint64_t* cdrain = sf_ready + STAGES;          // MX: the copier's last copies are done

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), 256);
        }
        mbar_init(smem_u32(drain), 1);
        for (int t = 0; t < kScaleStages; ++t) {
            mbar_init(smem_u32(&sc_full[t]), 1);
            mbar_init(smem_u32(&sc_empty[t]), 1);
        }
        if (MX) {
            for (int st = 0; st < STAGES; ++st)
                mbar_init(smem_u32(&sf_ready[st]), 1);
            mbar_init(smem_u32(cdrain), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tmx);
        tma_prefetch_map(&tmy);
    }
    if (warp == 1) {
        tmem_alloc<C::TMEM_COLS>(smem_u32(tmem_slot));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touched only this CTA's shared memory and TMEM; global
    // memory is read and written only after the preceding grids are done.
    // Meanwhile the producer warms L2 with the first ring's worth of tiles.
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        WorkIter<BN, TM> w0(p);
        Seg s0;
        if (w0.next(s0)) {
            const int n = s0.kb1 - s0.kb0 < STAGES ? s0.kb1 - s0.kb0 : STAGES;
            for (int i = 0; i < n; ++i) {
                prefetch_operand<XR>(&tmx, p.x_mn, (s0.kb0 + i) * KE, s0.x0, s0.b * p.x_bmul);
                prefetch_operand<BN>(&tmy, p.y_mn, (s0.kb0 + i) * KE, s0.y0, s0.b * p.y_bmul);
            }
        }
    }
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0;       // bit s: stage s has a load this thread issued
            uint32_t fill_parity = 0;  // bit s: parity of that fill
            // bytes the two data loads credit: packed 6- and 4-bit elements count
            // their global bytes, width / 8 of the shared ones
            const uint32_t data_tx = (p.x_box_bytes + C::Y_BYTES) * (p.ab_packed_bits ? p.ab_packed_bits : 8) / 8;
            int sst = 0;  // MX: scale stage ring
            uint32_t sphase = 0, sc_filled = 0, sc_parity = 0;
            // Swapped operands (few rows of A): X = B is streamed once, every CTA
            // re-reads all of Y = A.  Marking B evict_first and A evict_last keeps
            // A in L2 under the stream (8-bit skinny products 8 % faster, 16-bit 2 %).
            const bool hints = SWAP && !p.x_mn && !p.y_mn;
            const uint64_t pol_x = l2_policy_evict_first(), pol_y = l2_policy_evict_last();
            bool first = true, ok = true;
            WorkIter<BN, TM> w(p);
            Seg s;
            while (ok && w.next(s)) {
                for (int kb = s.kb0; kb < s.kb1; ++kb) {
                    if (MX && (kb == s.kb0 || kb % kScaleKb == 0)) {
                        // the next scale stage: atoms of k-blocks [kb, kg0 + 8) of the
                        // row blocks of x0 and y0, contiguous in the packed layout
                        if (!wait_bounded(smem_u32(&sc_empty[sst]), sphase ^ 1, abort_flag, p.wait_limit)) {
                            raise_timeout(p, abort_flag);
                            ok = false;
                            break;
                        }
                        const int kg0 = kb - kb % kScaleKb;
                        const int n = p.num_kb - kg0 < kScaleKb ? p.num_kb - kg0 : kScaleKb;
                        const uint32_t sb = smem_u32(&sc_full[sst]);
                        const uint32_t sd = smem_u32(sfs + sst * C::SC_STAGE_BYTES);
                        mbar_arrive_expect_tx(sb, static_cast<uint32_t>(2 * 512 * n));
                        bulk_load(sd, p.sf_x + s.b * p.sf_x_bstride + (static_cast<int64_t>(s.x0 / BM) * p.num_kb + kg0) * 512,
                                  static_cast<uint32_t>(512 * n), sb);
                        bulk_load(sd + kScaleKb * 512,
                                  p.sf_y + s.b * p.sf_y_bstride + (static_cast<int64_t>(s.y0 / BM) * p.num_kb + kg0) * 512,
                                  static_cast<uint32_t>(512 * n), sb);
                        sc_filled |= 1u << sst;
                        sc_parity = (sc_parity & ~(1u << sst)) | (sphase << sst);
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
                        const uint32_t fb = smem_u32(&full[stage]);
                        mbar_arrive_expect_tx(fb, data_tx);
                        if (hints) {
                            tma_load_3d_hint(smem_u32(xs + stage * C::X_BYTES), &tmx, fb, kb * KE, s.x0,
                                             s.b * p.x_bmul, pol_x);
                            tma_load_3d_hint(smem_u32(ys + stage * C::Y_BYTES), &tmy, fb, kb * KE, s.y0,
                                             s.b * p.y_bmul, pol_y);
                        } else {
                            load_operand<XR>(smem_u32(xs + stage * C::X_BYTES), &tmx, fb, p.x_mn, kb * KE, s.x0,
                                             s.b * p.x_bmul);
                            load_operand<BN>(smem_u32(ys + stage * C::Y_BYTES), &tmy, fb, p.y_mn, kb * KE, s.y0,
                                             s.b * p.y_bmul);
                        }
                        filled |= 1u << stage;
                        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // Let every load this thread issued land before the CTA can exit.
            for (int st = 0; st < kScaleStages; ++st) {
                if (sc_filled & (1u << st)) {
                    const uint32_t par = (sc_parity >> st) & 1u;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(smem_u32(&sc_full[st]), par) &&
                           static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
                    }
                }
            }
            for (int st = 0; st < STAGES; ++st) {
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
        // ------------------------------------------------------------ MMA issuer
        // An MMA issue blocks until the tensor core accepts it, about one MMA
        // ahead of the one executing, so the work between k-blocks is kept to
        // additions (stage addresses, descriptor words) and the waits' fast path.
        if (lane == 0) {
            const uint32_t idesc = (MX ? idesc_mx(BM, BN) : C::IDESC) | p.idesc_bits;
            const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
            const DescWords dx = desc_words(smem_u32(xs), p.x_mn != 0);
            const DescWords dy = desc_words(smem_u32(ys), p.y_mn != 0);
            uint32_t fa = full0, ea = empty0, xlo = dx.lo, ylo = dy.lo;
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool skip_release = p.fault == 2 && blockIdx.x == 0;  // test hook: lose one stage release
            bool ok = true;
            WorkIter<BN, TM> w(p);
            Seg s;
            while (ok && w.next(s)) {
                const int buf = local & 1;
                const uint32_t use = static_cast<uint32_t>(local >> 1);
                if (!wait_bounded(smem_u32(&tempty[buf]), (use & 1) ^ 1, abort_flag, p.wait_limit)) {
                    raise_timeout(p, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS);
                // MX: a Y tile that starts half-way into its 128-row atom reads
                // the atom's upper columns
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
                        const uint32_t sft = tmem_base + static_cast<uint32_t>(C::SF_COL + 8 * stage);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            tc_mma_mx(d_tmem, xlo + k * dx.kstep, dx.hi, ylo + k * dy.kstep, dy.hi,
                                      idesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4), sft,
                                      sft + 4 + y_sf_off, (k > 0 || kb != s.kb0) ? 1u : 0u);
                    } else if constexpr (WS) {
                        tc_mma_ws<F8>(d_tmem, xlo, dx.hi, ylo, dy.hi, idesc, kb != s.kb0);
#pragma unroll
                        for (int k = 1; k < BK / 16; ++k)
                            tc_mma_ws<F8>(d_tmem, xlo + k * dx.kstep, dx.hi, ylo + k * dy.kstep, dy.hi, idesc, 1u);
                    } else {
                        tc_mma_w<F8>(d_tmem, xlo, dx.hi, ylo, dy.hi, idesc, kb != s.kb0);
#pragma unroll
                        for (int k = 1; k < BK / 16; ++k)
                            tc_mma_w<F8>(d_tmem, xlo + k * dx.kstep, dx.hi, ylo + k * dy.kstep, dy.hi, idesc, 1u);
                    }
                    if (!skip_release)
                        tc_commit(ea);
                    skip_release = false;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                        fa = full0;
                        ea = empty0;
                        xlo = dx.lo;
                        ylo = dy.lo;
                    } else {
                        fa += 8;
                        ea += 8;
                        xlo += C::X_BYTES >> 4;
                        ylo += C::Y_BYTES >> 4;
                    }
                }
                if (!ok)
                    break;
                tc_commit(smem_u32(&tfull[buf]));
                ++local;
            }
            // No MMA may still be running when TMEM is released.
            tc_commit(smem_u32(drain));
            const long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(drain), 0) &&
                   static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
            }
        }
    } else if (warp >= 10) {
        // ------------------------------------------------------------ scale copier (block-scaled)
        // Copies each data stage's two scale atoms from the scale ring into the
        // stage's TMEM slot and signals sf_ready[stage] when the copies are done.
        // A stage's data lands only after its previous MMAs released it, so
        // waiting for the data also frees the slot.
        if (MX && lane == 0) {
            const uint32_t sf_smem0 = smem_u32(sfs);
            int stage = 0, sst = 0;
            uint32_t phase = 0, sphase = 0, sc_cur = 0;
            bool issued = false, ok = true;
            WorkIter<BN, TM> w(p);
            Seg s;
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
                    const uint32_t sft = tmem_base + static_cast<uint32_t>(C::SF_COL + 8 * stage);
                    const uint32_t j = static_cast<uint32_t>(kb % kScaleKb);
                    tc_cp_atom(sft, atom_desc(sc_cur + j * 512));
                    tc_cp_atom(sft + 4, atom_desc(sc_cur + (kScaleKb + j) * 512));
                    tc_commit(smem_u32(&sf_ready[stage]));
                    issued = true;
                    if (kb % kScaleKb == kScaleKb - 1 || kb == s.kb1 - 1) {
                        // the scale stage's last copies: free it once they are done
                        tc_commit(smem_u32(&sc_empty[sst]));
                        if (++sst == kScaleStages) {
                            sst = 0;
                            sphase ^= 1;
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (issued) {
                // no copy may still be running when TMEM is released
                tc_commit(smem_u32(cdrain));
                const long long t0 = clock64();
                while (!mbar_try_wait(smem_u32(cdrain), 0) &&
                       static_cast<unsigned long long>(clock64() - t0) <= p.wait_limit) {
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Eight warps: warp w reads TMEM lanes 32*(w%4).. (the only quadrant it
        // may access) and half of the tile's columns.
        const int ew = warp - 2;
        const int q = warp & 3;
        const int c_begin = (ew >> 2) * (C::ACC_COLS / 2);
        // this quadrant's tile rows and the tile column of its TMEM column 0
        const int row_off = TM == 128 ? 32 * q : (WS ? (TM == 64 ? 32 * (q & 1) : 0) : 16 * q);
        const int row_cap = (TM == 64 && !WS) ? 16 : 32;
        const int col_off = WS && TM == 64 ? (q >> 1) * (BN / 2) : (WS && TM == 32 ? q * (BN / 4) : 0);
        float* stage_buf = epi + ew * 32 * 32;
        int local = 0;
        WorkIter<BN, TM> w(p);
        Seg s;
        while (w.next(s)) {
            const int buf = local & 1;
            const uint32_t use = static_cast<uint32_t>(local >> 1);
            if (!wait_bounded(smem_u32(&tfull[buf]), use & 1, abort_flag, p.wait_limit)) {
                raise_timeout(p, abort_flag);
                break;
            }
            tc_fence_after();
            {
                const uint32_t tacc = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS);
                if (p.out_type == kOutF16)
                    epilogue_store<SWAP, kOutF16>(p, s, tacc, q, c_begin, c_begin + C::ACC_COLS / 2, lane, stage_buf,
                                              row_off, row_cap, col_off);
                else if (p.out_type == kOutBF16)
                    epilogue_store<SWAP, kOutBF16>(p, s, tacc, q, c_begin, c_begin + C::ACC_COLS / 2, lane, stage_buf,
                                              row_off, row_cap, col_off);
                else
                    epilogue_store<SWAP, kOutF32>(p, s, tacc, q, c_begin, c_begin + C::ACC_COLS / 2, lane, stage_buf,
                                              row_off, row_cap, col_off);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[buf]));
            ++local;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<C::TMEM_COLS>(tmem_base);
    }
}

template <int BN, bool SWAP, int XR = 128, int KIND = kKind16, int TM = 128, bool WS = false>
cudaError_t configure_kind()
{
    return cudaFuncSetAttribute(tc05_gemm_kernel<BN, SWAP, XR, KIND, TM, WS>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN, SWAP, XR, KIND, TM, WS>::SMEM);
}

template <int BN, bool SWAP, int XR = 128, int KIND = kKind16, int TM = 128, bool WS = false>
cudaError_t launch_kind(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int grid,
                        cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(threads_of(KIND), 1, 1);
    cfg.dynamicSmemBytes = Cfg<BN, SWAP, XR, KIND, TM, WS>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc05_gemm_kernel<BN, SWAP, XR, KIND, TM, WS>, tmx, tmy, p);
}

}  // namespace
}  // namespace gnt
