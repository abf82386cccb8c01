// tc05_small.cu -- instances of the one-CTA tcgen05 kernel (tc05_kernel.cuh)
// with other instruction shapes: 64-row tiles on the plain M = 64 MMA, and
// 64- or 32-row tiles on the weight-stationary MMA (tcgen05.mma.ws), for
// products with few rows of A.  "Blackwell Tensor Cores" names both forms next
// to the 128-row shape its example uses; the accumulator layouts they produce
// in Tensor Memory were measured with coded inputs (row i of A and column j of
// B tagged, every TMEM word decoded) and are written out in the kernel's
// configuration.
#include "tc05_kernel.cuh"

namespace gnt {

namespace {

using namespace tc;

template <int BN, int TM, bool WS>
cudaError_t configure_small()
{
    cudaError_t e = configure_kind<BN, false, TM, kKind16, TM, WS>();
    return e == cudaSuccess ? configure_kind<BN, false, TM, kKind8, TM, WS>() : e;
}

template <int BN, int TM, bool WS>
cudaError_t launch_small(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int grid, int kind,
                         cudaStream_t stream)
{
    if (kind == kKind8)
        return launch_kind<BN, false, TM, kKind8, TM, WS>(tmx, tmy, p, grid, stream);
    return launch_kind<BN, false, TM, kKind16, TM, WS>(tmx, tmy, p, grid, stream);
}

}  // namespace

cudaError_t tc05_small_configure()
{
    cudaError_t e = configure_small<64, 64, false>();
    if (e == cudaSuccess) e = configure_small<128, 64, false>();
    if (e == cudaSuccess) e = configure_small<256, 64, false>();
    if (e == cudaSuccess) e = configure_small<128, 64, true>();
    if (e == cudaSuccess) e = configure_small<256, 64, true>();
    if (e == cudaSuccess) e = configure_small<256, 32, true>();
    return e;
}

cudaError_t tc05_small_launch(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int bn, int tm,
                              bool ws, int grid, int kind, cudaStream_t stream)
{
    if (kind != 0 && kind != 1)
        return cudaErrorInvalidValue;
    if (!ws && tm == 64) {
        switch (bn) {
        case 64: return launch_small<64, 64, false>(tmx, tmy, p, grid, kind, stream);
        case 128: return launch_small<128, 64, false>(tmx, tmy, p, grid, kind, stream);
        case 256: return launch_small<256, 64, false>(tmx, tmy, p, grid, kind, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    if (ws && tm == 64) {
        if (bn == 128)
            return launch_small<128, 64, true>(tmx, tmy, p, grid, kind, stream);
        if (bn == 256)
            return launch_small<256, 64, true>(tmx, tmy, p, grid, kind, stream);
        return cudaErrorInvalidValue;
    }
    if (ws && tm == 32 && bn == 256)
        return launch_small<256, 32, true>(tmx, tmy, p, grid, kind, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gnt
