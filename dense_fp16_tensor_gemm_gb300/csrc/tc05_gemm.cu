// tc05_gemm.cu -- the instances of the one-CTA tcgen05 kernel (tc05_kernel.cuh)
// with 128-row tiles, and their host-side configure / launch entry points.
#include "tc05_kernel.cuh"

namespace gnt {

namespace {

using namespace tc;

template <int BN, bool SWAP, int XR = 128>
cudaError_t configure_one()
{
    cudaError_t e = configure_kind<BN, SWAP, XR, kKind16>();
    return e == cudaSuccess ? configure_kind<BN, SWAP, XR, kKind8>() : e;
}

template <int BN, bool SWAP, int XR = 128>
cudaError_t launch_one(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int grid, int kind,
                       cudaStream_t stream)
{
    if (kind == kKind8)
        return launch_kind<BN, SWAP, XR, kKind8>(tmx, tmy, p, grid, stream);
    return launch_kind<BN, SWAP, XR, kKind16>(tmx, tmy, p, grid, stream);
}

}  // namespace

cudaError_t tc05_configure(int bn, bool swap)
{
    if (swap) {
        if (bn != 64)
            return cudaErrorInvalidValue;
        cudaError_t e = configure_one<64, true>();
        if (e == cudaSuccess)
            e = configure_one<64, true, 112>();
        return e == cudaSuccess ? configure_kind<64, true, 128, kKindMx>() : e;
    }
    cudaError_t e;
    switch (bn) {
    case 64:
        e = configure_one<64, false>();
        return e == cudaSuccess ? configure_kind<64, false, 128, kKindMx>() : e;
    case 128:
        e = configure_one<128, false>();
        return e == cudaSuccess ? configure_kind<128, false, 128, kKindMx>() : e;
    case 256: return configure_one<256, false>();
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t tc05_launch(const CUtensorMap& tmx, const CUtensorMap& tmy, const TcParams& p, int bn, bool swap,
                        int grid, int kind, cudaStream_t stream)
{
    if (kind == kKindMx) {
        // block-scaled: 128-row X tiles (no row split), Y tiles of 64 or 128
        if (swap)
            return bn == 64 ? launch_kind<64, true, 128, kKindMx>(tmx, tmy, p, grid, stream) : cudaErrorInvalidValue;
        if (bn == 64)
            return launch_kind<64, false, 128, kKindMx>(tmx, tmy, p, grid, stream);
        if (bn == 128)
            return launch_kind<128, false, 128, kKindMx>(tmx, tmy, p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (swap) {
        if (bn != 64)
            return cudaErrorInvalidValue;
        if (p.x_box_bytes <= 112 * 128)
            return launch_one<64, true, 112>(tmx, tmy, p, grid, kind, stream);
        return launch_one<64, true>(tmx, tmy, p, grid, kind, stream);
    }
    switch (bn) {
    case 64: return launch_one<64, false>(tmx, tmy, p, grid, kind, stream);
    case 128: return launch_one<128, false>(tmx, tmy, p, grid, kind, stream);
    case 256: return launch_one<256, false>(tmx, tmy, p, grid, kind, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gnt
