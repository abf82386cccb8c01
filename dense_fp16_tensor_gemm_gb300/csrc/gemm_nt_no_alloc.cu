// gemm_nt_no_alloc.cu -- gemm_nt_f16_f32_batched_no_alloc: the CTA-pair kernel
// with its scratch in a fixed array inside the library, for callers that must
// not allocate device memory (code under stream capture, applications whose
// pool allocator owns all device memory, paths that cannot take a first-call
// allocation).  See include/gemm_nt.h for the contract.
#include <mutex>

#include <cuda_runtime.h>

#include "gemm_nt.h"
#include "internal.h"

namespace {

// Scratch for the split path: the slices of up to kSlicePairs CTA pairs
// (8 MiB) followed by the counters of up to kCounterTiles split tiles (4 KiB).
constexpr int kSlicePairs = 16;
constexpr int kCounterTiles = 64;
constexpr size_t kSliceBytes = static_cast<size_t>(kSlicePairs) * 4 * gnt::kPairSliceBytes;
constexpr size_t kCounterBytes = static_cast<size_t>(kCounterTiles) * 2 * 8 * sizeof(uint32_t);

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kSliceBytes + kCounterBytes];

constexpr int kMaxDevices = 64;

// Host code cannot use g_no_alloc_scratch's name as a device address: the
// device address is looked up with the device current, once it has succeeded,
// and again on the next call after a failed lookup.
struct ScratchAddress {
    std::mutex mu;
    unsigned char* ptr = nullptr;
};
ScratchAddress g_address[kMaxDevices];

int current_scratch(gnt::PairScratch* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return GEMM_ERR_LAUNCH;
    ScratchAddress& a = g_address[dev];
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(a.mu);
        if (a.ptr == nullptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr)
                return GEMM_ERR_LAUNCH;
            a.ptr = static_cast<unsigned char*>(p);
        }
        base = a.ptr;
    }
    out->slices = reinterpret_cast<float*>(base);
    out->slice_pairs = kSlicePairs;
    out->counters = reinterpret_cast<uint32_t*>(base + kSliceBytes);
    out->counter_tiles = kCounterTiles;
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_nt_f16_f32_batched_no_alloc(const void* A, const void* B, float* Out, int64_t M,
                                                          int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                                          int64_t ldo, int64_t strideA, int64_t strideB,
                                                          int64_t strideO, int64_t batch, gemm_stream_t stream)
{
    return static_cast<gemm_status_t>(gnt::run_pair_no_alloc(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB,
                                                             strideO, batch, current_scratch,
                                                             reinterpret_cast<cudaStream_t>(stream)));
}
