// gemm_nt_api.cu -- the C ABI of libgemm_nt (declared in include/gemm_nt.h):
// argument validation, kernel selection, TMA tensor-map construction, per-device
// state and the status word.
//
// The product is the one of the TIRx guides' worked examples ("Warp Matrix
// Instructions" and "Blackwell Tensor Cores"): Out = A @ B.T, fp16 inputs, fp32
// accumulation, Out overwritten.  The 128-byte swizzle of the tensor maps is the
// guides' swizzle "mode 3" (1024-byte period), which the tcgen05 kernel's
// shared-memory descriptors expect.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "gemm_nt.h"
#include "internal.h"

namespace gnt {

__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitLimit = 4000000000ull;  // ~2 s of SM clock

std::atomic<unsigned long long> g_wait_limit{0};
std::atomic<int> g_fault{0};

// Set up once per device by the first call that succeeds in it: a set-up that
// failed (a CUDA error) is tried again by the next call.
struct DeviceState {
    std::mutex init_mu;
    std::atomic<bool> ready{false};  // set-up done (supported or not)
    bool supported = false;
    int num_sms = 0;
    int max_pairs = 0;  // CTA pairs of the pair kernel resident at once
    uint32_t* status = nullptr;
    // host-buffer pipeline: copy streams and events, created by the first call
    // that succeeds in creating them
    std::atomic<bool> pipe_ready{false};
    std::mutex pipe_mu;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev[2 + 2 * 16];  // start, done, per-chunk input and output events
};

DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// Per-device one-time setup: capability check, SM count, kernel attributes and
// the address of the status word.
gemm_status_t device_state(DeviceState** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return GEMM_ERR_LAUNCH;
    DeviceState& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(d.init_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            const bool supported = major == 10 && minor == 3;
            if (supported) {
                void* sym = nullptr;
                int max_pairs = 0;
                e = cudaGetSymbolAddress(&sym, g_status_word);
                if (e == cudaSuccess) e = cudaMemset(sym, 0, sizeof(uint32_t));
                if (e == cudaSuccess) e = tc05_configure(64, false);
                if (e == cudaSuccess) e = tc05_configure(128, false);
                if (e == cudaSuccess) e = tc05_configure(256, false);
                if (e == cudaSuccess) e = tc05_configure(64, true);
                if (e == cudaSuccess) e = tc05_small_configure();
                if (e == cudaSuccess) e = tc05_pair_configure(&max_pairs);
                if (e != cudaSuccess)
                    return GEMM_ERR_LAUNCH;
                d.status = static_cast<uint32_t*>(sym);
                d.max_pairs = max_pairs;
            }
            d.num_sms = sms;
            d.supported = supported;
            d.ready.store(true, std::memory_order_release);
        }
    }
    if (!d.supported)
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return GEMM_OK;
}

// Stream-K workspace of the pair kernel, one per (device, stream) so that calls
// on different streams never share one; allocated and zeroed on first use and
// kept until the process exits (about 38 MB with 76 pairs).
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

gemm_status_t stream_workspace(cudaStream_t stream, size_t bytes, void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace& w = g_ws[std::make_pair(dev, stream)];
    if (w.bytes < bytes) {
        if (w.ptr) {
            if (cudaStreamSynchronize(stream) != cudaSuccess || cudaFree(w.ptr) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            w.ptr = nullptr;
            w.bytes = 0;
        }
        if (cudaMalloc(&w.ptr, bytes) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        if (cudaMemset(w.ptr, 0, bytes) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        w.bytes = bytes;
    }
    *out = w.ptr;
    return GEMM_OK;
}

// After a kernel gave up (bounded wait), its stream-K counters may be left
// non-zero: clear every workspace of the current device.
void reset_workspaces()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    for (auto& kv : g_ws)
        if (kv.first.first == dev && kv.second.ptr)
            cudaMemset(kv.second.ptr, 0, kv.second.bytes);
}

struct Problem {
    const void* A;
    const void* B;
    void* Out;
    int64_t M, N, K, lda, ldb, ldo, batch, sA, sB, sO;
    int ab_type = GEMM_DTYPE_F16;   // element type of A and B
    int out_type = GEMM_DTYPE_F32;  // element type of Out
    int a_major = GEMM_MAJOR_K;     // A(i,k) at A[i*lda + k] (K) or A[k*lda + i] (MN)
    int b_major = GEMM_MAJOR_K;
    // block scales of A and B in the packed atom layout (8-bit inputs only);
    // null for unscaled products
    const void* SA = nullptr;
    const void* SB = nullptr;

    bool mx() const { return SA != nullptr || SB != nullptr; }

    bool a_mn() const { return a_major == GEMM_MAJOR_MN; }
    bool b_mn() const { return b_major == GEMM_MAJOR_MN; }
    // stored matrices: (rows, cols) row-major with pitch lda / ldb
    int64_t a_rows() const { return a_mn() ? K : M; }
    int64_t a_cols() const { return a_mn() ? M : K; }
    int64_t b_rows() const { return b_mn() ? K : N; }
    int64_t b_cols() const { return b_mn() ? N : K; }

    int64_t out_esize() const { return out_type == GEMM_DTYPE_F32 ? 4 : 2; }
    // the 8-bit MMA kinds: 8-bit floats, and the 6- and 4-bit ones (stored packed)
    bool is_f8() const { return ab_type >= GEMM_DTYPE_E4M3 && ab_type <= GEMM_DTYPE_E2M1; }
    // 6- and 4-bit floats, packed along K (two per byte, or four per three bytes)
    bool is_packed() const { return ab_type >= GEMM_DTYPE_E2M3 && ab_type <= GEMM_DTYPE_E2M1; }
    int ab_bits() const
    {
        return ab_type == GEMM_DTYPE_E2M1 ? 4 : (is_packed() ? 6 : (is_f8() ? 8 : 16));
    }
    // bytes of n elements of A or B (n a multiple of the packing group)
    int64_t ab_bytes(int64_t n) const { return n * ab_bits() / 8; }
    // kernel kind of tc05_launch: 0 16-bit, 1 8-bit, 2 8-bit block-scaled
    int kind() const { return mx() ? 2 : (is_f8() ? 1 : 0); }
    int64_t ab_esize() const { return is_f8() ? 1 : 2; }
    // k-blocks of one 128-byte stage row: 64 elements of 16 bits, 128 of 8
    int64_t kblocks() const { return (K + 127 / ab_esize()) / (128 / ab_esize()); }
    int kernel_out() const { return out_type == GEMM_DTYPE_F16 ? kOutF16 : (out_type == GEMM_DTYPE_BF16 ? kOutBF16 : kOutF32); }
    // A/B format fields of the instruction descriptor (bits 7-9, 10-12): 1 is
    // bf16 for kind::f16 and E5M2 for kind::f8f6f4; 0 is fp16 or E4M3.
    uint32_t ab_fmt() const
    {
        // kind::f8f6f4 codes: E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5
        uint32_t f = 0;
        switch (ab_type) {
        case GEMM_DTYPE_BF16: f = 1; break;
        case GEMM_DTYPE_E5M2: f = 1; break;
        case GEMM_DTYPE_E2M3: f = 3; break;
        case GEMM_DTYPE_E3M2: f = 4; break;
        case GEMM_DTYPE_E2M1: f = 5; break;
        default: f = 0;
        }
        return (f << 7) | (f << 10);
    }
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Bytes of one packed block-scale matrix: 512-byte atoms for every 128 rows
// and every 128 elements of K.
int64_t mx_scale_bytes(int64_t rows, int64_t K)
{
    return ((rows + 127) / 128) * ((K + 127) / 128) * 512;
}

// Byte span [lo, hi) touched by a strided batch of row-major matrices.
void span(const void* base, int64_t esize, int64_t batch, int64_t stride, int64_t rows, int64_t ld,
          int64_t cols, uintptr_t& lo, uintptr_t& hi)
{
    const int64_t last = (batch - 1) * stride + (rows - 1) * ld + cols;
    lo = reinterpret_cast<uintptr_t>(base);
    hi = lo + static_cast<uintptr_t>(last * esize);
}

// The same for elements of `bits` bits (the end rounded up to a byte).
void span_bits(const void* base, int bits, int64_t batch, int64_t stride, int64_t rows, int64_t ld, int64_t cols,
               uintptr_t& lo, uintptr_t& hi)
{
    const int64_t last = (batch - 1) * stride + (rows - 1) * ld + cols;
    lo = reinterpret_cast<uintptr_t>(base);
    hi = lo + static_cast<uintptr_t>((last * bits + 7) / 8);
}

gemm_status_t validate(const Problem& q)
{
    if (q.M < 0 || q.N < 0 || q.K < 0 || q.batch < 0)
        return GEMM_ERR_INVALID_VALUE;
    if (q.M > INT32_MAX || q.N > INT32_MAX || q.K > INT32_MAX || q.batch > INT32_MAX)
        return GEMM_ERR_INVALID_VALUE;
    if (q.M == 0 || q.N == 0 || q.batch == 0)
        return GEMM_OK;
    if (!q.Out)
        return GEMM_ERR_INVALID_VALUE;
    if (q.K > 0 && (!q.A || !q.B))
        return GEMM_ERR_INVALID_VALUE;
    if (q.a_major != GEMM_MAJOR_K && q.a_major != GEMM_MAJOR_MN)
        return GEMM_ERR_INVALID_VALUE;
    if (q.b_major != GEMM_MAJOR_K && q.b_major != GEMM_MAJOR_MN)
        return GEMM_ERR_INVALID_VALUE;
    if (q.ldo < q.N || (q.K > 0 && (q.lda < q.a_cols() || q.ldb < q.b_cols())))
        return GEMM_ERR_INVALID_VALUE;
    if (q.sA < 0 || q.sB < 0 || q.sO < 0)
        return GEMM_ERR_INVALID_VALUE;
    // 64-bit extent limits (keep every byte offset below 2^62)
    const double lim = 4.0e18;
    if (static_cast<double>(q.batch) * static_cast<double>(std::max(q.sO, q.ldo * q.M)) * 4.0 > lim ||
        static_cast<double>(q.batch) * static_cast<double>(std::max(q.sA, q.lda * q.a_rows())) * 2.0 > lim ||
        static_cast<double>(q.batch) * static_cast<double>(std::max(q.sB, q.ldb * q.b_rows())) * 2.0 > lim)
        return GEMM_ERR_INVALID_VALUE;
    if (q.ab_type != GEMM_DTYPE_F16 && q.ab_type != GEMM_DTYPE_BF16 && !q.is_f8())
        return GEMM_ERR_INVALID_VALUE;
    if (q.out_type != GEMM_DTYPE_F32 && q.out_type != GEMM_DTYPE_F16 && q.out_type != GEMM_DTYPE_BF16)
        return GEMM_ERR_INVALID_VALUE;
    if (!aligned(q.Out, static_cast<uintptr_t>(q.out_esize())) ||
        (q.K > 0 && (!aligned(q.A, static_cast<uintptr_t>(q.ab_esize())) ||
                     !aligned(q.B, static_cast<uintptr_t>(q.ab_esize())))))
        return GEMM_ERR_INVALID_VALUE;
    if (q.batch > 1 && q.sO < (q.M - 1) * q.ldo + q.N)
        return GEMM_ERR_OVERLAP;
    if (q.is_packed() && q.K > 0) {
        // rows and batches start on whole bytes (fp4: even pitches; fp6: multiples of 4), K-major
        const int64_t g = q.ab_bits() == 4 ? 2 : 4;
        if (q.a_mn() || q.b_mn() || q.lda % g || q.ldb % g || q.sA % g || q.sB % g)
            return GEMM_ERR_INVALID_VALUE;
    }
    if (q.mx() && q.K > 0) {
        if (!q.SA || !q.SB || !q.is_f8() || q.a_mn() || q.b_mn())
            return GEMM_ERR_INVALID_VALUE;
        if (!aligned(q.SA, 16) || !aligned(q.SB, 16))
            return GEMM_ERR_INVALID_VALUE;
    }
    if (q.K > 0) {
        uintptr_t olo, ohi, alo, ahi, blo, bhi;
        span(q.Out, q.out_esize(), q.batch, q.sO, q.M, q.ldo, q.N, olo, ohi);
        span_bits(q.A, q.ab_bits(), q.batch, q.sA, q.a_rows(), q.lda, q.a_cols(), alo, ahi);
        span_bits(q.B, q.ab_bits(), q.batch, q.sB, q.b_rows(), q.ldb, q.b_cols(), blo, bhi);
        if ((olo < ahi && alo < ohi) || (olo < bhi && blo < ohi))
            return GEMM_ERR_OVERLAP;
        if (q.mx()) {
            const uintptr_t sa = reinterpret_cast<uintptr_t>(q.SA), sb = reinterpret_cast<uintptr_t>(q.SB);
            const uintptr_t na = static_cast<uintptr_t>(mx_scale_bytes(q.M, q.K)) * (q.sA == 0 ? 1 : q.batch);
            const uintptr_t nb = static_cast<uintptr_t>(mx_scale_bytes(q.N, q.K)) * (q.sB == 0 ? 1 : q.batch);
            if ((olo < sa + na && sa < ohi) || (olo < sb + nb && sb < ohi))
                return GEMM_ERR_OVERLAP;
        }
    }
    return GEMM_OK;
}

// Conditions for TMA tensor maps over A and B: 16-byte aligned bases and
// row / batch strides that are multiples of 16 bytes and below 2^40 bytes.
bool tma_ok(const Problem& q)
{
    if (q.is_packed()) {
        // the unpacking tensor-map types: 32-byte aligned bases, pitches and batch
        // strides in multiples of 32 bytes, K a multiple of 128, below 2^40 bytes
        if (!aligned(q.A, 32) || !aligned(q.B, 32) || q.K % 128)
            return false;
        if (q.ab_bytes(q.lda) % 32 || q.ab_bytes(q.ldb) % 32)
            return false;
        if (q.batch > 1 && (q.ab_bytes(q.sA) % 32 || q.ab_bytes(q.sB) % 32))
            return false;
        if (q.batch > 1 && ((q.sA != 0 && q.sA < q.a_rows() * q.lda) || (q.sB != 0 && q.sB < q.b_rows() * q.ldb)))
            return false;
        const int64_t lim = int64_t(1) << 40;
        return q.ab_bytes(q.lda) < lim && q.ab_bytes(q.ldb) < lim && q.ab_bytes(q.sA) < lim && q.ab_bytes(q.sB) < lim;
    }
    if (!aligned(q.A, 16) || !aligned(q.B, 16))
        return false;
    const int64_t v = 16 / q.ab_esize();  // elements in 16 bytes
    if ((q.lda % v) || (q.ldb % v))
        return false;
    if (q.batch > 1 && ((q.sA % v) || (q.sB % v)))
        return false;
    // 8-bit operands are staged K-major only (MN-major ones run on the warp kernel)
    if (q.is_f8() && (q.a_mn() || q.b_mn()))
        return false;
    // a batch dimension in a tensor map must step over whole matrices
    if (q.batch > 1 && ((q.sA != 0 && q.sA < q.a_rows() * q.lda) || (q.sB != 0 && q.sB < q.b_rows() * q.ldb)))
        return false;
    const int64_t lim = (int64_t(1) << 40) / q.ab_esize();  // strides below 2^40 bytes
    if (q.lda >= lim || q.ldb >= lim || q.sA >= lim || q.sB >= lim)
        return false;
    return true;
}

gemm_path_t select_path(const Problem& q)
{
    if (q.is_packed() && !q.mx())  // no warp kernel for packed 6- and 4-bit inputs
        return q.M <= 64 && q.N >= 1024 ? GEMM_PATH_SKINNY
                                        : (q.M > 128 && q.N > 128 ? GEMM_PATH_TC05_PAIR : GEMM_PATH_TC05);
    if (q.mx()) {  // block-scaled: no warp kernel; swapped for small M, pairs for large tiles
        if (q.M <= 64 && q.N >= 1024)
            return GEMM_PATH_SKINNY;
        return q.M > 128 && q.N > 128 ? GEMM_PATH_TC05_PAIR : GEMM_PATH_TC05;
    }
    if (!tma_ok(q))
        return GEMM_PATH_MMASYNC;
    if (q.M <= 64 && q.N >= 1024)
        return GEMM_PATH_SKINNY;
    if (q.M > 128 && q.N > 128)
        return GEMM_PATH_TC05_PAIR;
    return GEMM_PATH_TC05;
}

// Tensor maps depend only on the address and geometry, so each host thread
// keeps the last few it encoded (no lock needed) and repeat calls skip the
// driver's encoder.
struct MapKey {
    const void* base;
    int64_t rows, K, ld, batch, stride;
    int box_rows;
    int dtype;
    bool mn;
    bool operator==(const MapKey& o) const
    {
        return base == o.base && rows == o.rows && K == o.K && ld == o.ld && batch == o.batch &&
               stride == o.stride && box_rows == o.box_rows && dtype == o.dtype && mn == o.mn;
    }
};

struct MapCache {
    static constexpr int kEntries = 16;
    MapKey key[kEntries];
    CUtensorMap map[kEntries];
    int bmul[kEntries];
    int count = 0, next = 0;
};

thread_local MapCache t_maps;

// An operand of `rows` rows (M or N) and K columns of `dtype` (a gemm_dtype_t
// input type).  K-major: dims {K, rows, batch}, box {one 128-byte row of K,
// box_rows}.  MN-major (stored as (K, rows) with pitch ld; 16-bit types only):
// dims {rows, K, batch}, box {64 rows, 64 K}; box_rows is then ignored.
bool encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t ld, int64_t batch,
                int64_t stride, int box_rows, int* bmul, int dtype, bool mn)
{
    const bool f8 = dtype == GEMM_DTYPE_E4M3 || dtype == GEMM_DTYPE_E5M2;
    const bool packed = dtype >= GEMM_DTYPE_E2M3 && dtype <= GEMM_DTYPE_E2M1;
    const int bits = dtype == GEMM_DTYPE_E2M1 ? 4 : (packed ? 6 : (f8 ? 8 : 16));
    auto enc = encode_fn();
    if (!enc)
        return false;
    const bool batched = batch > 1 && stride > 0;
    const int64_t inner = mn ? rows : K, outer = mn ? K : rows;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                          static_cast<cuuint64_t>(batched ? batch : 1)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * bits / 8),
                             static_cast<cuuint64_t>((batched ? stride : outer * ld) * bits / 8)};
    // one 128-byte shared row per box row: 64 elements of 16 bits, 128 of 8 bits,
    // or 128 packed 6- or 4-bit elements, which the unpacking types spread to 16
    // elements per 16-byte chunk (the layout the 8-bit MMA kind reads them in)
    cuuint32_t box[3] = {static_cast<cuuint32_t>(bits == 16 ? 64 : 128), static_cast<cuuint32_t>(mn ? 64 : box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    *bmul = batched ? 1 : 0;
    const CUtensorMapDataType ty =
        packed ? (bits == 4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B)
               : (f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                     : (dtype == GEMM_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16));
    CUresult r = enc(map, ty, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Block scales of `mats` matrices (rows row blocks of 128, K of K) as a 4-D
// tensor {128 bytes, 4 rows, K block group, row block}: one atom is {128, 4},
// and a box takes box_kg consecutive K block groups of box_rb consecutive row
// blocks (unswizzled, so shared memory receives the atoms in that order).
bool encode_scale_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t mats, int box_rb,
                      int box_kg)
{
    auto enc = encode_fn();
    const int64_t kg = (K + 127) / 128, rb = (rows + 127) / 128 * mats;
    if (!enc || kg <= 0 || rb <= 0 || kg > (int64_t(1) << 31) || rb > (int64_t(1) << 31))
        return false;
    cuuint64_t dims[4] = {128, 4, static_cast<cuuint64_t>(kg), static_cast<cuuint64_t>(rb)};
    cuuint64_t strides[3] = {128, 512, static_cast<cuuint64_t>(kg * 512)};
    if (box_kg < 1 || box_kg > kg || box_rb < 1 || box_rb > rb)
        return false;
    cuuint32_t box[4] = {128, 4, static_cast<cuuint32_t>(box_kg), static_cast<cuuint32_t>(box_rb)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same scales as a 5-D tensor {128 bytes, 4 rows, 4 copies, K block group,
// row block} whose copy dimension has stride 0: a box {128, 4, 4, 1, box_rb}
// lands each of box_rb consecutive atoms of one K block group four times over,
// as [row block][copy][atom] (the source of one non-replicating TMEM copy).
bool encode_scale_rep_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t mats, int box_rb)
{
    auto enc = encode_fn();
    const int64_t kg = (K + 127) / 128, rb = (rows + 127) / 128 * mats;
    if (!enc || kg <= 0 || rb <= 0 || kg > (int64_t(1) << 31) || rb > (int64_t(1) << 31) || box_rb < 1 ||
        box_rb > rb)
        return false;
    cuuint64_t dims[5] = {128, 4, 4, static_cast<cuuint64_t>(kg), static_cast<cuuint64_t>(rb)};
    cuuint64_t strides[4] = {128, 0, 512, static_cast<cuuint64_t>(kg * 512)};
    cuuint32_t box[5] = {128, 4, 4, 1, static_cast<cuuint32_t>(box_rb)};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t ld, int64_t batch,
              int64_t stride, int box_rows, int* bmul, int dtype = GEMM_DTYPE_F16, bool mn = false)
{
    const MapKey k{base, rows, K, ld, batch, stride, box_rows, dtype, mn};
    MapCache& c = t_maps;
    for (int i = 0; i < c.count; ++i) {
        if (c.key[i] == k) {
            *map = c.map[i];
            *bmul = c.bmul[i];
            return true;
        }
    }
    if (!encode_map(map, base, rows, K, ld, batch, stride, box_rows, bmul, dtype, mn))
        return false;
    const int slot = c.next;
    c.key[slot] = k;
    c.map[slot] = *map;
    c.bmul[slot] = *bmul;
    c.next = (slot + 1) % MapCache::kEntries;
    if (c.count < MapCache::kEntries)
        ++c.count;
    return true;
}

gemm_status_t zero_out(const Problem& q, cudaStream_t stream)
{
    if (q.sO == q.M * q.ldo || q.batch == 1) {
        const int64_t rows = q.batch == 1 ? q.M : q.M * q.batch;
        if (cudaMemset2DAsync(q.Out, q.ldo * q.out_esize(), 0, q.N * q.out_esize(), rows, stream) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        return GEMM_OK;
    }
    for (int64_t b = 0; b < q.batch; ++b)
        if (cudaMemset2DAsync(static_cast<uint8_t*>(q.Out) + b * q.sO * q.out_esize(), q.ldo * q.out_esize(), 0,
                              q.N * q.out_esize(), q.M, stream) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

unsigned long long wait_limit()
{
    const unsigned long long v = g_wait_limit.load();
    return v ? v : kDefaultWaitLimit;
}

// tm < 128: tiles of tm rows of A on the plain M = 64 MMA or (ws) on the
// weight-stationary one; not swapped, unscaled, A K-major.
gemm_status_t run_tc05(const Problem& q, const DeviceState& d, bool swap, cudaStream_t stream, int tm = 128,
                       bool ws = false)
{
    // X: the operand on the MMA's M side (128-row tiles); Y: the N side.
    const void* xp = swap ? q.B : q.A;
    const void* yp = swap ? q.A : q.B;
    const int64_t xrows = swap ? q.N : q.M, yrows = swap ? q.M : q.N;
    const int64_t xld = swap ? q.ldb : q.lda, yld = swap ? q.lda : q.ldb;
    const int64_t xs = swap ? q.sB : q.sA, ys = swap ? q.sA : q.sB;
    const bool x_mn = swap ? q.b_mn() : q.a_mn(), y_mn = swap ? q.a_mn() : q.b_mn();
    int bn;
    if (tm < 128) {
        if (swap || q.mx() || x_mn)
            return GEMM_ERR_NOT_SUPPORTED;
        if (ws)
            bn = tm == 32 ? 256 : (yrows <= 128 ? 128 : 256);
        else
            bn = yrows <= 64 ? 64 : (yrows <= 128 ? 128 : 256);
    } else if (swap) {
        if (yrows > 64)
            return GEMM_ERR_NOT_SUPPORTED;
        bn = 64;
    } else if (q.mx()) {
        bn = yrows <= 64 ? 64 : 128;  // two accumulators and the scale slots fit TMEM
    } else {
        bn = yrows <= 64 ? 64 : (yrows <= 128 ? 128 : 256);
    }
    TcParams p{};
    p.ab_packed_bits = q.is_packed() ? q.ab_bits() : 0;
    // Row split (swapped operands, one batch, one column tile, 64..128 rows of
    // X per CTA): every CTA takes an even share of the rows over all of K, with
    // an X box just tall enough for that share (a multiple of 8 rows).
    // (K-major X only: an MN-major box is whole 64-row chunks.)
    const bool rowsplit = swap && !x_mn && !q.mx() && q.batch == 1 && yrows <= bn &&
                          xrows >= 64 * static_cast<int64_t>(d.num_sms) && xrows <= 128 * static_cast<int64_t>(d.num_sms);
    int xbox = tm;
    if (rowsplit) {
        const int64_t share = (xrows + d.num_sms - 1) / d.num_sms;
        xbox = static_cast<int>(std::min<int64_t>(128, (share + 7) / 8 * 8));
    }
    p.x_box_bytes = xbox * 128;
    CUtensorMap tmx, tmy;
    if (!make_map(&tmx, xp, xrows, q.K, xld, q.batch, xs, xbox, &p.x_bmul, q.ab_type, x_mn) ||
        !make_map(&tmy, yp, yrows, q.K, yld, q.batch, ys, bn, &p.y_bmul, q.ab_type, y_mn))
        return GEMM_ERR_LAUNCH;
    p.out = q.Out;
    p.out_type = q.kernel_out();
    p.x_mn = x_mn ? 1 : 0;
    p.y_mn = y_mn ? 1 : 0;
    p.idesc_bits = q.ab_fmt() | (x_mn ? 1u << 15 : 0u) | (y_mn ? 1u << 16 : 0u);
    p.ldo = q.ldo;
    p.stride_o = q.sO;
    p.rows_x = static_cast<int>(xrows);
    p.rows_y = static_cast<int>(yrows);
    p.batch = static_cast<int>(q.batch);
    p.tiles_x = static_cast<int>((xrows + tm - 1) / tm);
    p.tiles_y = static_cast<int>((yrows + bn - 1) / bn);
    p.num_kb = static_cast<int>(q.kblocks());
    const int64_t tpb = static_cast<int64_t>(p.tiles_x) * p.tiles_y;
    const int64_t ntiles = tpb * q.batch;
    if (ntiles > INT32_MAX)
        return GEMM_ERR_NOT_SUPPORTED;
    p.tiles_per_batch = static_cast<int>(tpb);
    p.num_tiles = static_cast<int>(ntiles);
    p.group_x = 16;
    p.total_iters = static_cast<long long>(ntiles) * p.num_kb;
    p.vec4 = (!swap && aligned(q.Out, static_cast<uintptr_t>(4 * q.out_esize())) && q.ldo % 4 == 0 &&
              (q.batch == 1 || q.sO % 4 == 0))
                 ? 1
                 : 0;
    p.status = d.status;
    p.wait_limit = wait_limit();
    p.fault = g_fault.load();
    int grid;
    if (rowsplit) {
        // no partial sums, nothing to zero
        p.mode = kModeRowSplit;
        grid = d.num_sms;
    } else if ((swap || tm < 128) && q.out_type == GEMM_DTYPE_F32 && ntiles < d.num_sms &&
               p.total_iters >= 2 * static_cast<long long>(d.num_sms) &&
               !(q.mx() && 2 * ntiles >= d.num_sms)) {
        // Stream-K when there are too few tiles to fill the GPU: each CTA takes
        // an even share of the (tile, k-block) iterations; tiles cut between
        // CTAs are summed with atomics into a zeroed Out.  Block-scaled
        // products keep whole tiles down to half as many tiles as SMs (30.9
        // against 32.8 us at 64 x 16384 x 8192, 128 tiles).
        p.mode = kModeStreamK;
        grid = d.num_sms;
        gemm_status_t z = zero_out(q, stream);
        if (z != GEMM_OK)
            return z;
    } else {
        p.mode = kModeTiles;
        grid = static_cast<int>(std::min<int64_t>(ntiles, d.num_sms));
    }
    if (q.mx()) {
        // scale atoms follow the operands: X = B when swapped
        const void* sx = swap ? q.SB : q.SA;
        const void* sy = swap ? q.SA : q.SB;
        p.sf_x = static_cast<const uint8_t*>(sx);
        p.sf_y = static_cast<const uint8_t*>(sy);
        p.sf_x_bstride = xs == 0 ? 0 : mx_scale_bytes(xrows, q.K);
        p.sf_y_bstride = ys == 0 ? 0 : mx_scale_bytes(yrows, q.K);
    }
    const cudaError_t le = tm < 128 ? tc05_small_launch(tmx, tmy, p, bn, tm, ws, grid, q.kind(), stream)
                                    : tc05_launch(tmx, tmy, p, bn, swap, grid, q.kind(), stream);
    if (le != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

// Tile width of the CTA-pair kernel: 256 columns, or 224 / 192 when that fits
// the number of tiles better to a whole number of rounds over the pairs.  The
// cost of a width is (rounds) x (width), the MMA work on the critical path,
// with a mild surcharge for narrower tiles, which move more bytes per MMA cycle
// (32 KB per 512 cycles at 256, 30 KB per 448 at 224, 28 KB per 384 at 192).
int pair_tile_width(int64_t M, int64_t N, int64_t batch, int pairs)
{
    static const int widths[3] = {256, 224, 192};
    static const double surcharge[3] = {1.0, 1.036, 1.084};
    int best = 256;
    double best_cost = 0;
    for (int i = 0; i < 3; ++i) {
        const int64_t tiles = batch * ((M + 255) / 256) * ((N + widths[i] - 1) / widths[i]);
        const int64_t rounds = (tiles + pairs - 1) / pairs;
        const double cost = static_cast<double>(rounds) * widths[i] * surcharge[i];
        if (i == 0 || cost < best_cost) {
            best = widths[i];
            best_cost = cost;
        }
    }
    return best;
}

// The split (stream-K) rule of the pair kernel, shared by both of its hosts:
// far fewer tiles than pairs and K long enough.
bool pair_split(int64_t ntiles, int num_kb, int pairs, int out_type)
{
    return out_type == GEMM_DTYPE_F32 && ntiles < pairs / 2 && num_kb >= 96;
}

int pair_plan_width(const Problem& q, const DeviceState& d)
{
    if (q.mx()) {
        // block-scaled: one 256-column accumulator with the direct epilogue
        // (Out rows 32-byte aligned, no split), else two 192-column ones;
        // either leaves TMEM room for the scale slots
        const bool direct = aligned(q.Out, static_cast<uintptr_t>(8 * q.out_esize())) && q.ldo % 8 == 0 &&
                            (q.batch == 1 || q.sO % 8 == 0);
        const int64_t tiles256 = q.batch * ((q.M + 255) / 256) * ((q.N + 255) / 256);
        return direct && !pair_split(tiles256, static_cast<int>(q.kblocks()), d.max_pairs, q.out_type) ? 256 : 192;
    }
    if (q.b_mn())
        return 256;  // each CTA's half of B must be whole 64-row chunks
    const int64_t tiles256 = q.batch * ((q.M + 255) / 256) * ((q.N + 255) / 256);
    if (pair_split(tiles256, static_cast<int>(q.kblocks()), d.max_pairs, q.out_type))
        return 256;
    return pair_tile_width(q.M, q.N, q.batch, d.max_pairs);
}

// CTA pairs: 256 x PBN tiles; each CTA loads its 128 rows of A and PBN/2 of
// the tile's PBN rows of B.  A split (stream-K) launch takes its scratch from
// `fixed` when given (memory the caller owns; nothing is allocated), else from
// the per-stream workspace.
gemm_status_t run_tc05_pair(const Problem& q, const DeviceState& d, cudaStream_t stream,
                            const PairScratch* fixed = nullptr)
{
    if (d.max_pairs < 1)
        return GEMM_ERR_NOT_SUPPORTED;
    TcParams p{};
    p.ab_packed_bits = q.is_packed() ? q.ab_bits() : 0;
    const int pbn = pair_plan_width(q, d);
    CUtensorMap tma, tmb;
    if (!make_map(&tma, q.A, q.M, q.K, q.lda, q.batch, q.sA, 128, &p.x_bmul, q.ab_type,
                  q.a_mn()) ||
        !make_map(&tmb, q.B, q.N, q.K, q.ldb, q.batch, q.sB, pbn / 2, &p.y_bmul, q.ab_type,
                  q.b_mn()))
        return GEMM_ERR_LAUNCH;
    p.out = q.Out;
    p.out_type = q.kernel_out();
    p.x_mn = q.a_mn() ? 1 : 0;
    p.y_mn = q.b_mn() ? 1 : 0;
    p.idesc_bits = q.ab_fmt() | (q.a_mn() ? 1u << 15 : 0u) | (q.b_mn() ? 1u << 16 : 0u);
    p.ldo = q.ldo;
    p.stride_o = q.sO;
    p.rows_x = static_cast<int>(q.M);
    p.rows_y = static_cast<int>(q.N);
    p.batch = static_cast<int>(q.batch);
    p.tiles_x = static_cast<int>((q.M + 255) / 256);
    p.tiles_y = static_cast<int>((q.N + pbn - 1) / pbn);
    p.num_kb = static_cast<int>(q.kblocks());
    const int64_t tpb = static_cast<int64_t>(p.tiles_x) * p.tiles_y;
    const int64_t ntiles = tpb * q.batch;
    if (ntiles > INT32_MAX)
        return GEMM_ERR_NOT_SUPPORTED;
    p.tiles_per_batch = static_cast<int>(tpb);
    p.num_tiles = static_cast<int>(ntiles);
    p.group_x = 8;
    p.mode = kModeTiles;
    p.total_iters = static_cast<long long>(ntiles) * p.num_kb;
    p.vec4 = (aligned(q.Out, static_cast<uintptr_t>(4 * q.out_esize())) && q.ldo % 4 == 0 &&
              (q.batch == 1 || q.sO % 4 == 0))
                 ? 1
                 : 0;
    p.status = d.status;
    p.wait_limit = wait_limit();
    p.fault = g_fault.load();
    // Stream-K when there are far fewer tiles than pairs and K is long (e.g.
    // 512 x 512 x 8192: 4 tiles for 76 pairs): every tile is cut into at most
    // kMaxPieces k ranges spread over the pairs; the warp that finishes a
    // portion last sums its slices.  That sum sits on the critical path (a few
    // microseconds), so the last partial round of a large problem is left to
    // whole tiles.
    constexpr int64_t kMaxPieces = 4;
    const int P = d.max_pairs;
    const int64_t rem = pair_split(ntiles, p.num_kb, P, q.out_type) ? ntiles : 0;
    const int64_t sk_pairs = std::min<int64_t>(P, rem * kMaxPieces);
    int pairs = static_cast<int>(std::min<int64_t>(ntiles, P));
    p.sk_first = p.num_tiles;
    p.sk_iters = 0;
    p.sk_pairs = 0;
    if (rem != 0) {
        pairs = static_cast<int>(std::max<int64_t>(pairs, sk_pairs));
        if (fixed) {
            // slices are indexed by the pair over every launched pair
            if (pairs > fixed->slice_pairs || rem > fixed->counter_tiles)
                return GEMM_ERR_SCRATCH_TOO_SMALL;
            // the counters must start at zero; the slices are fully rewritten
            if (cudaMemsetAsync(fixed->counters, 0, static_cast<size_t>(rem) * 2 * 8 * sizeof(uint32_t), stream) !=
                cudaSuccess)
                return GEMM_ERR_LAUNCH;
            p.ws = fixed->slices;
            p.ws_flags = fixed->counters;
        } else {
            void* ws = nullptr;
            gemm_status_t st = stream_workspace(stream, pair_workspace_bytes(P), &ws);
            if (st != GEMM_OK)
                return st;
            p.ws = static_cast<float*>(ws);
            p.ws_flags =
                reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + static_cast<size_t>(P) * 4 * kPairSliceBytes);
        }
        p.sk_first = static_cast<int>(ntiles - rem);
        p.sk_iters = rem * p.num_kb;
        p.sk_pairs = static_cast<int>(sk_pairs);
    }
    // Out rows 32-byte aligned: the epilogue stores without staging -- for
    // inputs whose rows TMA delivers at full speed (every row on a 128-byte
    // line).  With rows off their lines (e.g. a 2000-byte pitch) the staged
    // epilogue runs faster (179 against 210 us on a 16 x 3001 x 2048 x 1000
    // product); block-scaled tiles keep the choice their width was planned with.
    const int64_t ab_bits = q.ab_bits();
    const auto on_lines = [ab_bits](const void* base, int64_t ld, int64_t stride, int64_t batch) {
        return aligned(base, 128) && (ld * ab_bits / 8) % 128 == 0 && (batch == 1 || (stride * ab_bits / 8) % 128 == 0);
    };
    const bool direct = p.sk_pairs == 0 && aligned(q.Out, static_cast<uintptr_t>(8 * q.out_esize())) &&
                        q.ldo % 8 == 0 && (q.batch == 1 || q.sO % 8 == 0) &&
                        (q.mx() || (on_lines(q.A, q.lda, q.sA, q.batch) && on_lines(q.B, q.ldb, q.sB, q.batch)));
    if (q.mx()) {
        // each CTA stages its A rows' atom and the tile's two B atoms through
        // tensor maps over the packed scales
        // boxes of up to 8 K block groups and 2 B row blocks, never larger than
        // the scale tensors themselves
        CUtensorMap tmsa, tmsb;
        const int64_t mats_b = q.sB == 0 ? 1 : q.batch;
        p.sf_box_kg = static_cast<int>(std::min<int64_t>(8, (q.K + 127) / 128));
        p.sf_box_rb = static_cast<int>(std::min<int64_t>(2, (q.N + 127) / 128 * mats_b));
        // 256-wide tiles take B's scales per data stage, four times over
        const bool rep_b = pbn == 256 && direct;
        if (!encode_scale_map(&tmsa, q.SA, q.M, q.K, q.sA == 0 ? 1 : q.batch, 1, p.sf_box_kg) ||
            !(rep_b ? encode_scale_rep_map(&tmsb, q.SB, q.N, q.K, mats_b, p.sf_box_rb)
                    : encode_scale_map(&tmsb, q.SB, q.N, q.K, mats_b, p.sf_box_rb, p.sf_box_kg)))
            return GEMM_ERR_LAUNCH;
        p.sf_x_bstride = q.sA == 0 ? 0 : mx_scale_bytes(q.M, q.K);
        p.sf_y_bstride = q.sB == 0 ? 0 : mx_scale_bytes(q.N, q.K);
        if (tc05_pair_launch(tma, tmb, p, pairs, pbn, direct, q.kind(), stream, &tmsa, &tmsb) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        return GEMM_OK;
    }
    if (tc05_pair_launch(tma, tmb, p, pairs, pbn, direct, q.kind(), stream) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

gemm_status_t run_mmasync(const Problem& q, cudaStream_t stream)
{
    if ((q.M + 63) / 64 > 65535)
        return GEMM_ERR_NOT_SUPPORTED;
    MmaParams p{};
    p.A = static_cast<const uint16_t*>(q.A);
    p.B = static_cast<const uint16_t*>(q.B);
    p.out = q.Out;
    p.out_type = q.kernel_out();
    p.M = static_cast<int>(q.M);
    p.N = static_cast<int>(q.N);
    p.K = static_cast<int>(q.K);
    p.batch = static_cast<int>(q.batch);
    p.lda = q.lda;
    p.ldb = q.ldb;
    p.ldo = q.ldo;
    p.stride_a = q.sA;
    p.stride_b = q.sB;
    p.stride_o = q.sO;
    const uintptr_t v8 = static_cast<uintptr_t>(8 * q.ab_esize());  // 8 elements
    p.vec_a = aligned(q.A, v8) && q.lda % 8 == 0 && (q.batch == 1 || q.sA % 8 == 0);
    p.vec_b = aligned(q.B, v8) && q.ldb % 8 == 0 && (q.batch == 1 || q.sB % 8 == 0);
    p.a_mn = q.a_mn() ? 1 : 0;
    p.b_mn = q.b_mn() ? 1 : 0;
    return mmasync_launch(p, q.ab_type, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// The host link carries ~210 GB/s in and ~190 GB/s out (measured on GB300),
// so a call is bound by its input copies; what follows the last input chunk
// (that chunk's product and its Out copy) is the part not overlapped, which 16
// chunks keep short.
constexpr int kPipeChunks = 16;

// Host buffers in, host buffer out, with the copies overlapped with the
// products: the problem is cut into up to sixteen chunks (rows of A and Out for a
// single product, whole batches otherwise).  One library stream copies inputs
// to the device, the caller's stream runs each chunk's product once its inputs
// have arrived, a second library stream copies each chunk's Out back as soon as
// it is done, and the caller's stream finally waits for that last copy.
gemm_status_t from_host_pipelined(const void* A_host, const void* B_host, float* Out_host, uint16_t* dA,
                                  uint16_t* dB, float* dOut, int64_t M, int64_t N, int64_t K, int64_t batch,
                                  cudaStream_t stream);

gemm_status_t run(const Problem& q, gemm_path_t path, cudaStream_t stream)
{
    gemm_status_t st = validate(q);
    if (st != GEMM_OK)
        return st;
    if (q.M == 0 || q.N == 0 || q.batch == 0)
        return GEMM_OK;
    if (path < GEMM_PATH_AUTO || path > GEMM_PATH_TC05_WS)
        return GEMM_ERR_INVALID_VALUE;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != GEMM_OK)
        return st;
    if (q.K == 0)
        return zero_out(q, stream);
    if (path == GEMM_PATH_AUTO)
        path = select_path(q);
    if ((q.mx() || q.is_packed()) && path == GEMM_PATH_MMASYNC)
        return GEMM_ERR_NOT_SUPPORTED;
    switch (path) {
    case GEMM_PATH_MMASYNC:
        return run_mmasync(q, stream);
    case GEMM_PATH_TC05:
        if (!tma_ok(q))
            return GEMM_ERR_NOT_SUPPORTED;
        return run_tc05(q, *d, false, stream);
    case GEMM_PATH_SKINNY:
        if (!tma_ok(q))
            return GEMM_ERR_NOT_SUPPORTED;
        return run_tc05(q, *d, true, stream);
    case GEMM_PATH_TC05_PAIR:
        if (!tma_ok(q))
            return GEMM_ERR_NOT_SUPPORTED;
        return run_tc05_pair(q, *d, stream);
    case GEMM_PATH_TC05_M64:
    case GEMM_PATH_TC05_WS:
        if (!tma_ok(q) || q.mx())
            return GEMM_ERR_NOT_SUPPORTED;
        return run_tc05(q, *d, false, stream, path == GEMM_PATH_TC05_WS && q.M <= 32 ? 32 : 64,
                        path == GEMM_PATH_TC05_WS);
    default:
        return GEMM_ERR_NOT_SUPPORTED;
    }
}

// A single large product: Out is needed back in full, and each of its blocks
// needs a row block of A and one of B, so A and B are both cut into kBlockSplit
// row blocks and copied A0, B0, A1, B1, ...; Out block (i, j) is computed as
// soon as A_i and B_j are in and copied back at once (a 2-D copy).  The first
// result travels back after 2/kBlockSplit of the inputs instead of all of B,
// so the output copies, the longer half of the traffic, start early.
constexpr int kBlockSplit = 4;

gemm_status_t from_host_blocks(const void* A_host, const void* B_host, float* Out_host, uint16_t* dA, uint16_t* dB,
                               float* dOut, int64_t M, int64_t N, int64_t K, DeviceState& d, cudaStream_t stream)
{
    const int64_t per_a = (M + kBlockSplit - 1) / kBlockSplit, per_b = (N + kBlockSplit - 1) / kBlockSplit;
    const int64_t pa = (per_a + 255) / 256 * 256, pb = (per_b + 255) / 256 * 256;
    const int na = static_cast<int>((M + pa - 1) / pa), nb = static_cast<int>((N + pb - 1) / pb);
    cudaEvent_t ev_start = d.ev[0], ev_done = d.ev[1];
    cudaEvent_t* ev_a = d.ev + 2;
    cudaEvent_t* ev_b = ev_a + kBlockSplit;
    cudaEvent_t* ev_o = ev_b + kBlockSplit;  // kBlockSplit^2 of them
    static_assert(2 + 2 * kBlockSplit + kBlockSplit * kBlockSplit <= 2 + 2 * kPipeChunks, "event pool");
    std::lock_guard<std::mutex> lock(d.pipe_mu);
    if (cudaEventRecord(ev_start, stream) != cudaSuccess || cudaStreamWaitEvent(d.h2d, ev_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(d.d2h, ev_start, 0) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    const uint8_t* ha = static_cast<const uint8_t*>(A_host);
    const uint8_t* hb = static_cast<const uint8_t*>(B_host);
    const size_t row = static_cast<size_t>(K) * 2;
    for (int s = 0; s < std::max(na, nb); ++s) {
        if (s < na) {
            const int64_t r0 = s * pa, rows = std::min(pa, M - r0);
            if (cudaMemcpyAsync(reinterpret_cast<uint8_t*>(dA) + r0 * row, ha + r0 * row, rows * row,
                                cudaMemcpyHostToDevice, d.h2d) != cudaSuccess ||
                cudaEventRecord(ev_a[s], d.h2d) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
        }
        if (s < nb) {
            const int64_t r0 = s * pb, rows = std::min(pb, N - r0);
            if (cudaMemcpyAsync(reinterpret_cast<uint8_t*>(dB) + r0 * row, hb + r0 * row, rows * row,
                                cudaMemcpyHostToDevice, d.h2d) != cudaSuccess ||
                cudaEventRecord(ev_b[s], d.h2d) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
        }
    }
    // blocks in the order their inputs complete: step s brings A_s and B_s
    int k = 0;
    for (int s = 0; s < std::max(na, nb); ++s) {
        for (int t = 0; t < 2 * s + 1; ++t) {
            // (s, 0..s) then (0..s-1, s)
            const int i = t <= s ? s : t - s - 1;
            const int j = t <= s ? t : s;
            if (i >= na || j >= nb)
                continue;
            const int64_t r0 = i * pa, rows = std::min(pa, M - r0), c0 = j * pb, cols = std::min(pb, N - c0);
            if (cudaStreamWaitEvent(stream, ev_a[i], 0) != cudaSuccess ||
                cudaStreamWaitEvent(stream, ev_b[j], 0) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            const Problem q{dA + r0 * K, dB + c0 * K, dOut + r0 * N + c0, rows, cols, K, K, K, N, 1, 0, 0, 0};
            gemm_status_t st = run(q, GEMM_PATH_AUTO, stream);
            if (st != GEMM_OK)
                return st;
            if (cudaEventRecord(ev_o[k], stream) != cudaSuccess || cudaStreamWaitEvent(d.d2h, ev_o[k], 0) != cudaSuccess ||
                cudaMemcpy2DAsync(Out_host + r0 * N + c0, N * sizeof(float), dOut + r0 * N + c0, N * sizeof(float),
                                  cols * sizeof(float), rows, cudaMemcpyDeviceToHost, d.d2h) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            ++k;
        }
    }
    if (cudaEventRecord(ev_done, d.d2h) != cudaSuccess || cudaStreamWaitEvent(stream, ev_done, 0) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

gemm_status_t from_host_pipelined(const void* A_host, const void* B_host, float* Out_host, uint16_t* dA,
                                  uint16_t* dB, float* dOut, int64_t M, int64_t N, int64_t K, int64_t batch,
                                  cudaStream_t stream)
{
    DeviceState* d = nullptr;
    gemm_status_t st = device_state(&d);
    if (st != GEMM_OK)
        return st;
    if (!d->pipe_ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(d->pipe_mu);
        if (!d->pipe_ready.load(std::memory_order_relaxed)) {
            cudaError_t e = d->h2d ? cudaSuccess : cudaStreamCreateWithFlags(&d->h2d, cudaStreamNonBlocking);
            if (e == cudaSuccess && !d->d2h) e = cudaStreamCreateWithFlags(&d->d2h, cudaStreamNonBlocking);
            for (auto& ev : d->ev)
                if (e == cudaSuccess && !ev) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            d->pipe_ready.store(true, std::memory_order_release);
        }
    }
    if (batch == 1 && M >= 2048 && N >= 2048 && K > 0)
        return from_host_blocks(A_host, B_host, Out_host, dA, dB, dOut, M, N, K, *d, stream);
    // chunks: [first, first + count) of batches, or of rows when batch == 1
    const bool by_rows = batch == 1;
    const int64_t units = by_rows ? M : batch;
    int64_t per = units;
    if (by_rows && M >= 1024)
        per = std::max<int64_t>(256, ((M + kPipeChunks - 1) / kPipeChunks + 255) / 256 * 256);
    else if (!by_rows)
        per = (batch + kPipeChunks - 1) / kPipeChunks;
    const int nchunks = static_cast<int>((units + per - 1) / per);
    const uint8_t* ha = static_cast<const uint8_t*>(A_host);
    const uint8_t* hb = static_cast<const uint8_t*>(B_host);
    uint8_t* ho = reinterpret_cast<uint8_t*>(Out_host);

    std::lock_guard<std::mutex> lock(d->pipe_mu);  // the events are shared by calls on this device
    cudaEvent_t ev_start = d->ev[0], ev_done = d->ev[1];
    cudaEvent_t* ev_in = d->ev + 2;
    cudaEvent_t* ev_out = d->ev + 2 + kPipeChunks;
    if (cudaEventRecord(ev_start, stream) != cudaSuccess || cudaStreamWaitEvent(d->h2d, ev_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(d->d2h, ev_start, 0) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    const size_t a_unit = static_cast<size_t>(by_rows ? K : M * K) * 2;  // bytes per row / per batch of A
    const size_t b_unit = static_cast<size_t>(N * K) * 2;                // bytes per batch of B
    const size_t o_unit = static_cast<size_t>(by_rows ? N : M * N) * 4;
    if (by_rows && K > 0 && cudaMemcpyAsync(dB, hb, b_unit, cudaMemcpyHostToDevice, d->h2d) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    for (int c = 0; c < nchunks; ++c) {
        const int64_t first = c * per, count = std::min(per, units - first);
        if (K > 0) {
            if (cudaMemcpyAsync(reinterpret_cast<uint8_t*>(dA) + first * a_unit, ha + first * a_unit, count * a_unit,
                                cudaMemcpyHostToDevice, d->h2d) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            if (!by_rows && cudaMemcpyAsync(reinterpret_cast<uint8_t*>(dB) + first * b_unit, hb + first * b_unit,
                                            count * b_unit, cudaMemcpyHostToDevice, d->h2d) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
        }
        if (cudaEventRecord(ev_in[c], d->h2d) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
    }
    for (int c = 0; c < nchunks; ++c) {
        const int64_t first = c * per, count = std::min(per, units - first);
        if (cudaStreamWaitEvent(stream, ev_in[c], 0) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        Problem q = by_rows ? Problem{dA + first * K, dB, dOut + first * N, count, N, K, K, K, N, 1, 0, 0, 0}
                            : Problem{dA + first * M * K, dB + first * N * K, dOut + first * M * N, M, N, K, K, K, N,
                                      count, M * K, N * K, M * N};
        st = run(q, GEMM_PATH_AUTO, stream);
        if (st != GEMM_OK)
            return st;
        if (cudaEventRecord(ev_out[c], stream) != cudaSuccess || cudaStreamWaitEvent(d->d2h, ev_out[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(ho + first * o_unit, reinterpret_cast<uint8_t*>(dOut) + first * o_unit, count * o_unit,
                            cudaMemcpyDeviceToHost, d->d2h) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
    }
    if (cudaEventRecord(ev_done, d->d2h) != cudaSuccess || cudaStreamWaitEvent(stream, ev_done, 0) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

}  // namespace

// The CTA-pair kernel with its split scratch taken from memory the caller of
// this function owns (no allocation): arguments are checked before any CUDA
// call, then `scratch` gives the current device's fixed scratch, and the work
// is planned and launched by run_tc05_pair, as on the automatic path.
int run_pair_no_alloc(const void* A, const void* B, float* Out, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldo, int64_t strideA, int64_t strideB, int64_t strideO, int64_t batch,
                      PairScratchFn scratch, cudaStream_t stream)
{
    const Problem q{A, B, Out, M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    gemm_status_t st = validate(q);
    if (st != GEMM_OK)
        return st;
    if (q.M == 0 || q.N == 0 || q.batch == 0)
        return GEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != GEMM_OK)
        return st;
    PairScratch fixed{};
    st = static_cast<gemm_status_t>(scratch(&fixed));
    if (st != GEMM_OK)
        return st;
    if (q.K == 0)
        return zero_out(q, stream);
    if (!tma_ok(q) || d->max_pairs < 1)
        return GEMM_ERR_NOT_SUPPORTED;
    return run_tc05_pair(q, *d, stream, &fixed);
}

}  // namespace gnt

using gnt::Problem;

extern "C" {

gemm_status_t gemm_nt_f16_f32(const void* A, const void* B, float* Out, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldo, gemm_stream_t stream)
{
    Problem q{A, B, Out, M, N, K, lda, ldb, ldo, 1, 0, 0, 0};
    return gnt::run(q, GEMM_PATH_AUTO, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_nt_f16_f32_batched(const void* A, const void* B, float* Out, int64_t M, int64_t N, int64_t K,
                                      int64_t lda, int64_t ldb, int64_t ldo, int64_t strideA, int64_t strideB,
                                      int64_t strideO, int64_t batch, gemm_stream_t stream)
{
    Problem q{A, B, Out, M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    return gnt::run(q, GEMM_PATH_AUTO, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_nt_f16_f32_batched_path(const void* A, const void* B, float* Out, int64_t M, int64_t N,
                                           int64_t K, int64_t lda, int64_t ldb, int64_t ldo, int64_t strideA,
                                           int64_t strideB, int64_t strideO, int64_t batch, gemm_path_t path,
                                           gemm_stream_t stream)
{
    Problem q{A, B, Out, M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    return gnt::run(q, path, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_nt_batched_ex(const void* A, const void* B, void* Out, gemm_dtype_t ab_type, gemm_dtype_t out_type,
                                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldo, int64_t strideA,
                                 int64_t strideB, int64_t strideO, int64_t batch, gemm_path_t path,
                                 gemm_stream_t stream)
{
    Problem q{A, B, Out, M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    q.ab_type = static_cast<int>(ab_type);
    q.out_type = static_cast<int>(out_type);
    return gnt::run(q, path, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_nt_batched_major(const void* A, gemm_major_t a_major, const void* B, gemm_major_t b_major,
                                    void* Out, gemm_dtype_t ab_type, gemm_dtype_t out_type, int64_t M, int64_t N,
                                    int64_t K, int64_t lda, int64_t ldb, int64_t ldo, int64_t strideA, int64_t strideB,
                                    int64_t strideO, int64_t batch, gemm_path_t path, gemm_stream_t stream)
{
    Problem q{A, B, Out, M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    q.ab_type = static_cast<int>(ab_type);
    q.out_type = static_cast<int>(out_type);
    q.a_major = static_cast<int>(a_major);
    q.b_major = static_cast<int>(b_major);
    return gnt::run(q, path, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_nt_mx(const void* A, const void* SA, const void* B, const void* SB, void* Out,
                         gemm_dtype_t ab_type, gemm_dtype_t out_type, int64_t M, int64_t N, int64_t K, int64_t lda,
                         int64_t ldb, int64_t ldo, int64_t strideA, int64_t strideB, int64_t strideO, int64_t batch,
                         gemm_path_t path, gemm_stream_t stream)
{
    if (K > 0 && M > 0 && N > 0 && batch > 0 && (!SA || !SB))
        return GEMM_ERR_INVALID_VALUE;
    Problem q{A, B, Out, M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    q.ab_type = static_cast<int>(ab_type);
    q.out_type = static_cast<int>(out_type);
    q.SA = SA;
    q.SB = SB;
    if (!q.is_f8())
        return GEMM_ERR_INVALID_VALUE;
    return gnt::run(q, path, reinterpret_cast<cudaStream_t>(stream));
}

int64_t gemm_nt_mx_scale_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0)
        return -1;
    return gnt::mx_scale_bytes(rows, K);
}

gemm_status_t gemm_nt_mx_pack_scales(const void* plain, int64_t ld, int64_t stride, void* packed, int64_t rows,
                                     int64_t K, int64_t batch, gemm_stream_t stream)
{
    if (rows < 0 || K < 0 || batch < 0 || ld < 0 || stride < 0)
        return GEMM_ERR_INVALID_VALUE;
    if (rows == 0 || K == 0 || batch == 0)
        return GEMM_OK;
    const int64_t kb = (K + 31) / 32;
    if (!plain || !packed || ld < kb || (batch > 1 && stride != 0 && stride < (rows - 1) * ld + kb))
        return GEMM_ERR_INVALID_VALUE;
    if (rows > INT32_MAX || K > INT32_MAX || batch > INT32_MAX)
        return GEMM_ERR_INVALID_VALUE;
    gnt::DeviceState* d = nullptr;
    gemm_status_t st = gnt::device_state(&d);
    if (st != GEMM_OK)
        return st;
    return gnt::mx_pack_launch(static_cast<const uint8_t*>(plain), ld, stride, static_cast<uint8_t*>(packed), rows, K,
                               batch, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_LAUNCH;
}

gemm_status_t gemm_nt_f16_f32_from_host(const void* A_host, const void* B_host, float* Out_host, void* dA,
                                        void* dB, float* dOut, int64_t M, int64_t N, int64_t K, int64_t batch,
                                        gemm_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0 || batch < 0)
        return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0 || batch == 0)
        return GEMM_OK;
    if (!Out_host || !dOut || (K > 0 && (!A_host || !B_host || !dA || !dB)))
        return GEMM_ERR_INVALID_VALUE;
    Problem q{dA, dB, dOut, M, N, K, K, K, N, batch, M * K, N * K, M * N};
    gemm_status_t st = gnt::validate(q);
    if (st != GEMM_OK)
        return st;
    return gnt::from_host_pipelined(A_host, B_host, Out_host, static_cast<uint16_t*>(dA), static_cast<uint16_t*>(dB),
                                    dOut, M, N, K, batch, reinterpret_cast<cudaStream_t>(stream));
}

gemm_path_t gemm_nt_select_path(const void* A, const void* B, const float* Out, int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldb, int64_t ldo, int64_t strideA, int64_t strideB,
                                int64_t strideO, int64_t batch)
{
    Problem q{A, B, const_cast<float*>(Out), M, N, K, lda, ldb, ldo, batch, strideA, strideB, strideO};
    return gnt::select_path(q);
}

gemm_status_t gemm_nt_check(gemm_stream_t stream)
{
    gnt::DeviceState* d = nullptr;
    gemm_status_t st = gnt::device_state(&d);
    if (st != GEMM_OK)
        return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    uint32_t word = 0;
    if (cudaMemcpy(&word, d->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    if (word) {
        const uint32_t zero = 0;
        if (cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        gnt::reset_workspaces();
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

const char* gemm_nt_error_string(gemm_status_t status)
{
    switch (status) {
    case GEMM_OK: return "success";
    case GEMM_ERR_INVALID_VALUE: return "invalid argument";
    case GEMM_ERR_MISALIGNED: return "misaligned operand (reserved: never returned)";
    case GEMM_ERR_OVERLAP: return "output overlaps an input or itself";
    case GEMM_ERR_LAUNCH: return "CUDA runtime or driver call failed";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_NOT_SUPPORTED: return "the requested kernel cannot take these arguments";
    case GEMM_ERR_SCRATCH_TOO_SMALL:
        return "the call needs more scratch than the no-allocation entry point's fixed array holds";
    }
    return "unknown status";
}

gemm_status_t gemm_nt_probe_m16n8k16(const void* A, const void* B, uint32_t* ar, uint32_t* br, float* dr,
                                     gemm_stream_t stream)
{
    if (!A || !B || !ar || !br || !dr)
        return GEMM_ERR_INVALID_VALUE;
    if (!gnt::aligned(A, 2) || !gnt::aligned(B, 2) || !gnt::aligned(ar, 4) || !gnt::aligned(br, 4) ||
        !gnt::aligned(dr, 4))
        return GEMM_ERR_INVALID_VALUE;
    gnt::DeviceState* d = nullptr;
    gemm_status_t st = gnt::device_state(&d);
    if (st != GEMM_OK)
        return st;
    return gnt::probe_launch(static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), ar, br, dr,
                             reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_LAUNCH;
}

void gemm_nt_debug_set_wait_limit(uint64_t cycles) { gnt::g_wait_limit.store(cycles); }

void gemm_nt_debug_set_fault(int fault) { gnt::g_fault.store(fault); }

}  // extern "C"
