/*
 * gemm_nt.h -- C ABI of the GB300 (sm_103a) fp16 -> fp32 matrix product
 *
 *     Out = A @ B.T
 *
 * with A (M,K) and B (N,K) row-major IEEE binary16, Out (M,N) row-major float32,
 * float32 accumulation.  This is the product computed by the two worked examples
 * of the Apache TVM TIRx programming guides: "Warp Matrix Instructions" (opening
 * paragraph and "From Shared Memory to a Matrix Product": A (16,16), B (8,16),
 * ldmatrix + mma.sync m16n8k16, fp32 accumulators) and "Blackwell Tensor Cores"
 * ("The Accumulator's Lifetime": A (128,64), B (64,64), tcgen05.mma kind::f16
 * with the fp32 accumulator in Tensor Memory).  Both examples start a fresh
 * accumulator (C = 0, accum=False), so Out is overwritten: there is no alpha,
 * beta or C input.
 *
 * The pages run each kernel as compiled(a, b, out) on torch CUDA tensors (the
 * listings that compile the kernel and compare it with torch, in "Warp Matrix
 * Instructions" and "Blackwell Tensor Cores") and define no C interface.  The
 * entry points here take that call's three operands as device pointers, in the
 * same order (A, B, Out), followed by the sizes, the leading dimensions, the
 * batch strides and batch count where there are any, and the stream.  Status
 * codes 0-6 are those of the plain and batched products; 7 and 8 belong to the
 * entry points that choose a kernel or allocate nothing.
 *
 * Conventions shared by every entry point
 *   - Pointers A, B, Out are DEVICE pointers owned by the caller.  A and B hold
 *     fp16 bit patterns (__half / uint16_t).  The library keeps no reference to
 *     them after the call's work has run.
 *   - Sizes and leading dimensions are in ELEMENTS; rows are contiguous:
 *       A[i,k] = A[i*lda + k],  B[j,k] = B[j*ldb + k],  Out[i,j] = Out[i*ldo + j].
 *     Batched forms add b*strideA, b*strideB, b*strideO elements for batch b.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t / CUstream;
 *     NULL = the legacy default stream).  Argument errors are detected on the
 *     host, return immediately and launch nothing.
 *   - Empty cases: M == 0, N == 0 or batch == 0 -> GEMM_OK, nothing launched.
 *     K == 0 -> Out is filled with zeros (the empty sum).
 *   - Any alignment is accepted.  The tensor-core kernels need 16-byte aligned
 *     A/B bases and lda, ldb (and strideA, strideB) multiples of 8 elements;
 *     other inputs run on the warp-MMA kernel, which accepts any layout.
 *   - Device-side failures (a bounded wait inside a kernel that ran out) are
 *     recorded in a per-device status word and reported by gemm_nt_check().
 *   - Thread safety: all entry points may be called concurrently from several
 *     host threads.  Calls whose Out ranges overlap must not run concurrently.
 *   - Only devices of compute capability 10.3 (GB300, sm_103a) are supported.
 *   - Per-device set-up (kernel attributes, the status word's address) is done
 *     once, by the first call on a device that passes the argument checks (a
 *     set-up that failed is tried again by the next call), and kept for the
 *     life of the process: after cudaDeviceReset() on a device, make no further
 *     call on that device.
 */
#ifndef GEMM_NT_H
#define GEMM_NT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t and CUstream. */
struct CUstream_st;
typedef struct CUstream_st *gemm_stream_t;

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,      /* null pointer, negative size, ld < row length, ... */
    GEMM_ERR_MISALIGNED = 2,         /* reserved, never returned: layouts the tensor-core kernels
                                        cannot read run on the warp-MMA kernel instead */
    GEMM_ERR_OVERLAP = 3,            /* Out overlaps A or B, or batches of Out overlap */
    GEMM_ERR_LAUNCH = 4,             /* a CUDA runtime/driver call failed (launch, tensor map,
                                        synchronisation, per-device set-up) */
    GEMM_ERR_DEVICE_TIMEOUT = 5,     /* a kernel's bounded wait ran out; Out is undefined */
    GEMM_ERR_UNSUPPORTED_DEVICE = 6, /* current device is not compute capability 10.3 */
    /* Codes 7 and 8 belong to entry points beyond the plain and batched products: */
    GEMM_ERR_NOT_SUPPORTED = 7,      /* the requested kernel cannot take these arguments */
    GEMM_ERR_SCRATCH_TOO_SMALL = 8   /* gemm_nt_f16_f32_batched_no_alloc: the call needs more
                                        scratch than the library's fixed array holds */
} gemm_status_t;

/* Element types of gemm_nt_batched_ex. */
typedef enum gemm_dtype {
    GEMM_DTYPE_F16 = 0,  /* IEEE binary16 */
    GEMM_DTYPE_BF16 = 1, /* bfloat16: the upper half of an IEEE binary32 */
    GEMM_DTYPE_F32 = 2,  /* IEEE binary32 (Out only) */
    GEMM_DTYPE_E4M3 = 3, /* 8-bit float, 4 exponent bits (bias 7), 3 fraction bits, no infinities,
                            largest value 448 (A and B only) */
    GEMM_DTYPE_E5M2 = 4, /* 8-bit float, 5 exponent bits (bias 15), 2 fraction bits: the upper byte
                            of an IEEE binary16 (A and B only) */
    /* 6- and 4-bit floats (A and B only), no infinities or NaN, packed along K with
       little-endian bit order: element k of a row occupies bits [b*k, b*k + b) of the
       row's bit string (b = 6 or 4; byte i holds bits [8i, 8i + 8)), so fp4 holds
       element 2t in the low nibble of byte t and element 2t+1 in its high nibble: */
    GEMM_DTYPE_E2M3 = 5, /* sign bit 5, 2 exponent bits (bias 1), 3 fraction bits; largest 7.5 */
    GEMM_DTYPE_E3M2 = 6, /* sign bit 5, 3 exponent bits (bias 3), 2 fraction bits; largest 28 */
    GEMM_DTYPE_E2M1 = 7  /* sign bit 3, 2 exponent bits (bias 1), 1 fraction bit; largest 6 */
} gemm_dtype_t;

/* Kernel choice.  GEMM_PATH_AUTO lets the library pick (see gemm_nt_select_path). */
typedef enum gemm_path {
    GEMM_PATH_AUTO = 0,
    GEMM_PATH_TC05 = 1,     /* persistent tcgen05 kernel, TMEM accumulator, one CTA per tile */
    GEMM_PATH_SKINNY = 2,   /* tcgen05 with swapped operands and split K, for small M */
    GEMM_PATH_MMASYNC = 3,  /* ldmatrix + mma.sync m16n8k16 warp kernel, any layout */
    GEMM_PATH_TC05_PAIR = 4, /* tcgen05 on a CTA pair (cta_group::2), 256-row tiles */
    GEMM_PATH_TC05_M64 = 5,  /* one CTA per 64-row tile, plain M = 64 tcgen05.mma (few rows of A) */
    GEMM_PATH_TC05_WS = 6    /* one CTA per 32- or 64-row tile, weight-stationary tcgen05.mma.ws
                                (M = 32 when M <= 32, else 64) */
} gemm_path_t;

/*
 * Out = A @ B.T for one problem.
 *   A   : M x K, leading dimension lda >= K
 *   B   : N x K, leading dimension ldb >= K
 *   Out : M x N float32, leading dimension ldo >= N; must not overlap A or B.
 * Returns GEMM_OK once the work is enqueued on `stream`.
 */
gemm_status_t gemm_nt_f16_f32(const void *A, const void *B, float *Out,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldo,
                              gemm_stream_t stream);

/*
 * Strided batch of independent products: for b < batch,
 *   Out_b = A_b @ B_b.T,  A_b = A + b*strideA,  B_b = B + b*strideB,  Out_b = Out + b*strideO.
 * strideA or strideB may be 0 (the operand is shared by every batch); strideO
 * must separate the batches of Out (strideO >= (M-1)*ldo + N when batch > 1).
 */
gemm_status_t gemm_nt_f16_f32_batched(const void *A, const void *B, float *Out,
                                      int64_t M, int64_t N, int64_t K,
                                      int64_t lda, int64_t ldb, int64_t ldo,
                                      int64_t strideA, int64_t strideB, int64_t strideO,
                                      int64_t batch, gemm_stream_t stream);

/*
 * As gemm_nt_f16_f32_batched, on an explicitly chosen kernel.  Returns
 * GEMM_ERR_NOT_SUPPORTED (and launches nothing) if that kernel cannot take the
 * arguments, e.g. a tensor-core path with unaligned A.  GEMM_PATH_TC05_M64 and
 * GEMM_PATH_TC05_WS ("Blackwell Tensor Cores" names the M = 64 and the
 * weight-stationary tcgen05.mma forms beside its 128-row example) put 64 rows
 * of A (32 on the weight-stationary form when M <= 32) on each tile's MMA
 * side; they take the same inputs as GEMM_PATH_TC05 except block scales and
 * an MN-major A (GEMM_ERR_NOT_SUPPORTED).  GEMM_PATH_AUTO never picks them.
 * A path value outside gemm_path_t: GEMM_ERR_INVALID_VALUE.
 */
gemm_status_t gemm_nt_f16_f32_batched_path(const void *A, const void *B, float *Out,
                                           int64_t M, int64_t N, int64_t K,
                                           int64_t lda, int64_t ldb, int64_t ldo,
                                           int64_t strideA, int64_t strideB, int64_t strideO,
                                           int64_t batch, gemm_path_t path,
                                           gemm_stream_t stream);

/*
 * The strided batched product with other element types: A and B both fp16 or
 * both bf16 ("Warp Matrix Instructions", "Other Fragment Shapes and
 * Transfers", names the float16 and bfloat16 forms of the warp MMA; the
 * tcgen05 kind::f16 MMA of "Blackwell Tensor Cores" takes either), products
 * accumulated in fp32 as always, and Out stored as fp32, or rounded to nearest
 * even into fp16 or bf16 (Out's element size is then 2 bytes; ldo and strideO
 * still count elements).  Same conventions, layouts and error behaviour as
 * gemm_nt_f16_f32_batched_path; gemm_nt_f16_f32_batched_path(...) equals
 * gemm_nt_batched_ex(..., GEMM_DTYPE_F16, GEMM_DTYPE_F32, ...).  An fp16 Out
 * overflows to infinity beyond 65504.  Products that would split K across CTAs
 * (few output tiles, long K) run on whole tiles when Out is not fp32, since
 * the partial sums are kept in fp32 only.
 *
 * A and B may also both be 8-bit floats (E4M3 or E5M2; lda, ldb and the batch
 * strides then count bytes), or both one of the 6- and 4-bit floats E2M3,
 * E3M2, E2M1, packed along K (lda, ldb and the batch strides count elements
 * and must start every row on a byte: multiples of 2 for E2M1, of 4 for the
 * 6-bit types; K-major only, else GEMM_ERR_INVALID_VALUE).  The packed types run
 * on the tcgen05 kernels only (kind::f8f6f4, whose tensor maps spread every 16
 * packed elements to a 16-byte chunk of shared memory), which need K a
 * multiple of 128, A and B 32-byte aligned, and pitches and batch strides of
 * whole multiples of 32 bytes; other layouts, and the warp kernel path, give
 * GEMM_ERR_NOT_SUPPORTED.  "Blackwell Tensor Cores" names the block-scaled
 * low-precision forms of the tcgen05 MMA beside kind::f16; these run on its
 * kind::f8f6f4 form without scale factors (products exact, fp32 accumulation),
 * at twice the fp16 rate.  The tensor-core kernels want 16-byte aligned bases
 * and pitches that are multiples of 16; other layouts, and MN-major 8-bit
 * operands (gemm_nt_batched_major), run on the warp kernel, which widens the
 * 8-bit values to fp16 (exact).  Any other dtype value: GEMM_ERR_INVALID_VALUE.
 */
gemm_status_t gemm_nt_batched_ex(const void *A, const void *B, void *Out,
                                 gemm_dtype_t ab_type, gemm_dtype_t out_type,
                                 int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldo,
                                 int64_t strideA, int64_t strideB, int64_t strideO,
                                 int64_t batch, gemm_path_t path, gemm_stream_t stream);

/* Storage order of one operand of gemm_nt_batched_major.  The operand is the
 * logical (rows, K) matrix of the product (A: rows = M; B: rows = N).
 *   GEMM_MAJOR_K : element (r, k) at base[r*ld + k], ld >= K  -- row-major (rows, K),
 *                  the layout of every other entry point;
 *   GEMM_MAJOR_MN: element (r, k) at base[k*ld + r], ld >= rows -- row-major (K, rows),
 *                  i.e. the operand's transpose stored row-major. */
typedef enum gemm_major {
    GEMM_MAJOR_K = 0,
    GEMM_MAJOR_MN = 1
} gemm_major_t;

/*
 * The product Out[b] = A[b] @ B[b].T with each operand stored K-major or
 * MN-major: with B MN-major, B is given as a row-major (K, N) matrix and the
 * call computes the plain row-major product A @ B ("NN"); with A MN-major too,
 * A is given as (K, M) and the call computes A.T @ B ("TN").  "Warp Matrix
 * Instructions" ("Other Fragment Shapes and Transfers") names ldmatrix's
 * .trans form, and "copy -> ldstmatrix" ("Algorithm" step 3) selects it for a
 * column-major shared tile whose column stride is a multiple of 8 elements:
 * the warp kernel stages an MN-major operand that way.  The tcgen05 kernels
 * (the pages show them K-major only) read it through the instruction
 * descriptor's transpose bit and an MN-major 128-byte-swizzled shared-memory
 * descriptor, as the PTX ISA defines them.
 *
 * Arguments as gemm_nt_batched_ex, plus a_major and b_major; lda and ldb are
 * the row pitches of the stored matrices (ld >= K for K-major, ld >= M or N
 * for MN-major) and strideA / strideB the batch strides, all in elements.
 * gemm_nt_batched_ex(...) equals this call with both operands GEMM_MAJOR_K.
 * The tensor-core kernels need 16-byte aligned A/B bases and ld, strides that
 * are multiples of 8 elements (else the warp kernel runs, as for K-major).
 * An MN-major operand on the CTA-pair kernel always uses 256-wide tiles, and
 * the skinny kernel's row split (an even share of rows per CTA) is K-major
 * only.  Any other major value: GEMM_ERR_INVALID_VALUE.
 */
gemm_status_t gemm_nt_batched_major(const void *A, gemm_major_t a_major, const void *B,
                                    gemm_major_t b_major, void *Out,
                                    gemm_dtype_t ab_type, gemm_dtype_t out_type,
                                    int64_t M, int64_t N, int64_t K,
                                    int64_t lda, int64_t ldb, int64_t ldo,
                                    int64_t strideA, int64_t strideB, int64_t strideO,
                                    int64_t batch, gemm_path_t path, gemm_stream_t stream);

/*
 * Block-scaled 8-bit product ("Blackwell Tensor Cores", on the other TMEM
 * operations: tcgen05.cp brings the scale factors of a block-scaled MMA into
 * Tensor Memory; the MMA reference it points to lists block scaling).  A and B
 * are E4M3, E5M2, E2M3, E3M2 or E2M1 (both the same), K-major, as in
 * gemm_nt_batched_ex; every
 * run of 32 consecutive K elements of a row of A (of B) shares one scale, an
 * E8M0 byte e standing for 2^(e-127) (255 is NaN), and
 *   Out[b,i,j] = sum_k (A[b,i,k] * 2^(sa[b,i,k/32]-127)) * (B[b,j,k] * 2^(sb[b,j,k/32]-127))
 * accumulated in fp32 on the tcgen05 kind::mxf8f6f4 MMA, Out fp32, fp16 or
 * bf16.
 *
 * SA and SB hold the scales in the packed atom layout (device memory, 16-byte
 * aligned): for each 128 rows and each 128 elements of K one 512-byte atom
 * whose byte 16*r + 4*q + s is the scale of row 32*q + r of the row block, K
 * block s of the K block group; atoms stored row block-major, so atom
 * (rb, kg) is at byte (rb * ceil(K/128) + kg) * 512; rows and K blocks past
 * the matrix are ignored (any value but 255).  One matrix of scales takes
 * gemm_nt_mx_scale_bytes(rows, K) bytes; the matrices of a batch follow one
 * another, except that an operand with batch stride 0 (shared by every batch)
 * has one matrix of scales.  gemm_nt_mx_pack_scales makes this layout from
 * the plain one.
 *
 * path: GEMM_PATH_AUTO, GEMM_PATH_TC05 (128 x 64 or 128 x 128 tiles),
 * GEMM_PATH_SKINNY (M <= 64) or GEMM_PATH_TC05_PAIR (256 x 256 tiles on CTA
 * pairs when Out rows are 32-byte aligned and K is not split, else 256 x 192);
 * AUTO takes SKINNY for M <= 64 and N >= 1024, the pairs for M and N
 * above 128, else TC05.  The warp kernel takes no scales
 * (GEMM_ERR_NOT_SUPPORTED), nor does any kernel a layout the tensor-core
 * kernels cannot read (unaligned bases, pitches not multiples of 16 bytes).  Null SA / SB with K > 0, a 16-bit ab_type, or
 * unaligned SA / SB: GEMM_ERR_INVALID_VALUE; Out overlapping A, B, SA or SB:
 * GEMM_ERR_OVERLAP.  Other arguments and errors as gemm_nt_batched_ex.
 */
gemm_status_t gemm_nt_mx(const void *A, const void *SA, const void *B, const void *SB, void *Out,
                         gemm_dtype_t ab_type, gemm_dtype_t out_type,
                         int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldo,
                         int64_t strideA, int64_t strideB, int64_t strideO,
                         int64_t batch, gemm_path_t path, gemm_stream_t stream);

/* Bytes of one packed scale matrix for `rows` rows and K elements of K:
 * ceil(rows/128) * ceil(K/128) * 512; -1 for negative arguments. */
int64_t gemm_nt_mx_scale_bytes(int64_t rows, int64_t K);

/*
 * Packs block scales on the device: `plain` holds, for each of `batch`
 * matrices (batch stride `stride` bytes, 0 = one shared matrix), `rows` rows of
 * ceil(K/32) E8M0 bytes with row pitch `ld` bytes (ld >= ceil(K/32));
 * `packed` receives batch * gemm_nt_mx_scale_bytes(rows, K) bytes in the
 * layout gemm_nt_mx reads (padding atoms filled with 127).  Stream-ordered;
 * GEMM_ERR_INVALID_VALUE for null pointers or pitches too small.
 */
gemm_status_t gemm_nt_mx_pack_scales(const void *plain, int64_t ld, int64_t stride, void *packed,
                                     int64_t rows, int64_t K, int64_t batch, gemm_stream_t stream);

/*
 * Host-side pipeline for callers whose data lives in host memory: copies A and
 * B (packed: lda = ldb = K, strideA = M*K, strideB = N*K) from host to the
 * caller's device buffers dA, dB, runs the batched product into dOut (packed,
 * ldo = N, strideO = M*N) and copies dOut back to host Out.  The work is cut
 * into up to sixteen chunks (row blocks of A and Out when batch == 1, groups of
 * batches otherwise) so that copies in both directions overlap the products:
 * inputs travel on a library-owned copy stream, each chunk's product runs on
 * `stream` once its inputs have arrived, and its Out travels back on a second
 * library-owned stream; `stream` finally waits for the last copy, so
 * synchronising `stream` is enough before reading Out.  For the copies to be
 * asynchronous the host buffers must be pinned.  No device memory is
 * allocated; the two copy streams and ten events are created once per device,
 * on the first call (make that first call outside any stream capture).  Calls
 * on one device are enqueued one at a time (an internal lock).
 */
gemm_status_t gemm_nt_f16_f32_from_host(const void *A_host, const void *B_host, float *Out_host,
                                        void *dA, void *dB, float *dOut,
                                        int64_t M, int64_t N, int64_t K, int64_t batch,
                                        gemm_stream_t stream);

/*
 * Same product as gemm_nt_f16_f32_batched, for callers that must not allocate
 * device memory.  (The source pages have no counterpart to this entry point;
 * it exists for users of this library.)  Code running inside CUDA stream
 * capture may not call cudaMalloc, applications whose device memory is owned by
 * their own pool allocator may forbid any other allocation, and latency-
 * critical code cannot afford an allocation on its first call - yet the
 * automatic path allocates a workspace (about 38 MB per stream, once) when it
 * splits a problem with few output tiles and a long K across the GPU.
 *
 * This entry point always runs the CTA-pair tensor-core kernel (so A and B
 * must meet the tensor-core alignment rule, else GEMM_ERR_NOT_SUPPORTED) and
 * plans the split exactly as the automatic path does, but takes its scratch
 * from one fixed array inside the library: 8 MiB for the partial results of
 * up to 16 CTA pairs plus 4 KiB of counters for up to 64 split tiles.  Every
 * GPU that loads the library holds that array until the process exits.  A call
 * whose split would need more (a problem of 5 to about 37 tiles of 256 x 256
 * with K >= 6144 on a 152-SM GB300) returns GEMM_ERR_SCRATCH_TOO_SMALL and
 * launches nothing; problems that are not split use no scratch at all.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Argument
 * errors are returned before any CUDA call, as for every entry point.  The
 * first call on a device whose arguments pass the checks (and are not empty)
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  A lookup that
 * failed is tried again on the next call.  The address is kept for the life of
 * the process, so after cudaDeviceReset() on a device make no further call on
 * it.  Before each split launch the counters are cleared on `stream`
 * (cudaMemsetAsync, which allocates nothing).  All calls share the one array:
 * calls that may overlap on the GPU (different streams, or several host threads
 * without ordering) race on it and give wrong results, so order them on one
 * stream.
 */
gemm_status_t gemm_nt_f16_f32_batched_no_alloc(const void *A, const void *B, float *Out,
                                               int64_t M, int64_t N, int64_t K,
                                               int64_t lda, int64_t ldb, int64_t ldo,
                                               int64_t strideA, int64_t strideB, int64_t strideO,
                                               int64_t batch, gemm_stream_t stream);

/*
 * The kernel GEMM_PATH_AUTO would choose for these arguments (host-only: reads
 * no device state and makes no CUDA call).  Pointers are used only for their
 * alignment.
 */
gemm_path_t gemm_nt_select_path(const void *A, const void *B, const float *Out,
                                int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldb, int64_t ldo,
                                int64_t strideA, int64_t strideB, int64_t strideO,
                                int64_t batch);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: GEMM_ERR_DEVICE_TIMEOUT if any kernel launched since the last check hit
 * its bounded-wait limit, GEMM_ERR_LAUNCH if the synchronisation failed, else GEMM_OK.
 */
gemm_status_t gemm_nt_check(gemm_stream_t stream);

/* Static, human-readable text for a status code ("unknown status" for a value
 * outside gemm_status_t).  Never NULL. */
const char *gemm_nt_error_string(gemm_status_t status);

/*
 * Diagnostic: one warp executes the warp example of "Warp Matrix Instructions"
 * ("From Shared Memory to a Matrix Product") on device inputs A (16x16, row-
 * major fp16) and B (8x16): stage to shared memory, ldmatrix.x4 / .x2, one
 * mma.sync m16n8k16 with C = 0.  It writes the raw per-lane registers to device
 * buffers ar (32x4 uint32), br (32x2 uint32), dr (32x4 float), lane-major, so
 * the fragment maps can be checked.
 */
gemm_status_t gemm_nt_probe_m16n8k16(const void *A, const void *B, uint32_t *ar, uint32_t *br,
                                     float *dr, gemm_stream_t stream);

/*
 * Test hooks for the bounded waits (not for production use).  Sets, for the
 * calling process, the wait limit in SM clock cycles of the tcgen05 kernels
 * (0 restores the default of about two seconds) and a fault to inject into the
 * next launches on CTA 0: 0 none, 1 the producer drops its first stage, 2 the
 * MMA thread skips its first stage release.  With a fault injected the kernel
 * gives up after the limit and gemm_nt_check() returns GEMM_ERR_DEVICE_TIMEOUT.
 */
void gemm_nt_debug_set_wait_limit(uint64_t cycles);
void gemm_nt_debug_set_fault(int fault);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_NT_H */
