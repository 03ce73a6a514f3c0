/*
 * w4a16.h -- C ABI of libw4a16, the W4A16 group-quantized linear layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (one weight-only int4 linear layer, activations in fp16/bf16):
 *
 *     y[m, n] = sum_k x[m, k] * (q[k, n] - z[k / g, n]) * s[k / g, n]
 *
 *   x   [M, K]    activations, fp16 or bf16, row-major
 *   q   [K, N]    4-bit weight codes 0..15, stored packed (see qweight)
 *   s   [K/g, N]  one scale per group of g rows of K and per column, same
 *                 dtype as x
 *   z   [K/g, N]  4-bit zero-points 0..15, stored packed (see qzeros); the
 *                 symmetric layer has no zero-point tensor and uses z = 8,
 *                 the "code - 8" recentring described on "qsa_prompt_attn:
 *                 Q4_0 KV on tensor cores" (section "What")
 *   y   [M, N]    output, same dtype as x, rounded to nearest-even from an
 *                 FP32 accumulator
 *
 * Packed layouts (words are read as uint32 bit patterns):
 *   qweight int32 [K/8, N]    nibble j (bits 4j..4j+3) of word [w, n] holds
 *                             q[8w + j, n]
 *   qzeros  int32 [K/g, N/8]  the zero-point of column n sits in word
 *                             [t, n/8] at bits 4*(n%8). This is the packed
 *                             zero-point layout of "Keep W4A16 zero-points
 *                             packed at 4 bits instead of expanding to 2
 *                             bytes" (section "Change"); that page's point is
 *                             that the kernel reads zero-points in this form,
 *                             0.5 byte per group and column, and never an
 *                             expanded activation-dtype copy of them.
 *
 * Conventions for every entry point below:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; tensors
 *     are dense and row-major. The library never allocates or frees device
 *     memory and never synchronises, except w4a16_device_status, which
 *     synchronises the given stream.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *   - All argument checks run on the host BEFORE anything is launched; a
 *     failed check returns an error status and launches nothing.
 *   - A launch error is returned as W4A16_ERR_CUDA. The library does not
 *     clear CUDA's sticky error state.
 *   - The library runs only on compute capability 10.3 (GB300); any other
 *     device gives W4A16_ERR_DEVICE.
 *   - Shape limits: N % 8 == 0, K % g == 0, g in {32, 64, 128, 256}, all
 *     dimensions > 0 and < 2^31, base pointers 16-byte aligned. Products of
 *     dimensions are not limited: every offset is computed in 64 bits, so
 *     tensors past 2^32 elements or 4 GiB are fine.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_ABI_VERSION 1

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_NULL = 1,        /* a required pointer is NULL                          */
    W4A16_ERR_SHAPE = 2,       /* a dimension is out of range or inconsistent         */
    W4A16_ERR_DTYPE = 3,       /* unknown activation dtype                            */
    W4A16_ERR_ALIGN = 4,       /* a base pointer is not 16-byte aligned               */
    W4A16_ERR_UNSUPPORTED = 5, /* valid request this build does not implement         */
    W4A16_ERR_DEVICE = 6,      /* no CUDA device, or not compute capability 10.3      */
    W4A16_ERR_WORKSPACE = 7,   /* workspace missing or smaller than required          */
    W4A16_ERR_CUDA = 8,        /* a CUDA runtime call or a launch failed              */
    W4A16_ERR_TIMEOUT = 9      /* a device-side pipeline wait ran out (see below)     */
} w4a16_status;

typedef enum {
    W4A16_F16 = 0,
    W4A16_BF16 = 1
} w4a16_dtype;

/* Same type as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* w4a16_stream;

/* Which kernel a workspace query is for. */
typedef enum {
    W4A16_OP_GEMV = 0,
    W4A16_OP_GEMM = 1
} w4a16_op;

/*
 * w4a16_pack -- pack 4-bit codes eight to a 32-bit word.
 *
 * src  uint8 [rows, cols]; only the low 4 bits of each byte are used.
 * dim  0: pack along rows -> dst int32 [rows/8, cols]; nibble j of word
 *         [w, c] is src[8w + j, c] (the qweight layout, rows = K);
 *      1: pack along cols -> dst int32 [rows, cols/8]; column c goes to word
 *         [r, c/8] at bits 4*(c%8) (the qzeros layout of "Keep W4A16
 *         zero-points packed at 4 bits instead of expanding to 2 bytes",
 *         section "Change", rows = K/g, cols = N).
 * The packed dimension must be a multiple of 8. Bit-exact; deterministic.
 * Errors: NULL, SHAPE (non-positive or not a multiple of 8), ALIGN (either
 * pointer not 16-byte aligned), DEVICE, CUDA.
 */
w4a16_status w4a16_pack(const uint8_t* src, int32_t* dst, int64_t rows, int64_t cols, int dim,
                        w4a16_stream stream);

/*
 * w4a16_unpack -- inverse of w4a16_pack. `rows`, `cols` and `dim` describe the
 * UNPACKED tensor dst uint8 [rows, cols] (values 0..15); src is the packed
 * int32 tensor of w4a16_pack's output shape. This is the inverse that the
 * zero-point page names as unpacking along the packed dimension. Errors as
 * for w4a16_pack.
 */
w4a16_status w4a16_unpack(const int32_t* src, uint8_t* dst, int64_t rows, int64_t cols, int dim,
                          w4a16_stream stream);

/*
 * w4a16_workspace_bytes -- bytes of device workspace `op` needs for this shape
 * on the current device. For the GEMV: the FP32 partial-sum slots of the
 * GEMV kernel (8 KB per SM), then those of the few-row tensor-core kernel
 * that w4a16_mxfp4_gemv runs for 5..16 rows of large layers (128 KB per SM;
 * both sizes depend only on the device), then the ticket words of whichever
 * kernel needs more for this shape (one per column block, or four per 128
 * columns; rounded up to 256 bytes). For the GEMM
 * with M <= 128: FP32 partial slots of 128 KB per SM, followed by four 32-bit
 * tickets per 128 columns (rounded up to 256 bytes); 0 for the GEMM with
 * M > 128. The same sizes serve w4a16_mxfp4_gemv and w4a16_mxfp4_gemm with
 * g = 32. Returns 0 for shapes the op rejects and when no GB300 is current.
 */
size_t w4a16_workspace_bytes(w4a16_op op, int64_t M, int64_t N, int64_t K, int64_t g);

/*
 * w4a16_gemv -- decode path, 1 <= M <= 16.
 *
 * One row (and two rows of a layer of at most 4 * 2^20 weights) is
 * converted with FP32 FMAs; 2..16 rows otherwise go through warp-level
 * m16n8k16 tensor-core MMAs: (q - z) formed exactly in 16 bits as the A
 * operand, x as B, FP32 accumulators scaled once per 32-row chunk (measured
 * at N = 43008, K = 5376: 39.3 us at M = 4 against 58.9 us with FMAs, 59 us
 * at M = 16 against 67.5 us on the few-row tensor-core kernel of w4a16_gemm).
 *
 * Streams qweight, scales and qzeros once with 128-bit coalesced loads; the
 * loads of the next 32-row chunk of K are in flight while the current one is
 * converted, which is the overlap whose absence the zero-point page blames for
 * its batch-4, g=128 regression (section "Known regression"). A persistent
 * grid (one CTA per SM at most) takes equal shares of (column block, K chunk)
 * items, so every SM streams the same bytes (for small layers, a whole number
 * of CTAs per column block when that is cheaper); a column block shared by several CTAs is finished by the last of
 * them to arrive, which sums the partial vectors in ascending CTA order: the
 * result is deterministic.
 *
 * The kernel is launched with programmatic stream serialization. Its prologue
 * (barrier setup and an L2 prefetch of its first weight chunks, a cache hint
 * that delivers no data to the kernel) may overlap the end of the preceding
 * kernel on `stream`; every read of x, qweight, scales, qzeros and the
 * workspace, and every write, happens after that kernel has completed and
 * its memory operations are visible, exactly as for an ordinary launch.
 *
 * x        [M, K] dtype `dt`
 * qweight  int32 [K/8, N]
 * scales   [K/g, N] dtype `dt`
 * qzeros   int32 [K/g, N/8], or NULL for the symmetric layer (z = 8)
 * y        [M, N] dtype `dt`, written (not accumulated into)
 * workspace, workspace_bytes   device scratch of at least
 *          w4a16_workspace_bytes(W4A16_OP_GEMV, M, N, K, g) bytes, 16-byte
 *          aligned, owned by the caller. It must be zero-filled before its
 *          first use; every call leaves its ticket words at zero again and
 *          writes partial sums only below the ticket region, so one
 *          workspace sized for the largest N serves any later call of any
 *          shape. Two calls that may run at the same time (different
 *          streams) must not share a workspace, and the GEMV and the GEMM
 *          must not share one: the GEMM's partial-sum region covers the
 *          GEMV's ticket words (the MXFP4 GEMV and GEMM use the same layouts
 *          as these two and may share with them respectively).
 * Errors: NULL, SHAPE (M outside 1..16, N % 8, K % g), UNSUPPORTED (g not in
 * {32, 64, 128, 256}), DTYPE, ALIGN, WORKSPACE (NULL, unaligned or too small),
 * DEVICE, CUDA.
 */
w4a16_status w4a16_gemv(const void* x, const int32_t* qweight, const void* scales,
                        const int32_t* qzeros, void* y, int64_t M, int64_t N, int64_t K,
                        int64_t g, w4a16_dtype dt, void* workspace, size_t workspace_bytes,
                        w4a16_stream stream);

/*
 * w4a16_gemv_noalloc -- w4a16_gemv for callers that cannot allocate device
 * memory. (No counterpart on the pages this library follows.)
 *
 * Some callers have no way to obtain scratch memory: a plugin loaded into a
 * host program that owns every device allocation and hands plugins no
 * allocator; a serving process that has already reserved all device memory
 * for its own pools; a latency-critical loop where cudaMalloc, which can
 * synchronise the device and take unbounded time, is not allowed. This entry
 * point takes the same arguments as w4a16_gemv minus the workspace and uses a
 * fixed 4 MiB scratch array compiled into the library instead. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * - The array lives in every GPU that loads the library, until the process
 *   exits.
 * - The first call on a device looks up the array's device address once
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture on the device. A first call made while `stream`
 *   is being captured does not look the address up: it returns
 *   W4A16_ERR_CUDA and enqueues nothing.
 * - Every call on a device uses the same array and clears its ticket words
 *   (an asynchronous memset on `stream`) before the kernel. Two calls that can
 *   run at the same time on one device (different streams) race on the array
 *   and give wrong results: serialise them.
 * - A shape whose scratch (w4a16_workspace_bytes(W4A16_OP_GEMV, ...)) exceeds
 *   4 MiB is rejected with W4A16_ERR_WORKSPACE; the partial-sum region takes
 *   8 KB per SM and each column block a 4-byte ticket (column blocks are at
 *   least 64 columns wide), so on a 152-SM GB300 every N up to about 47
 *   million columns fits.
 * It runs the same kernel and plan as w4a16_gemv, so its results are
 * identical to w4a16_gemv's. Other errors as for w4a16_gemv.
 */
w4a16_status w4a16_gemv_noalloc(const void* x, const int32_t* qweight, const void* scales,
                                const int32_t* qzeros, void* y, int64_t M, int64_t N, int64_t K,
                                int64_t g, w4a16_dtype dt, w4a16_stream stream);

/*
 * w4a16_gemm -- prefill path, any M >= 1.
 *
 * M <= 128 runs an operand-swapped kernel: 128 weight columns per tile, the
 * dequantised weight tile as the MMA's 128-row operand and x (padded to 32,
 * 64 or 128 rows) as the other, so no MMA work is spent on 256-row tiles. The
 * dequantised tile is written straight into tensor memory and the MMA reads
 * it there. Its (column block, K step) pairs (256 deep up to 64 padded rows of
 * x, 128 above) are split into equal contiguous ranges,
 * one per SM (stream-K); a column block split between CTAs is finished by the
 * last of them, which sums their FP32 partials from the workspace in
 * ascending CTA order (deterministic). This path needs a workspace of
 * w4a16_workspace_bytes(W4A16_OP_GEMM, M, N, K, g) bytes with the GEMV's
 * ownership and zero-fill rules (W4A16_ERR_WORKSPACE otherwise); after a
 * W4A16_ERR_TIMEOUT reported by w4a16_device_status, zero it again. It is
 * launched with programmatic stream serialization like w4a16_gemv: its
 * prologue (barrier setup, tensor-memory allocation, tensor-map prefetch) may
 * overlap the end of the preceding kernel on `stream`, and every read and
 * write of caller memory follows that kernel's completion.
 * Larger M runs the kernel described next and needs no workspace.
 *
 * Clusters of two CTAs (one per SM) own 256 x 256 output tiles of a
 * persistent grid. Per 64-deep K step each CTA brings its 128 rows of x and
 * the packed weights of its 128 columns into shared memory with TMA, sixteen
 * warps dequantise the weight tile ONCE into a shared bf16/fp16 operand tile
 * that every MMA of the tile consumes (the cooperative shared tile of "ROCm
 * KQuantGemmKWmmaQ4K/Q6K: redesign around a cooperative shared tile",
 * section "Confirmed mechanism"), and one thread issues
 * tcgen05.mma.cta_group::2 (M=256, N=256) over both CTAs' operands with the
 * FP32 accumulator in tensor memory. M and N tails are handled by TMA zero
 * fill on loads and predicated stores. The dequantised weight is (q - z) * s
 * rounded once to the activation dtype.
 *
 * Arguments and errors as w4a16_gemv, except M >= 1 with no upper limit.
 * W4A16_ERR_TIMEOUT is never returned here; a pipeline wait that runs out
 * sets a device flag that w4a16_device_status reports.
 */
w4a16_status w4a16_gemm(const void* x, const int32_t* qweight, const void* scales,
                        const int32_t* qzeros, void* y, int64_t M, int64_t N, int64_t K,
                        int64_t g, w4a16_dtype dt, void* workspace, size_t workspace_bytes,
                        w4a16_stream stream);

/*
 * w4a16_dequant -- dense dequantised copy of the packed weights:
 *
 *     w[k, n] = RN((q[k, n] - z[k / g, n]) * s[k / g, n])
 *
 * in dtype `dt`, row-major [K, N]: the dense dequantised weight copy that
 * "Keep W4A16 zero-points packed at 4 bits instead of expanding to 2 bytes"
 * (section "Change") builds at load time beside the skinny GEMM. (q - z) is exact in 16-bit
 * arithmetic and the product is rounded once, so the result is bit-exact.
 *
 * qweight  int32 [K/8, N]; scales [K/g, N] dtype `dt`; qzeros int32
 *          [K/g, N/8] or NULL (symmetric, z = 8)
 * w        [K, N] dtype `dt`, written (device memory owned by the caller)
 * Errors: NULL, SHAPE (N % 8, K % g, non-positive), UNSUPPORTED (g), DTYPE,
 * ALIGN, DEVICE, CUDA. Streams each operand once; bound by HBM bandwidth.
 */
w4a16_status w4a16_dequant(const int32_t* qweight, const void* scales, const int32_t* qzeros, void* w, int64_t N,
                           int64_t K, int64_t g, w4a16_dtype dt, w4a16_stream stream);

/*
 * MXFP4 weights -- "Add BF16xFP4 MoE GEMM stage1 kernel" (section "Technical
 * Details"): bf16 activations, weights stored as 4-bit E2M1 codes with one
 * E8M0 exponent byte e per 32 consecutive K rows of a column, decoded in
 * software to bf16 before the contraction, FP32 accumulation. The weight is
 *
 *     W[k, n] = RN_bf16( E2M1(q[k, n]) * 2^(e[k / 32, n] - 127) )
 *
 * where code q has the sign in bit 3, a 2-bit exponent field E (bias 1) in
 * bits 2..1 and a mantissa bit m in bit 0 (E = 0: m / 2, otherwise
 * 2^(E - 1) (1 + m/2)): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. Byte 0 means
 * 2^-127 and byte 255 NaN (every weight of that block is NaN). Every W is
 * exact in bf16 except where it exceeds the bf16 range (+-inf).
 *
 * qweight  int32 [K/8, N], the W4A16 word layout: nibble j of word [w, n] is
 *          the code of row 8w + j
 * escale   uint8 [K/32, N]: exponent byte of block b, column n at b * N + n
 * x        bf16 [M, K]; y bf16 [M, N], written (not accumulated into)
 * Shapes: N % 16 == 0 (each exponent row starts 16-byte aligned), K % 32 == 0.
 * Every pointer 16-byte aligned device memory owned by the caller.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA, WORKSPACE (GEMV only).
 */

/*
 * w4a16_mxfp4_dequant -- dense bf16 copy W [K, N] (row-major) of MXFP4
 * weights. Bit-exact. Streams each operand once; bound by HBM bandwidth.
 */
w4a16_status w4a16_mxfp4_dequant(const int32_t* qweight, const uint8_t* escale, void* w, int64_t N, int64_t K,
                                 w4a16_stream stream);

/*
 * w4a16_mxfp4_gemv -- decode path for MXFP4 weights, 1 <= M <= 16: the
 * w4a16_gemv kernel with the E2M1 decode in place of the 4-bit integer one
 * (each 32-row chunk is one exponent block; its scale 2^(e - 127) is applied
 * in FP32 once per chunk). Same persistent grid, deterministic fix-up and
 * programmatic launch, and the same conversion choice: FP32 FMAs for one row
 * (and two rows of a layer of at most 4 * 2^20 weights), warp-level
 * tensor-core MMAs on fp16 operands otherwise (each chunk's x rows are first
 * rescaled to fp16 by a power of two per row, undone in FP32). 9..16 rows of
 * a layer with at least 48 * 2^20 weights run the few-row tensor-core kernel
 * of w4a16_mxfp4_gemm instead, where the 16-row rescale costs more than the
 * MMAs save (43008 x 5376, M = 12: 110.5 against 77.3 us; M = 8 stays on the
 * GEMV: 59.4 against 77.1 us).
 * Workspace: at least w4a16_workspace_bytes(W4A16_OP_GEMV, M, N, K, 32) bytes,
 * with the same ownership and zero-fill rules as for w4a16_gemv.
 */
w4a16_status w4a16_mxfp4_gemv(const void* x, const int32_t* qweight, const uint8_t* escale, void* y, int64_t M,
                              int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                              w4a16_stream stream);

/*
 * w4a16_mxfp4_gemm -- prefill path for MXFP4 weights, any M >= 1: the
 * w4a16_gemm kernels (operand-swapped and stream-K for M <= 128, CTA pairs
 * above) with the E2M1 decode writing the bf16 operand tile. Workspace as for
 * w4a16_gemm (needed for M <= 128, sized by w4a16_workspace_bytes(
 * W4A16_OP_GEMM, M, N, K, 32)). A pipeline wait that runs out sets the device
 * flag that w4a16_device_status reports.
 */
w4a16_status w4a16_mxfp4_gemm(const void* x, const int32_t* qweight, const uint8_t* escale, void* y, int64_t M,
                              int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                              w4a16_stream stream);

/*
 * w4a16_device_status -- synchronise `stream`, then read and clear the
 * device-side error word of the current device. Every wait on an mbarrier
 * inside the GEMM pipeline gives up after about two seconds; the kernel then
 * records W4A16_ERR_TIMEOUT there, drains its own copies in flight, frees its
 * tensor memory and returns, so the CUDA context stays usable. Returns
 * W4A16_OK when nothing was recorded, W4A16_ERR_CUDA if synchronisation
 * failed.
 */
w4a16_status w4a16_device_status(w4a16_stream stream);

/*
 * w4a16_selftest_wait_timeout -- exercise the device-side failure path. (No
 * counterpart on the pages this library follows.)
 *
 * Launches, asynchronously on `stream`, one warp that waits on an mbarrier
 * nothing will complete, with the same bounded wait the GEMV uses. After about
 * two seconds the wait gives up, records W4A16_ERR_TIMEOUT in the device error
 * word and the kernel exits normally, so the CUDA context stays usable; a
 * following w4a16_device_status(stream) returns W4A16_ERR_TIMEOUT (and clears
 * the word). Touches no caller memory. Errors: DEVICE, CUDA (launch failed).
 */
w4a16_status w4a16_selftest_wait_timeout(w4a16_stream stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* w4a16_status_string(w4a16_status status);

/* W4A16_ABI_VERSION of the compiled library. */
int w4a16_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
