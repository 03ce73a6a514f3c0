// Launchers shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

struct DeviceProps {
    int device = -1;
    int sms = 0;
    int cc_major = 0;
    int cc_minor = 0;
    size_t smem_optin = 0;
};

// Properties of the current device, cached per device ordinal.
cudaError_t current_device_props(DeviceProps* out);

// Raise `kernel`'s dynamic shared memory limit on `device` (the current
// device) to at least `bytes`. Thread-safe; the limit only ever grows, so a
// launch that needs less is never refused because another thread set a
// smaller limit in between.
cudaError_t ensure_dynamic_smem(const void* kernel, int device, size_t bytes);

cudaError_t launch_pack(const uint8_t* src, uint32_t* dst, int64_t rows, int64_t cols, int dim,
                        const DeviceProps& dp, cudaStream_t s);
cudaError_t launch_unpack(const uint32_t* src, uint8_t* dst, int64_t rows, int64_t cols, int dim,
                          const DeviceProps& dp, cudaStream_t s);

struct GemvPlan {
    int mt = 0;             // row template (>= M)
    int cols = 0;           // columns per lane
    int cb = 0;             // columns per column block (32 * cols)
    int box_cols = 0;       // columns per tensor copy of weights and scales (cb, or 96 for 288-column blocks)
    int n_cb = 0;           // column blocks
    int warps = 0;          // warps per CTA (streaming warps + one reduction warp)
    int grid = 0;           // persistent CTAs (one per SM at most)
    long long items = 0;    // column blocks x 32-row chunks of K
    long long items_split = 0;   // items of the blocks shared stream-K by all CTAs ([0, whole_first))
    int whole_first = 0;    // first of the blocks handed out whole
    int whole_per_cta = 0;  // whole blocks per CTA (after its stream-K share)
    int cluster = 0;        // CTAs per column block summed through distributed shared memory (0: tickets)
    bool mma = false;       // products through warp-level tensor-core MMAs (W4A16, 2..16 rows)
    bool fact = false;      // zero-point applied per chunk through chunk sums of x
    bool xpre = false;      // with fact: the chunk sums computed once per CTA up front
    size_t smem_bytes = 0;  // dynamic shared memory per CTA
    size_t ticket_bytes = 0;
    size_t partial_bytes = 0;
    int device = -1;
};

GemvPlan plan_gemv(int M, int N, int K, int g, const DeviceProps& dp);
// The GEMV plan for MXFP4 weights (no zero-points); same workspace size as
// plan_gemv(M, N, K, 32, dp).
GemvPlan plan_mx_gemv(int M, int N, int K, const DeviceProps& dp);
// The CUDA-core kernel's own scratch: plan.partial_bytes of partial-sum slots
// (a size fixed per device) and plan.ticket_bytes of ticket words.
size_t gemv_workspace_bytes(const GemvPlan& plan);

// `partials`: plan.partial_bytes of partial-sum slots; `tickets`: ticket words
// (zero before the first call; every call leaves them zero).
cudaError_t launch_gemv(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y,
                        int M, int N, int K, int g, bool bf16, const GemvPlan& plan, float* partials,
                        uint32_t* tickets, cudaStream_t s);

// w4a16_mxfp4_gemv converts 2..16 rows with tensor-core MMAs like the int4
// GEMV, but rescales every chunk's x rows to fp16 first; with 16 rows that
// costs more than the MMAs save on large layers, so 9..16 rows of a layer
// with at least kMxTensorMinWeights weights go to the few-row tensor-core
// kernel. Measured (us, GEMV / tensor-core kernel): 43008 x 5376 M=8 59.4 /
// 77.1, M=12 110.5 / 77.3; 16384 x 5376 M=12 47.1 / 36.0; 8192 x 4096 M=12
// 19.1 / 21.7, M=16 20.0 / 21.7. (w4a16_gemv hands nothing over.)
constexpr int kGemvTensorMinM = 9;
constexpr long long kMxTensorMinWeights = 48ll << 20;
inline bool mx_gemv_uses_tensor_cores(long long M, long long N, long long K) {
    return M >= kGemvTensorMinM && N * K >= kMxTensorMinWeights;
}

// Size of the GEMV's built-in scratch array (w4a16_gemv_noalloc).
constexpr size_t kGemvNoAllocScratchBytes = size_t(4) << 20;

// Device address of that array on `device` (which must be current); looked up
// once per device and cached. With may_look_up false (the caller's stream is
// being captured) an address not yet cached is not looked up:
// cudaErrorStreamCaptureUnsupported.
cudaError_t gemv_noalloc_scratch(int device, bool may_look_up, void** ptr);

cudaError_t launch_gemm(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y,
                        int M, int N, int K, int g, bool bf16, const DeviceProps& dp, cudaStream_t s);

// Read and clear the device-side error word of the GEMM pipeline (after a sync).
cudaError_t read_and_clear_device_error(uint32_t* out, cudaStream_t s);
// Read and clear the device-side error word of the GEMV rings (no sync).
cudaError_t read_and_clear_gemv_error(uint32_t* out);
cudaError_t launch_wait_selftest(cudaStream_t s);
// GEMMs with at most this many rows of x run the operand-swapped kernel
// (weights as the 128-row MMA operand, x padded to 32..128 rows; it cannot take
// more); measured at N = 43008, K = 5376: 109-133 us for M = 1..128 against
// 174-180 us on the CTA-pair kernel, which runs M >= 129 (180 us at M = 192,
// where the operand-swapped kernel with 256 padded rows took 247 us).
#ifndef W4A16_SKINNY_MAX_M
#define W4A16_SKINNY_MAX_M 128
#endif
constexpr int kSkinnyMaxM = W4A16_SKINNY_MAX_M;
// The operand-swapped kernel splits its work stream-K; its workspace holds FP32
// partial slots (two per CTA; the size depends only on the device) followed by
// one ticket word per column block and epilogue warp (zero before the first
// call; every call leaves them zero).
size_t skinny_partial_bytes(const DeviceProps& dp);
size_t skinny_ticket_bytes(int N);
size_t skinny_workspace_bytes(int N, const DeviceProps& dp);   // partials, then tickets
cudaError_t launch_gemm_skinny(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                               int N, int K, int g, bool bf16, float* partials, uint32_t* tickets,
                               const DeviceProps& dp, cudaStream_t s);
cudaError_t read_and_clear_skinny_error(uint32_t* out);
cudaError_t launch_dequant(const uint32_t* qw, const void* sc, const uint32_t* qz, void* out, int N, int K, int g,
                           bool bf16, const DeviceProps& dp, cudaStream_t s);

// MXFP4 weights (E2M1 codes, E8M0 bytes [K/32, N]); bf16 activations and outputs.
cudaError_t launch_mx_dequant(const uint32_t* qw, const uint8_t* es, void* out, int N, int K, const DeviceProps& dp,
                              cudaStream_t s);
cudaError_t launch_mx_gemm(const void* x, const uint32_t* qw, const uint8_t* es, void* y, int M, int N, int K,
                           const DeviceProps& dp, cudaStream_t s);
cudaError_t launch_mx_gemm_skinny(const void* x, const uint32_t* qw, const uint8_t* es, void* y, int M, int N, int K,
                                  float* partials, uint32_t* tickets, const DeviceProps& dp, cudaStream_t s);
cudaError_t launch_mx_gemv(const void* x, const uint32_t* qw, const uint8_t* es, void* y, int M, int N, int K,
                           const GemvPlan& plan, float* partials, uint32_t* tickets, cudaStream_t s);

// Workspace of the GEMV entry points (w4a16_mxfp4_gemv runs either the GEMV
// kernel or, for 5..16 rows of a large layer, the few-row tensor-core kernel):
// both kernels' partial-sum regions (sizes fixed per device), then one ticket
// region both use. Every call leaves the tickets at zero and no partial region covers
// them, so one workspace sized for the largest N serves calls of any shape.
struct GemvWorkspace {
    size_t cuda_partials = 0, tensor_partials = 0, tickets = 0;
    size_t total() const { return cuda_partials + tensor_partials + tickets; }
    float* cuda_part(void* ws) const { return static_cast<float*>(ws); }
    float* tensor_part(void* ws) const { return reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cuda_partials); }
    uint32_t* ticket_words(void* ws) const {
        return reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + cuda_partials + tensor_partials);
    }
};
inline GemvWorkspace gemv_workspace(const GemvPlan& plan, int N, const DeviceProps& dp) {
    GemvWorkspace w;
    w.cuda_partials = plan.partial_bytes;
    w.tensor_partials = skinny_partial_bytes(dp);
    w.tickets = plan.ticket_bytes > skinny_ticket_bytes(N) ? plan.ticket_bytes : skinny_ticket_bytes(N);
    return w;
}

}  // namespace w4a16
