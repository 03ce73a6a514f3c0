// C ABI of libw4a16: argument validation, device gate, dispatch.
// Declarations and the contract of every entry point are in include/w4a16.h.
#include "w4a16.h"

#include "internal.h"

#include <map>
#include <mutex>
#include <utility>

namespace w4a16 {

cudaError_t current_device_props(DeviceProps* out) {
    static std::mutex mu;
    static DeviceProps cache[64];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].device != dev) {
        DeviceProps p;
        p.device = dev;
        if ((e = cudaDeviceGetAttribute(&p.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&p.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&p.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
        int optin = 0;
        if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
        p.smem_optin = static_cast<size_t>(optin);
        cache[dev] = p;
    }
    *out = cache[dev];
    return cudaSuccess;
}

cudaError_t ensure_dynamic_smem(const void* kernel, int device, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> set;   // largest limit set per (kernel, device)
    std::lock_guard<std::mutex> lock(mu);
    size_t& cur = set[{kernel, device}];
    if (cur >= bytes) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) cur = bytes;
    return e;
}

}  // namespace w4a16

namespace {

using w4a16::DeviceProps;

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_group(int64_t g) { return g == 32 || g == 64 || g == 128 || g == 256; }

// Device gate: a CUDA device must be current and be compute capability 10.3.
w4a16_status device_gate(DeviceProps* dp) {
    if (w4a16::current_device_props(dp) != cudaSuccess) {
        cudaGetLastError();   // the failed query is not the caller's error
        return W4A16_ERR_DEVICE;
    }
    if (dp->cc_major != 10 || dp->cc_minor != 3) return W4A16_ERR_DEVICE;
    return W4A16_OK;
}

w4a16_status check_pack_args(const void* src, const void* dst, int64_t rows, int64_t cols, int dim) {
    if (!src || !dst) return W4A16_ERR_NULL;
    if (dim != 0 && dim != 1) return W4A16_ERR_SHAPE;
    if (rows <= 0 || cols <= 0 || rows > kMaxDim || cols > kMaxDim) return W4A16_ERR_SHAPE;
    if ((dim == 0 ? rows : cols) % 8 != 0) return W4A16_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(dst)) return W4A16_ERR_ALIGN;
    return W4A16_OK;
}

w4a16_status check_layer_args(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros,
                              const void* y, int64_t M, int64_t N, int64_t K, int64_t g, w4a16_dtype dt,
                              int64_t max_m) {
    if (!x || !qweight || !scales || !y) return W4A16_ERR_NULL;
    if (dt != W4A16_F16 && dt != W4A16_BF16) return W4A16_ERR_DTYPE;
    if (M < 1 || N < 1 || K < 1 || g < 1) return W4A16_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return W4A16_ERR_SHAPE;
    if (max_m > 0 && M > max_m) return W4A16_ERR_SHAPE;
    if (N % 8 != 0 || K % g != 0) return W4A16_ERR_SHAPE;
    if (!supported_group(g)) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) ||
        (qzeros && !aligned16(qzeros)))
        return W4A16_ERR_ALIGN;
    return W4A16_OK;
}

// MXFP4 weights: qweight int32 [K/8, N]; exponent bytes [K/32, N] (N % 16:
// every row of the byte tensor starts 16-byte aligned).
w4a16_status check_mx_weights(const int32_t* qweight, const uint8_t* escale, int64_t N, int64_t K) {
    if (!qweight || !escale) return W4A16_ERR_NULL;
    if (N < 1 || K < 1 || N > kMaxDim || K > kMaxDim) return W4A16_ERR_SHAPE;
    if (N % 16 != 0 || K % 32 != 0) return W4A16_ERR_SHAPE;
    if (!aligned16(qweight) || !aligned16(escale)) return W4A16_ERR_ALIGN;
    return W4A16_OK;
}

// ... and bf16 x [M, K], y [M, N]
w4a16_status check_mx_args(const void* x, const int32_t* qweight, const uint8_t* escale, const void* y, int64_t M,
                           int64_t N, int64_t K, int64_t max_m) {
    if (!x || !y) return W4A16_ERR_NULL;
    w4a16_status st = check_mx_weights(qweight, escale, N, K);
    if (st != W4A16_OK) return st;
    if (M < 1 || M > kMaxDim || (max_m > 0 && M > max_m)) return W4A16_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(y)) return W4A16_ERR_ALIGN;
    return W4A16_OK;
}

w4a16_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

}  // namespace

extern "C" {

int w4a16_abi_version(void) { return W4A16_ABI_VERSION; }

const char* w4a16_status_string(w4a16_status status) {
    switch (status) {
        case W4A16_OK: return "W4A16_OK";
        case W4A16_ERR_NULL: return "W4A16_ERR_NULL";
        case W4A16_ERR_SHAPE: return "W4A16_ERR_SHAPE";
        case W4A16_ERR_DTYPE: return "W4A16_ERR_DTYPE";
        case W4A16_ERR_ALIGN: return "W4A16_ERR_ALIGN";
        case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED";
        case W4A16_ERR_DEVICE: return "W4A16_ERR_DEVICE";
        case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE";
        case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
        case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT";
    }
    return "W4A16_ERR_UNKNOWN";
}

w4a16_status w4a16_pack(const uint8_t* src, int32_t* dst, int64_t rows, int64_t cols, int dim,
                        w4a16_stream stream) {
    w4a16_status st = check_pack_args(src, dst, rows, cols, dim);
    if (st != W4A16_OK) return st;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    return from_cuda(w4a16::launch_pack(src, reinterpret_cast<uint32_t*>(dst), rows, cols, dim, dp,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_unpack(const int32_t* src, uint8_t* dst, int64_t rows, int64_t cols, int dim,
                          w4a16_stream stream) {
    w4a16_status st = check_pack_args(src, dst, rows, cols, dim);
    if (st != W4A16_OK) return st;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    return from_cuda(w4a16::launch_unpack(reinterpret_cast<const uint32_t*>(src), dst, rows, cols, dim, dp,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

size_t w4a16_workspace_bytes(w4a16_op op, int64_t M, int64_t N, int64_t K, int64_t g) {
    if (op != W4A16_OP_GEMV && op != W4A16_OP_GEMM) return 0;
    if (M < 1 || N < 8 || N % 8 || K < 1 || K > kMaxDim || N > kMaxDim || M > kMaxDim || !supported_group(g) || K % g)
        return 0;
    if (op == W4A16_OP_GEMV && M > 16) return 0;
    if (op == W4A16_OP_GEMM && M > w4a16::kSkinnyMaxM) return 0;
    DeviceProps dp;
    if (device_gate(&dp) != W4A16_OK) return 0;
    if (op == W4A16_OP_GEMM) return w4a16::skinny_workspace_bytes((int)N, dp);
    return w4a16::gemv_workspace(w4a16::plan_gemv((int)M, (int)N, (int)K, (int)g, dp), (int)N, dp).total();
}

w4a16_status w4a16_gemv(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros, void* y,
                        int64_t M, int64_t N, int64_t K, int64_t g, w4a16_dtype dt, void* workspace,
                        size_t workspace_bytes, w4a16_stream stream) {
    w4a16_status st = check_layer_args(x, qweight, scales, qzeros, y, M, N, K, g, dt, 16);
    if (st != W4A16_OK) return st;
    if (!workspace || !aligned16(workspace)) return W4A16_ERR_WORKSPACE;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    const w4a16::GemvPlan plan = w4a16::plan_gemv((int)M, (int)N, (int)K, (int)g, dp);
    const w4a16::GemvWorkspace wl = w4a16::gemv_workspace(plan, (int)N, dp);
    if (workspace_bytes < wl.total()) return W4A16_ERR_WORKSPACE;
    return from_cuda(w4a16::launch_gemv(x, reinterpret_cast<const uint32_t*>(qweight), scales,
                                        reinterpret_cast<const uint32_t*>(qzeros), y, (int)M, (int)N, (int)K, (int)g,
                                        dt == W4A16_BF16, plan, wl.cuda_part(workspace), wl.ticket_words(workspace),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_gemv_noalloc(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros,
                                void* y, int64_t M, int64_t N, int64_t K, int64_t g, w4a16_dtype dt,
                                w4a16_stream stream) {
    w4a16_status st = check_layer_args(x, qweight, scales, qzeros, y, M, N, K, g, dt, 16);
    if (st != W4A16_OK) return st;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    const w4a16::GemvPlan plan = w4a16::plan_gemv((int)M, (int)N, (int)K, (int)g, dp);
    if (w4a16::gemv_workspace_bytes(plan) > w4a16::kGemvNoAllocScratchBytes) return W4A16_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The first call on a device looks the array's address up, which must not
    // happen inside a stream capture: refuse it there instead.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return W4A16_ERR_CUDA;
    void* scratch = nullptr;
    if (w4a16::gemv_noalloc_scratch(dp.device, cap == cudaStreamCaptureStatusNone, &scratch) != cudaSuccess)
        return W4A16_ERR_CUDA;
    // the ticket words must start at zero; the partial sums are written before they are read
    if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + plan.partial_bytes, 0, plan.ticket_bytes, s) != cudaSuccess)
        return W4A16_ERR_CUDA;
    return from_cuda(w4a16::launch_gemv(x, reinterpret_cast<const uint32_t*>(qweight), scales,
                                        reinterpret_cast<const uint32_t*>(qzeros), y, (int)M, (int)N, (int)K, (int)g,
                                        dt == W4A16_BF16, plan, static_cast<float*>(scratch),
                                        reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scratch) + plan.partial_bytes),
                                        s));
}

w4a16_status w4a16_gemm(const void* x, const int32_t* qweight, const void* scales, const int32_t* qzeros, void* y,
                        int64_t M, int64_t N, int64_t K, int64_t g, w4a16_dtype dt, void* workspace,
                        size_t workspace_bytes, w4a16_stream stream) {
    w4a16_status st = check_layer_args(x, qweight, scales, qzeros, y, M, N, K, g, dt, 0);
    if (st != W4A16_OK) return st;
    if (M <= w4a16::kSkinnyMaxM && (!workspace || !aligned16(workspace))) return W4A16_ERR_WORKSPACE;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    if (M <= w4a16::kSkinnyMaxM) {
        if (workspace_bytes < w4a16::skinny_workspace_bytes((int)N, dp)) return W4A16_ERR_WORKSPACE;
        return from_cuda(w4a16::launch_gemm_skinny(
            x, reinterpret_cast<const uint32_t*>(qweight), scales, reinterpret_cast<const uint32_t*>(qzeros), y,
            (int)M, (int)N, (int)K, (int)g, dt == W4A16_BF16, static_cast<float*>(workspace),
            reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + w4a16::skinny_partial_bytes(dp)), dp,
            reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(w4a16::launch_gemm(x, reinterpret_cast<const uint32_t*>(qweight), scales,
                                        reinterpret_cast<const uint32_t*>(qzeros), y, (int)M, (int)N, (int)K, (int)g,
                                        dt == W4A16_BF16, dp, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_device_status(w4a16_stream stream) {
    DeviceProps dp;
    w4a16_status st = device_gate(&dp);
    if (st != W4A16_OK) return st;
    uint32_t v = 0, u = 0, k = 0;
    if (w4a16::read_and_clear_device_error(&v, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess ||
        w4a16::read_and_clear_gemv_error(&u) != cudaSuccess || w4a16::read_and_clear_skinny_error(&k) != cudaSuccess)
        return W4A16_ERR_CUDA;
    return (v | u | k) ? W4A16_ERR_TIMEOUT : W4A16_OK;
}

w4a16_status w4a16_dequant(const int32_t* qweight, const void* scales, const int32_t* qzeros, void* w, int64_t N,
                           int64_t K, int64_t g, w4a16_dtype dt, w4a16_stream stream) {
    if (!qweight || !scales || !w) return W4A16_ERR_NULL;
    if (dt != W4A16_F16 && dt != W4A16_BF16) return W4A16_ERR_DTYPE;
    if (N < 1 || K < 1 || g < 1 || N > kMaxDim || K > kMaxDim) return W4A16_ERR_SHAPE;
    if (N % 8 != 0 || K % g != 0) return W4A16_ERR_SHAPE;
    if (!supported_group(g)) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(qweight) || !aligned16(scales) || !aligned16(w) || (qzeros && !aligned16(qzeros)))
        return W4A16_ERR_ALIGN;
    DeviceProps dp;
    w4a16_status st = device_gate(&dp);
    if (st != W4A16_OK) return st;
    return from_cuda(w4a16::launch_dequant(reinterpret_cast<const uint32_t*>(qweight), scales,
                                           reinterpret_cast<const uint32_t*>(qzeros), w, (int)N, (int)K, (int)g,
                                           dt == W4A16_BF16, dp, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_mxfp4_dequant(const int32_t* qweight, const uint8_t* escale, void* w, int64_t N, int64_t K,
                                 w4a16_stream stream) {
    if (!w) return W4A16_ERR_NULL;
    w4a16_status st = check_mx_weights(qweight, escale, N, K);
    if (st != W4A16_OK) return st;
    if (!aligned16(w)) return W4A16_ERR_ALIGN;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    return from_cuda(w4a16::launch_mx_dequant(reinterpret_cast<const uint32_t*>(qweight), escale, w, (int)N, (int)K,
                                              dp, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_mxfp4_gemv(const void* x, const int32_t* qweight, const uint8_t* escale, void* y, int64_t M,
                              int64_t N, int64_t K, void* workspace, size_t workspace_bytes, w4a16_stream stream) {
    w4a16_status st = check_mx_args(x, qweight, escale, y, M, N, K, 16);
    if (st != W4A16_OK) return st;
    if (!workspace || !aligned16(workspace)) return W4A16_ERR_WORKSPACE;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    const w4a16::GemvPlan plan = w4a16::plan_mx_gemv((int)M, (int)N, (int)K, dp);
    const w4a16::GemvWorkspace wl = w4a16::gemv_workspace(plan, (int)N, dp);
    if (workspace_bytes < wl.total()) return W4A16_ERR_WORKSPACE;
    if (w4a16::mx_gemv_uses_tensor_cores(M, N, K))
        return from_cuda(w4a16::launch_mx_gemm_skinny(x, reinterpret_cast<const uint32_t*>(qweight), escale, y, (int)M,
                                                      (int)N, (int)K, wl.tensor_part(workspace),
                                                      wl.ticket_words(workspace), dp,
                                                      reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(w4a16::launch_mx_gemv(x, reinterpret_cast<const uint32_t*>(qweight), escale, y, (int)M, (int)N,
                                           (int)K, plan, wl.cuda_part(workspace), wl.ticket_words(workspace),
                                           reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_mxfp4_gemm(const void* x, const int32_t* qweight, const uint8_t* escale, void* y, int64_t M,
                              int64_t N, int64_t K, void* workspace, size_t workspace_bytes, w4a16_stream stream) {
    w4a16_status st = check_mx_args(x, qweight, escale, y, M, N, K, 0);
    if (st != W4A16_OK) return st;
    if (M <= w4a16::kSkinnyMaxM && (!workspace || !aligned16(workspace))) return W4A16_ERR_WORKSPACE;
    DeviceProps dp;
    if ((st = device_gate(&dp)) != W4A16_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(qweight);
    if (M <= w4a16::kSkinnyMaxM) {
        if (workspace_bytes < w4a16::skinny_workspace_bytes((int)N, dp)) return W4A16_ERR_WORKSPACE;
        return from_cuda(w4a16::launch_mx_gemm_skinny(
            x, qw, escale, y, (int)M, (int)N, (int)K, static_cast<float*>(workspace),
            reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + w4a16::skinny_partial_bytes(dp)), dp, s));
    }
    return from_cuda(w4a16::launch_mx_gemm(x, qw, escale, y, (int)M, (int)N, (int)K, dp, s));
}

w4a16_status w4a16_selftest_wait_timeout(w4a16_stream stream) {
    DeviceProps dp;
    w4a16_status st = device_gate(&dp);
    if (st != W4A16_OK) return st;
    return w4a16::launch_wait_selftest(reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A16_OK
                                                                                          : W4A16_ERR_CUDA;
}

}  // extern "C"
