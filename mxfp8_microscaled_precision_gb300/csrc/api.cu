// api.cu -- the extern "C" entry points of libmxq (declared in include/mxq.h).
//
// Each call validates its arguments on the host, checks that the current
// device is a GB300 (sm_103), and launches one kernel on the caller's
// stream.  Nothing is allocated per call.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

// Device status word: kernels record a timed-out bounded wait here.
__device__ unsigned int g_mxq_device_status = 0u;
// What the last mxq_get_device_status found in the status word (read and
// cleared in one atomic exchange on the device).
__device__ unsigned int g_mxq_status_taken = 0u;

namespace mxq {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_have[kMaxDevices] = {};
DeviceInfo g_info[kMaxDevices];
std::mutex g_status_mu;   // one mxq_get_device_status at a time per process

// Moves the status word into g_mxq_status_taken and clears it, atomically: a
// timeout recorded by a kernel still running elsewhere is either taken here
// or stays for the next call.
__global__ void status_take_kernel(unsigned int* status) { g_mxq_status_taken = atomicExch(status, 0u); }

}  // namespace

cudaError_t current_device_info(DeviceInfo* info) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_have[dev]) {
            DeviceInfo d;
            d.device = dev;
            if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
                return e;
            int optin = 0;
            if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
                return e;
            d.smem_optin = static_cast<size_t>(optin);
            g_info[dev] = d;
            g_have[dev] = true;
        }
        *info = g_info[dev];
    }
    // The status word's address belongs to the current context, which a device
    // reset replaces: it is looked up on every call, never cached.
    info->status = nullptr;
    if (info->cc_major == 10 && info->cc_minor == 3) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_mxq_device_status)) != cudaSuccess) return e;
        info->status = static_cast<unsigned int*>(p);
    }
    return cudaSuccess;
}

}  // namespace mxq

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device check shared by every launching call.
mxq_status device_ok(mxq::DeviceInfo* info) {
    if (mxq::current_device_info(info) != cudaSuccess) return MXQ_ERR_CUDA;
    if (info->cc_major != 10 || info->cc_minor != 3 || info->status == nullptr)
        return MXQ_ERR_UNSUPPORTED_DEVICE;
    return MXQ_OK;
}

inline mxq_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MXQ_OK;
    if (e == cudaErrorInvalidValue) return MXQ_ERR_INVALID_ARG;
    return MXQ_ERR_CUDA;
}

// What a validated dense GEMM asks for.
enum DenseWork { kNothing = 0, kZeroFill = 1, kLaunch = 2 };

// Argument checks of the dense BF16-output GEMMs (see mxq_gemm_bf16out).
mxq_status check_dense(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q, const void* b_s,
                       mxq_fp8_format b_fmt, int64_t M, int64_t N, int64_t K, int b_mn_major, const void* y,
                       int64_t ldy, DenseWork* work) {
    *work = kNothing;
    if (M < 0 || N < 0 || K < 0 || (b_mn_major != 0 && b_mn_major != 1)) return MXQ_ERR_INVALID_ARG;
    if ((a_fmt != MXQ_FP8_E4M3 && a_fmt != MXQ_FP8_E5M2) || (b_fmt != MXQ_FP8_E4M3 && b_fmt != MXQ_FP8_E5M2))
        return MXQ_ERR_INVALID_ARG;
    if (K % 32 != 0 || N % 16 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (b_mn_major && N % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M > (int64_t(1) << 31) - 128 || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - 128)
        return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return MXQ_OK;
    if (!y || ldy < N || ldy % 8 != 0 || !aligned16(y)) return MXQ_ERR_INVALID_ARG;
    if (K == 0) {  // empty contraction: y = 0
        *work = kZeroFill;
        return MXQ_OK;
    }
    if (!a_q || !a_s || !b_q || !b_s) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(a_s) || !aligned16(b_q) || !aligned16(b_s))
        return MXQ_ERR_INVALID_ARG;
    *work = kLaunch;
    return MXQ_OK;
}

cudaError_t zero_fill(void* y, int64_t ldy, int64_t M, int64_t N, mxq_stream_t stream) {
    return cudaMemset2DAsync(y, static_cast<size_t>(ldy) * 2, 0, static_cast<size_t>(N) * 2,
                             static_cast<size_t>(M), reinterpret_cast<cudaStream_t>(stream));
}

// Argument checks of the grouped-rows GEMMs; MXQ_OK with *launch false when
// there is nothing to compute.
mxq_status check_grouped_rows(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q,
                              const void* b_s, mxq_fp8_format b_fmt, const int64_t* group_offsets, int32_t G,
                              int64_t M_total, int64_t N, int64_t K, const void* y, int64_t ldy, bool* launch) {
    *launch = false;
    if ((a_fmt != MXQ_FP8_E4M3 && a_fmt != MXQ_FP8_E5M2) || (b_fmt != MXQ_FP8_E4M3 && b_fmt != MXQ_FP8_E5M2))
        return MXQ_ERR_INVALID_ARG;
    if (G < 1 || M_total < 0 || N < 0 || K < 0) return MXQ_ERR_INVALID_ARG;
    if (G > 1024) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (N % 128 != 0 || K % 32 != 0 || K == 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M_total > (int64_t(1) << 31) - 128 || static_cast<int64_t>(G) * N > (int64_t(1) << 31) - 256 ||
        K > (int64_t(1) << 31) - 128)
        return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M_total == 0 || N == 0) return MXQ_OK;
    if (!a_q || !a_s || !b_q || !b_s || !group_offsets || !y) return MXQ_ERR_INVALID_ARG;
    if (ldy < N || ldy % 8 != 0) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(a_s) || !aligned16(b_q) || !aligned16(b_s) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(group_offsets) & 7u) != 0)
        return MXQ_ERR_INVALID_ARG;
    *launch = true;
    return MXQ_OK;
}

// Argument checks and launch of the grouped-rows GEMMs (a_bands_cap 0: A scales
// MMA-tiled over all rows; > 0: group-tiled).
mxq_status grouped_rows_gemm(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q,
                             const void* b_s, mxq_fp8_format b_fmt, const int64_t* group_offsets, int32_t G,
                             int64_t M_total, int64_t N, int64_t K, int64_t a_bands_cap, void* y, int64_t ldy,
                             mxq_stream_t stream) {
    bool launch = false;
    mxq_status st = check_grouped_rows(a_q, a_s, a_fmt, b_q, b_s, b_fmt, group_offsets, G, M_total, N, K, y, ldy,
                                       &launch);
    if (st != MXQ_OK || !launch) return st;
    mxq::DeviceInfo dev;
    st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_grouped_gemm(dev, a_q, a_s, b_q, b_s, group_offsets, G, M_total, N, K, a_bands_cap,
                                              y, ldy, static_cast<int>(a_fmt), static_cast<int>(b_fmt),
                                              reinterpret_cast<cudaStream_t>(stream)));
}

// Bands of a group-tiled A-scale buffer that hold any routing of M_total rows
// over G experts, and its bytes.
int64_t group_tiled_bands(int64_t M_total, int32_t G) { return (M_total + 127) / 128 + G; }

int64_t group_tiled_bytes(int64_t M_total, int32_t G, int64_t K) {
    return group_tiled_bands(M_total, G) * ((K / 32 + 3) / 4) * 512;
}

}  // namespace

extern "C" {

int mxq_abi_version(void) { return MXQ_ABI_VERSION; }

const char* mxq_status_string(mxq_status s) {
    switch (s) {
        case MXQ_OK: return "ok";
        case MXQ_ERR_INVALID_ARG: return "invalid argument";
        case MXQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MXQ_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103 / GB300)";
        case MXQ_ERR_CUDA: return "CUDA error";
        case MXQ_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

size_t mxq_scale_bytes(int64_t rows, int64_t cols, mxq_scale_layout layout) {
    if (rows < 0 || cols < 0 || cols % 32 != 0) return 0;
    const int64_t groups = cols / 32;
    if (layout == MXQ_SCALE_ROWMAJOR) return static_cast<size_t>(rows * groups);
    if (layout == MXQ_SCALE_MMA_TILED)
        return static_cast<size_t>(((rows + 127) / 128 * 128) * ((groups + 3) / 4 * 4));
    return 0;
}

mxq_status mxq_quant_1x32_dual_batched(const void* x, int64_t batch, int64_t rows, int64_t cols,
                                       int64_t ld, int64_t batch_stride, void* q_row, void* s_row,
                                       void* q_col, void* s_col, mxq_scale_layout layout,
                                       mxq_fp8_format fmt, mxq_stream_t stream) {
    if (layout != MXQ_SCALE_ROWMAJOR && layout != MXQ_SCALE_MMA_TILED) return MXQ_ERR_INVALID_ARG;
    if (fmt != MXQ_FP8_E4M3 && fmt != MXQ_FP8_E5M2) return MXQ_ERR_INVALID_ARG;
    if (batch < 0 || rows < 0 || cols < 0) return MXQ_ERR_INVALID_ARG;
    const bool row = q_row != nullptr || s_row != nullptr;
    const bool col = q_col != nullptr || s_col != nullptr;
    if (!row && !col) return MXQ_ERR_INVALID_ARG;
    if (cols % 32 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (col && rows % 32 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (batch > 65535) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (batch == 0 || rows == 0 || cols == 0) return MXQ_OK;
    if (!x || (row && (!q_row || !s_row)) || (col && (!q_col || !s_col))) return MXQ_ERR_INVALID_ARG;
    if (ld < cols || ld % 8 != 0) return MXQ_ERR_INVALID_ARG;
    if (batch > 1 && (batch_stride < rows * ld || batch_stride % 8 != 0)) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(x) || (row && (!aligned16(q_row) || !aligned16(s_row))) ||
        (col && (!aligned16(q_col) || !aligned16(s_col))))
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_quant_1x32(dev, x, batch, rows, cols, ld, batch > 1 ? batch_stride : rows * ld,
                                            row ? q_row : nullptr, row ? s_row : nullptr,
                                            col ? q_col : nullptr, col ? s_col : nullptr,
                                            layout == MXQ_SCALE_MMA_TILED, static_cast<int>(fmt),
                                            reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_quant_1x32_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q_row,
                               void* s_row, void* q_col, void* s_col, mxq_scale_layout layout,
                               mxq_stream_t stream) {
    return mxq_quant_1x32_dual_batched(x, 1, rows, cols, ld, 0, q_row, s_row, q_col, s_col, layout,
                                       MXQ_FP8_E4M3, stream);
}

mxq_status mxq_quant_1x32_cols_grouped(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                       const int64_t* group_offsets, int32_t G, int64_t capacity,
                                       void* q_col, void* s_col, mxq_scale_layout layout,
                                       mxq_stream_t stream) {
    return mxq_quant_1x32_cols_grouped_fmt(x, rows, cols, ld, group_offsets, G, capacity, q_col, s_col, layout,
                                           MXQ_FP8_E4M3, stream);
}

mxq_status mxq_quant_1x32_cols_grouped_fmt(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                           const int64_t* group_offsets, int32_t G, int64_t capacity,
                                           void* q_col, void* s_col, mxq_scale_layout layout, mxq_fp8_format fmt,
                                           mxq_stream_t stream) {
    if (layout != MXQ_SCALE_ROWMAJOR && layout != MXQ_SCALE_MMA_TILED) return MXQ_ERR_INVALID_ARG;
    if (fmt != MXQ_FP8_E4M3 && fmt != MXQ_FP8_E5M2) return MXQ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || G < 1 || capacity < 0) return MXQ_ERR_INVALID_ARG;
    if (G > 1024) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (cols % 32 != 0 || capacity % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (capacity < rows + 127 * static_cast<int64_t>(G)) return MXQ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0 || capacity == 0) return MXQ_OK;   // no tokens: every slot is empty
    if (!x || !group_offsets || !q_col || !s_col) return MXQ_ERR_INVALID_ARG;
    if (ld < cols || ld % 8 != 0) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q_col) || !aligned16(s_col) ||
        (reinterpret_cast<uintptr_t>(group_offsets) & 7u) != 0)
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_quant_cols_grouped(dev, x, rows, cols, ld, group_offsets, G, capacity, q_col,
                                                    s_col, layout == MXQ_SCALE_MMA_TILED, static_cast<int>(fmt),
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_quant_32x32(const void* w, int64_t n, int64_t k, int64_t ld, void* q, void* s_fwd,
                           void* s_bwd, mxq_scale_layout layout, mxq_stream_t stream) {
    return mxq_quant_32x32_fmt(w, n, k, ld, q, s_fwd, s_bwd, layout, MXQ_FP8_E4M3, stream);
}

mxq_status mxq_quant_32x32_fmt(const void* w, int64_t n, int64_t k, int64_t ld, void* q, void* s_fwd,
                               void* s_bwd, mxq_scale_layout layout, mxq_fp8_format fmt, mxq_stream_t stream) {
    if (layout != MXQ_SCALE_ROWMAJOR && layout != MXQ_SCALE_MMA_TILED) return MXQ_ERR_INVALID_ARG;
    if (fmt != MXQ_FP8_E4M3 && fmt != MXQ_FP8_E5M2) return MXQ_ERR_INVALID_ARG;
    if (n < 0 || k < 0) return MXQ_ERR_INVALID_ARG;
    if (n % 32 != 0 || k % 32 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (n == 0 || k == 0) return MXQ_OK;
    if (!w || !q) return MXQ_ERR_INVALID_ARG;
    if (ld < k || ld % 8 != 0) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || (s_fwd && !aligned16(s_fwd)) || (s_bwd && !aligned16(s_bwd)))
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_quant_32x32(dev, w, n, k, ld, q, s_fwd, s_bwd,
                                             layout == MXQ_SCALE_MMA_TILED, static_cast<int>(fmt),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_gemm_bf16out(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                            int64_t M, int64_t N, int64_t K, int b_mn_major, void* y, int64_t ldy,
                            mxq_scale_layout layout, mxq_stream_t stream) {
    // The tensor cores read only MMA-tiled scales; the row-major layout is
    // refused before anything else (an unsupported configuration).
    if (layout != MXQ_SCALE_MMA_TILED) return MXQ_ERR_INVALID_ARG;
    return mxq_gemm_bf16out_fmt(a_q, a_s, MXQ_FP8_E4M3, b_q, b_s, MXQ_FP8_E4M3, M, N, K, b_mn_major, y, ldy,
                                stream);
}

mxq_status mxq_gemm_bf16out_fmt(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q,
                                const void* b_s, mxq_fp8_format b_fmt, int64_t M, int64_t N, int64_t K,
                                int b_mn_major, void* y, int64_t ldy, mxq_stream_t stream) {
    DenseWork work;
    mxq_status st = check_dense(a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, b_mn_major, y, ldy, &work);
    if (st != MXQ_OK || work == kNothing) return st;
    mxq::DeviceInfo dev;
    st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    if (work == kZeroFill) return from_cuda(zero_fill(y, ldy, M, N, stream));
    return from_cuda(mxq::launch_gemm(dev, a_q, a_s, b_q, b_s, M, N, K, b_mn_major != 0, y, ldy,
                                      static_cast<int>(a_fmt), static_cast<int>(b_fmt),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_gemm_bf16out_multi(const mxq_gemm_desc* gemms, int32_t count, int b_mn_major,
                                  mxq_stream_t stream) {
    if (count < 0 || count > 4 || (count > 0 && !gemms)) return MXQ_ERR_INVALID_ARG;
    mxq::DenseGemm launch[4];
    int n_launch = 0;
    bool any_zero = false;
    for (int i = 0; i < count; ++i) {   // every GEMM is checked before anything runs
        const mxq_gemm_desc& g = gemms[i];
        DenseWork work;
        const mxq_status st = check_dense(g.a_q, g.a_s, g.a_fmt, g.b_q, g.b_s, g.b_fmt, g.M, g.N, g.K, b_mn_major,
                                          g.y, g.ldy, &work);
        if (st != MXQ_OK) return st;
        if (work == kZeroFill) any_zero = true;
        if (work == kLaunch)
            launch[n_launch++] = mxq::DenseGemm{g.a_q, g.a_s, g.b_q, g.b_s, g.M, g.N, g.K, g.y, g.ldy,
                                                static_cast<int>(g.a_fmt), static_cast<int>(g.b_fmt)};
    }
    if (n_launch == 0 && !any_zero) return MXQ_OK;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    for (int i = 0; i < count; ++i)
        if (gemms[i].K == 0 && gemms[i].M > 0 && gemms[i].N > 0) {
            const cudaError_t e = zero_fill(gemms[i].y, gemms[i].ldy, gemms[i].M, gemms[i].N, stream);
            if (e != cudaSuccess) return from_cuda(e);
        }
    if (n_launch == 0) return MXQ_OK;
    return from_cuda(mxq::launch_gemm_multi(dev, launch, n_launch, b_mn_major != 0,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_gemm_mxfp8out(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                             int64_t M, int64_t N, int64_t K, int b_mn_major, void* y, int64_t ldy,
                             void* y_q, void* y_s, mxq_stream_t stream) {
    if (M < 0 || N < 0 || K < 0 || (b_mn_major != 0 && b_mn_major != 1)) return MXQ_ERR_INVALID_ARG;
    if (K % 32 != 0 || K == 0 || N % 32 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (b_mn_major && N % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M > (int64_t(1) << 31) - 128 || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - 128)
        return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return MXQ_OK;
    if (y && (ldy < N || ldy % 8 != 0 || !aligned16(y))) return MXQ_ERR_INVALID_ARG;
    if (!a_q || !a_s || !b_q || !b_s || !y_q || !y_s) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(a_s) || !aligned16(b_q) || !aligned16(b_s) || !aligned16(y_q) ||
        !aligned16(y_s))
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_gemm_quant(dev, a_q, a_s, b_q, b_s, M, N, K, b_mn_major != 0, y, ldy, y_q,
                                            y_s, reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_fsdp_payload_layout(mxq_fsdp_recipe recipe, int64_t n, int64_t k, int32_t world,
                                   int64_t* offsets, int64_t* payload_bytes) {
    if ((recipe != MXQ_FSDP_1X32_DUAL && recipe != MXQ_FSDP_32X32) || !offsets || !payload_bytes)
        return MXQ_ERR_INVALID_ARG;
    if (world < 1 || n <= 0 || k <= 0 || n > (int64_t(1) << 31) || k > (int64_t(1) << 31))
        return MXQ_ERR_UNSUPPORTED_SHAPE;
    return mxq::fsdp_payload_layout(static_cast<int>(recipe), n, k, world, offsets, payload_bytes)
               ? MXQ_OK
               : MXQ_ERR_UNSUPPORTED_SHAPE;
}

mxq_status mxq_fsdp_unpack(mxq_fsdp_recipe recipe, int64_t n, int64_t k, int32_t world, const void* gathered,
                           void* q_fwd, void* s_fwd, void* q_bwd, void* s_bwd, mxq_stream_t stream) {
    int64_t off[4], payload = 0;
    const mxq_status lay = mxq_fsdp_payload_layout(recipe, n, k, world, off, &payload);
    if (lay != MXQ_OK) return lay;
    if (static_cast<int64_t>(world) * payload / 16 >= (int64_t(1) << 31)) return MXQ_ERR_UNSUPPORTED_SHAPE;
    const bool dual = recipe == MXQ_FSDP_1X32_DUAL;
    if (!gathered || !q_fwd || !s_fwd || !s_bwd || (dual != (q_bwd != nullptr))) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(gathered) || !aligned16(q_fwd) || !aligned16(s_fwd) || !aligned16(s_bwd) ||
        (dual && !aligned16(q_bwd)))
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_fsdp_unpack(dev, static_cast<int>(recipe), n, k, world, gathered, q_fwd, s_fwd,
                                             q_bwd, s_bwd, reinterpret_cast<cudaStream_t>(stream)));
}

size_t mxq_grouped_gemm_workspace_size(int32_t G, int64_t M_total, int64_t N, int64_t K) {
    if (G < 1 || G > 1024 || M_total < 0 || N < 0 || K <= 0 || K % 32 != 0 || M_total > (int64_t(1) << 31) - 128 ||
        K > (int64_t(1) << 31) - 128)
        return 0;
    return static_cast<size_t>(group_tiled_bytes(M_total, G, K));
}

mxq_status mxq_grouped_gemm(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                            const int64_t* group_offsets, int32_t G, int64_t M_total, int64_t N,
                            int64_t K, void* y, void* workspace, size_t workspace_bytes, mxq_stream_t stream) {
    return mxq_grouped_gemm_fmt(a_q, a_s, MXQ_FP8_E4M3, b_q, b_s, MXQ_FP8_E4M3, group_offsets, G, M_total, N, K, y,
                                N, workspace, workspace_bytes, stream);
}

mxq_status mxq_grouped_gemm_fmt(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q,
                                const void* b_s, mxq_fp8_format b_fmt, const int64_t* group_offsets, int32_t G,
                                int64_t M_total, int64_t N, int64_t K, void* y, int64_t ldy, void* workspace,
                                size_t workspace_bytes, mxq_stream_t stream) {
    if ((workspace == nullptr) != (workspace_bytes == 0)) return MXQ_ERR_INVALID_ARG;
    bool launch = false;
    mxq_status st = check_grouped_rows(a_q, a_s, a_fmt, b_q, b_s, b_fmt, group_offsets, G, M_total, N, K, y, ldy,
                                       &launch);
    if (st != MXQ_OK) return st;
    if (workspace != nullptr &&
        (!aligned16(workspace) || workspace_bytes < static_cast<size_t>(group_tiled_bytes(M_total, G, K))))
        return MXQ_ERR_INVALID_ARG;
    if (!launch) return MXQ_OK;
    mxq::DeviceInfo dev;
    st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int64_t bands = 0;
    const void* sa = a_s;
    if (workspace != nullptr) {   // A scales group-tiled in the workspace, then tiles from each expert's first row
        bands = group_tiled_bands(M_total, G);
        const cudaError_t e = mxq::launch_scale_regroup_rows(dev, a_s, M_total, K, group_offsets, G, bands,
                                                             workspace, s);
        if (e != cudaSuccess) return from_cuda(e);
        sa = workspace;
    }
    return from_cuda(mxq::launch_grouped_gemm(dev, a_q, sa, b_q, b_s, group_offsets, G, M_total, N, K, bands, y, ldy,
                                              static_cast<int>(a_fmt), static_cast<int>(b_fmt), s));
}

mxq_status mxq_grouped_gemm_group_tiled(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q,
                                        const void* b_s, mxq_fp8_format b_fmt, const int64_t* group_offsets,
                                        int32_t G, int64_t M_total, int64_t N, int64_t K, int64_t a_bands_cap,
                                        void* y, int64_t ldy, mxq_stream_t stream) {
    if (G >= 1 && M_total >= 0 && a_bands_cap < (M_total + 127) / 128 + G) return MXQ_ERR_INVALID_ARG;
    return grouped_rows_gemm(a_q, a_s, a_fmt, b_q, b_s, b_fmt, group_offsets, G, M_total, N, K, a_bands_cap, y,
                             ldy, stream);
}

mxq_status mxq_scale_regroup_rows(const void* s_tiled, int64_t rows, int64_t cols, const int64_t* group_offsets,
                                  int32_t G, int64_t bands_cap, void* s_out, mxq_stream_t stream) {
    if (G < 1 || rows < 0 || cols < 0) return MXQ_ERR_INVALID_ARG;
    if (G > 1024) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (cols % 32 != 0 || rows > (int64_t(1) << 31) - 128 || cols > (int64_t(1) << 31) - 128)
        return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (bands_cap < (rows + 127) / 128 + G) return MXQ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MXQ_OK;
    if (!s_tiled || !s_out || !group_offsets) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(s_tiled) || !aligned16(s_out) || (reinterpret_cast<uintptr_t>(group_offsets) & 7u) != 0)
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_scale_regroup_rows(dev, s_tiled, rows, cols, group_offsets, G, bands_cap, s_out,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}


mxq_status mxq_grouped_gemm_wgrad(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                                  const int64_t* group_offsets, int32_t G, int64_t M_total,
                                  int64_t capacity, int64_t M, int64_t N, void* y, int64_t ldy,
                                  mxq_stream_t stream) {
    return mxq_grouped_gemm_wgrad_fmt(a_q, a_s, MXQ_FP8_E4M3, b_q, b_s, MXQ_FP8_E4M3, group_offsets, G, M_total,
                                      capacity, M, N, y, ldy, stream);
}

mxq_status mxq_grouped_gemm_wgrad_fmt(const void* a_q, const void* a_s, mxq_fp8_format a_fmt, const void* b_q,
                                      const void* b_s, mxq_fp8_format b_fmt, const int64_t* group_offsets,
                                      int32_t G, int64_t M_total, int64_t capacity, int64_t M, int64_t N, void* y,
                                      int64_t ldy, mxq_stream_t stream) {
    if ((a_fmt != MXQ_FP8_E4M3 && a_fmt != MXQ_FP8_E5M2) || (b_fmt != MXQ_FP8_E4M3 && b_fmt != MXQ_FP8_E5M2))
        return MXQ_ERR_INVALID_ARG;
    if (G < 1 || M_total < 0 || M < 0 || N < 0 || capacity < 0) return MXQ_ERR_INVALID_ARG;
    if (G > 1024) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (N % 16 != 0 || capacity % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (capacity < M_total + 127 * static_cast<int64_t>(G)) return MXQ_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 128 || N > (int64_t(1) << 31) - 256 || capacity > (int64_t(1) << 31) - 128 ||
        static_cast<int64_t>(G) * M > (int64_t(1) << 40))
        return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return MXQ_OK;
    if (!a_q || !a_s || !b_q || !b_s || !group_offsets || !y) return MXQ_ERR_INVALID_ARG;
    if (ldy < N || ldy % 8 != 0) return MXQ_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(a_s) || !aligned16(b_q) || !aligned16(b_s) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(group_offsets) & 7u) != 0)
        return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    if (capacity == 0) {  // every expert is empty: y = 0
        return from_cuda(cudaMemset2DAsync(y, static_cast<size_t>(ldy) * 2, 0, static_cast<size_t>(N) * 2,
                                           static_cast<size_t>(G) * static_cast<size_t>(M),
                                           reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(mxq::launch_grouped_gemm_wgrad(dev, a_q, a_s, b_q, b_s, group_offsets, G, M_total,
                                                    capacity, M, N, y, ldy, static_cast<int>(a_fmt), static_cast<int>(b_fmt),
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

mxq_status mxq_get_device_status(mxq_stream_t stream) {
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(mxq::g_status_mu);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MXQ_ERR_CUDA;
    mxq::status_take_kernel<<<1, 1, 0, s>>>(dev.status);
    if (cudaGetLastError() != cudaSuccess) return MXQ_ERR_CUDA;
    unsigned int v = 0u;
    if (cudaMemcpyFromSymbolAsync(&v, g_mxq_status_taken, sizeof v, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MXQ_ERR_CUDA;
    return v != 0u ? MXQ_ERR_TIMEOUT : MXQ_OK;
}

mxq_status mxq_debug_wait_timeout(uint32_t timeout_us, mxq_stream_t stream) {
    if (timeout_us < 1u || timeout_us > 1000000u) return MXQ_ERR_INVALID_ARG;
    mxq::DeviceInfo dev;
    mxq_status st = device_ok(&dev);
    if (st != MXQ_OK) return st;
    return from_cuda(mxq::launch_wait_probe(dev, static_cast<uint64_t>(timeout_us) * 1000ull,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
