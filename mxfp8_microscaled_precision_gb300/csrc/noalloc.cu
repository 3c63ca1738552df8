// noalloc.cu -- mxq_grouped_gemm_noalloc: the grouped GEMM with its
// per-expert A-scale workspace taken from a fixed array that the library
// itself holds in device memory, for callers that cannot allocate.
//
// mxq_grouped_gemm can use a caller-supplied workspace (A's scales re-tiled
// per expert, so that no 128-row tile spans two experts).  Some callers have
// no way to provide one: code that only receives its input and output buffers
// from a host framework or serving runtime whose allocator owns all device
// memory and hands out nothing else, and code that must not call cudaMalloc /
// cudaFree because those calls can synchronize the whole device.  This entry
// point gives them the same computation with the scratch bytes in a
// file-scope __device__ array instead.
//
// The array is module data: every GPU that loads this library holds its
// kNoallocScratchBytes until the process exits, and all calls share it.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

// Scratch of the allocation-free grouped GEMM (A's scales tiled per expert).
constexpr size_t kNoallocScratchBytes = MXQ_GROUPED_NOALLOC_MAX_WORKSPACE;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device

// The device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and kept.
cudaError_t scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

mxq_status mxq_grouped_gemm_noalloc(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                                    const int64_t* group_offsets, int32_t G, int64_t M_total, int64_t N, int64_t K,
                                    void* y, mxq_stream_t stream) {
    const size_t need = mxq_grouped_gemm_workspace_size(G, M_total, N, K);
    // A zero size means arguments mxq_grouped_gemm refuses: it reports which,
    // before anything runs, and never touches a workspace.
    if (need == 0)
        return mxq_grouped_gemm_fmt(a_q, a_s, MXQ_FP8_E4M3, b_q, b_s, MXQ_FP8_E4M3, group_offsets, G, M_total, N,
                                    K, y, N, nullptr, 0, stream);
    if (need > kNoallocScratchBytes) return MXQ_ERR_UNSUPPORTED_SHAPE;   // past the array's fixed size
    mxq::DeviceInfo info;
    if (mxq::current_device_info(&info) != cudaSuccess) return MXQ_ERR_CUDA;
    if (info.cc_major != 10 || info.cc_minor != 3) return MXQ_ERR_UNSUPPORTED_DEVICE;
    void* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return MXQ_ERR_CUDA;
    return mxq_grouped_gemm_fmt(a_q, a_s, MXQ_FP8_E4M3, b_q, b_s, MXQ_FP8_E4M3, group_offsets, G, M_total, N, K,
                                y, N, scratch, kNoallocScratchBytes, stream);
}

}  // extern "C"
