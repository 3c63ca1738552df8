// fsdp.cu -- the all-gather payload of a pre-quantized weight under fully
// sharded data parallelism (MindSpeed RFC "Add MXFP8-32x32 quantization
// support to FSDP", section 3.3.2): each rank quantizes its 128-row-aligned
// shard of the weight straight into one contiguous payload (the quantizers
// write at the offsets given here, so packing costs no copy); the collective
// concatenates the ranks' payloads; `fsdp_unpack_kernel` then rebuilds the
// full-weight operands the GEMMs read.  The 1x32 dual recipe moves four
// tensors (row payload, row scales, column payload, column scales), the 32x32
// recipe three (one payload, two scales).
//
// Where each shard tensor lands in the full operand:
//   row payload  [n_s, K]          -> rows r*n_s.. of [N, K]           (contiguous)
//   row scales   tiled [n_s, K/32] -> 128-row bands of [N, K/32]       (contiguous)
//   col payload  [K, n_s]          -> columns r*n_s.. of [K, N]        (K strided rows)
//   col scales   tiled [K, n_s/32] -> atoms r*n_s/128.. of every band  (strided)
// (n_s = N / world, a multiple of 128, so no scale atom spans two ranks.)

#include <cuda_runtime.h>

#include <cstdint>

#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // 16-byte chunks in flight per thread

struct CopyPlan {
    uint8_t* dst;
    int64_t src_off;       // offset of the tensor inside one rank's payload
    int64_t dst_rank_off;  // bytes between consecutive ranks' blocks in dst
    int64_t dst_stride;    // bytes between rows in dst
    uint32_t row_chunks;   // 16-byte chunks per row
    uint32_t chunks;       // chunks per rank (rows * row_chunks)
};

struct UnpackArgs {
    const uint8_t* src;
    int64_t payload;       // bytes of one rank's payload
    uint32_t world;
    int n_plans;
    CopyPlan plan[4];
};

int64_t tiled_bytes(int64_t rows, int64_t cols) {
    return (rows + 127) / 128 * 128 * ((cols / 32 + 3) / 4 * 4);
}

// One copy per 16-byte chunk, kUnroll chunks per thread in flight; the chunk
// index runs over ranks, rows and row chunks of one tensor at a time.
__global__ void __launch_bounds__(kThreads) fsdp_unpack_kernel(const __grid_constant__ UnpackArgs a) {
    for (int t = 0; t < a.n_plans; ++t) {
        const CopyPlan& p = a.plan[t];
        const uint32_t total = p.chunks * a.world;
        const uint32_t span = static_cast<uint32_t>(kThreads * kUnroll);
        for (uint32_t base = blockIdx.x * span; base < total; base += gridDim.x * span) {
            uint4 v[kUnroll];
            uint8_t* d[kUnroll];
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
                const uint32_t i = base + j * kThreads + threadIdx.x;
                d[j] = nullptr;
                if (i < total) {
                    const uint32_t rank = i / p.chunks;
                    const uint32_t rem = i - rank * p.chunks;
                    const uint32_t row = rem / p.row_chunks;
                    const uint32_t col = rem - row * p.row_chunks;
                    const uint8_t* s = a.src + rank * a.payload + p.src_off + static_cast<int64_t>(rem) * 16;
                    v[j] = __ldcs(reinterpret_cast<const uint4*>(s));
                    d[j] = p.dst + rank * p.dst_rank_off + row * p.dst_stride + static_cast<int64_t>(col) * 16;
                }
            }
#pragma unroll
            for (int j = 0; j < kUnroll; ++j)
                if (d[j] != nullptr) *reinterpret_cast<uint4*>(d[j]) = v[j];
        }
    }
}

}  // namespace

bool fsdp_payload_layout(int recipe, int64_t n, int64_t k, int32_t world, int64_t offsets[4],
                         int64_t* payload_bytes) {
    if (world < 1 || n <= 0 || k <= 0 || n % (128 * static_cast<int64_t>(world)) != 0 || k % 32 != 0)
        return false;
    if (recipe != 0 && recipe != 1) return false;
    const int64_t ns = n / world;
    const int64_t q = ns * k;
    const int64_t sf = tiled_bytes(ns, k);
    const int64_t sb = tiled_bytes(k, ns);
    offsets[0] = 0;
    offsets[1] = q;
    if (recipe == 0) {
        offsets[2] = q + sf;
        offsets[3] = 2 * q + sf;
        *payload_bytes = 2 * q + sf + sb;
    } else {
        offsets[2] = -1;
        offsets[3] = q + sf;
        *payload_bytes = q + sf + sb;
    }
    return true;
}

cudaError_t launch_fsdp_unpack(const DeviceInfo& dev, int recipe, int64_t n, int64_t k, int32_t world,
                               const void* gathered, void* q_fwd, void* s_fwd, void* q_bwd, void* s_bwd,
                               cudaStream_t stream) {
    int64_t off[4], payload = 0;
    if (!fsdp_payload_layout(recipe, n, k, world, off, &payload)) return cudaErrorInvalidValue;
    const int64_t ns = n / world;
    const int64_t kb = (k + 127) / 128;  // 128-row bands of the column scales
    UnpackArgs a{};
    a.src = static_cast<const uint8_t*>(gathered);
    a.payload = payload;
    a.world = static_cast<uint32_t>(world);
    auto add = [&](void* dst, int64_t src_off, int64_t rows, int64_t row_bytes, int64_t dst_stride,
                   int64_t dst_rank_off) {
        CopyPlan& p = a.plan[a.n_plans++];
        p.dst = static_cast<uint8_t*>(dst);
        p.src_off = src_off;
        p.dst_rank_off = dst_rank_off;
        p.dst_stride = dst_stride;
        p.row_chunks = static_cast<uint32_t>(row_bytes / 16);
        p.chunks = static_cast<uint32_t>(rows * (row_bytes / 16));
    };
    const int64_t sf = off[recipe == 0 ? 2 : 3] - off[1];
    add(q_fwd, off[0], 1, ns * k, 0, ns * k);
    add(s_fwd, off[1], 1, sf, 0, sf);
    if (recipe == 0) add(q_bwd, off[2], k, ns, n, ns);
    add(s_bwd, off[3], kb, ns / 128 * 512, n / 128 * 512, ns / 128 * 512);
    int64_t most = 0;
    for (int t = 0; t < a.n_plans; ++t) {
        const int64_t c = static_cast<int64_t>(a.plan[t].chunks) * world;
        if (c >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // 32-bit chunk indices
        most = c > most ? c : most;
    }
    const int64_t span = kThreads * kUnroll;
    int64_t grid = (most + span - 1) / span;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    fsdp_unpack_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace mxq
