// mxq_internal.h -- host-side launchers shared between the C ABI (api.cu)
// and the kernel translation units.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxq {

// Per-device facts the launchers need.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;            // max dynamic shared memory per block
    unsigned int* status = nullptr;   // device status word (timeouts)
};

// Returns cudaSuccess and fills `info` for the current device.
cudaError_t current_device_info(DeviceInfo* info);

// 2-D tensor map over a row-major matrix [outer, inner] of 1- or 2-byte
// elements with the given row stride, box [box_outer, box_inner].
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, bool two_byte_elems, uint64_t inner,
                          uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                          uint32_t box_outer, bool swizzle_128b);

// 3-D tensor map [outer, mid, inner], box [1, box_mid, box_inner], no swizzle.
// BF16 [rows, cols] (row stride ld elements) for 32 x 32 tiled stores with the
// 64-byte swizzle.
bool encode_tensor_map_bf16_store(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                                  uint64_t ld);
// Bytes [rows, cols] (row stride ld bytes) for 32 x 32 tiled stores, no swizzle.
bool encode_tensor_map_u8_store(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t ld);
bool encode_tensor_map_3d(CUtensorMap* map, const void* base, bool two_byte_elems, uint64_t inner,
                          uint64_t mid, uint64_t outer, uint64_t mid_stride_bytes,
                          uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_mid);

// 1x32 quantization of `batch` matrices [rows, cols] (row stride ld, matrix
// stride batch_stride elements); outputs of matrix b follow each other.
// fmt: 0 = E4M3, 1 = E5M2.
cudaError_t launch_quant_1x32(const DeviceInfo& dev, const void* x, int64_t batch, int64_t rows,
                              int64_t cols, int64_t ld, int64_t batch_stride, void* q_row,
                              void* s_row, void* q_col, void* s_col, bool tiled, int fmt,
                              cudaStream_t stream);

// Token-axis 1x32 quantization inside each expert (zero-padded, 128-aligned slots).
cudaError_t launch_quant_cols_grouped(const DeviceInfo& dev, const void* x, int64_t rows,
                                      int64_t cols, int64_t ld, const int64_t* offsets, int G,
                                      int64_t capacity, void* q_col, void* s_col, bool tiled, int fmt,
                                      cudaStream_t stream);

// 32x32 block quantization (fmt: 0 = E4M3, 1 = E5M2).
cudaError_t launch_quant_32x32(const DeviceInfo& dev, const void* w, int64_t n, int64_t k,
                               int64_t ld, void* q, void* s_fwd, void* s_bwd, bool tiled, int fmt,
                               cudaStream_t stream);

// One dense GEMM y = A B^T of a multi-GEMM launch (fields as in mxq_gemm_bf16out_fmt).
struct DenseGemm {
    const void* a_q;
    const void* a_s;
    const void* b_q;
    const void* b_s;
    int64_t M, N, K;
    void* y;
    int64_t ldy;
    int a_fmt, b_fmt;
};

// 1 to 4 dense GEMMs (all with B K-major, or all MN-major) in one persistent
// launch over their output tiles.  cudaErrorInvalidValue for a bad count or
// shapes whose tensor maps cannot be encoded.
cudaError_t launch_gemm_multi(const DeviceInfo& dev, const DenseGemm* gemms, int count, bool b_mn_major,
                              cudaStream_t stream);

// Dense block-scaled GEMM (see mxq_gemm_bf16out).  Returns cudaErrorInvalidValue
// when a tensor map cannot be encoded for the given shapes.
cudaError_t launch_gemm(const DeviceInfo& dev, const void* a_q, const void* a_s, const void* b_q,
                        const void* b_s, int64_t M, int64_t N, int64_t K, bool b_mn_major, void* y,
                        int64_t ldy, int a_fmt, int b_fmt, cudaStream_t stream);

// Dense GEMM whose epilogue also writes the 1x32 E4M3 quantization of the BF16
// output (y may be null: quantized output only).
cudaError_t launch_gemm_quant(const DeviceInfo& dev, const void* a_q, const void* a_s, const void* b_q,
                              const void* b_s, int64_t M, int64_t N, int64_t K, bool b_mn_major, void* y,
                              int64_t ldy, void* y_q, void* y_s, cudaStream_t stream);

// All-gather payload of a pre-quantized weight shard: tensor byte offsets in
// one rank's payload (offsets[2] = -1 for the 32x32 recipe) and its size.
// False when the shape is not supported (n % (128*world), k % 32).
bool fsdp_payload_layout(int recipe, int64_t n, int64_t k, int32_t world, int64_t offsets[4],
                         int64_t* payload_bytes);
cudaError_t launch_fsdp_unpack(const DeviceInfo& dev, int recipe, int64_t n, int64_t k, int32_t world,
                               const void* gathered, void* q_fwd, void* s_fwd, void* q_bwd, void* s_bwd,
                               cudaStream_t stream);

// a_bands_cap: 0 = A scales MMA-tiled over all rows; > 0 = group-tiled (see
// mxq_scale_regroup_rows) in a buffer of a_bands_cap bands.
cudaError_t launch_grouped_gemm(const DeviceInfo& dev, const void* a_q, const void* a_s,
                                const void* b_q, const void* b_s, const int64_t* offsets, int G,
                                int64_t M_total, int64_t N, int64_t K, int64_t a_bands_cap, void* y,
                                int64_t ldy, int a_fmt, int b_fmt, cudaStream_t stream);

// Group-tiled copy of the MMA-tiled scales of a row quantization (see
// mxq_scale_regroup_rows).
cudaError_t launch_scale_regroup_rows(const DeviceInfo& dev, const void* s_tiled, int64_t rows, int64_t cols,
                                      const int64_t* offsets, int G, int64_t bands_cap, void* s_out,
                                      cudaStream_t stream);

// Grouped contraction (MoE weight gradient): y[g] = A_g B_g^T where the K range
// of expert g is its 128-aligned token slot; A [M, capacity], B [N, capacity].
cudaError_t launch_grouped_gemm_wgrad(const DeviceInfo& dev, const void* a_q, const void* a_s,
                                      const void* b_q, const void* b_s, const int64_t* offsets, int G,
                                      int64_t M_total, int64_t capacity, int64_t M, int64_t N, void* y,
                                      int64_t ldy, int a_fmt, int b_fmt, cudaStream_t stream);

cudaError_t launch_wait_probe(const DeviceInfo& dev, uint64_t limit_ns, cudaStream_t stream);

}  // namespace mxq
