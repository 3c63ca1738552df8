// quant.cu -- MXFP8 quantizers for sm_103a.
//
//  * 1x32 (row and/or column copy): one E8M0 scale per 32 consecutive
//    elements along the quantized axis (torchtitan-npu low-precision
//    tutorial, "MXFP8 与 HiF8 架构原理速览"; the dual-axis form of the MindSpeed
//    RFC "Add MXFP8-32x32 quantization support to FSDP", section 3.3.3).
//  * 32x32: one scale per 32x32 tile and a single payload shared by the
//    forward and backward GEMMs (same RFC, sections 3.1 and 3.3.3).
//
// Both are HBM-bound.  A CTA of 256 threads owns a 128x128 BF16 tile:
// every thread issues its eight 16-byte loads up front, the amax of a
// 32-group is reduced over the four lanes that hold it with two shuffles,
// the exponent is the exact rceil rule evaluated on the BF16 bits of amax,
// the scaling by 2^-e is an exact multiply, and one cvt.rn.satfinite
// instruction rounds two values to E4M3.  The column copy is produced from
// the same tile staged in shared memory, so the input is read once.
// Scales go out either plain or in the MMA-tiled layout; the tiled
// permutation is fused into the scale stores (and writes its zero padding).

#include <cuda_runtime.h>

#include <cstdint>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr int kLoadsPerThread = kTile * kTile / 8 / kThreads;  // 8 x 16-byte loads

// E8M0 exponent of a finite, non-negative amax given as BF16 bits
// (sign cleared): e = ceil(log2(amax/448)), clamped below at -127.
// With amax = 1.m * 2^(E-127): amax/448 = (1.m/1.75) * 2^(E-135), and the
// ceiling steps up exactly when the 7-bit mantissa exceeds 1.75 (m > 96).
// Subnormal and zero amax (E == 0) fall below -127 and are clamped.
__device__ __forceinline__ int rceil_exponent(uint32_t amax_bits) {
    const int E = static_cast<int>(amax_bits >> 7);
    const int m = static_cast<int>(amax_bits & 0x7Fu);
    const int e = E - 135 + (m > 96 ? 1 : 0);
    return e < -127 ? -127 : e;
}

// 2^-e as a float for e in [-127, 120] (always a normal number).
__device__ __forceinline__ float pow2_neg(int e) { return __int_as_float((127 - e) << 23); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t abs_max_bits(uint32_t w, uint32_t m) {
    m = max(m, w & 0x7FFFu);
    return max(m, (w >> 16) & 0x7FFFu);
}

// Quantize 8 BF16 values (4 words) with scale 2^-e -> 8 E4M3 bytes.
__device__ __forceinline__ uint2 quant8(const uint4 v, float sc) {
    uint2 o;
    o.x = cvt_e4m3x2(bf16_lo(v.x) * sc, bf16_hi(v.x) * sc) |
          (cvt_e4m3x2(bf16_lo(v.y) * sc, bf16_hi(v.y) * sc) << 16);
    o.y = cvt_e4m3x2(bf16_lo(v.z) * sc, bf16_hi(v.z) * sc) |
          (cvt_e4m3x2(bf16_lo(v.w) * sc, bf16_hi(v.w) * sc) << 16);
    return o;
}

// Payload of a group holding NaN or Inf: every byte 0x7F | sign.
__device__ __forceinline__ uint32_t nan_bytes4(uint32_t w0, uint32_t w1) {
    return 0x7F7F7F7Fu | ((w0 >> 8) & 0x80u) | ((w0 >> 16) & 0x8000u) | ((w1 << 8) & 0x800000u) |
           (w1 & 0x80000000u);
}

__device__ __forceinline__ uint2 nan8(const uint4 v) {
    return make_uint2(nan_bytes4(v.x, v.y), nan_bytes4(v.z, v.w));
}

__device__ __forceinline__ void store_scale(uint8_t* s, int64_t r, int64_t g, int64_t groups,
                                            bool tiled, uint8_t code) {
    if (tiled)
        s[tiled_scale_offset(r, g, groups)] = code;
    else
        s[r * groups + g] = code;
}

// ---------------------------------------------------------------------------------
// 1x32 quantization: row copy and/or column copy of one 128x128 tile.
// Thread t loads rows (t/16 + 16 i), i = 0..7, 16-byte chunk (t % 16) of the
// tile; the four chunks of one 32-group sit in four consecutive lanes.
template <bool kRow, bool kCol, bool kTiled>
__global__ void __launch_bounds__(kThreads) quant_1x32_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col,
    uint8_t* __restrict__ s_col) {
    // Column pass staging: 128 rows x 128 BF16 (row stride 256 bytes).
    __shared__ __align__(16) uint32_t tile[kCol ? kTile * kTile / 2 : 1];

    const int t = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTile;
    const int chunk = t & 15;
    const int64_t col = c0 + chunk * 8;
    const bool col_ok = col < cols;
    const int64_t groups = cols >> 5;

    uint4 v[kLoadsPerThread];
#pragma unroll
    for (int i = 0; i < kLoadsPerThread; ++i) {
        const int64_t r = r0 + (t >> 4) + 16 * i;
        if (col_ok && r < rows)
            v[i] = __ldg(reinterpret_cast<const uint4*>(x + r * ld + col));
        else
            v[i] = make_uint4(0u, 0u, 0u, 0u);
    }

    if constexpr (kCol) {
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i)
            reinterpret_cast<uint4*>(tile)[((t >> 4) + 16 * i) * 16 + chunk] = v[i];
    }

    if constexpr (kRow) {
        const int64_t g = col >> 5;  // group of this chunk
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i) {
            const int64_t r = r0 + (t >> 4) + 16 * i;
            uint32_t m = abs_max_bits(v[i].x, 0u);
            m = abs_max_bits(v[i].y, m);
            m = abs_max_bits(v[i].z, m);
            m = abs_max_bits(v[i].w, m);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            const bool valid = col_ok && r < rows;
            uint8_t code;
            uint2 out;
            if (m >= 0x7F80u) {  // NaN or Inf in the group
                code = 0xFF;
                out = nan8(v[i]);
            } else {
                const int e = rceil_exponent(m);
                code = static_cast<uint8_t>(e + 127);
                out = quant8(v[i], pow2_neg(e));
            }
            if (valid) *reinterpret_cast<uint2*>(q_row + r * cols + col) = out;
            if ((chunk & 3) == 0) {
                if (valid)
                    store_scale(s_row, r, g, groups, kTiled, code);
                else if (kTiled)  // zero padding of the tiled layout
                    store_scale(s_row, r, g, groups, true, 0);
            }
        }
    }

    if constexpr (kCol) {
        __syncthreads();
        // Thread t: column pair p = t % 64 (columns 2p, 2p+1 of the tile) and
        // 32-row group gi = t / 64.  A warp reads 128 contiguous bytes of one
        // tile row per step, so the shared-memory reads are conflict-free.
        const int p = t & 63;
        const int gi = t >> 6;
        const int64_t cA = c0 + 2 * p;               // output row of q_col
        const int64_t rbase = r0 + 32 * gi;          // first input row of the group
        const int64_t rgroups = rows >> 5;           // groups per q_col row
        const int64_t g_out = rbase >> 5;
        const bool ok = cA < cols && rbase < rows;   // rows % 32 == 0 in column mode
        uint32_t w[32];
        uint32_t mlo = 0u, mhi = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            w[j] = tile[(32 * gi + j) * 64 + p];
            mlo = max(mlo, w[j] & 0x7FFFu);
            mhi = max(mhi, (w[j] >> 16) & 0x7FFFu);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t m = half ? mhi : mlo;
            const int64_t c = cA + half;
            uint8_t code;
            uint32_t o[8];
            if (m >= 0x7F80u) {
                code = 0xFF;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t b = 0x7F7F7F7Fu;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t hbits = half ? (w[4 * j + u] >> 16) : (w[4 * j + u] & 0xFFFFu);
                        b |= ((hbits >> 15) & 1u) << (8 * u + 7);
                    }
                    o[j] = b;
                }
            } else {
                const int e = rceil_exponent(m);
                const float sc = pow2_neg(e);
                code = static_cast<uint8_t>(e + 127);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float f[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        f[u] = (half ? bf16_hi(w[4 * j + u]) : bf16_lo(w[4 * j + u])) * sc;
                    o[j] = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
                }
            }
            if (ok) {
                uint4* dst = reinterpret_cast<uint4*>(q_col + c * rows + rbase);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                store_scale(s_col, c, g_out, rgroups, kTiled, code);
            } else if (kTiled) {
                store_scale(s_col, c, g_out, rgroups, true, 0);
            }
        }
    }
}

// ---------------------------------------------------------------------------------
// 32x32 block quantization of one 128x128 tile of w [n, k]: 16 blocks.
template <bool kTiled>
__global__ void __launch_bounds__(kThreads) quant_32x32_kernel(
    const uint16_t* __restrict__ w, int64_t n, int64_t k, int64_t ld, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s_fwd, uint8_t* __restrict__ s_bwd) {
    __shared__ uint32_t blk_amax[4][4];  // [32-row block][32-col block] of this tile
    const int t = threadIdx.x;
    if (t < 16) blk_amax[t >> 2][t & 3] = 0u;

    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTile;
    const int chunk = t & 15;
    const int gcol = chunk >> 2;  // 32-column block within the tile
    const int64_t col = c0 + chunk * 8;
    const bool col_ok = col < k;

    uint4 v[kLoadsPerThread];
#pragma unroll
    for (int i = 0; i < kLoadsPerThread; ++i) {
        const int64_t r = r0 + (t >> 4) + 16 * i;
        if (col_ok && r < n)
            v[i] = __ldg(reinterpret_cast<const uint4*>(w + r * ld + col));
        else
            v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();  // blk_amax initialised

    // Row i of this thread lies in 32-row block i/2 of the tile.
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t m = 0u;
#pragma unroll
        for (int i = 2 * b; i < 2 * b + 2; ++i) {
            m = abs_max_bits(v[i].x, m);
            m = abs_max_bits(v[i].y, m);
            m = abs_max_bits(v[i].z, m);
            m = abs_max_bits(v[i].w, m);
        }
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        if ((chunk & 3) == 0) atomicMax(&blk_amax[b][gcol], m);
    }
    __syncthreads();

    const int64_t kgroups = k >> 5, ngroups = n >> 5;
#pragma unroll
    for (int i = 0; i < kLoadsPerThread; ++i) {
        const int64_t r = r0 + (t >> 4) + 16 * i;
        const uint32_t m = blk_amax[i >> 1][gcol];
        const bool valid = col_ok && r < n;
        uint8_t code;
        uint2 out;
        if (m >= 0x7F80u) {
            code = 0xFF;
            out = nan8(v[i]);
        } else {
            const int e = rceil_exponent(m);
            code = static_cast<uint8_t>(e + 127);
            out = quant8(v[i], pow2_neg(e));
        }
        if (valid) *reinterpret_cast<uint2*>(q + r * k + col) = out;
        if (s_fwd && (chunk & 3) == 0) {
            if (valid)
                store_scale(s_fwd, r, col >> 5, kgroups, kTiled, code);
            else if (kTiled)
                store_scale(s_fwd, r, col >> 5, kgroups, true, 0);
        }
    }

    // s_bwd [k, n/32]: row c (a column of w), group = 32-row block of w.
    if (s_bwd) {
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
            const int idx = t + kThreads * e2;   // 0..511
            const int cl = idx & 127, b = idx >> 7;
            const int64_t c = c0 + cl;
            const int64_t gi = (r0 >> 5) + b;
            const bool valid = c < k && gi < ngroups;
            const uint32_t m = blk_amax[b][cl >> 5];
            uint8_t code = 0;
            if (valid) code = (m >= 0x7F80u) ? 0xFF : static_cast<uint8_t>(rceil_exponent(m) + 127);
            if (valid || kTiled) store_scale(s_bwd, c, gi, ngroups, kTiled, code);
        }
    }
}

template <bool kRow, bool kCol>
cudaError_t launch_1x32_t(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q_row,
                          void* s_row, void* q_col, void* s_col, bool tiled, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((cols + kTile - 1) / kTile),
                    static_cast<unsigned>((rows + kTile - 1) / kTile));
    auto xp = static_cast<const uint16_t*>(x);
    auto qr = static_cast<uint8_t*>(q_row);
    auto sr = static_cast<uint8_t*>(s_row);
    auto qc = static_cast<uint8_t*>(q_col);
    auto sc = static_cast<uint8_t*>(s_col);
    if (tiled)
        quant_1x32_kernel<kRow, kCol, true><<<grid, kThreads, 0, stream>>>(xp, rows, cols, ld, qr, sr,
                                                                           qc, sc);
    else
        quant_1x32_kernel<kRow, kCol, false><<<grid, kThreads, 0, stream>>>(xp, rows, cols, ld, qr,
                                                                            sr, qc, sc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_1x32(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q_row,
                              void* s_row, void* q_col, void* s_col, bool tiled,
                              cudaStream_t stream) {
    const bool row = q_row != nullptr, col = q_col != nullptr;
    if (row && col)
        return launch_1x32_t<true, true>(x, rows, cols, ld, q_row, s_row, q_col, s_col, tiled, stream);
    if (row)
        return launch_1x32_t<true, false>(x, rows, cols, ld, q_row, s_row, q_col, s_col, tiled, stream);
    return launch_1x32_t<false, true>(x, rows, cols, ld, q_row, s_row, q_col, s_col, tiled, stream);
}

cudaError_t launch_quant_32x32(const void* w, int64_t n, int64_t k, int64_t ld, void* q,
                               void* s_fwd, void* s_bwd, bool tiled, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((k + kTile - 1) / kTile),
                    static_cast<unsigned>((n + kTile - 1) / kTile));
    auto wp = static_cast<const uint16_t*>(w);
    auto qp = static_cast<uint8_t*>(q);
    auto sf = static_cast<uint8_t*>(s_fwd);
    auto sb = static_cast<uint8_t*>(s_bwd);
    if (tiled)
        quant_32x32_kernel<true><<<grid, kThreads, 0, stream>>>(wp, n, k, ld, qp, sf, sb);
    else
        quant_32x32_kernel<false><<<grid, kThreads, 0, stream>>>(wp, n, k, ld, qp, sf, sb);
    return cudaGetLastError();
}

}  // namespace mxq
