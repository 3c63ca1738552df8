// quant.cu -- MXFP8 quantizers for sm_103a.
//
//  * 1x32 (row and/or column copy): one E8M0 scale per 32 consecutive
//    elements along the quantized axis (torchtitan-npu low-precision
//    tutorial, "MXFP8 与 HiF8 架构原理速览"; the dual-axis form of the MindSpeed
//    RFC "Add MXFP8-32x32 quantization support to FSDP", section 3.3.3).
//  * 32x32: one scale per 32x32 tile and a single payload shared by the
//    forward and backward GEMMs (same RFC, sections 3.1 and 3.3.3).
//
// Both are HBM-bound.  Persistent CTAs of 256 threads stream 128x128 BF16
// tiles through a two-slot shared-memory ring filled by TMA, so the loads of
// the next tiles overlap the quantization and stores of the current one.
// The amax of a 32-group is reduced over the four lanes that hold it with
// two shuffles (row groups) or by one thread over a shared-memory column
// (column groups); the exponent is the exact rceil rule evaluated on the
// BF16 bits of amax; the scaling by 2^-e is an exact multiply; one
// cvt.rn.satfinite instruction rounds two values to E4M3.  The column copy
// reads the same staged tile, so the input is read from HBM once.  Scales
// go out plain or in the MMA-tiled layout; the tiled permutation is fused
// into the scale stores (which also write its zero padding).

#include <cuda_runtime.h>

#include <cstdint>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr int kLoadsPerThread = kTile * kTile / 8 / kThreads;  // 8 x 16-byte chunks
constexpr int kRing = 2;                                        // tile slots per CTA
constexpr int kTileBytes = kTile * kTile * 2;                   // 32 KB of BF16
constexpr int kCtasPerSm = 3;
constexpr int kSmemBytes = kRing * kTileBytes + 1024 + 256;     // ring + alignment + barriers

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

// Shared-memory ring of TMA-filled tiles, shared by both quantizers.
struct Ring {
    uint8_t* buf;        // kRing slots of kTileBytes, 1024-byte aligned
    uint32_t bar0;       // kRing full barriers (8 bytes apart)
    volatile int* abort_flag;
};

__device__ __forceinline__ Ring ring_setup(uint8_t* smem_raw) {
    Ring r;
    r.buf = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
    r.bar0 = smem_u32(r.buf + kRing * kTileBytes);
    r.abort_flag = reinterpret_cast<volatile int*>(r.buf + kRing * kTileBytes + 8 * kRing);
    return r;
}

// Issue the TMA load of tile `tile` (tiles_c tiles per 128-row band) into slot s.
__device__ __forceinline__ void ring_load(const Ring& r, const CUtensorMap* map, int s, int64_t tile,
                                          int64_t tiles_c) {
    const uint32_t bar = r.bar0 + 8u * s;
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_2d(smem_u32(r.buf + s * kTileBytes), map, static_cast<int32_t>((tile % tiles_c) * kTile),
                static_cast<int32_t>((tile / tiles_c) * kTile), bar);
}

// Thread 0 initialises the barriers and issues the first kRing loads.
__device__ __forceinline__ void ring_start(const Ring& r, const CUtensorMap* map, int64_t n_tiles,
                                           int64_t tiles_c) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) mbar_init(r.bar0 + 8u * s, 1);
        *r.abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(map);
        for (int s = 0; s < kRing; ++s) {
            const int64_t tile = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (tile < n_tiles) ring_load(r, map, s, tile, tiles_c);
        }
    }
    __syncthreads();
}

// Waits for slot i % kRing; the verdict is block-uniform (false: give up).
__device__ __forceinline__ bool ring_wait(const Ring& r, int i, const WaitGuard& g) {
    const uint32_t bar = r.bar0 + 8u * (i % kRing);
    const uint32_t parity = static_cast<uint32_t>(i / kRing) & 1u;
    const bool ok = mbar_try_wait(bar, parity) || mbar_wait(bar, parity, g);
    return !__syncthreads_or(!ok);
}

// After every thread is done with slot i % kRing: refill it with the tile
// kRing iterations ahead.
__device__ __forceinline__ void ring_release(const Ring& r, const CUtensorMap* map, int i, int64_t tile,
                                             int64_t n_tiles, int64_t tiles_c) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const int64_t next = tile + static_cast<int64_t>(kRing) * gridDim.x;
        if (next < n_tiles) ring_load(r, map, i % kRing, next, tiles_c);
    }
}

// After a timeout, let the loads still in flight land before the CTA exits.
__device__ __forceinline__ void ring_drain(const Ring& r, int i, int64_t tile, int64_t n_tiles,
                                           const WaitGuard& g) {
    if (threadIdx.x != 0 || !*r.abort_flag) return;
    WaitGuard g2 = g;
    volatile int never = 0;
    g2.abort_flag = &never;
    for (int j = 0; j < kRing; ++j) {
        const int64_t t = tile + static_cast<int64_t>(j) * gridDim.x;
        if (t < n_tiles)
            (void)mbar_wait(r.bar0 + 8u * ((i + j) % kRing), static_cast<uint32_t>((i + j) / kRing) & 1u, g2);
    }
}

// ---------------------------------------------------------------------------------
// 1x32 quantization: row copy and/or column copy, tile by tile.
// Row pass: thread t takes rows (t/16 + 16 i), i = 0..7, 16-byte chunk t % 16
// of the tile; the four chunks of one 32-group sit in four consecutive lanes.
// Column pass: thread t takes the column pair t % 64 and the 32-row group
// t / 64; a warp reads 128 contiguous bytes of one tile row per step, so the
// shared-memory reads are conflict-free.
template <bool kRow, bool kCol, bool kTiled>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quant_1x32_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col,
    uint8_t* __restrict__ s_col, int64_t tiles_c, int64_t n_tiles, unsigned int* status,
    uint64_t wait_limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const Ring ring = ring_setup(smem_raw);
    const WaitGuard guard{ring.abort_flag, status, wait_limit_ns};
    ring_start(ring, &tmap, n_tiles, tiles_c);

    const int t = threadIdx.x;
    const int chunk = t & 15;
    const int64_t groups = cols >> 5;
    const int64_t rgroups = rows >> 5;
    int i = 0;
    int64_t tile = blockIdx.x;
    for (; tile < n_tiles; tile += gridDim.x, ++i) {
        if (!ring_wait(ring, i, guard)) break;
        const uint8_t* buf = ring.buf + (i % kRing) * kTileBytes;
        const int64_t r0 = (tile / tiles_c) * kTile;
        const int64_t c0 = (tile % tiles_c) * kTile;

        if constexpr (kRow) {
            const int64_t col = c0 + chunk * 8;
            const bool col_ok = col < cols;
            const int64_t g = col >> 5;
#pragma unroll
            for (int j = 0; j < kLoadsPerThread; ++j) {
                const int lr = (t >> 4) + 16 * j;
                const uint4 v = reinterpret_cast<const uint4*>(buf)[lr * 16 + chunk];
                const int64_t r = r0 + lr;
                uint32_t m = abs_max_bits(v.x, 0u);
                m = abs_max_bits(v.y, m);
                m = abs_max_bits(v.z, m);
                m = abs_max_bits(v.w, m);
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                const bool valid = col_ok && r < rows;
                uint8_t code;
                uint2 out;
                if (m >= 0x7F80u) {  // NaN or Inf in the group
                    code = 0xFF;
                    out = nan8(v);
                } else {
                    const int e = rceil_exponent(m);
                    code = static_cast<uint8_t>(e + 127);
                    out = quant8(v, pow2_neg(e));
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
            const uint32_t* tw = reinterpret_cast<const uint32_t*>(buf);
            const int p = t & 63;
            const int gi = t >> 6;
            const int64_t cA = c0 + 2 * p;              // output row of q_col
            const int64_t rbase = r0 + 32 * gi;         // first input row of the group
            const int64_t g_out = rbase >> 5;
            const bool ok = cA < cols && rbase < rows;  // rows % 32 == 0 in column mode
            uint32_t w[32];
            uint32_t mlo = 0u, mhi = 0u;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                w[j] = tw[(32 * gi + j) * 64 + p];
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
                            const uint32_t h = half ? (w[4 * j + u] >> 16) : (w[4 * j + u] & 0xFFFFu);
                            b |= ((h >> 15) & 1u) << (8 * u + 7);
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
        ring_release(ring, &tmap, i, tile, n_tiles, tiles_c);
    }
    ring_drain(ring, i, tile, n_tiles, guard);
}

// ---------------------------------------------------------------------------------
// 32x32 block quantization of w [n, k], one 128x128 tile (16 blocks) at a time.
template <bool kTiled>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quant_32x32_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t n, int64_t k, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s_fwd, uint8_t* __restrict__ s_bwd, int64_t tiles_c, int64_t n_tiles,
    unsigned int* status, uint64_t wait_limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t blk_amax[2][4][4];  // [tile parity][32-row block][32-col block]
    const Ring ring = ring_setup(smem_raw);
    const WaitGuard guard{ring.abort_flag, status, wait_limit_ns};
    const int t = threadIdx.x;
    if (t < 32) reinterpret_cast<uint32_t*>(blk_amax)[t] = 0u;
    ring_start(ring, &tmap, n_tiles, tiles_c);

    const int chunk = t & 15;
    const int gcol = chunk >> 2;  // 32-column block within the tile
    const int64_t kgroups = k >> 5, ngroups = n >> 5;
    int i = 0;
    int64_t tile = blockIdx.x;
    for (; tile < n_tiles; tile += gridDim.x, ++i) {
        if (!ring_wait(ring, i, guard)) break;
        const uint4* buf = reinterpret_cast<const uint4*>(ring.buf + (i % kRing) * kTileBytes);
        uint32_t(*am)[4] = blk_amax[i & 1];
        const int64_t r0 = (tile / tiles_c) * kTile;
        const int64_t c0 = (tile % tiles_c) * kTile;
        const int64_t col = c0 + chunk * 8;
        const bool col_ok = col < k;

        uint4 v[kLoadsPerThread];
#pragma unroll
        for (int j = 0; j < kLoadsPerThread; ++j) v[j] = buf[((t >> 4) + 16 * j) * 16 + chunk];
        // Row (t/16 + 16 j) lies in 32-row block j/2 of the tile.
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t m = 0u;
#pragma unroll
            for (int j = 2 * b; j < 2 * b + 2; ++j) {
                m = abs_max_bits(v[j].x, m);
                m = abs_max_bits(v[j].y, m);
                m = abs_max_bits(v[j].z, m);
                m = abs_max_bits(v[j].w, m);
            }
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            if ((chunk & 3) == 0) atomicMax(&am[b][gcol], m);
        }
        __syncthreads();
        // The other parity's block maxima belong to the next tile: clear them now.
        if (t < 16) reinterpret_cast<uint32_t*>(blk_amax[(i + 1) & 1])[t] = 0u;

#pragma unroll
        for (int j = 0; j < kLoadsPerThread; ++j) {
            const int64_t r = r0 + (t >> 4) + 16 * j;
            const uint32_t m = am[j >> 1][gcol];
            const bool valid = col_ok && r < n;
            uint8_t code;
            uint2 out;
            if (m >= 0x7F80u) {
                code = 0xFF;
                out = nan8(v[j]);
            } else {
                const int e = rceil_exponent(m);
                code = static_cast<uint8_t>(e + 127);
                out = quant8(v[j], pow2_neg(e));
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
                const uint32_t m = am[b][cl >> 5];
                uint8_t code = 0;
                if (valid) code = (m >= 0x7F80u) ? 0xFF : static_cast<uint8_t>(rceil_exponent(m) + 127);
                if (valid || kTiled) store_scale(s_bwd, c, gi, ngroups, kTiled, code);
            }
        }
        ring_release(ring, &tmap, i, tile, n_tiles, tiles_c);
    }
    ring_drain(ring, i, tile, n_tiles, guard);
}

// Sets the dynamic shared-memory limit once per device and thread.
template <class Kern>
cudaError_t configure_once(Kern kern, int device, int* configured) {
    if (*configured == device) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) *configured = device;
    return e;
}

int64_t grid_for(const DeviceInfo& dev, int64_t n_tiles) {
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * kCtasPerSm;
    return n_tiles < cap ? n_tiles : cap;
}

template <bool kRow, bool kCol, bool kTiled>
cudaError_t launch_1x32_t(const DeviceInfo& dev, const CUtensorMap& map, int64_t rows, int64_t cols,
                          void* q_row, void* s_row, void* q_col, void* s_col, cudaStream_t stream) {
    auto kern = quant_1x32_kernel<kRow, kCol, kTiled>;
    static thread_local int configured = -1;
    cudaError_t e = configure_once(kern, dev.device, &configured);
    if (e != cudaSuccess) return e;
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t n_tiles = tiles_c * ((rows + kTile - 1) / kTile);
    kern<<<static_cast<unsigned>(grid_for(dev, n_tiles)), kThreads, kSmemBytes, stream>>>(
        map, rows, cols, static_cast<uint8_t*>(q_row), static_cast<uint8_t*>(s_row),
        static_cast<uint8_t*>(q_col), static_cast<uint8_t*>(s_col), tiles_c, n_tiles, dev.status,
        kDefaultWaitLimitNs);
    return cudaGetLastError();
}

template <bool kRow, bool kCol>
cudaError_t launch_1x32_l(const DeviceInfo& dev, const CUtensorMap& map, int64_t rows, int64_t cols,
                          void* q_row, void* s_row, void* q_col, void* s_col, bool tiled,
                          cudaStream_t stream) {
    if (tiled) return launch_1x32_t<kRow, kCol, true>(dev, map, rows, cols, q_row, s_row, q_col, s_col, stream);
    return launch_1x32_t<kRow, kCol, false>(dev, map, rows, cols, q_row, s_row, q_col, s_col, stream);
}

template <bool kTiled>
cudaError_t launch_32x32_t(const DeviceInfo& dev, const CUtensorMap& map, int64_t n, int64_t k, void* q,
                           void* s_fwd, void* s_bwd, cudaStream_t stream) {
    auto kern = quant_32x32_kernel<kTiled>;
    static thread_local int configured = -1;
    cudaError_t e = configure_once(kern, dev.device, &configured);
    if (e != cudaSuccess) return e;
    const int64_t tiles_c = (k + kTile - 1) / kTile;
    const int64_t n_tiles = tiles_c * ((n + kTile - 1) / kTile);
    kern<<<static_cast<unsigned>(grid_for(dev, n_tiles)), kThreads, kSmemBytes, stream>>>(
        map, n, k, static_cast<uint8_t*>(q), static_cast<uint8_t*>(s_fwd), static_cast<uint8_t*>(s_bwd),
        tiles_c, n_tiles, dev.status, kDefaultWaitLimitNs);
    return cudaGetLastError();
}

// BF16 [rows, cols] with row stride ld elements, 128 x 128 boxes, no swizzle.
bool bf16_tile_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols, int64_t ld) {
    return encode_tensor_map_2d(map, x, true, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                                static_cast<uint64_t>(ld) * 2, kTile, kTile, false);
}

}  // namespace

cudaError_t launch_quant_1x32(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols,
                              int64_t ld, void* q_row, void* s_row, void* q_col, void* s_col,
                              bool tiled, cudaStream_t stream) {
    CUtensorMap map;
    if (!bf16_tile_map(&map, x, rows, cols, ld)) return cudaErrorInvalidValue;
    const bool row = q_row != nullptr, col = q_col != nullptr;
    if (row && col) return launch_1x32_l<true, true>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tiled, stream);
    if (row) return launch_1x32_l<true, false>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tiled, stream);
    return launch_1x32_l<false, true>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tiled, stream);
}

cudaError_t launch_quant_32x32(const DeviceInfo& dev, const void* w, int64_t n, int64_t k, int64_t ld,
                               void* q, void* s_fwd, void* s_bwd, bool tiled, cudaStream_t stream) {
    CUtensorMap map;
    if (!bf16_tile_map(&map, w, n, k, ld)) return cudaErrorInvalidValue;
    if (tiled) return launch_32x32_t<true>(dev, map, n, k, q, s_fwd, s_bwd, stream);
    return launch_32x32_t<false>(dev, map, n, k, q, s_fwd, s_bwd, stream);
}

}  // namespace mxq
