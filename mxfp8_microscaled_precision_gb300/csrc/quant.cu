// quant.cu -- MXFP8 quantizers for sm_103a.
//
//  * 1x32 (row and/or column copy): one E8M0 scale per 32 consecutive
//    elements along the quantized axis (torchtitan-npu low-precision
//    tutorial, "MXFP8 与 HiF8 架构原理速览"; the dual-axis form of the MindSpeed
//    RFC "Add MXFP8-32x32 quantization support to FSDP", section 3.3.3).
//  * 32x32: one scale per 32x32 tile and a single payload shared by the
//    forward and backward GEMMs (same RFC, sections 3.1 and 3.3.3).
//
// Both are HBM-bound.  Work is cut into 128x128 BF16 tiles; a CTA of 256
// threads quantizes a tile.  Kernels that only need the row copy (and the
// 32x32 kernel) load their tile straight into registers with 16-byte loads
// issued up front, one tile per CTA.  Kernels that also produce the column
// copy are persistent and stream tiles through a three-slot shared-memory
// ring filled by TMA, so the loads of the next tiles overlap the work on the
// current one; the column groups are read back from the staged tile, so the
// input is read from HBM once.  The amax of a row group is reduced with
// packed 16x2 maxima and two shuffles over the four lanes that hold it; a
// column group is reduced by one thread.  The exponent is the exact rceil
// rule evaluated on the BF16 bits of amax; the scaling by 2^-e is an exact
// multiply; one cvt.rn.satfinite instruction rounds two values to E4M3.
// Scales go out plain or in the MMA-tiled layout; the tiled permutation is
// fused into the scale stores (which also write its zero padding).

#include <cuda_runtime.h>

#include <cstdint>

#include "mxq_device.cuh"
#include "mxq_internal.h"
#include "mxq_quant_math.cuh"

namespace mxq {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr int kLoadsPerThread = kTile * kTile / 8 / kThreads;  // 8 x 16-byte chunks
constexpr int kRing = 2;                                        // tile slots per CTA
constexpr int kTileBytes = kTile * kTile * 2;                   // 32 KB of BF16
constexpr int kCtasPerSm = 3;                                   // ring kernels
constexpr int kSmemBytes = kRing * kTileBytes + 1024 + 256;     // ring + alignment + barriers

// FP8 pair of the two BF16 values of a word (as FP32, exactly).
template <int kFmt>
__device__ __forceinline__ uint32_t cvt_pair(uint32_t w) {
    return cvt_fp8x2<kFmt>(bf16_lo(w), bf16_hi(w));
}

// Quantize 8 finite BF16 values (4 words) with scale 2^-e -> 8 FP8 bytes; s2 is
// 2^-e as a BF16 pair (pow2_neg_bf16 in both halves).  The BF16 product is
// exact: x * 2^-e has x's 8 significant bits and |x * 2^-e| <= the format's
// largest value, except when it falls below 2^-126, where both the exact and
// the rounded product convert to a signed zero (far below half the smallest
// E4M3 / E5M2 subnormal).
template <int kFmt = 0>
__device__ __forceinline__ uint2 quant8(const uint4 v, uint32_t s2) {
    uint2 o;
    o.x = cvt_pair<kFmt>(mul_bf16x2(v.x, s2)) | (cvt_pair<kFmt>(mul_bf16x2(v.y, s2)) << 16);
    o.y = cvt_pair<kFmt>(mul_bf16x2(v.z, s2)) | (cvt_pair<kFmt>(mul_bf16x2(v.w, s2)) << 16);
    return o;
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

// Tile numbering of a batch of matrices: tile = b * tiles_per_batch +
// (row band) * tiles_c + (column block).
struct TileGrid {
    int64_t tiles_c, tiles_per_batch, n_tiles;
    __device__ __forceinline__ void at(int64_t tile, int64_t& b, int64_t& r0, int64_t& c0) const {
        b = tile / tiles_per_batch;
        const int64_t local = tile - b * tiles_per_batch;
        r0 = (local / tiles_c) * kTile;
        c0 = (local % tiles_c) * kTile;
    }
};

// Issue the TMA load of `tile` into slot s (3-D map {cols, rows, batch}).
__device__ __forceinline__ void ring_load(const Ring& r, const CUtensorMap* map, int s, int64_t tile,
                                          const TileGrid& tg) {
    int64_t b, r0, c0;
    tg.at(tile, b, r0, c0);
    const uint32_t bar = r.bar0 + 8u * s;
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_3d(smem_u32(r.buf + s * kTileBytes), map, static_cast<int32_t>(c0), static_cast<int32_t>(r0),
                static_cast<int32_t>(b), bar);
}

// Thread 0 initialises the barriers and issues the first kRing loads.
__device__ __forceinline__ void ring_start(const Ring& r, const CUtensorMap* map, const TileGrid& tg) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) mbar_init(r.bar0 + 8u * s, 1);
        *r.abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(map);
        for (int s = 0; s < kRing; ++s) {
            const int64_t tile = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (tile < tg.n_tiles) ring_load(r, map, s, tile, tg);
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
                                             const TileGrid& tg) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const int64_t next = tile + static_cast<int64_t>(kRing) * gridDim.x;
        fence_proxy_async_smem();   // the slot's reads (and writes) come before the TMA refill
        if (next < tg.n_tiles) ring_load(r, map, i % kRing, next, tg);
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
// Row copy of one 128x128 tile held in registers.  Thread t holds rows
// (t/16 + 16 j), j = 0..7, 16-byte chunk t % 16 of the tile; the four chunks
// of one 32-group sit in four consecutive lanes.
// `chunk_of(j)` returns chunk j (registers or shared memory).
template <bool kTiled, int kFmt, class ChunkOf>
__device__ __forceinline__ void row_pass(ChunkOf chunk_of, int64_t r0, int64_t c0, int64_t rows,
                                         int64_t cols, uint8_t* __restrict__ q_row,
                                         uint8_t* __restrict__ s_row) {
    const int t = threadIdx.x;
    const int chunk = t & 15;
    const int64_t groups = cols >> 5;
    const int64_t col = c0 + chunk * 8;
    const bool col_ok = col < cols;
    const int64_t rows_left = rows - r0 - (t >> 4);  // chunk j is in a real row if 16 j < rows_left
    uint8_t* qp = q_row + (r0 + (t >> 4)) * cols + col;
    const int64_t qstep = 16 * cols;
    // Tiled: the tile's scales fill one 512-byte atom; row r and group g sit at
    // 16*(r%32) + 4*((r%128)/32) + g%4, i.e. 16*(t/16) + 256*(j%2) + 4*(j/2) + chunk/4.
    uint8_t* sp = kTiled ? s_row + ((r0 >> 7) * ((groups + 3) >> 2) + (c0 >> 7)) * 512 + ((t >> 4) << 4) +
                               (chunk >> 2)
                         : s_row + (r0 + (t >> 4)) * groups + (col >> 5);
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        const uint4 v = chunk_of(j);
        uint32_t m = amax8_bits(v);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        const bool valid = col_ok && 16 * j < rows_left;
        uint8_t code;
        uint2 out;
        if (m >= 0x7F80u) {  // NaN or Inf in the group
            code = 0xFF;
            out = nan8(v);
        } else {
            const int e = rceil_exponent<kFmt>(m);
            code = static_cast<uint8_t>(e + 127);
            out = quant8<kFmt>(v, pow2_neg_bf16(e) * 0x10001u);
        }
        if (valid) *reinterpret_cast<uint2*>(qp + j * qstep) = out;
        if ((chunk & 3) == 0 && (valid || kTiled)) {  // tiled padding gets 0
            uint8_t* dst = kTiled ? sp + 256 * (j & 1) + 4 * (j >> 1) : sp + j * 16 * groups;
            *dst = valid ? code : 0;
        }
    }
}

// Row copy of a staged tile (the dual kernels; the tile is 128 rows of 256
// bytes): lane l of warp w owns the 32-column group l % 4 of tile rows
// 16 w + l / 4 and 16 w + 8 + l / 4, reads it as four 16-byte chunks, reduces,
// scales and converts it in registers and stores it as one 32-byte run, so four
// lanes write a row's 128 contiguous bytes.  A lane reads its chunks in the
// order i ^ rot, rot = (group & 2) | (row & 1): the 8 lanes of a load phase (two
// rows, four groups) then hit 8 different 16-byte bank groups.  A group's scale
// byte goes to its place in the plain or tiled layout (tiled padding gets 0).
template <bool kTiled, int kFmt>
__device__ __forceinline__ void row_pass_tile(uint32_t tile, int64_t r0, int64_t c0, int64_t rows, int64_t cols,
                                              uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row) {
    const int t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    const int g = lane & 3;                  // 32-column group of the tile
    const int64_t col = c0 + 32 * g;
    const int64_t groups = cols >> 5;
    const bool col_ok = col < cols;
    const bool v8 = (reinterpret_cast<uintptr_t>(q_row) & 31u) == 0;   // runs are 32-byte aligned
    const int rot = (g & 2) | ((lane >> 2) & 1);
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int r = 16 * warp + 8 * it + (lane >> 2);
        const int64_t row = r0 + r;
        const bool valid = col_ok && row < rows;
        const uint32_t rowaddr = tile + static_cast<uint32_t>(r * 256 + 64 * g);
        uint4 v[4];   // v[i]: chunk i ^ rot of the group
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = lds128(rowaddr + 16u * static_cast<uint32_t>(i ^ rot));
        uint32_t a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = max_abs_bf16x2(max_abs_bf16x2(v[i].x, v[i].y), max_abs_bf16x2(v[i].z, v[i].w));
        const uint32_t m2 = max_abs_bf16x2(max_abs_bf16x2(a[0], a[1]), max_abs_bf16x2(a[2], a[3])) & 0x7FFF7FFFu;
        const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
        uint8_t code;
        uint32_t o[8];   // o[2 i], o[2 i + 1]: the payload bytes of chunk i ^ rot
        if (m >= 0x7F80u) {  // NaN or Inf in the group
            code = 0xFF;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint2 n = nan8(v[i]);
                o[2 * i] = n.x;
                o[2 * i + 1] = n.y;
            }
        } else {
            const int e = rceil_exponent<kFmt>(m);
            code = static_cast<uint8_t>(e + 127);
            const uint32_t s2 = pow2_neg_bf16(e) * 0x10001u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint2 q = quant8<kFmt>(v[i], s2);
                o[2 * i] = q.x;
                o[2 * i + 1] = q.y;
            }
        }
        // back to chunk order: undo the XOR with rot one bit at a time
        if (rot & 1) {
#pragma unroll
            for (int k = 0; k < 8; k += 4) {
                uint32_t x = o[k]; o[k] = o[k + 2]; o[k + 2] = x;
                x = o[k + 1]; o[k + 1] = o[k + 3]; o[k + 3] = x;
            }
        }
        if (rot & 2) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t x = o[k]; o[k] = o[k + 4]; o[k + 4] = x;
            }
        }
        if (valid) {
            uint8_t* dst = q_row + row * cols + col;
            if (v8) {
                stg256(dst, o);
            } else {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
        if (valid || kTiled) store_scale(s_row, row, col >> 5, groups, kTiled, valid ? code : 0);
    }
}

// Loads this thread's 8 chunks of tile (r0, c0) straight from global memory
// (zeros outside the matrix).
__device__ __forceinline__ void load_tile_chunks(uint4 (&v)[kLoadsPerThread], const uint16_t* __restrict__ x,
                                                 int64_t r0, int64_t c0, int64_t rows, int64_t cols,
                                                 int64_t ld) {
    const int t = threadIdx.x;
    const int64_t col = c0 + (t & 15) * 8;
    const int64_t rows_left = rows - r0 - (t >> 4);
    const uint16_t* xp = x + (r0 + (t >> 4)) * ld + col;
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        if (col < cols && 16 * j < rows_left)
            v[j] = __ldg(reinterpret_cast<const uint4*>(xp + j * 16 * ld));
        else
            v[j] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Output strides between the matrices of a batch (bytes), input stride (elements).
struct BatchStrides {
    int64_t x, q_row, s_row, q_col, s_col;
};

// Row copy only: one tile per CTA, loaded straight into registers.
template <bool kTiled, int kFmt>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ld,
                                                              uint8_t* __restrict__ q_row,
                                                              uint8_t* __restrict__ s_row, TileGrid tg,
                                                              BatchStrides bs) {
    int64_t b, r0, c0;
    tg.at(blockIdx.x, b, r0, c0);
    uint4 v[kLoadsPerThread];
    load_tile_chunks(v, x + b * bs.x, r0, c0, rows, cols, ld);
    row_pass<kTiled, kFmt>([&](int j) { return v[j]; }, r0, c0, rows, cols, q_row + b * bs.q_row,
                     s_row + b * bs.s_row);
}

// Column copy of one staged tile: thread t takes the column pair t % 64 and
// the 32-token group t / 64; a warp reads 128 contiguous bytes of one staged
// row per step (conflict-free).  The group's first token is tok0 + 32 (t/64)
// in the output (row stride out_ld, out_ld/32 scale groups); groups at or past
// tok_limit are not written (tiled layout: their scale is padding, 0).
template <bool kTiled, int kFmt>
__device__ __forceinline__ void col_pass(const uint32_t* tw_ptr, int64_t c0, int64_t cols, int64_t out_ld,
                                         int64_t tok0, int64_t tok_limit, uint8_t* __restrict__ q_col,
                                         uint8_t* __restrict__ s_col) {
    const uint32_t tw = smem_u32(tw_ptr);   // the staged tile is in shared memory
    const int t = threadIdx.x;
    const int p = t & 63;
    const int gi = t >> 6;
    const int64_t cA = c0 + 2 * p;              // output row of q_col
    const int64_t tok = tok0 + 32 * gi;         // first token of the group
    const int64_t ogroups = out_ld >> 5;
    const int64_t g_out = tok >> 5;
    const bool ok = cA < cols && tok < tok_limit;
    uint32_t w[32];
    uint32_t m2 = 0u;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        w[j] = lds32(tw + 4u * static_cast<uint32_t>((32 * gi + j) * 64 + p));
        m2 = max_abs_bf16x2(m2, w[j]);
    }
    m2 &= 0x7FFF7FFFu;                          // column cA's amax in the low half, cA+1's in the high
    uint8_t* q0 = q_col + cA * out_ld + tok;
    // Runs start at multiples of 32 tokens in rows of a multiple of 32 bytes, so
    // they are 32-byte aligned whenever the output is (uniform over the call).
    const bool v8 = (reinterpret_cast<uintptr_t>(q_col) & 31u) == 0;
    // Scale bytes of rows cA and cA+1 (same 32-row block: cA is even).
    uint8_t* s0 = kTiled ? s_col + tiled_scale_offset(cA, g_out, ogroups) : s_col + cA * ogroups + g_out;
    const int64_t s_next = kTiled ? 16 : ogroups;
    const uint32_t mh[2] = {m2 & 0xFFFFu, m2 >> 16};
    uint8_t code[2];
    uint32_t o[2][8];
    if (mh[0] < 0x7F80u && mh[1] < 0x7F80u) {
        // Both groups finite: scale both columns of a word with one BF16 multiply
        // (exact, see quant8), then pair consecutive tokens of each column.
        const int e0 = rceil_exponent<kFmt>(mh[0]), e1 = rceil_exponent<kFmt>(mh[1]);
        code[0] = static_cast<uint8_t>(e0 + 127);
        code[1] = static_cast<uint8_t>(e1 + 127);
        const uint32_t s2 = pow2_neg_bf16(e0) | (pow2_neg_bf16(e1) << 16);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t p0 = mul_bf16x2(w[4 * j], s2), p1 = mul_bf16x2(w[4 * j + 1], s2);
            const uint32_t p2 = mul_bf16x2(w[4 * j + 2], s2), p3 = mul_bf16x2(w[4 * j + 3], s2);
            o[0][j] = cvt_fp8x2<kFmt>(bf16_lo(p0), bf16_lo(p1)) | (cvt_fp8x2<kFmt>(bf16_lo(p2), bf16_lo(p3)) << 16);
            o[1][j] = cvt_fp8x2<kFmt>(bf16_hi(p0), bf16_hi(p1)) | (cvt_fp8x2<kFmt>(bf16_hi(p2), bf16_hi(p3)) << 16);
        }
    } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (mh[half] >= 0x7F80u) {   // NaN or Inf in the group: 0x7F | sign per element
                code[half] = 0xFF;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t bt = 0x7F7F7F7Fu;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t h = half ? (w[4 * j + u] >> 16) : (w[4 * j + u] & 0xFFFFu);
                        bt |= ((h >> 15) & 1u) << (8 * u + 7);
                    }
                    o[half][j] = bt;
                }
            } else {
                const int e = rceil_exponent<kFmt>(mh[half]);
                const float sc = pow2_neg(e);
                code[half] = static_cast<uint8_t>(e + 127);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float f[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        f[u] = (half ? bf16_hi(w[4 * j + u]) : bf16_lo(w[4 * j + u])) * sc;
                    o[half][j] = cvt_fp8x2<kFmt>(f[0], f[1]) | (cvt_fp8x2<kFmt>(f[2], f[3]) << 16);
                }
            }
        }
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        if (ok) {
            uint8_t* dst = q0 + half * out_ld;
            if (v8) {   // the 32-byte run in one store (a lane writes one row per store)
                stg256(dst, o[half]);
            } else {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[half][0], o[half][1], o[half][2], o[half][3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[half][4], o[half][5], o[half][6], o[half][7]);
            }
        }
        if (ok || kTiled) s0[half * s_next] = ok ? code[half] : 0;
    }
}

// Column copy (with or without the row copy): persistent, TMA-fed ring.
// Column pass: thread t takes the column pair t % 64 and the 32-row group
// t / 64; a warp reads 128 contiguous bytes of one staged row per step, so
// the shared-memory reads are conflict-free.  Row pass: row_pass_tile.
template <bool kRow, bool kTiled, int kFmt>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quant_cols_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col,
    uint8_t* __restrict__ s_col, TileGrid tg, BatchStrides bs, unsigned int* status,
    uint64_t wait_limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const Ring ring = ring_setup(smem_raw);
    const WaitGuard guard{ring.abort_flag, status, wait_limit_ns};
    ring_start(ring, &tmap, tg);

    int i = 0;
    int64_t tile = blockIdx.x;
    for (; tile < tg.n_tiles; tile += gridDim.x, ++i) {
        if (!ring_wait(ring, i, guard)) break;
        const uint8_t* buf = ring.buf + (i % kRing) * kTileBytes;
        int64_t b, r0, c0;
        tg.at(tile, b, r0, c0);
        if constexpr (kRow)
            row_pass_tile<kTiled, kFmt>(smem_u32(buf), r0, c0, rows, cols, q_row + b * bs.q_row, s_row + b * bs.s_row);
        col_pass<kTiled, kFmt>(reinterpret_cast<const uint32_t*>(buf), c0, cols, rows, r0, rows,
                         q_col + b * bs.q_col, s_col + b * bs.s_col);
        ring_release(ring, &tmap, i, tile, tg);
    }
    ring_drain(ring, i, tile, tg.n_tiles, guard);
}

// Token-axis (column) quantization inside each expert for the MoE weight
// gradient.  Expert g's tokens go to the slot [P_g, P_g + L_g) of q_col
// [cols, capacity], L_g = m_g rounded up to 128, P_g = sum of earlier L; each
// 32-token group starts at the expert's first token and is zero-padded past
// its last.  The slots are computed from the device offsets by every CTA (in
// shared memory); the CTAs then walk the (slot block, column block) tiles.
// Persistent and fed by the TMA ring: a tile is 128 tokens of one expert's
// slot x 128 columns, loaded from the tokens' rows of x (rows past the
// expert's last token are zeroed in shared memory before the column pass).
struct GroupedTile {
    int64_t pos, c0, row0, valid;   // slot position, first column, first row of x, real rows (1..128)
};

__device__ __forceinline__ GroupedTile grouped_tile(int64_t tl, int64_t tiles_c, const int64_t* s_off,
                                                    const int64_t* s_slot, int G) {
    GroupedTile gt;
    gt.pos = (tl / tiles_c) * kTile;
    gt.c0 = (tl % tiles_c) * kTile;
    int lo = 0, hi = G;  // owner: largest g with s_slot[g] <= pos
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_slot[mid] <= gt.pos) lo = mid; else hi = mid;
    }
    gt.row0 = s_off[lo] + (gt.pos - s_slot[lo]);
    const int64_t left = s_off[lo + 1] - gt.row0;
    gt.valid = left < kTile ? left : kTile;
    return gt;
}

template <bool kTiled, int kFmt>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quant_cols_grouped_ring_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, const int64_t* __restrict__ offsets,
    int G, int64_t capacity, uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col, unsigned int* status,
    uint64_t wait_limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const Ring ring = ring_setup(smem_raw);
    const WaitGuard guard{ring.abort_flag, status, wait_limit_ns};
    int64_t* s_off = reinterpret_cast<int64_t*>(ring.buf + kRing * kTileBytes + 64);   // [G+1]
    int64_t* s_slot = s_off + (G + 1);                                                  // [G+1]
    const int t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    for (int g = t; g <= G; g += kThreads) {
        int64_t o = offsets[g];
        s_off[g] = o < 0 ? 0 : (o > rows ? rows : o);  // malformed offsets stay in bounds
    }
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of the slot lengths, 32 experts at a time
        int64_t carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int64_t len = 0;
            if (g < G) {
                const int64_t m = s_off[g + 1] - s_off[g];
                len = m > 0 ? (m + kTile - 1) / kTile * kTile : 0;
            }
            int64_t incl = len;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            if (g < G) s_slot[g] = carry + incl - len;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) s_slot[G] = carry;
    }
    __syncthreads();
    const int64_t used = s_slot[G] < capacity ? s_slot[G] : capacity;
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t n_tiles = (used / kTile) * tiles_c;

    auto issue = [&](int slot, int64_t tl) {
        const GroupedTile gt = grouped_tile(tl, tiles_c, s_off, s_slot, G);
        const uint32_t bar = ring.bar0 + 8u * slot;
        mbar_arrive_expect_tx(bar, kTileBytes);
        tma_load_3d(smem_u32(ring.buf + slot * kTileBytes), &tmap, static_cast<int32_t>(gt.c0),
                    static_cast<int32_t>(gt.row0), 0, bar);
    };
    if (t == 0) {
        for (int sl = 0; sl < kRing; ++sl) mbar_init(ring.bar0 + 8u * sl, 1);
        *ring.abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmap);
        for (int sl = 0; sl < kRing; ++sl) {
            const int64_t tl = blockIdx.x + static_cast<int64_t>(sl) * gridDim.x;
            if (tl < n_tiles) issue(sl, tl);
        }
    }
    __syncthreads();

    int i = 0;
    int64_t tl = blockIdx.x;
    for (; tl < n_tiles; tl += gridDim.x, ++i) {
        if (!ring_wait(ring, i, guard)) break;
        uint8_t* buf = ring.buf + (i % kRing) * kTileBytes;
        const GroupedTile gt = grouped_tile(tl, tiles_c, s_off, s_slot, G);
        if (gt.valid < kTile) {   // tokens of the next expert (or past x) read as zero
            uint4* b4 = reinterpret_cast<uint4*>(buf);
            for (int u = static_cast<int>(gt.valid) * 16 + t; u < kTile * 16; u += kThreads)
                b4[u] = make_uint4(0u, 0u, 0u, 0u);
            __syncthreads();
        }
        col_pass<kTiled, kFmt>(reinterpret_cast<const uint32_t*>(buf), gt.c0, cols, capacity, gt.pos, capacity,
                               q_col, s_col);
        __syncthreads();
        if (t == 0) {
            const int64_t next = tl + static_cast<int64_t>(kRing) * gridDim.x;
            fence_proxy_async_smem();   // the slot's reads and zeroing come before the TMA refill
            if (next < n_tiles) issue(i % kRing, next);
        }
    }
    ring_drain(ring, i, tl, n_tiles, guard);
}

// ---------------------------------------------------------------------------------
// 32x32 block quantization of w [n, k]: one 128x128 tile (16 blocks) per CTA;
// payload E4M3 (kFmt 0) or E5M2 (kFmt 1).
template <bool kTiled, int kFmt>
__global__ void __launch_bounds__(kThreads) quant_32x32_kernel(const uint16_t* __restrict__ w, int64_t n,
                                                               int64_t k, int64_t ld, uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ s_fwd,
                                                               uint8_t* __restrict__ s_bwd, int64_t tiles_c) {
    __shared__ uint32_t blk_amax[4][4];  // [32-row block][32-col block] of this tile
    const int t = threadIdx.x;
    if (t < 16) blk_amax[t >> 2][t & 3] = 0u;
    const int64_t tile = blockIdx.x;
    const int64_t r0 = (tile / tiles_c) * kTile, c0 = (tile % tiles_c) * kTile;
    const int chunk = t & 15;
    const int gcol = chunk >> 2;  // 32-column block within the tile
    uint4 v[kLoadsPerThread];
    load_tile_chunks(v, w, r0, c0, n, k, ld);
    __syncthreads();  // blk_amax cleared

    // Chunk j (row t/16 + 16 j) lies in 32-row block j/2 of the tile.
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t m = max(amax8_bits(v[2 * b]), amax8_bits(v[2 * b + 1]));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        if ((chunk & 3) == 0) atomicMax(&blk_amax[b][gcol], m);
    }
    __syncthreads();

    const int64_t kgroups = k >> 5, ngroups = n >> 5;
    const int64_t col = c0 + chunk * 8;
    const bool col_ok = col < k;
    const int64_t rows_left = n - r0 - (t >> 4);
    uint8_t* qp = q + (r0 + (t >> 4)) * k + col;
    uint8_t* sp = nullptr;
    if (s_fwd)
        sp = kTiled ? s_fwd + ((r0 >> 7) * ((kgroups + 3) >> 2) + (c0 >> 7)) * 512 + ((t >> 4) << 4) + (chunk >> 2)
                    : s_fwd + (r0 + (t >> 4)) * kgroups + (col >> 5);
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        const uint32_t m = blk_amax[j >> 1][gcol];
        const bool valid = col_ok && 16 * j < rows_left;
        uint8_t code;
        uint2 out;
        if (m >= 0x7F80u) {
            code = 0xFF;
            out = nan8(v[j]);
        } else {
            const int e = rceil_exponent<kFmt>(m);
            code = static_cast<uint8_t>(e + 127);
            out = quant8<kFmt>(v[j], pow2_neg_bf16(e) * 0x10001u);
        }
        if (valid) *reinterpret_cast<uint2*>(qp + j * 16 * k) = out;
        if (sp && (chunk & 3) == 0 && (valid || kTiled)) {
            uint8_t* dst = kTiled ? sp + 256 * (j & 1) + 4 * (j >> 1) : sp + j * 16 * kgroups;
            *dst = valid ? code : 0;
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
            if (valid) code = (m >= 0x7F80u) ? 0xFF : static_cast<uint8_t>(rceil_exponent<kFmt>(m) + 127);
            if (valid || kTiled) store_scale(s_bwd, c, gi, ngroups, kTiled, code);
        }
    }
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

template <bool kRow, bool kTiled, int kFmt>
cudaError_t launch_cols_t(const DeviceInfo& dev, const CUtensorMap& map, int64_t rows, int64_t cols,
                          void* q_row, void* s_row, void* q_col, void* s_col, const TileGrid& tg,
                          const BatchStrides& bs, cudaStream_t stream) {
    auto kern = quant_cols_kernel<kRow, kTiled, kFmt>;
    static thread_local int configured = -1;
    cudaError_t e = configure_once(kern, dev.device, &configured);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid_for(dev, tg.n_tiles)), kThreads, kSmemBytes, stream>>>(
        map, rows, cols, static_cast<uint8_t*>(q_row), static_cast<uint8_t*>(s_row),
        static_cast<uint8_t*>(q_col), static_cast<uint8_t*>(s_col), tg, bs, dev.status, kDefaultWaitLimitNs);
    return cudaGetLastError();
}

template <int kFmt>
cudaError_t launch_1x32_fmt(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld,
                            int64_t batch, int64_t batch_stride, void* q_row, void* s_row, void* q_col,
                            void* s_col, bool tiled, const TileGrid& tg, const BatchStrides& bs,
                            cudaStream_t stream) {
    const bool row = q_row != nullptr, col = q_col != nullptr;
    if (!col) {  // row copy only: direct loads, one tile per CTA
        auto xp = static_cast<const uint16_t*>(x);
        auto qp = static_cast<uint8_t*>(q_row);
        auto sp = static_cast<uint8_t*>(s_row);
        if (tiled)
            quant_rows_kernel<true, kFmt><<<static_cast<unsigned>(tg.n_tiles), kThreads, 0, stream>>>(xp, rows, cols, ld, qp, sp, tg, bs);
        else
            quant_rows_kernel<false, kFmt><<<static_cast<unsigned>(tg.n_tiles), kThreads, 0, stream>>>(xp, rows, cols, ld, qp, sp, tg, bs);
        return cudaGetLastError();
    }
    CUtensorMap map;
    if (!encode_tensor_map_3d(&map, x, true, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                              static_cast<uint64_t>(batch), static_cast<uint64_t>(ld) * 2,
                              static_cast<uint64_t>(batch_stride) * 2, kTile, kTile))
        return cudaErrorInvalidValue;
    if (row)
        return tiled ? launch_cols_t<true, true, kFmt>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tg, bs, stream)
                     : launch_cols_t<true, false, kFmt>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tg, bs, stream);
    return tiled ? launch_cols_t<false, true, kFmt>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tg, bs, stream)
                 : launch_cols_t<false, false, kFmt>(dev, map, rows, cols, q_row, s_row, q_col, s_col, tg, bs, stream);
}

int64_t scale_bytes(int64_t rows, int64_t cols, bool tiled) {
    const int64_t groups = cols / 32;
    return tiled ? ((rows + 127) / 128 * 128) * ((groups + 3) / 4 * 4) : rows * groups;
}

}  // namespace

cudaError_t launch_quant_1x32(const DeviceInfo& dev, const void* x, int64_t batch, int64_t rows,
                              int64_t cols, int64_t ld, int64_t batch_stride, void* q_row,
                              void* s_row, void* q_col, void* s_col, bool tiled, int fmt,
                              cudaStream_t stream) {
    TileGrid tg;
    tg.tiles_c = (cols + kTile - 1) / kTile;
    tg.tiles_per_batch = tg.tiles_c * ((rows + kTile - 1) / kTile);
    tg.n_tiles = tg.tiles_per_batch * batch;
    BatchStrides bs;
    bs.x = batch_stride;
    bs.q_row = rows * cols;
    bs.s_row = scale_bytes(rows, cols, tiled);
    bs.q_col = cols * rows;
    bs.s_col = scale_bytes(cols, rows, tiled);
    if (fmt == 1)
        return launch_1x32_fmt<1>(dev, x, rows, cols, ld, batch, batch_stride, q_row, s_row, q_col, s_col, tiled, tg, bs, stream);
    return launch_1x32_fmt<0>(dev, x, rows, cols, ld, batch, batch_stride, q_row, s_row, q_col, s_col, tiled, tg, bs, stream);
}

cudaError_t launch_quant_cols_grouped(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols,
                                      int64_t ld, const int64_t* offsets, int G, int64_t capacity,
                                      void* q_col, void* s_col, bool tiled, int fmt, cudaStream_t stream) {
    const size_t smem = kRing * kTileBytes + 1024 + 64 + 2 * 8 * static_cast<size_t>(G + 1);
    auto qp = static_cast<uint8_t*>(q_col);
    auto sp = static_cast<uint8_t*>(s_col);
    const int64_t max_tiles = (capacity / kTile) * ((cols + kTile - 1) / kTile);
    if (max_tiles == 0) return cudaSuccess;
    CUtensorMap map;
    if (!encode_tensor_map_3d(&map, x, true, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), 1,
                              static_cast<uint64_t>(ld) * 2, static_cast<uint64_t>(ld) * 2 * static_cast<uint64_t>(rows),
                              kTile, kTile))
        return cudaErrorInvalidValue;
    auto run = [&](auto kern, int* configured, int* per_sm) -> cudaError_t {
        if (*configured != dev.device) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kRing * kTileBytes + 1024 + 64 + 16 * 1025));
            if (e != cudaSuccess) return e;
            *configured = dev.device;
        }
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
        if (e != cudaSuccess) return e;
        *per_sm = n < 1 ? 1 : n;
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * *per_sm;
        const unsigned grid = static_cast<unsigned>(max_tiles < cap ? max_tiles : cap);
        kern<<<grid, kThreads, smem, stream>>>(map, rows, cols, offsets, G, capacity, qp, sp, dev.status,
                                               kDefaultWaitLimitNs);
        return cudaGetLastError();
    };
    int per_sm = 0;
    if (tiled && fmt == 1) {
        static thread_local int configured = -1;
        return run(quant_cols_grouped_ring_kernel<true, 1>, &configured, &per_sm);
    }
    if (tiled) {
        static thread_local int configured = -1;
        return run(quant_cols_grouped_ring_kernel<true, 0>, &configured, &per_sm);
    }
    if (fmt == 1) {
        static thread_local int configured = -1;
        return run(quant_cols_grouped_ring_kernel<false, 1>, &configured, &per_sm);
    }
    static thread_local int configured = -1;
    return run(quant_cols_grouped_ring_kernel<false, 0>, &configured, &per_sm);
}

// ---- group-tiled scales (A operand of the grouped GEMM) ------------------------------

constexpr int kRegroupThreads = 256;
constexpr int kAtomsPerItem = 4;   // atoms of one band per warp work item

// Group-tiled copy of the MMA-tiled scales of a row quantization: the rows
// [off[g], off[g+1]) of group g form ceil(n_g / 128) bands of their own, from
// band B_g (the prefix of the band counts); bands at or past bands_cap are
// dropped.  A warp handles four atoms of one output band at a time.  Lane l's
// 16 bytes of an atom are the scales of rows l, 32 + l, 64 + l, 96 + l of its
// band (word j: row 32 j + l).
// Output row 32 j + l of band i of group g is row v = s + 32 j + l of the
// two-band source window that starts at band (off[g] + 128 i) / 128, where
// s = (off[g] + 128 i) % 128: source band v / 128, lane (s + l) % 32 -- the same
// for every j -- and word (v / 32) % 4.  So each lane loads its 16 bytes of the
// two source atoms, takes lane (s + l) % 32's eight words by shuffles and stores
// 16 bytes: coalesced on both sides.  Rows past the group's last are zero.
__global__ void __launch_bounds__(kRegroupThreads)
    scale_regroup_rows_kernel(const uint4* __restrict__ src, int64_t rows, int64_t k_atoms,
                              const int64_t* __restrict__ offsets, int G, int64_t bands_cap,
                              uint4* __restrict__ dst) {
    __shared__ int64_t s_off[1025];   // offsets clamped to [0, rows]
    __shared__ int s_band[1025];      // exclusive prefix of the groups' band counts
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= G; i += kRegroupThreads) {
        const int64_t o = offsets[i];
        s_off[i] = o < 0 ? 0 : (o > rows ? rows : o);
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int bands = 0;
            if (g < G && s_off[g + 1] > s_off[g]) bands = static_cast<int>((s_off[g + 1] - s_off[g] + 127) >> 7);
            int incl = bands;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            if (g < G) s_band[g] = carry + incl - bands;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) s_band[G] = carry;
    }
    __syncthreads();
    const int64_t bands = min(static_cast<int64_t>(s_band[G]), bands_cap);
    // Work item: kAtomsPerItem consecutive atoms of one output band (one group
    // lookup, all the item's loads in flight before the first shuffle).
    constexpr int kWarps = kRegroupThreads / 32;
    const int64_t kgroups = (k_atoms + kAtomsPerItem - 1) / kAtomsPerItem;
    const int64_t items = bands * kgroups;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * kWarps + warp; it < items;
         it += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int64_t b = it / kgroups, ka0 = (it - b * kgroups) * kAtomsPerItem;
        int g = 0, hi_g = G;  // the last group whose first band is <= b (never an empty one)
        while (hi_g - g > 1) {
            const int mid = (g + hi_g) >> 1;
            if (s_band[mid] <= b) g = mid; else hi_g = mid;
        }
        const int64_t r0 = s_off[g] + (b - s_band[g]) * 128, end = s_off[g + 1];
        const int64_t b0 = r0 >> 7;
        const int sh = static_cast<int>(r0 & 127);
        const bool two = sh != 0 && (b0 + 1) * 128 < rows;
        const int u = sh + lane, from = u & 31;
        uint4 x0[kAtomsPerItem], x1[kAtomsPerItem];
#pragma unroll
        for (int q = 0; q < kAtomsPerItem; ++q) {
            const int64_t ka = ka0 + q;
            x0[q] = x1[q] = make_uint4(0u, 0u, 0u, 0u);
            if (ka < k_atoms) {
                x0[q] = src[(b0 * k_atoms + ka) * 32 + lane];
                if (two) x1[q] = src[((b0 + 1) * k_atoms + ka) * 32 + lane];
            }
        }
#pragma unroll
        for (int q = 0; q < kAtomsPerItem; ++q) {
            const int64_t ka = ka0 + q;
            if (ka >= k_atoms) break;   // uniform across the warp
            uint32_t w0[4], w1[4];
            w0[0] = __shfl_sync(0xFFFFFFFFu, x0[q].x, from);
            w0[1] = __shfl_sync(0xFFFFFFFFu, x0[q].y, from);
            w0[2] = __shfl_sync(0xFFFFFFFFu, x0[q].z, from);
            w0[3] = __shfl_sync(0xFFFFFFFFu, x0[q].w, from);
            w1[0] = __shfl_sync(0xFFFFFFFFu, x1[q].x, from);
            w1[1] = __shfl_sync(0xFFFFFFFFu, x1[q].y, from);
            w1[2] = __shfl_sync(0xFFFFFFFFu, x1[q].z, from);
            w1[3] = __shfl_sync(0xFFFFFFFFu, x1[q].w, from);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = u + 32 * j;          // row in the two-band window
                const int k = (v >> 5) & 3;        // its word in the source lane's 16 bytes
                const uint32_t* w = (v >> 7) ? w1 : w0;
                const uint32_t val = k == 0 ? w[0] : k == 1 ? w[1] : k == 2 ? w[2] : w[3];
                o[j] = r0 + 32 * j + lane < end ? val : 0u;
            }
            dst[(b * k_atoms + ka) * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

cudaError_t launch_scale_regroup_rows(const DeviceInfo& dev, const void* s_tiled, int64_t rows, int64_t cols,
                                      const int64_t* offsets, int G, int64_t bands_cap, void* s_out,
                                      cudaStream_t stream) {
    const int64_t k_atoms = (cols / 32 + 3) / 4;
    const int64_t per_block = kRegroupThreads / 32;
    int64_t grid = (bands_cap * ((k_atoms + kAtomsPerItem - 1) / kAtomsPerItem) + per_block - 1) / per_block;
    const int64_t most = static_cast<int64_t>(dev.sm_count) * 3;   // resident blocks (80 registers a thread)
    if (grid > most) grid = most;
    if (grid <= 0) return cudaSuccess;
    scale_regroup_rows_kernel<<<static_cast<unsigned>(grid), kRegroupThreads, 0, stream>>>(
        static_cast<const uint4*>(s_tiled), rows, k_atoms, offsets, G, bands_cap, static_cast<uint4*>(s_out));
    return cudaGetLastError();
}

cudaError_t launch_quant_32x32(const DeviceInfo& dev, const void* w, int64_t n, int64_t k, int64_t ld,
                               void* q, void* s_fwd, void* s_bwd, bool tiled, int fmt, cudaStream_t stream) {
    (void)dev;
    const int64_t tiles_c = (k + kTile - 1) / kTile;
    const int64_t n_tiles = tiles_c * ((n + kTile - 1) / kTile);
    auto wp = static_cast<const uint16_t*>(w);
    auto qp = static_cast<uint8_t*>(q);
    auto sf = static_cast<uint8_t*>(s_fwd);
    auto sb = static_cast<uint8_t*>(s_bwd);
    auto kern = tiled ? (fmt == 0 ? quant_32x32_kernel<true, 0> : quant_32x32_kernel<true, 1>)
                      : (fmt == 0 ? quant_32x32_kernel<false, 0> : quant_32x32_kernel<false, 1>);
    kern<<<static_cast<unsigned>(n_tiles), kThreads, 0, stream>>>(wp, n, k, ld, qp, sf, sb, tiles_c);
    return cudaGetLastError();
}

}  // namespace mxq
