// gemm.cu -- block-scaled MXFP8 GEMMs with BF16 output for sm_103a.
//
//   y[m, n] = sum_k (qa[m,k] * 2^ea[m,k/32]) * (qb[n,k] * 2^eb[n,k/32])
//
// The FP8 matmul of the MXFP8 recipe (torchtitan-npu low-precision tutorial,
// "MXFP8 与 HiF8 架构原理速览": FP8 matmul, output restored to BF16) for the
// forward, dgrad and wgrad of linear layers, and its grouped form for MoE
// experts (same page; MindSpeed RFC "Add MXFP8-32x32 quantization support
// to FSDP", section 2.2, gate_up_proj / down_proj).  With the 32x32 recipe
// the dgrad reads the one shared weight payload N-major (RFC section 3.1).
//
// Two kernels.  Every launch the pair kernel can take runs on CTA pairs
// (clusters of two SMs, tcgen05 cta_group::2, 256 x 256 tiles; its own section
// below).  The single-CTA kernel takes the rest (more than 512 experts, a
// tensor map the driver refuses to encode, a device with one SM) and is the
// design the pair kernel extends.
//
// Single-CTA design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: A and B tiles (128-byte swizzle) and the
//               512-byte scale atoms, into a ring of STAGES shared-memory
//               slots guarded by full/empty mbarriers.
//   warp 1      allocates tensor memory; the whole warp runs the tile and
//               stage loops (warp-uniform, so counters and descriptors live in
//               uniform registers) and one elected lane issues, per stage,
//               tcgen05.cp of the scale atoms into that stage's TMEM columns
//               and the tcgen05.mma.kind::mxf8f6f4.block_scale instructions
//               (128 x BN x 32 each) into the TMEM accumulator.
//   warps 2-9   epilogue: one thread waits (suspending) for a finished
//               accumulator while the other epilogue warps sleep on a named
//               barrier; tcgen05.ld of the FP32 accumulator, which is then
//               released to the MMA warp; RNE to BF16 (and, in the quantizing
//               mode, the 1x32 MXFP8 quantization); BF16 tiles go out
//               through a per-warp shared-memory staging buffer (8 rows x 64
//               contiguous bytes per store instruction), the quantizing
//               epilogue with 16-byte stores per row.
// Every mbarrier wait is bounded (see mxq_device.cuh).

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "mxq_device.cuh"
#include "mxq_internal.h"
#include "mxq_quant_math.cuh"

namespace mxq {
namespace {

constexpr int kBM = 128;          // rows of A per tile (= TMEM lanes)
constexpr int kBK = 128;          // K elements (= bytes) per pipeline stage
constexpr int kUmmaK = 32;        // K of one MMA instruction (FP8)
constexpr int kRasterBand = 8;    // m-tiles per raster band (L2 reuse of B)
constexpr int kMaxGroups = 1024;
constexpr int kMaxProblems = 4;   // dense GEMMs of one launch

// Kernel modes.
constexpr int kDense = 0;         // y = A B^T
constexpr int kGroupedRows = 1;   // rows of A split by expert, one B per expert (MoE fwd, dgrad)
constexpr int kGroupedK = 2;      // contraction split by expert (MoE wgrad), y stacked per expert
constexpr int kDenseQuant = 3;    // dense, epilogue also emits the 1x32 MXFP8 quantization of y

// One GEMM of a launch (grouped modes: the only one).
struct Problem {
    const uint8_t* a_s;      // A scales, MMA-tiled
    const uint8_t* b_s;      // B scales, MMA-tiled
    uint16_t* y;             // bf16 output
    int64_t M, N, K, ldy;
    int64_t k_atoms;         // 4-group scale atoms per 128-row band = ceil(K/128)
    int64_t b_bands;         // 128-row bands of B scales that exist
    int64_t m_tiles, n_tiles;
    int64_t first_item;      // dense: the problem's first work item
    int num_kb;              // 128-deep K blocks
    uint32_t fmt_bits;       // operand formats in the instruction descriptor (0 = E4M3, E4M3)
    int y_tma;               // 1: TensorMaps::y of this problem maps y (32 x 32 tiled stores)
};

struct GemmArgs {
    Problem pr[kMaxProblems];
    int nprob;
    int64_t items;           // dense: work items (output tiles) of all problems
    int64_t M_total;         // grouped contraction: rows of the token-sorted inputs
    const int64_t* offsets;  // grouped: [G+1] on the device
    int G;
    int64_t a_bands_cap;     // grouped rows: 0 = A scales MMA-tiled over all rows; > 0 = group-tiled
                             // (each group's rows tiled on their own, at most this many bands)
    uint8_t* yq;             // quantizing epilogue: E4M3 payload [M, N] (row stride N)
    uint8_t* ys;             //   and its MMA-tiled scales [M, N/32]
    int yq_tma;              // 1: PairMaps::yq maps yq (32 x 32 tiled payload stores)
    unsigned int* status;
    uint64_t wait_limit_ns;
};

// Tensor maps of A and B per problem (a kernel parameter: TMA reads them there).
struct TensorMaps {
    CUtensorMap a[kMaxProblems];
    CUtensorMap b[kMaxProblems];
    CUtensorMap y[kMaxProblems];   // BF16 outputs, for tiled stores (Problem::y_tma)
};

// Compile-time configuration of one kernel instance.
//   BN = 128: two 128-column TMEM accumulators (the epilogue of tile t
//             overlaps the main loop of tile t+1), 4 epilogue warps.
//   BN = 256: one 256-column accumulator (two would leave no TMEM columns
//             for the scale factors); 8 epilogue warps drain it into
//             registers at once and release it before converting and
//             storing, so the next tile's MMAs start after the drain only.
// Shared memory after the ring: the grouped modes' schedule tables (grouped
// rows: tile prefix and first m-tiles; grouped contraction: slot starts and
// lengths), then, with BN = 256 and outside the quantizing epilogue, a 2 KB
// staging buffer per epilogue warp (see store_staged).
template <int BN, int STAGES, int kMode>
struct Cfg {
    static constexpr int kAccStages = BN == 128 ? 2 : 1;
    static constexpr int kEpiWarps = 4 * (BN / 128);   // each owns 32 lanes x 128 columns
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kBBytes = BN * kBK;            // per stage
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kSfbAtoms = BN / 128;
    static constexpr int kOffB = 0;                     // B first: see the N-major note below
    static constexpr int kOffA = kOffB + STAGES * kBBytes;
    static constexpr int kOffSfa = kOffA + STAGES * kABytes;
    static constexpr int kOffSfb = kOffSfa + STAGES * 512;
    static constexpr int kOffBar = kOffSfb + STAGES * 512 * kSfbAtoms;
    static constexpr int kNumBars = 2 * STAGES + 2 * kAccStages + 1;
    static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffEpiFlag = kOffAbort + 4;   // accumulator-ready verdict for the epilogue warps
    static constexpr int kOffSched = (kOffEpiFlag + 4 + 15) / 16 * 16;
    static constexpr int kSchedBytes = kMode == kGroupedRows || kMode == kGroupedK ? 4 * (kMaxGroups + 1) + 4 * kMaxGroups : 0;
    static constexpr bool kStaged = BN == 256 && kMode != kDenseQuant;
    static constexpr int kStageWarpBytes = 32 * 32 * 2;  // 32 rows x 32 BF16 columns
    static constexpr int kOffStage = (kOffSched + kSchedBytes + 1023) / 1024 * 1024;   // 64-byte swizzle atoms
    static constexpr int kBytes = kOffStage + (kStaged ? kEpiWarps * kStageWarpBytes : 0);
    static constexpr int kAlloc = kBytes + 1024;        // slack for 1024-byte alignment
    // TMEM columns: accumulators, then per-stage SFA and SFB slots.
    static constexpr int kTmemSfa = kAccStages * BN;
    static constexpr int kTmemSfb = kTmemSfa + 4 * STAGES;
    static constexpr int kTmemUsed = kTmemSfb + 4 * kSfbAtoms * STAGES;
    static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static_assert(kTmemUsed <= 512, "tensor memory budget");
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// Output-tile schedule.  Dense: raster bands of kRasterBand m-tiles, n-tiles
// inside a band.  Grouped rows: tiles of expert g cover the 128-row blocks that
// intersect [off[g], off[g+1]); n-tiles innermost.  Grouped contraction: every
// expert has the full m x n tile grid (rastered as dense); its K range is the
// expert's 128-aligned token slot.
struct TileInfo {
    int64_t m0;      // first row of the A tile (multiple of 128, or a group's first row + 128 i)
    int64_t a_band;  // 128-row band of the A scale atoms of the tile
    int64_t n0;      // first output column
    int64_t row_lo;  // rows [row_lo, row_hi) of this tile are stored
    int64_t row_hi;
    int64_t b_row;   // first row of the B tile in the (stacked) B matrix
    int64_t kb0;     // first 128-deep K block
    int nkb;         // K blocks of this tile (0: the tile is all zeros)
    int64_t y_row0;  // output row of A row 0 (grouped contraction: g * M)
    int prob;        // problem of the tile
};

struct Schedule {
    int64_t m_tiles, n_tiles, total;   // grouped modes (dense: per problem)
    // grouped modes only (shared memory)
    const int* prefix;    // [G+1] grouped rows: tile prefix; grouped K: slot start / 128
    const int* first_mt;  // [G]   grouped rows: first m-tile (group-tiled A scales: first band);
                          //       grouped K: slot length / 128
    int G;
};

// Group offset g, clamped to [0, limit] so that malformed offsets stay in bounds.
__device__ __forceinline__ int64_t clamped_offset(const GemmArgs& p, int g, int64_t limit) {
    const int64_t o = p.offsets[g];
    return o < 0 ? int64_t(0) : (o > limit ? limit : o);
}

// Problem of dense work item t (problems are laid out back to back).
__device__ __forceinline__ int problem_of(const GemmArgs& p, int64_t t) {
    int q = 0;
    while (q + 1 < p.nprob && t >= p.pr[q + 1].first_item) ++q;
    return q;
}

template <int BN, int kMode>
__device__ __forceinline__ TileInfo tile_info(const Schedule& s, const GemmArgs& p, int64_t t) {
    TileInfo ti;
    ti.kb0 = 0;
    ti.y_row0 = 0;
    ti.prob = 0;
    if constexpr (kMode != kGroupedRows) {
        int64_t g = 0;
        int64_t m_tiles = s.m_tiles, n_tiles = s.n_tiles;
        if constexpr (kMode == kGroupedK) {
            const int64_t per = s.m_tiles * s.n_tiles;
            g = t / per;
            t -= g * per;
        } else {
            ti.prob = problem_of(p, t);
            t -= p.pr[ti.prob].first_item;
            m_tiles = p.pr[ti.prob].m_tiles;
            n_tiles = p.pr[ti.prob].n_tiles;
        }
        const Problem& P = p.pr[ti.prob];
        ti.nkb = P.num_kb;
        const int64_t per_band = static_cast<int64_t>(kRasterBand) * n_tiles;
        const int64_t band = t / per_band, within = t - band * per_band;
        const int64_t mb = band * kRasterBand;
        const int64_t bh = min(static_cast<int64_t>(kRasterBand), m_tiles - mb);
        const int64_t m_blk = mb + within % bh, n_blk = within / bh;
        ti.m0 = m_blk * kBM;
        ti.a_band = m_blk;
        ti.n0 = n_blk * BN;
        ti.row_lo = ti.m0;
        ti.row_hi = min(ti.m0 + kBM, P.M);
        ti.b_row = ti.n0;
        if constexpr (kMode == kGroupedK) {
            ti.kb0 = s.prefix[g];
            ti.nkb = s.first_mt[g];
            ti.y_row0 = g * P.M;
        }
    } else {
        int lo = 0, hi = s.G;  // largest g with prefix[g] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s.prefix[mid] <= t) lo = mid; else hi = mid;
        }
        const int g = lo;
        const Problem& P = p.pr[0];
        ti.nkb = P.num_kb;
        const int64_t local = t - s.prefix[g];
        const int64_t n_blk = local % s.n_tiles;
        const int64_t first_row = clamped_offset(p, g, P.M);
        if (p.a_bands_cap > 0) {   // tiles from the group's first row
            ti.m0 = first_row + (local / s.n_tiles) * kBM;
            ti.a_band = s.first_mt[g] + local / s.n_tiles;
            ti.row_lo = ti.m0;
        } else {                   // tiles on the 128-row grid of all rows
            const int64_t m_blk = s.first_mt[g] + local / s.n_tiles;
            ti.m0 = m_blk * kBM;
            ti.a_band = m_blk;
            ti.row_lo = max(ti.m0, first_row);
        }
        ti.n0 = n_blk * BN;
        ti.row_hi = min(ti.m0 + kBM, clamped_offset(p, g + 1, P.M));
        ti.b_row = static_cast<int64_t>(g) * P.N + ti.n0;
    }
    return ti;
}

// One epilogue warp's share of a finished tile through its 2 KB shared-memory
// staging buffer: lane l holds output row row0 + l (y's row numbering) in v,
// FP32 columns n .. n+127.  Per 32-column chunk each lane writes its row's 64
// BF16 bytes to the buffer; 16-byte chunk j of staged row r sits at position
// j ^ ((r >> 1) & 3), which is the 64-byte swizzle of a tiled bulk copy.  When
// all 32 rows are stored, lane 0 stores the chunk with one tiled bulk copy
// (the tensor map clips columns past N and rows past the matrix) and the warp
// goes on; the buffer is rewritten only after that copy has read it (`pending`
// carries this across calls, so the wait for a tile's last chunk falls after
// the next tile's accumulator drain).  Otherwise the warp stores 8 rows x 64
// contiguous bytes per instruction, skipping rows outside [row_lo, row_hi)
// (tile-row numbering); writes (one row per lane) and reads (four lanes per
// row) of the buffer are conflict-free.
__device__ __forceinline__ void store_staged(const Problem& p, const uint32_t (&v)[4][32], uint32_t stage,
                                             int64_t row0, int64_t tile_row0, int64_t row_lo, int64_t row_hi,
                                             int64_t n, int lane, const CUtensorMap* ymap, bool& pending) {
    const uint32_t wrow = stage + 64u * static_cast<uint32_t>(lane);
    const uint32_t wswz = static_cast<uint32_t>((lane >> 1) & 3);
    const int rsub = lane >> 2;   // row within an 8-row group
    const int jj = lane & 3;      // 16-byte chunk within a 64-byte row
    // All 32 rows stored: one tiled store from the buffer (its layout is the
    // 64-byte swizzle); otherwise the rows in [row_lo, row_hi) one by one.
    const bool whole = p.y_tma && tile_row0 >= row_lo && tile_row0 + 32 <= row_hi;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            o[j].x = cvt_bf16x2(__uint_as_float(v[c][8 * j + 0]), __uint_as_float(v[c][8 * j + 1]));
            o[j].y = cvt_bf16x2(__uint_as_float(v[c][8 * j + 2]), __uint_as_float(v[c][8 * j + 3]));
            o[j].z = cvt_bf16x2(__uint_as_float(v[c][8 * j + 4]), __uint_as_float(v[c][8 * j + 5]));
            o[j].w = cvt_bf16x2(__uint_as_float(v[c][8 * j + 6]), __uint_as_float(v[c][8 * j + 7]));
        }
        if (pending) {   // the previous tiled store still reads the buffer
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            pending = false;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) sts128(wrow + 16u * (static_cast<uint32_t>(j) ^ wswz), o[j]);
        if (whole) {
            fence_proxy_async_smem();   // the buffer is read by the bulk copy (async proxy)
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(ymap, static_cast<int32_t>(n + 32 * c), static_cast<int32_t>(row0), stage);
                bulk_commit_group();
            }
            pending = true;
            continue;
        }
        __syncwarp();
        const int64_t col = n + 32 * c + 8 * jj;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 8 * i + rsub;
            const uint4 x = lds128_ordered(stage + 64u * static_cast<uint32_t>(r) +
                                           16u * (static_cast<uint32_t>(jj) ^ static_cast<uint32_t>((r >> 1) & 3)));
            if (tile_row0 + r >= row_lo && tile_row0 + r < row_hi && col + 8 <= p.N)
                *reinterpret_cast<uint4*>(p.y + (row0 + r) * p.ldy + col) = x;
        }
        __syncwarp();   // the buffer is rewritten by the next chunk
    }
}

// One epilogue thread's share of a finished tile: 128 accumulator columns
// (starting at n) of output row `row`, stored when row_lo <= row < row_hi.
// kDenseQuant rounds them to BF16 (stored when y is given) and writes their
// 1x32 MXFP8 quantization: 32-byte payload runs and one 4-byte word of a tiled
// scale atom (zero for rows or groups past the matrix: the layout's padding,
// written for every row of a band that lies in the matrix, tile_in).
template <int kMode>
__device__ __forceinline__ void store_row(const GemmArgs& a, const Problem& p, uint32_t (&v)[4][32], int64_t row, int64_t row_lo,
                                          int64_t row_hi, int64_t y_row0, int64_t n, bool tile_in) {
    if constexpr (kMode == kDenseQuant) {
        // Round to BF16, then quantize each 32-column group of this row in
        // registers (rceil E8M0 scale, E4M3 payload): the same bytes as
        // quantizing the BF16 output, without its round trip through HBM.
        const bool row_in = row >= row_lo && row < row_hi;
        const int64_t ngroups = p.N >> 5;
        const int64_t g0 = n >> 5;    // a multiple of 4
        uint32_t codes = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t nc = n + c * 32;
            const bool grp_ok = row_in && nc < p.N;
            uint32_t b[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                b[i] = cvt_bf16x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1]));
            if (grp_ok && p.y != nullptr) {
                uint4* yd = reinterpret_cast<uint4*>(p.y + row * p.ldy + nc);
#pragma unroll
                for (int q = 0; q < 4; ++q) yd[q] = make_uint4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
            }
            uint32_t m2 = 0u;
#pragma unroll
            for (int i = 0; i < 16; ++i) m2 = max_abs_bf16x2(m2, b[i]);
            m2 &= 0x7FFF7FFFu;
            const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
            uint32_t o[8];
            uint32_t code;
            if (m >= 0x7F80u) {  // NaN or Inf in the group
                code = 0xFFu;
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = nan_bytes4(b[2 * j], b[2 * j + 1]);
            } else {
                const int e = rceil_exponent<0>(m);
                // 2^-e in both BF16 halves: the BF16 product is exact (or, below 2^-126,
                // converts to the same signed zero as the exact value)
                const uint32_t s2 = pow2_neg_bf16(e) * 0x10001u;
                code = static_cast<uint32_t>(e + 127);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t p0 = mul_bf16x2(b[2 * j], s2), p1 = mul_bf16x2(b[2 * j + 1], s2);
                    o[j] = cvt_fp8x2<0>(bf16_lo(p0), bf16_hi(p0)) | (cvt_fp8x2<0>(bf16_lo(p1), bf16_hi(p1)) << 16);
                }
            }
            if (grp_ok) {
                uint4* qd = reinterpret_cast<uint4*>(a.yq + row * p.N + nc);
                qd[0] = make_uint4(o[0], o[1], o[2], o[3]);
                qd[1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
            codes |= (grp_ok ? code : 0u) << (8 * c);
        }
        // The 4 groups are 4 consecutive bytes of one tiled scale atom.
        if (tile_in && g0 < ((ngroups + 3) & ~static_cast<int64_t>(3)))
            *reinterpret_cast<uint32_t*>(a.ys + tiled_scale_offset(row, g0, ngroups)) = codes;
    } else {
        (void)tile_in;
        if (row >= row_lo && row < row_hi) {
            uint16_t* yrow = p.y + (y_row0 + row) * p.ldy;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int64_t nc = n + c * 32;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (nc + 8 * q + 8 <= p.N) {
                        uint4 o;
                        o.x = cvt_bf16x2(__uint_as_float(v[c][8 * q + 0]), __uint_as_float(v[c][8 * q + 1]));
                        o.y = cvt_bf16x2(__uint_as_float(v[c][8 * q + 2]), __uint_as_float(v[c][8 * q + 3]));
                        o.z = cvt_bf16x2(__uint_as_float(v[c][8 * q + 4]), __uint_as_float(v[c][8 * q + 5]));
                        o.w = cvt_bf16x2(__uint_as_float(v[c][8 * q + 6]), __uint_as_float(v[c][8 * q + 7]));
                        *reinterpret_cast<uint4*>(yrow + nc + 8 * q) = o;
                    }
                }
            }
        }
    }
}

// The quantizing epilogue of the pair kernel, staged like store_staged: for
// each 32-column chunk the warp's 32 rows write their BF16 values (when y is
// written; 64-byte swizzled rows, as store_staged) and their E4M3 payload bytes
// (32-byte rows) to shared memory, and each leaves with one tiled bulk store;
// the four scale codes a thread holds per 128 columns are one 4-byte word of a
// tiled scale atom, stored directly.  The arithmetic is store_row's.  When the
// warp's rows are not all stored (a ragged M) or a map is missing, store_row
// takes the tile.  `pending`: this warp's last bulk stores may still read the
// buffers.
__device__ __forceinline__ void store_quant_staged(const GemmArgs& a, const Problem& p, uint32_t (&v)[4][32],
                                                   uint32_t stage_y, uint32_t stage_q, int64_t row0,
                                                   int64_t row_lo, int64_t row_hi, int64_t n, int lane,
                                                   const CUtensorMap* ymap, const CUtensorMap* qmap,
                                                   bool tile_in, bool& pending) {
    const bool rows_whole = row0 >= row_lo && row0 + 32 <= row_hi;
    const bool with_y = p.y != nullptr;
    if (!rows_whole || !a.yq_tma || (with_y && !p.y_tma)) {
        store_row<kDenseQuant>(a, p, v, row0 + lane, row_lo, row_hi, 0, n, tile_in);
        return;
    }
    const int64_t row = row0 + lane;
    const int64_t ngroups = p.N >> 5;
    const int64_t g0 = n >> 5;    // a multiple of 4
    const uint32_t wrow = stage_y + 64u * static_cast<uint32_t>(lane);
    const uint32_t wswz = static_cast<uint32_t>((lane >> 1) & 3);
    const uint32_t qrow = stage_q + 32u * static_cast<uint32_t>(lane);
    uint32_t codes = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int64_t nc = n + c * 32;
        const bool grp_ok = nc < p.N;
        uint32_t b[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            b[i] = cvt_bf16x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1]));
        uint32_t m2 = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) m2 = max_abs_bf16x2(m2, b[i]);
        m2 &= 0x7FFF7FFFu;
        const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
        uint32_t o[8];
        uint32_t code;
        if (m >= 0x7F80u) {  // NaN or Inf in the group
            code = 0xFFu;
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = nan_bytes4(b[2 * j], b[2 * j + 1]);
        } else {
            const int e = rceil_exponent<0>(m);
            const uint32_t s2 = pow2_neg_bf16(e) * 0x10001u;
            code = static_cast<uint32_t>(e + 127);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t p0 = mul_bf16x2(b[2 * j], s2), p1 = mul_bf16x2(b[2 * j + 1], s2);
                o[j] = cvt_fp8x2<0>(bf16_lo(p0), bf16_hi(p0)) | (cvt_fp8x2<0>(bf16_lo(p1), bf16_hi(p1)) << 16);
            }
        }
        codes |= (grp_ok ? code : 0u) << (8 * c);
        if (pending) {   // the previous chunk's bulk stores still read the buffers
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            pending = false;
        }
        if (with_y) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                sts128(wrow + 16u * (static_cast<uint32_t>(j) ^ wswz),
                       make_uint4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]));
        }
        sts128(qrow, make_uint4(o[0], o[1], o[2], o[3]));
        sts128(qrow + 16u, make_uint4(o[4], o[5], o[6], o[7]));
        fence_proxy_async_smem();   // the buffers are read by the bulk copies (async proxy)
        __syncwarp();
        if (lane == 0 && grp_ok) {
            if (with_y) tma_store_2d(ymap, static_cast<int32_t>(nc), static_cast<int32_t>(row0), stage_y);
            tma_store_2d(qmap, static_cast<int32_t>(nc), static_cast<int32_t>(row0), stage_q);
            bulk_commit_group();
        }
        pending = grp_ok;
    }
    // The 4 groups are 4 consecutive bytes of one tiled scale atom.
    if (tile_in && g0 < ((ngroups + 3) & ~static_cast<int64_t>(3)))
        *reinterpret_cast<uint32_t*>(a.ys + tiled_scale_offset(row, g0, ngroups)) = codes;
}

// Wait for the accumulator hand-off between the MMA warp and the epilogue, on
// the critical path between tiles: busy polling without suspending the thread
// (measured 1-4% faster than the suspending probe), bounded, then the timed wait.
__device__ __forceinline__ bool spin_phase(uint32_t bar, uint32_t parity, const WaitGuard& g) {
    for (uint32_t i = 0; i < (1u << 20); ++i)
        if (mbar_test_wait(bar, parity)) return true;
    return mbar_wait(bar, parity, g);
}

// Fast path of a bounded wait: one probe inline, the polling loop out of line.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitGuard& g) {
    return mbar_try_wait(bar, parity) || mbar_wait(bar, parity, g);
}

template <int BN, int STAGES, bool kMnMajor, int kMode>
__global__ void __launch_bounds__(Cfg<BN, STAGES, kMode>::kThreads, 1)
    gemm_mxf8_kernel(const __grid_constant__ TensorMaps maps, const GemmArgs p) {
    using L = Cfg<BN, STAGES, kMode>;
    constexpr int kAcc = L::kAccStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t bar0 = sbase + L::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + kAcc + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * kAcc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
    volatile int* epi_flag = reinterpret_cast<volatile int*>(smem + L::kOffEpiFlag);
    const WaitGuard guard{abort_flag, p.status, p.wait_limit_ns};

    // ---- set-up -------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), L::kEpiWarps);  // one arrive per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int q = 0; q < p.nprob; ++q) {
            prefetch_tensormap(&maps.a[q]);
            prefetch_tensormap(&maps.b[q]);
        }
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kOffTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }

    Schedule sch;
    sch.m_tiles = p.pr[0].m_tiles;
    sch.n_tiles = p.pr[0].n_tiles;
    sch.G = p.G;
    if constexpr (kMode == kDense || kMode == kDenseQuant) {
        sch.total = p.items;
        sch.prefix = nullptr;
        sch.first_mt = nullptr;
    } else {
        // Tables built from the clamped offsets (tile_info reads the two offsets
        // of a grouped-row tile again, clamped the same way, for its row mask).
        int* s_prefix = reinterpret_cast<int*>(smem + L::kOffSched);
        int* s_first = s_prefix + (kMaxGroups + 1);
        const int64_t row_limit = kMode == kGroupedRows ? p.pr[0].M : p.M_total;
        if (warp == 0) {  // tile counts and their exclusive prefix, 32 groups at a time
            int carry = 0, band_carry = 0;
            for (int base = 0; base < p.G; base += 32) {
                const int g = base + lane;
                int cnt = 0, bands = 0;
                if (g < p.G) {
                    const int64_t lo = clamped_offset(p, g, row_limit), hi = clamped_offset(p, g + 1, row_limit);
                    if constexpr (kMode == kGroupedRows) {
                        if (p.a_bands_cap == 0) {
                            const int64_t fm = lo / kBM;
                            s_first[g] = static_cast<int>(fm);
                            cnt = hi > lo ? static_cast<int>((hi - 1) / kBM - fm + 1) * static_cast<int>(sch.n_tiles) : 0;
                        } else {
                            bands = hi > lo ? static_cast<int>((hi - lo + kBM - 1) / kBM) : 0;
                        }
                    } else {  // slot length in 128-token blocks
                        cnt = hi > lo ? static_cast<int>((hi - lo + kBK - 1) / kBK) : 0;
                        s_first[g] = cnt;
                    }
                }
                if (kMode == kGroupedRows && p.a_bands_cap > 0) {
                    // Group-tiled A scales: group g's bands start at band B_g (the
                    // prefix of the band counts); bands at or past the cap are dropped.
                    int bincl = bands;
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const int y = __shfl_up_sync(0xFFFFFFFFu, bincl, d);
                        if (lane >= d) bincl += y;
                    }
                    const int64_t first_band = band_carry + bincl - bands;
                    if (g < p.G) {
                        s_first[g] = static_cast<int>(first_band);
                        const int64_t kept = min(static_cast<int64_t>(bands), max(int64_t(0), p.a_bands_cap - first_band));
                        cnt = static_cast<int>(kept) * static_cast<int>(sch.n_tiles);
                    }
                    band_carry += __shfl_sync(0xFFFFFFFFu, bincl, 31);
                }
                int incl = cnt;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                    if (lane >= d) incl += y;
                }
                if (g < p.G) s_prefix[g] = carry + incl - cnt;
                carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
            if (lane == 0) s_prefix[p.G] = carry;
        }
        sch.prefix = s_prefix;
        sch.first_mt = s_first;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemSlot);
    if constexpr (kMode == kGroupedRows) sch.total = sch.prefix[p.G];
    if constexpr (kMode == kGroupedK) {
        sch.total = static_cast<int64_t>(p.G) * sch.m_tiles * sch.n_tiles;
        // the slots must fit the K extent of the operands
        if (static_cast<int64_t>(sch.prefix[p.G]) * kBK > p.pr[0].K) sch.total = 0;
    }
    // Work item of this CTA's r-th round.  Dense launches (whose problems come
    // longest K first) take the items of odd rounds in reverse CTA order, so
    // that CTAs that drew long tiles early draw the last short ones late; the
    // grouped modes go round-robin.
    auto item_of = [&](int64_t r) -> int64_t {
        const int64_t g = gridDim.x;
        if constexpr (kMode == kDense || kMode == kDenseQuant)
            return r * g + ((r & 1) ? g - 1 - blockIdx.x : blockIdx.x);
        return r * g + blockIdx.x;
    };

    if (warp == 0) {
        // ---- producer -------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            const uint32_t full0 = full_bar(0), empty0 = empty_bar(0);
            for (int64_t r = 0; r * gridDim.x < sch.total && !*abort_flag; ++r) {
                const int64_t t = item_of(r);
                if (t >= sch.total) continue;
                const TileInfo ti = tile_info<BN, kMode>(sch, p, t);
                const Problem& P = p.pr[ti.prob];
                const CUtensorMap* tma_a = &maps.a[ti.prob];
                const CUtensorMap* tma_b = &maps.b[ti.prob];
                const int64_t b_band0 = ti.b_row / 128;
                int sfb_atoms = 0;
#pragma unroll
                for (int j = 0; j < L::kSfbAtoms; ++j)
                    if (b_band0 + j < P.b_bands) ++sfb_atoms;
                const uint32_t bytes = L::kABytes + L::kBBytes + 512u + 512u * sfb_atoms;
                const uint8_t* sfa_src = P.a_s + (ti.a_band * P.k_atoms + ti.kb0) * 512;
                const uint8_t* sfb_src = P.b_s + (b_band0 * P.k_atoms + ti.kb0) * 512;
                const int64_t sfb_band_stride = P.k_atoms * 512;
                const int32_t ma = static_cast<int32_t>(ti.m0);
                const int32_t nb = static_cast<int32_t>(ti.b_row);
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    const uint32_t fb = full0 + 8u * stage;
                    if (!wait_phase(empty0 + 8u * stage, phase ^ 1u, guard)) break;
                    mbar_arrive_expect_tx(fb, bytes);
                    const uint32_t sa = sbase + L::kOffA + stage * L::kABytes;
                    const uint32_t sb = sbase + L::kOffB + stage * L::kBBytes;
                    const int32_t kx = static_cast<int32_t>((ti.kb0 + kb) * kBK);
                    tma_load_2d(sa, tma_a, kx, ma, fb);
                    if constexpr (!kMnMajor) {
                        tma_load_2d(sb, tma_b, kx, nb, fb);
                    } else {
                        // B stored [K, N]: boxes of 128 N-bytes x 128 K-rows, one per 128 columns.
#pragma unroll
                        for (int j = 0; j < BN / 128; ++j)
                            tma_load_2d(sb + j * 128 * kBK, tma_b, nb + 128 * j, kx, fb);
                    }
                    bulk_load(sbase + L::kOffSfa + stage * 512, sfa_src + kb * 512, 512u, fb);
                    for (int j = 0; j < sfb_atoms; ++j)
                        bulk_load(sbase + L::kOffSfb + (stage * L::kSfbAtoms + j) * 512,
                                  sfb_src + j * sfb_band_stride + kb * 512, 512u, fb);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (*abort_flag) {
                // Let copies already in flight land before the CTA exits.
                const int64_t n = issued < STAGES ? issued : STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (int64_t i = 0; i < n; ++i) {
                    if (--s < 0) { s = STAGES - 1; ph ^= 1u; }
                    WaitGuard g2 = guard;
                    volatile int never = 0;
                    g2.abort_flag = &never;
                    (void)mbar_wait(full_bar(s), ph, g2);
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer -----------------------------------------------------
        // The whole warp runs the loops (warp-uniform control flow, so counters
        // and descriptors stay in uniform registers); lane 0 waits on the
        // barriers and broadcasts the verdict, and one elected lane issues the
        // tensor-core instructions.
        {
            const uint64_t a_desc0 = make_smem_desc(sbase + L::kOffA, 16, 1024, 2);
            const uint64_t b_desc0 = kMnMajor ? make_smem_desc(sbase + L::kOffB, 128 * kBK, 1024, 2)
                                              : make_smem_desc(sbase + L::kOffB, 16, 1024, 2);
            const uint64_t sfa_desc0 = make_smem_desc(sbase + L::kOffSfa, 0, 128, 0);
            const uint64_t sfb_desc0 = make_smem_desc(sbase + L::kOffSfb, 0, 128, 0);
            constexpr uint32_t kBStepK = kMnMajor ? (kUmmaK * 128) >> 4 : kUmmaK >> 4;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t r = 0; r * gridDim.x < sch.total && ok; ++r) {
                const int64_t t = item_of(r);
                if (t >= sch.total) continue;
                int got = 1;
                if (lane == 0) got = spin_phase(tempty_bar(acc), acc_phase ^ 1u, guard) ? 1 : 0;
                if (!__shfl_sync(0xFFFFFFFFu, got, 0)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const int q = kMode == kDense || kMode == kDenseQuant ? problem_of(p, t) : 0;
                const int nkb = kMode == kGroupedK ? tile_info<BN, kMode>(sch, p, t).nkb : p.pr[q].num_kb;
                const int64_t K = p.pr[q].K;
                const uint32_t fmt_bits = p.pr[q].fmt_bits;
                for (int kb = 0; kb < nkb; ++kb) {
                    int fgot = 1;
                    if (lane == 0) fgot = wait_phase(full_bar(stage), phase, guard) ? 1 : 0;
                    if (!__shfl_sync(0xFFFFFFFFu, fgot, 0)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + L::kTmemSfa + 4 * stage;
                    const uint32_t sfb_t = tmem_base + L::kTmemSfb + 4 * L::kSfbAtoms * stage;
                    const uint64_t a_desc = a_desc0 + static_cast<uint64_t>((stage * L::kABytes) >> 4);
                    const uint64_t b_desc = b_desc0 + static_cast<uint64_t>((stage * L::kBBytes) >> 4);
                    const uint64_t sfa_d = sfa_desc0 + static_cast<uint64_t>((stage * 512) >> 4);
                    const uint64_t sfb_d = sfb_desc0 + static_cast<uint64_t>((stage * L::kSfbAtoms * 512) >> 4);
                    const int64_t k_left = kMode == kGroupedK ? static_cast<int64_t>(nkb - kb) * kBK
                                                              : K - static_cast<int64_t>(kb) * kBK;
                    const int ksub = k_left >= kBK ? kBK / kUmmaK : static_cast<int>(k_left) / kUmmaK;
                    if (elect_one()) {
                        tc_cp_32x128b_warpx4(sfa_t, sfa_d);
#pragma unroll
                        for (int a = 0; a < L::kSfbAtoms; ++a)
                            tc_cp_32x128b_warpx4(sfb_t + 4 * a, sfb_d + static_cast<uint64_t>((a * 512) >> 4));
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k)
                            if (k < ksub)
                                tc_mma_mxf8(d_tmem, a_desc + ((k * kUmmaK) >> 4), b_desc + k * kBStepK,
                                            make_idesc_mxf8(kBM, BN, kMnMajor ? 1u : 0u, k, k) | fmt_bits, sfa_t,
                                            sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
                        tc_commit(empty_bar(stage));  // frees the slot once these MMAs are done
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (elect_one()) tc_commit(tfull_bar(acc));
                __syncwarp();
                if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
            }
            // Drain: every MMA and copy issued above completes before teardown.
            if (lane == 0) {
                tc_commit(drain_bar);
                WaitGuard g2 = guard;
                volatile int never = 0;
                g2.abort_flag = &never;
                (void)mbar_wait(drain_bar, 0, g2);
            }
            __syncwarp();
        }
    } else {
        // ---- epilogue (warps 2 .. 2+kEpiWarps-1) ------------------------------
        // Warp w reads TMEM lanes 32*(w%4).. (its lane quarter) and the
        // 128-column half (w-2)/4 of the accumulator.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool pending = false;   // a tiled store of this warp may still read its buffer
        for (int64_t r = 0; r * gridDim.x < sch.total; ++r) {
            const int64_t t = item_of(r);
            if (t >= sch.total) continue;
            const TileInfo ti = tile_info<BN, kMode>(sch, p, t);
            // One thread waits for the finished accumulator with the suspending
            // try_wait; the other epilogue warps sleep on named barrier 1 meanwhile
            // (busy polling from every warp for a whole main loop measured 0-4%
            // slower: the polls take issue slots and shared-memory bandwidth).
            // Barrier 2 keeps the flag from being rewritten before every warp has
            // read it.  All warps follow one verdict, so the .sync.aligned
            // tensor-memory loads below always run with full warps.
            if (warp == 2 && lane == 0) *epi_flag = wait_phase(tfull_bar(acc), acc_phase, guard) ? 1 : 0;
            named_bar_sync(1, 32 * L::kEpiWarps);
            const int ok = *epi_flag;
            named_bar_sync(2, 32 * L::kEpiWarps);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + acc * BN + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + 32 * c, v[c]);
            tmem_ld_wait();
            // The accumulator is in registers: hand it back to the MMA warp now.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }

            if (ti.nkb == 0) {  // no K blocks (an empty expert): the tile is zero
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[c][j] = 0u;
            }
            const Problem& P = p.pr[ti.prob];
            if constexpr (L::kStaged)
                store_staged(P, v, sbase + L::kOffStage + (warp - 2) * L::kStageWarpBytes,
                             ti.y_row0 + ti.m0 + 32 * quad, ti.m0 + 32 * quad, ti.row_lo, ti.row_hi,
                             ti.n0 + half * 128, lane, &maps.y[ti.prob], pending);
            else
                store_row<kMode>(p, P, v, ti.m0 + 32 * quad + lane, ti.row_lo, ti.row_hi, ti.y_row0,
                                 ti.n0 + half * 128, ti.m0 < P.M);
        }
        if (lane == 0) bulk_wait_all();   // this warp's tiled stores complete before the CTA ends
        __syncwarp();
    }

    // ---- teardown -----------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

// ---- GEMMs on CTA pairs (clusters of two, tcgen05 cta_group::2) ----------------------
//
// Output tiles of 256 x 256 per pair of SMs.  CTA rank r of the pair owns the
// 128 rows of its half: it loads those rows of A, its 128-row half of the B
// tile (B rows b_row + 128 r; N-major B: columns n0 + 128 r) and its A scale
// atom; it also needs both B scale atoms (every CTA's tensor core reads the
// scales of all 256 B rows from its own tensor memory), so CTA r loads atom r
// and multicasts it to both.  All of it completes on the even CTA's full
// barrier.  Warp 1 of the even CTA runs the tile and stage loops warp-uniformly
// and one elected lane issues, per 128-deep stage, three pair scale copies and
// four 256 x 256 x 32 pair MMAs, then a commit that frees the stage's slot in
// both CTAs.  Against the single-CTA 128 x 256 tile this halves the operand
// bytes each SM stages per multiply-add and the instructions issued per
// multiply-add; a stage is 33.5 KB per CTA, six stages deep.  Each CTA's eight
// epilogue warps drain its 128 accumulator rows and arrive on the even CTA's
// accumulator-empty barrier.
//
// Modes: dense (1-4 GEMMs per launch, longest K first), dense with the
// quantizing epilogue, grouped rows (a pair tile is two 128-row tiles of one
// expert; when an expert has an odd number of row tiles the odd CTA of its last
// pair tile stores nothing), grouped contraction (a pair tile is 256 x 256 of
// one expert's weight gradient over that expert's token slot).
template <int kMode>
struct PairCfg {
    static constexpr bool kGrouped = kMode == kGroupedRows || kMode == kGroupedK;
    static constexpr int kMaxGroups = 512;             // larger G runs on the single-CTA kernel
    static constexpr int kStages = 6;
    static constexpr int kEpiWarps = 8;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kABytes = 128 * kBK;          // own A rows per stage
    static constexpr int kBBytes = 128 * kBK;          // own half of B per stage
    static constexpr int kSfbBytes = 2 * 512;          // scale atoms of all 256 B rows
    static constexpr int kStageBytes = kABytes + kBBytes + 512 + kSfbBytes;   // per CTA
    static constexpr int kOffB = 0;
    static constexpr int kOffA = kOffB + kStages * kBBytes;
    static constexpr int kOffSfa = kOffA + kStages * kABytes;
    static constexpr int kOffSfb = kOffSfa + kStages * 512;
    static constexpr int kOffBar = kOffSfb + kStages * kSfbBytes;
    static constexpr int kNumBars = 2 * kStages + 3;   // full, empty, accumulator full / empty, drain
    static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffEpiFlag = kOffAbort + 4;
    static constexpr int kOffSched = (kOffEpiFlag + 4 + 15) / 16 * 16;
    static constexpr int kSchedBytes = kGrouped ? 4 * (kMaxGroups + 1) + 4 * kMaxGroups : 0;
    static constexpr int kOffStage = (kOffSched + kSchedBytes + 1023) / 1024 * 1024;   // 64-byte swizzle atoms
    static constexpr int kStageWarpBytes = 32 * 32 * 2;                 // BF16 chunk of 32 rows
    static constexpr int kQStageWarpBytes = kMode == kDenseQuant ? 32 * 32 : 0;   // E4M3 chunk of 32 rows
    static constexpr int kOffQStage = kOffStage + kEpiWarps * kStageWarpBytes;
    static constexpr int kBytes = kOffQStage + kEpiWarps * kQStageWarpBytes;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr int kTmemSfa = 256;               // one 256-column accumulator, then the scales
    static constexpr int kTmemSfb = kTmemSfa + 4 * kStages;
    static constexpr int kTmemCols = 512;
    static_assert(kTmemSfb + 8 * kStages <= kTmemCols, "tensor memory budget");
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// Tensor maps of a pair launch (a kernel parameter: TMA reads them there).
// Scales: the MMA-tiled bytes of an operand viewed as rows of 256 bytes, one
// 512-byte atom = a box of 2 rows.
struct PairMaps {
    CUtensorMap yq;          // quantizing epilogue: the E4M3 payload [M, N]
    CUtensorMap a[kMaxProblems];
    CUtensorMap b[kMaxProblems];
    CUtensorMap sfa[kMaxProblems];
    CUtensorMap sfb[kMaxProblems];
    CUtensorMap y[kMaxProblems];
};

// What one CTA of a pair does for pair tile t.
struct PairTileInfo {
    int prob;
    int64_t m0;              // this CTA's first A row (a TMA coordinate; may lie past the matrix)
    int64_t a_band;          // this CTA's A scale band
    int64_t row_lo, row_hi;  // A rows [row_lo, row_hi) of this CTA are stored (empty: none)
    int64_t n0;              // first output column of the pair tile
    int64_t b_row;           // first B row of the pair tile in the (stacked) B matrix
    int64_t kb0;             // first 128-deep K block
    int nkb;                 // K blocks (0: the tile is zero)
    int64_t y_row0;          // output row of A row 0 (grouped contraction: g * M)
};

// Raster order inside one m x n grid of cluster tiles (kPairs x 256 rows by 256
// columns): bands of 1024 rows for pairs and of 2048 rows (four tile rows) for
// clusters of two pairs, n-tiles inside a band.
template <int kPairs>
__device__ __forceinline__ void pair_raster(int64_t local, int64_t m_tiles, int64_t n_tiles, int64_t& m0,
                                            int64_t& n0) {
    constexpr int kBand = kPairs == 2 ? 4 : kRasterBand / 2;
    const int64_t per_band = static_cast<int64_t>(kBand) * n_tiles;
    const int64_t band = local / per_band, within = local - band * per_band;
    const int64_t mb = band * kBand;
    const int64_t bh = min(static_cast<int64_t>(kBand), m_tiles - mb);
    m0 = (mb + within % bh) * (256 * kPairs);
    n0 = (within / bh) * 256;
}

// Schedule of the grouped pair modes (shared memory, built from the device
// offsets).  Grouped rows: prefix[g] = first pair tile of expert g (prefix[G]
// = all), first[g] = expert g's first A band (group-tiled scales) or first
// 128-row block.  Grouped contraction: prefix[g] = slot start / 128, first[g] =
// slot length / 128.
struct PairSchedule {
    const int* prefix;
    const int* first;
    int64_t m_tiles, n_tiles, total;
};

// t is a cluster tile; pp is the pair's index in its cluster (dense modes:
// the pairs of a cluster take consecutive 256-row tiles of one column of tiles).
template <int kMode, int kPairs = 1>
__device__ __forceinline__ PairTileInfo pair_tile_info(const PairSchedule& s, const GemmArgs& p, int64_t t,
                                                       uint32_t rank, uint32_t pp = 0) {
    PairTileInfo ti;
    ti.kb0 = 0;
    ti.y_row0 = 0;
    ti.prob = 0;
    if constexpr (kMode == kDense || kMode == kDenseQuant) {
        ti.prob = problem_of(p, t);
        const Problem& P = p.pr[ti.prob];
        int64_t m0p;
        pair_raster<kPairs>(t - P.first_item, P.m_tiles, P.n_tiles, m0p, ti.n0);
        ti.m0 = m0p + 256 * pp + 128 * rank;
        ti.a_band = ti.m0 / 128;
        ti.row_lo = ti.m0;
        ti.row_hi = min(ti.m0 + 128, P.M);
        ti.b_row = ti.n0;
        ti.nkb = P.num_kb;
    } else if constexpr (kMode == kGroupedK) {
        const Problem& P = p.pr[0];
        const int64_t per = s.m_tiles * s.n_tiles;
        const int64_t g = t / per;
        int64_t m0p;
        pair_raster<1>(t - g * per, s.m_tiles, s.n_tiles, m0p, ti.n0);
        ti.m0 = m0p + 128 * rank;
        ti.a_band = ti.m0 / 128;
        ti.row_lo = ti.m0;
        ti.row_hi = min(ti.m0 + 128, P.M);
        ti.b_row = ti.n0;
        ti.kb0 = s.prefix[g];
        ti.nkb = s.first[g];
        ti.y_row0 = g * P.M;
    } else {   // grouped rows
        const Problem& P = p.pr[0];
        int lo = 0, hi = p.G;  // largest g with prefix[g] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s.prefix[mid] <= t) lo = mid; else hi = mid;
        }
        const int g = lo;
        const int64_t local = t - s.prefix[g];
        ti.n0 = (local % s.n_tiles) * 256;
        const int64_t i = 2 * (local / s.n_tiles) + rank;   // this CTA's row tile of the expert
        const int64_t first_row = clamped_offset(p, g, P.M), end_row = clamped_offset(p, g + 1, P.M);
        int64_t tiles;
        if (p.a_bands_cap > 0) {   // row tiles from the expert's first row, group-tiled scales
            tiles = (end_row - first_row + kBM - 1) / kBM;
            tiles = min(tiles, max(int64_t(0), p.a_bands_cap - s.first[g]));
            const int64_t ii = i < tiles ? i : 0;
            ti.m0 = first_row + ii * kBM;
            ti.a_band = s.first[g] + ii;
            ti.row_lo = ti.m0;
        } else {                   // row tiles on the 128-row grid of all rows
            tiles = end_row > first_row ? (end_row - 1) / kBM - first_row / kBM + 1 : 0;
            const int64_t ii = i < tiles ? i : 0;
            ti.a_band = s.first[g] + ii;
            ti.m0 = ti.a_band * kBM;
            ti.row_lo = max(ti.m0, first_row);
        }
        ti.row_hi = i < tiles ? min(ti.m0 + kBM, end_row) : ti.row_lo;   // past the expert's tiles: nothing
        ti.b_row = static_cast<int64_t>(g) * P.N + ti.n0;
        ti.nkb = P.num_kb;
    }
    return ti;
}

// kCluster = 2: one pair per cluster.  kCluster = 4 (dense modes): two pairs
// per cluster take vertically adjacent pair tiles of one column of tiles, which
// read the same B tile: each CTA loads half of its 128 B rows per stage and
// multicasts them to itself and to the CTA of the same rank in the other pair,
// so a cluster reads each B tile from L2 once.  A stage's slot is then written
// by both pairs' producers, and is free when both pairs' MMAs have read it: the
// empty barriers take a commit from each pair.
template <bool kMnMajor, int kMode, int kCluster>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(PairCfg<kMode>::kThreads, 1)
    gemm_mxf8_pair_kernel(const __grid_constant__ PairMaps maps, const GemmArgs p) {
    using L = PairCfg<kMode>;
    constexpr int STAGES = L::kStages;
    constexpr int kPairs = kCluster / 2;
    static_assert(kCluster == 2 || (kCluster == 4 && !L::kGrouped), "clusters of two pairs: dense modes only");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = blockIdx.x % kCluster;   // rank in the (one-dimensional) cluster
    const uint32_t rank = crank & 1u;               // rank in the pair
    const uint32_t pp = crank >> 1;                 // the pair's index in the cluster
    const uint32_t lead = crank & ~1u;              // cluster rank of the pair's even CTA
    const bool leader = rank == 0;

    const uint32_t bar0 = sbase + L::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * STAGES);
    const uint32_t tempty_bar = bar0 + 8u * (2 * STAGES + 1);
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
    volatile int* epi_flag = reinterpret_cast<volatile int*>(smem + L::kOffEpiFlag);
    const WaitGuard guard{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);      // the even CTA's producer arrives (with both CTAs' bytes)
            mbar_init(empty_bar(s), kPairs);   // each pair's even CTA's multicast commit
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, 2 * L::kEpiWarps);   // every epilogue warp of both CTAs
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int q = 0; q < p.nprob; ++q) {
            prefetch_tensormap(&maps.a[q]);
            prefetch_tensormap(&maps.b[q]);
            prefetch_tensormap(&maps.sfa[q]);
            prefetch_tensormap(&maps.sfb[q]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(sbase + L::kOffTmemSlot, L::kTmemCols);
        tmem_relinquish_pair();
    }

    PairSchedule sch;
    sch.prefix = nullptr;
    sch.first = nullptr;
    sch.m_tiles = p.pr[0].m_tiles;
    sch.n_tiles = p.pr[0].n_tiles;
    sch.total = p.items;
    if constexpr (L::kGrouped) {
        // Tables from the clamped offsets (pair_tile_info reads the two offsets of
        // a grouped-row tile again, clamped the same way, for its rows).
        int* s_prefix = reinterpret_cast<int*>(smem + L::kOffSched);
        int* s_first = s_prefix + (L::kMaxGroups + 1);
        const int64_t row_limit = kMode == kGroupedRows ? p.pr[0].M : p.M_total;
        if (warp == 0) {  // 32 groups at a time: counts, then exclusive prefixes by warp scans
            int carry = 0, band_carry = 0;
            for (int base = 0; base < p.G; base += 32) {
                const int g = base + lane;
                int cnt = 0, bands = 0;
                int64_t lo = 0, hi = 0;
                if (g < p.G) {
                    lo = clamped_offset(p, g, row_limit);
                    hi = clamped_offset(p, g + 1, row_limit);
                }
                if constexpr (kMode == kGroupedRows) {
                    if (p.a_bands_cap == 0) {
                        const int64_t tiles = hi > lo ? (hi - 1) / kBM - lo / kBM + 1 : 0;
                        if (g < p.G) s_first[g] = static_cast<int>(lo / kBM);
                        cnt = static_cast<int>((tiles + 1) / 2) * static_cast<int>(sch.n_tiles);
                    } else {
                        bands = hi > lo ? static_cast<int>((hi - lo + kBM - 1) / kBM) : 0;
                        int bincl = bands;
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {
                            const int y = __shfl_up_sync(0xFFFFFFFFu, bincl, d);
                            if (lane >= d) bincl += y;
                        }
                        const int64_t first_band = band_carry + bincl - bands;
                        const int64_t kept = min(static_cast<int64_t>(bands), max(int64_t(0), p.a_bands_cap - first_band));
                        if (g < p.G) s_first[g] = static_cast<int>(first_band);
                        cnt = static_cast<int>((kept + 1) / 2) * static_cast<int>(sch.n_tiles);
                        band_carry += __shfl_sync(0xFFFFFFFFu, bincl, 31);
                    }
                } else {   // slot length in 128-token blocks
                    cnt = hi > lo ? static_cast<int>((hi - lo + kBK - 1) / kBK) : 0;
                    if (g < p.G) s_first[g] = cnt;
                }
                int incl = cnt;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                    if (lane >= d) incl += y;
                }
                if (g < p.G) s_prefix[g] = carry + incl - cnt;
                carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
            if (lane == 0) s_prefix[p.G] = carry;
        }
        sch.prefix = s_prefix;
        sch.first = s_first;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers initialised and tensor memory allocated
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemSlot);
    if constexpr (kMode == kGroupedRows) sch.total = sch.prefix[p.G];
    if constexpr (kMode == kGroupedK) {
        sch.total = static_cast<int64_t>(p.G) * sch.m_tiles * sch.n_tiles;
        if (static_cast<int64_t>(sch.prefix[p.G]) * kBK > p.pr[0].K) sch.total = 0;   // slots past the operands
    }
    const int64_t total = sch.total;
    const int64_t pair_id = blockIdx.x / kCluster;   // this cluster's index, and the count
    const int64_t n_pairs = gridDim.x / kCluster;
    // Item of this pair's r-th round: dense problems come longest K first, and
    // dense launches take odd rounds in reverse pair order.
    auto item_of = [&](int64_t r) -> int64_t {
        if constexpr (kMode == kDense || kMode == kDenseQuant)
            return r * n_pairs + ((r & 1) ? n_pairs - 1 - pair_id : pair_id);
        return r * n_pairs + pair_id;
    };

    if (warp == 0) {
        // ---- producer (both CTAs) --------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            const uint32_t full0 = leader ? full_bar(0) : mapa_shared(full_bar(0), lead);
            for (int64_t r = 0; r * n_pairs < total && !*abort_flag; ++r) {
                const int64_t t = item_of(r);
                if (t >= total) continue;
                const PairTileInfo ti = pair_tile_info<kMode, kPairs>(sch, p, t, rank, pp);
                const Problem& P = p.pr[ti.prob];
                const CUtensorMap* ma_map = &maps.a[ti.prob];
                const CUtensorMap* mb_map = &maps.b[ti.prob];
                const int32_t ma = static_cast<int32_t>(ti.m0);
                const int32_t nb = static_cast<int32_t>(ti.b_row + 128 * rank);
                const int32_t sfa_row = static_cast<int32_t>(2 * (ti.a_band * P.k_atoms + ti.kb0));
                const int32_t sfb_row0 = static_cast<int32_t>(2 * ((ti.b_row / 128) * P.k_atoms + ti.kb0));
                const int32_t sfb_row1 = static_cast<int32_t>(2 * ((ti.b_row / 128 + 1) * P.k_atoms + ti.kb0));
                bool stop = false;
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if (!wait_phase(empty_bar(stage), phase ^ 1u, guard)) { stop = true; break; }
                    const uint32_t fb = full0 + 8u * stage;
                    if (leader) mbar_arrive_expect_tx(fb, 2u * L::kStageBytes);
                    const uint32_t ssb = sbase + L::kOffSfb + stage * L::kSfbBytes;
                    const int32_t kx = static_cast<int32_t>((ti.kb0 + kb) * kBK);
                    tma_load_2d_pair(sbase + L::kOffA + stage * L::kABytes, ma_map, kx, ma, fb);
                    if constexpr (kPairs == 1) {
                        if constexpr (!kMnMajor)
                            tma_load_2d_pair(sbase + L::kOffB + stage * L::kBBytes, mb_map, kx, nb, fb);
                        else   // B stored [K, N]: this CTA's 128 columns x 128 K-rows
                            tma_load_2d_pair(sbase + L::kOffB + stage * L::kBBytes, mb_map, nb, kx, fb);
                    } else {   // half pp of this CTA's B (64 rows: N rows, or K rows when N-major), both pairs
                        const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (2 + rank)));
                        const uint32_t bdst = sbase + L::kOffB + stage * L::kBBytes + pp * (L::kBBytes / 2);
                        if constexpr (!kMnMajor)
                            tma_load_2d_pair_mc(bdst, mb_map, kx, nb + 64 * static_cast<int32_t>(pp), fb, mask);
                        else
                            tma_load_2d_pair_mc(bdst, mb_map, nb, kx + 64 * static_cast<int32_t>(pp), fb, mask);
                    }
                    tma_load_2d_pair(sbase + L::kOffSfa + stage * 512, &maps.sfa[ti.prob], 0, sfa_row + 2 * kb, fb);
                    // Every CTA of the cluster needs the same two B scale atoms (the
                    // scales of all 256 B rows): each CTA loads its share once and
                    // multicasts it to all.  Pairs: atom `rank` to both CTAs.  Two
                    // pairs: row crank & 1 of atom crank >> 1 to all four.
                    if constexpr (kPairs == 1) {
                        tma_load_2d_pair_mc(ssb + 512 * rank, &maps.sfb[ti.prob], 0,
                                            (rank ? sfb_row1 : sfb_row0) + 2 * kb, fb, 0x3);
                    } else {
                        const int32_t srow = ((crank >> 1) ? sfb_row1 : sfb_row0) + 2 * kb + static_cast<int32_t>(crank & 1);
                        tma_load_2d_pair_mc(ssb + 256 * crank, &maps.sfb[ti.prob], 0, srow, fb, 0xF);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (stop) break;
            }
            if (*abort_flag) {
                // Loads in flight complete on the even CTA's barrier, which the odd
                // CTA cannot wait on: give them a bounded while to land.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer (even CTA; warp-uniform loops, one elected lane issues) -----------
        if (leader) {
            const uint64_t a_desc0 = make_smem_desc(sbase + L::kOffA, 16, 1024, 2);
            const uint64_t b_desc0 = kMnMajor ? make_smem_desc(sbase + L::kOffB, 128 * kBK, 1024, 2)
                                              : make_smem_desc(sbase + L::kOffB, 16, 1024, 2);
            const uint64_t sfa_desc0 = make_smem_desc(sbase + L::kOffSfa, 0, 128, 0);
            const uint64_t sfb_desc0 = make_smem_desc(sbase + L::kOffSfb, 0, 128, 0);
            constexpr uint32_t kBStepK = kMnMajor ? (kUmmaK * 128) >> 4 : kUmmaK >> 4;
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t r = 0; r * n_pairs < total && ok; ++r) {
                const int64_t t = item_of(r);
                if (t >= total) continue;
                int got = 1;
                if (lane == 0) got = spin_phase(tempty_bar, acc_phase ^ 1u, guard) ? 1 : 0;
                if (!__shfl_sync(0xFFFFFFFFu, got, 0)) { ok = false; break; }
                tc_fence_after();
                const int q = kMode == kDense || kMode == kDenseQuant ? problem_of(p, t) : 0;
                const int nkb = kMode == kGroupedK ? pair_tile_info<kMode>(sch, p, t, 0u).nkb : p.pr[q].num_kb;
                const int64_t K = p.pr[q].K;
                const uint32_t fmt_bits = p.pr[q].fmt_bits;
                for (int kb = 0; kb < nkb; ++kb) {
                    int fgot = 1;
                    if (lane == 0) fgot = wait_phase(full_bar(stage), phase, guard) ? 1 : 0;
                    if (!__shfl_sync(0xFFFFFFFFu, fgot, 0)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + L::kTmemSfa + 4 * stage;
                    const uint32_t sfb_t = tmem_base + L::kTmemSfb + 8 * stage;
                    const uint64_t a_desc = a_desc0 + static_cast<uint64_t>((stage * L::kABytes) >> 4);
                    const uint64_t b_desc = b_desc0 + static_cast<uint64_t>((stage * L::kBBytes) >> 4);
                    const uint64_t sfa_d = sfa_desc0 + static_cast<uint64_t>((stage * 512) >> 4);
                    const uint64_t sfb_d = sfb_desc0 + static_cast<uint64_t>((stage * L::kSfbBytes) >> 4);
                    const int64_t k_left = kMode == kGroupedK ? static_cast<int64_t>(nkb - kb) * kBK
                                                              : K - static_cast<int64_t>(kb) * kBK;
                    const int ksub = k_left >= kBK ? kBK / kUmmaK : static_cast<int>(k_left) / kUmmaK;
                    if (elect_one()) {
                        // this stage's scale atoms into its tensor-memory columns (each CTA its own)
                        tc_cp_32x128b_warpx4_pair(sfa_t, sfa_d);
                        tc_cp_32x128b_warpx4_pair(sfb_t, sfb_d);
                        tc_cp_32x128b_warpx4_pair(sfb_t + 4, sfb_d + static_cast<uint64_t>(512 >> 4));
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k)
                            if (k < ksub)
                                tc_mma_mxf8_pair(tmem_base, a_desc + ((k * kUmmaK) >> 4), b_desc + k * kBStepK,
                                                 make_idesc_mxf8(256, 256, kMnMajor ? 1u : 0u, k, k) | fmt_bits,
                                                 sfa_t, sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
                        // frees the slot in every CTA of the cluster (each counts the commits of all pairs)
                        tc_commit_pair_multicast(empty_bar(stage), kCluster == 4 ? 0xF : 0x3);
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (elect_one()) tc_commit_pair_multicast(tfull_bar, static_cast<uint16_t>(0x3u << lead));
                __syncwarp();
                acc_phase ^= 1u;
            }
            // Drain: every MMA and copy issued above completes before teardown.
            if (lane == 0) {
                tc_commit_pair(drain_bar);
                WaitGuard g2 = guard;
                volatile int never = 0;
                g2.abort_flag = &never;
                (void)mbar_wait(drain_bar, 0, g2);
            }
            __syncwarp();
        }
    } else {
        // ---- epilogue (both CTAs; warps 2..9) ----------------------------------------
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t tempty_leader = leader ? tempty_bar : mapa_shared(tempty_bar, lead);
        uint32_t acc_phase = 0;
        bool pending = false;   // a tiled store of this warp may still read its buffer
        for (int64_t r = 0; r * n_pairs < total; ++r) {
            const int64_t t = item_of(r);
            if (t >= total) continue;
            const PairTileInfo ti = pair_tile_info<kMode, kPairs>(sch, p, t, rank, pp);
            const Problem& P = p.pr[ti.prob];
            // One thread waits (suspending), the other epilogue warps sleep on a
            // named barrier; barrier 2 keeps the verdict until every warp read it.
            if (warp == 2 && lane == 0) *epi_flag = wait_phase(tfull_bar, acc_phase, guard) ? 1 : 0;
            named_bar_sync(1, 32 * L::kEpiWarps);
            const int ok = *epi_flag;
            named_bar_sync(2, 32 * L::kEpiWarps);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + 32 * c, v[c]);
            tmem_ld_wait();
            // The accumulator is in registers: hand it back to the MMA warp now.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(tempty_bar);
                else mbar_arrive_cluster(tempty_leader);
            }
            acc_phase ^= 1u;
            if (ti.nkb == 0) {  // no K blocks (an empty expert): the tile is zero
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[c][j] = 0u;
            }
            if constexpr (kMode == kDenseQuant)
                store_quant_staged(p, P, v, sbase + L::kOffStage + (warp - 2) * L::kStageWarpBytes,
                                   sbase + L::kOffQStage + (warp - 2) * L::kQStageWarpBytes, ti.m0 + 32 * quad,
                                   ti.row_lo, ti.row_hi, ti.n0 + half * 128, lane, &maps.y[ti.prob], &maps.yq,
                                   ti.m0 < P.M, pending);
            else
                store_staged(P, v, sbase + L::kOffStage + (warp - 2) * L::kStageWarpBytes,
                             ti.y_row0 + ti.m0 + 32 * quad, ti.m0 + 32 * quad, ti.row_lo, ti.row_hi,
                             ti.n0 + half * 128, lane, &maps.y[ti.prob], pending);
        }
        if (lane == 0) bulk_wait_all();   // this warp's tiled stores complete before the CTA ends
        __syncwarp();
    }

    // ---- teardown: nothing may still target the peer when either CTA leaves ----
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, L::kTmemCols);
    }
}

// Row-major u8 matrix [rows, cols] (cols contiguous), box [box_rows, 128 bytes],
// 128-byte swizzle.
bool make_tma_u8(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    return encode_tensor_map_2d(map, ptr, false, cols, rows, cols, 128u, box_rows, true);
}

template <int BN, int STAGES, bool kMnMajor, int kMode>
cudaError_t launch_t(const DeviceInfo& dev, const TensorMaps& maps, const GemmArgs& args, int64_t max_tiles,
                     cudaStream_t stream) {
    using L = Cfg<BN, STAGES, kMode>;
    auto kern = gemm_mxf8_kernel<BN, STAGES, kMnMajor, kMode>;
    static thread_local int configured_device = -1;  // attribute set once per device and thread
    if (configured_device != dev.device) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev.device;
    }
    int64_t grid = dev.sm_count;
    if (max_tiles >= 0 && max_tiles < grid) grid = max_tiles;
    if (grid <= 0) return cudaSuccess;
    kern<<<static_cast<unsigned>(grid), L::kThreads, L::kAlloc, stream>>>(maps, args);
    return cudaGetLastError();
}

constexpr int kBN = 256;
constexpr int kStages = 4;

// Tensor maps of the dense modes: A boxes of 128 rows x 128 K-bytes; B K-major
// [N, K] boxes of 256 rows, MN-major [K, N] boxes of 128 N-bytes x 128 K-rows.
bool make_dense_maps(CUtensorMap* ta, CUtensorMap* tb, const void* a_q, const void* b_q, int64_t M, int64_t N,
                     int64_t K, bool b_mn_major) {
    if (!make_tma_u8(ta, a_q, static_cast<uint64_t>(M), static_cast<uint64_t>(K), kBM)) return false;
    if (!b_mn_major) return make_tma_u8(tb, b_q, static_cast<uint64_t>(N), static_cast<uint64_t>(K), kBN);
    return make_tma_u8(tb, b_q, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kBK);
}

// kind::mxf8f6f4 format codes: E4M3 = 0, E5M2 = 1 (A at bits 7-9, B at 10-12).
uint32_t fmt_bits_of(int a_fmt, int b_fmt) {
    return (static_cast<uint32_t>(a_fmt) << 7) | (static_cast<uint32_t>(b_fmt) << 10);
}

Problem make_problem(const void* a_s, const void* b_s, void* y, int64_t M, int64_t N, int64_t K, int64_t ldy,
                     int64_t k_atoms, int64_t b_bands, uint32_t fmt_bits) {
    Problem q{};
    q.a_s = static_cast<const uint8_t*>(a_s);
    q.b_s = static_cast<const uint8_t*>(b_s);
    q.y = static_cast<uint16_t*>(y);
    q.M = M; q.N = N; q.K = K; q.ldy = ldy;
    q.k_atoms = k_atoms;
    q.b_bands = b_bands;
    q.m_tiles = (M + kBM - 1) / kBM;
    q.n_tiles = (N + kBN - 1) / kBN;
    q.num_kb = static_cast<int>((K + kBK - 1) / kBK);
    q.fmt_bits = fmt_bits;
    return q;
}

GemmArgs base_args(const DeviceInfo& dev) {
    GemmArgs a{};
    a.nprob = 1;
    a.status = dev.status;
    a.wait_limit_ns = kDefaultWaitLimitNs;
    return a;
}

// Tiled-store map of a BF16 output [rows, N] with row stride ldy; the problem
// keeps row-by-row stores when there is no output or the rows exceed the 32-bit
// box coordinates.
void set_store_map(CUtensorMap* map, Problem* q, const void* y, int64_t rows, int64_t N, int64_t ldy) {
    q->y_tma = 0;
    if (y != nullptr && rows > 0 && rows < (int64_t(1) << 31) - 32 &&
        encode_tensor_map_bf16_store(map, y, static_cast<uint64_t>(N), static_cast<uint64_t>(rows),
                                     static_cast<uint64_t>(ldy)))
        q->y_tma = 1;
}

// Dense problems of one launch, ordered by K descending (stable), their work
// items laid out back to back.
bool fill_dense(const DenseGemm* gemms, int count, bool b_mn_major, TensorMaps* maps, GemmArgs* args) {
    int order[kMaxProblems];
    for (int i = 0; i < count; ++i) order[i] = i;
    for (int i = 1; i < count; ++i)
        for (int j = i; j > 0 && gemms[order[j]].K > gemms[order[j - 1]].K; --j) {
            const int t = order[j]; order[j] = order[j - 1]; order[j - 1] = t;
        }
    int64_t items = 0;
    for (int i = 0; i < count; ++i) {
        const DenseGemm& g = gemms[order[i]];
        if (!make_dense_maps(&maps->a[i], &maps->b[i], g.a_q, g.b_q, g.M, g.N, g.K, b_mn_major)) return false;
        args->pr[i] = make_problem(g.a_s, g.b_s, g.y, g.M, g.N, g.K, g.ldy, (g.K + 127) / 128, (g.N + 127) / 128,
                                   fmt_bits_of(g.a_fmt, g.b_fmt));
        set_store_map(&maps->y[i], &args->pr[i], g.y, g.M, g.N, g.ldy);
        args->pr[i].first_item = items;
        items += args->pr[i].m_tiles * args->pr[i].n_tiles;
    }
    args->nprob = count;
    args->items = items;
    return true;
}

// MMA-tiled scales of an operand with `bands` 128-row bands of k_atoms atoms,
// as rows of 256 bytes (one atom = a 2 x 256 box at row 2 (band k_atoms + kb)).
bool make_tma_scales(CUtensorMap* map, const void* ptr, int64_t bands, int64_t k_atoms, uint32_t box_rows = 2) {
    return encode_tensor_map_2d(map, ptr, false, 256u, static_cast<uint64_t>(bands * k_atoms * 2), 256u, 256u,
                                box_rows, false);
}

// Scale maps and the scale-row range check of a pair launch: an operand with
// `bands` 128-row bands of k_atoms atoms (rows up to three bands past the end
// are addressed, and read as zeros).
bool pair_scale_map(CUtensorMap* map, const void* ptr, int64_t bands, int64_t k_atoms, uint32_t box_rows = 2) {
    if ((bands + 4) * k_atoms * 2 >= (int64_t(1) << 31)) return false;
    return make_tma_scales(map, ptr, bands, k_atoms, box_rows);
}

// The problems of one dense pair launch (K descending, as fill_dense orders
// them), their 256 x 256 pair tiles laid out back to back.  False when a tensor
// map cannot be encoded or a scale map's rows exceed its 32-bit coordinates
// (the single-CTA kernel then runs the launch).
bool fill_dense_pair(const DenseGemm* gemms, int count, bool b_mn_major, int pairs, PairMaps* maps,
                     GemmArgs* args) {
    const uint32_t b_box = static_cast<uint32_t>(128 / pairs);   // B rows (or K rows) one CTA loads per stage
    int order[kMaxProblems];
    for (int i = 0; i < count; ++i) order[i] = i;
    for (int i = 1; i < count; ++i)
        for (int j = i; j > 0 && gemms[order[j]].K > gemms[order[j - 1]].K; --j) {
            const int t = order[j]; order[j] = order[j - 1]; order[j - 1] = t;
        }
    int64_t items = 0;
    for (int i = 0; i < count; ++i) {
        const DenseGemm& g = gemms[order[i]];
        const int64_t k_atoms = (g.K + 127) / 128;
        const int64_t a_bands = (g.M + 127) / 128, b_bands = (g.N + 127) / 128;
        if (!make_tma_u8(&maps->a[i], g.a_q, static_cast<uint64_t>(g.M), static_cast<uint64_t>(g.K), 128)) return false;
        if (!b_mn_major) {
            if (!make_tma_u8(&maps->b[i], g.b_q, static_cast<uint64_t>(g.N), static_cast<uint64_t>(g.K), b_box))
                return false;
        } else if (!make_tma_u8(&maps->b[i], g.b_q, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.N), b_box)) {
            return false;
        }
        if (!pair_scale_map(&maps->sfa[i], g.a_s, a_bands, k_atoms) ||
            !pair_scale_map(&maps->sfb[i], g.b_s, b_bands, k_atoms, pairs == 2 ? 1u : 2u))
            return false;
        args->pr[i] = make_problem(g.a_s, g.b_s, g.y, g.M, g.N, g.K, g.ldy, k_atoms, b_bands,
                                   fmt_bits_of(g.a_fmt, g.b_fmt));
        args->pr[i].m_tiles = (g.M + 256 * pairs - 1) / (256 * pairs);   // cluster tiles
        args->pr[i].n_tiles = (g.N + 255) / 256;
        set_store_map(&maps->y[i], &args->pr[i], g.y, g.M, g.N, g.ldy);
        args->pr[i].first_item = items;
        items += args->pr[i].m_tiles * args->pr[i].n_tiles;
    }
    args->nprob = count;
    args->items = items;
    return true;
}

// Clusters of kCluster CTAs of the pair kernel that the device holds at once
// (set up once per device and thread).  Pairs always cover every SM; clusters
// of four need four SMs of one GPC, and a GPC whose SM count is not a multiple
// of four leaves SMs idle (on GB300: 36 clusters, 144 of the 152 SMs).
template <bool kMnMajor, int kMode, int kCluster>
cudaError_t pair_clusters(const DeviceInfo& dev, int64_t* clusters) {
    using L = PairCfg<kMode>;
    auto kern = gemm_mxf8_pair_kernel<kMnMajor, kMode, kCluster>;
    static thread_local int configured_device = -1;
    static thread_local int64_t max_clusters = 0;
    if (configured_device != dev.device) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (e != cudaSuccess) return e;
        int64_t n = dev.sm_count / kCluster;
        if (kCluster > 2 && n > 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(kCluster * n), 1, 1);
            cfg.blockDim = dim3(L::kThreads, 1, 1);
            cfg.dynamicSmemBytes = L::kAlloc;
            int active = 0;
            e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
            if (e != cudaSuccess) return e;
            n = min(n, static_cast<int64_t>(active));
        }
        max_clusters = n;
        configured_device = dev.device;
    }
    *clusters = max_clusters;
    return cudaSuccess;
}

template <bool kMnMajor, int kMode, int kCluster = 2>
cudaError_t launch_pair_t(const DeviceInfo& dev, const PairMaps& maps, const GemmArgs& args, int64_t max_tiles,
                          cudaStream_t stream) {
    using L = PairCfg<kMode>;
    int64_t units = 0;
    const cudaError_t e = pair_clusters<kMnMajor, kMode, kCluster>(dev, &units);
    if (e != cudaSuccess) return e;
    if (max_tiles >= 0 && max_tiles < units) units = max_tiles;
    if (units <= 0) return cudaSuccess;
    gemm_mxf8_pair_kernel<kMnMajor, kMode, kCluster>
        <<<static_cast<unsigned>(kCluster * units), L::kThreads, L::kAlloc, stream>>>(maps, args);
    return cudaGetLastError();
}

// Pairs per cluster for a dense launch of `pair_tiles` 256 x 256 tiles.
// Clusters of two pairs read each B tile (and its scales) from L2 once per
// cluster instead of once per pair, and their launches move fewer bytes through
// L2 and DRAM.  Per tile that is a little faster at full clock, and under the
// power cap that a long run of large GEMMs reaches the lower draw also buys a
// higher SM clock.  Against that they leave 8 of GB300's 152 SMs idle, and a
// launch of few waves loses more to the coarser last wave.  Launches of at least
// kQuadMinPairTiles tiles (about 20 waves of pairs) take clusters of two pairs
// where the device holds them; MXQ_GEMM_CLUSTER=2 or 4 overrides the choice.
constexpr int64_t kQuadMinPairTiles = 1536;

template <bool kMnMajor, int kMode>
int dense_pairs_per_cluster(const DeviceInfo& dev, int64_t pair_tiles) {
    const char* env = std::getenv("MXQ_GEMM_CLUSTER");
    bool quad = pair_tiles >= kQuadMinPairTiles;
    if (env != nullptr && (env[0] == '2' || env[0] == '4') && env[1] == '\0') quad = env[0] == '4';
    if (!quad) return 1;
    int64_t quads = 0;
    if (pair_clusters<kMnMajor, kMode, 4>(dev, &quads) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return quads > 0 ? 2 : 1;
}

// A dense launch on CTA pairs; *done false when the pair kernel cannot take it.
template <int kMode>
cudaError_t try_pair(const DeviceInfo& dev, const DenseGemm* gemms, int count, bool b_mn_major, uint8_t* yq,
                     uint8_t* ys, cudaStream_t stream, bool* done) {
    *done = false;
    if (dev.sm_count < 2) return cudaSuccess;
    int64_t pair_tiles = 0;
    for (int i = 0; i < count; ++i) pair_tiles += ((gemms[i].M + 255) / 256) * ((gemms[i].N + 255) / 256);
    const int pairs = b_mn_major ? dense_pairs_per_cluster<true, kMode>(dev, pair_tiles)
                                 : dense_pairs_per_cluster<false, kMode>(dev, pair_tiles);
    PairMaps maps;
    GemmArgs args = base_args(dev);
    if (!fill_dense_pair(gemms, count, b_mn_major, pairs, &maps, &args)) return cudaSuccess;
    args.yq = yq;
    args.ys = ys;
    args.yq_tma = 0;
    if (yq != nullptr && gemms[0].M > 0 && gemms[0].M < (int64_t(1) << 31) - 32 &&
        encode_tensor_map_u8_store(&maps.yq, yq, static_cast<uint64_t>(gemms[0].N),
                                   static_cast<uint64_t>(gemms[0].M), static_cast<uint64_t>(gemms[0].N)))
        args.yq_tma = 1;
    *done = true;
    if (pairs == 2) {
        if (b_mn_major) return launch_pair_t<true, kMode, 4>(dev, maps, args, args.items, stream);
        return launch_pair_t<false, kMode, 4>(dev, maps, args, args.items, stream);
    }
    if (b_mn_major) return launch_pair_t<true, kMode>(dev, maps, args, args.items, stream);
    return launch_pair_t<false, kMode>(dev, maps, args, args.items, stream);
}

}  // namespace

cudaError_t launch_gemm_multi(const DeviceInfo& dev, const DenseGemm* gemms, int count, bool b_mn_major,
                              cudaStream_t stream) {
    if (count < 1 || count > kMaxProblems) return cudaErrorInvalidValue;
    bool done = false;
    const cudaError_t e = try_pair<kDense>(dev, gemms, count, b_mn_major, nullptr, nullptr, stream, &done);
    if (done || e != cudaSuccess) return e;
    TensorMaps maps;
    GemmArgs args = base_args(dev);
    if (!fill_dense(gemms, count, b_mn_major, &maps, &args)) return cudaErrorInvalidValue;
    if (b_mn_major)
        return launch_t<kBN, kStages, true, kDense>(dev, maps, args, args.items, stream);
    return launch_t<kBN, kStages, false, kDense>(dev, maps, args, args.items, stream);
}

cudaError_t launch_gemm(const DeviceInfo& dev, const void* a_q, const void* a_s, const void* b_q,
                        const void* b_s, int64_t M, int64_t N, int64_t K, bool b_mn_major, void* y,
                        int64_t ldy, int a_fmt, int b_fmt, cudaStream_t stream) {
    const DenseGemm g{a_q, a_s, b_q, b_s, M, N, K, y, ldy, a_fmt, b_fmt};
    return launch_gemm_multi(dev, &g, 1, b_mn_major, stream);
}

cudaError_t launch_gemm_quant(const DeviceInfo& dev, const void* a_q, const void* a_s, const void* b_q,
                              const void* b_s, int64_t M, int64_t N, int64_t K, bool b_mn_major, void* y,
                              int64_t ldy, void* y_q, void* y_s, cudaStream_t stream) {
    const DenseGemm g{a_q, a_s, b_q, b_s, M, N, K, y, ldy, 0, 0};
    bool done = false;
    const cudaError_t e = try_pair<kDenseQuant>(dev, &g, 1, b_mn_major, static_cast<uint8_t*>(y_q),
                                                static_cast<uint8_t*>(y_s), stream, &done);
    if (done || e != cudaSuccess) return e;
    TensorMaps maps;
    GemmArgs args = base_args(dev);
    if (!fill_dense(&g, 1, b_mn_major, &maps, &args)) return cudaErrorInvalidValue;
    args.yq = static_cast<uint8_t*>(y_q);
    args.ys = static_cast<uint8_t*>(y_s);
    if (b_mn_major)
        return launch_t<kBN, kStages, true, kDenseQuant>(dev, maps, args, args.items, stream);
    return launch_t<kBN, kStages, false, kDenseQuant>(dev, maps, args, args.items, stream);
}

cudaError_t launch_grouped_gemm(const DeviceInfo& dev, const void* a_q, const void* a_s,
                                const void* b_q, const void* b_s, const int64_t* offsets, int G,
                                int64_t M_total, int64_t N, int64_t K, int64_t a_bands_cap, void* y,
                                int64_t ldy, int a_fmt, int b_fmt, cudaStream_t stream) {
    if (G <= PairCfg<kGroupedRows>::kMaxGroups && dev.sm_count >= 2) {   // CTA pairs
        PairMaps pm;
        const int64_t k_atoms = (K + 127) / 128;
        const int64_t a_bands = a_bands_cap > 0 ? a_bands_cap : (M_total + 127) / 128;
        const int64_t b_bands = static_cast<int64_t>(G) * N / 128;
        if (make_tma_u8(&pm.a[0], a_q, static_cast<uint64_t>(M_total), static_cast<uint64_t>(K), kBM) &&
            make_tma_u8(&pm.b[0], b_q, static_cast<uint64_t>(G) * static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                        128) &&
            pair_scale_map(&pm.sfa[0], a_s, a_bands, k_atoms) && pair_scale_map(&pm.sfb[0], b_s, b_bands, k_atoms)) {
            GemmArgs args = base_args(dev);
            args.pr[0] = make_problem(a_s, b_s, y, M_total, N, K, ldy, k_atoms, b_bands, fmt_bits_of(a_fmt, b_fmt));
            args.pr[0].n_tiles = (N + 255) / 256;
            set_store_map(&pm.y[0], &args.pr[0], y, M_total, N, ldy);
            args.offsets = offsets;
            args.G = G;
            args.a_bands_cap = a_bands_cap;
            return launch_pair_t<false, kGroupedRows>(dev, pm, args, -1, stream);
        }
    }
    TensorMaps maps;
    if (!make_tma_u8(&maps.a[0], a_q, static_cast<uint64_t>(M_total), static_cast<uint64_t>(K), kBM))
        return cudaErrorInvalidValue;
    if (!make_tma_u8(&maps.b[0], b_q, static_cast<uint64_t>(G) * static_cast<uint64_t>(N),
                     static_cast<uint64_t>(K), kBN))
        return cudaErrorInvalidValue;
    GemmArgs args = base_args(dev);
    args.pr[0] = make_problem(a_s, b_s, y, M_total, N, K, ldy, (K + 127) / 128, static_cast<int64_t>(G) * N / 128,
                              fmt_bits_of(a_fmt, b_fmt));
    set_store_map(&maps.y[0], &args.pr[0], y, M_total, N, ldy);
    args.offsets = offsets;
    args.G = G;
    args.a_bands_cap = a_bands_cap;
    return launch_t<kBN, kStages, false, kGroupedRows>(dev, maps, args, -1, stream);
}

cudaError_t launch_grouped_gemm_wgrad(const DeviceInfo& dev, const void* a_q, const void* a_s,
                                      const void* b_q, const void* b_s, const int64_t* offsets, int G,
                                      int64_t M_total, int64_t capacity, int64_t M, int64_t N, void* y,
                                      int64_t ldy, int a_fmt, int b_fmt, cudaStream_t stream) {
    if (G <= PairCfg<kGroupedK>::kMaxGroups && dev.sm_count >= 2) {   // CTA pairs
        PairMaps pm;
        const int64_t k_atoms = capacity / 128;
        if (make_tma_u8(&pm.a[0], a_q, static_cast<uint64_t>(M), static_cast<uint64_t>(capacity), kBM) &&
            make_tma_u8(&pm.b[0], b_q, static_cast<uint64_t>(N), static_cast<uint64_t>(capacity), 128) &&
            pair_scale_map(&pm.sfa[0], a_s, (M + 127) / 128, k_atoms) &&
            pair_scale_map(&pm.sfb[0], b_s, (N + 127) / 128, k_atoms)) {
            GemmArgs args = base_args(dev);
            args.pr[0] = make_problem(a_s, b_s, y, M, N, capacity, ldy, k_atoms, (N + 127) / 128,
                                      fmt_bits_of(a_fmt, b_fmt));
            args.pr[0].m_tiles = (M + 255) / 256;   // pair tiles per expert
            args.pr[0].n_tiles = (N + 255) / 256;
            set_store_map(&pm.y[0], &args.pr[0], y, static_cast<int64_t>(G) * M, N, ldy);   // y[g] stacked
            args.M_total = M_total;
            args.offsets = offsets;
            args.G = G;
            return launch_pair_t<false, kGroupedK>(dev, pm, args, -1, stream);
        }
    }
    TensorMaps maps;
    if (!make_tma_u8(&maps.a[0], a_q, static_cast<uint64_t>(M), static_cast<uint64_t>(capacity), kBM))
        return cudaErrorInvalidValue;
    if (!make_tma_u8(&maps.b[0], b_q, static_cast<uint64_t>(N), static_cast<uint64_t>(capacity), kBN))
        return cudaErrorInvalidValue;
    GemmArgs args = base_args(dev);
    args.pr[0] = make_problem(a_s, b_s, y, M, N, capacity, ldy, capacity / 128, (N + 127) / 128,
                              fmt_bits_of(a_fmt, b_fmt));
    set_store_map(&maps.y[0], &args.pr[0], y, static_cast<int64_t>(G) * M, N, ldy);   // y[g] stacked
    args.M_total = M_total;
    args.offsets = offsets;
    args.G = G;
    return launch_t<kBN, kStages, false, kGroupedK>(dev, maps, args, -1, stream);
}

// ---- bounded-wait probe ---------------------------------------------------------------

namespace {
__global__ void wait_probe_kernel(unsigned int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitGuard g{&abort_flag, status, limit_ns};
    if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, g);  // nobody arrives
    __syncthreads();
}
}  // namespace

cudaError_t launch_wait_probe(const DeviceInfo& dev, uint64_t limit_ns, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(dev.status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mxq
