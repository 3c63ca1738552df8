/*
 * mxq.h -- C ABI of libmxq: MXFP8 microscaled quantization and block-scaled
 * FP8 GEMMs with BF16 output, for NVIDIA GB300 (sm_103a).
 *
 * What is computed (sources, by page and section):
 *   - "torchtitan-npu MXFP8/HiF8 low-precision training tutorial", section
 *     "MXFP8 与 HiF8 架构原理速览": MXFP8 is per-block dynamic quantization in
 *     which every 32 consecutive elements share one E8M0 (power-of-two)
 *     scale; the FP8 matmul returns BF16.  Linear layers and MoE expert
 *     layers (grouped matmul) are quantized.  Section "常用环境变量"
 *     (MXFP8_DUAL_AXIS_FORWARD): the forward quantizes along both axes.
 *     Section "第 3 步": the scale rule is "mxfp8_rceil".
 *   - MindSpeed RFC "Add MXFP8-32x32 quantization support to FSDP":
 *     section 3.1 (block size [1,32,32]: 32 along input_dim and output_dim,
 *     token_dim unblocked; forward and backward share one weight), section
 *     3.3.1 (E4M3 elements, dynamic scaling), section 3.3.3 (dual-axis
 *     quantization gives separate forward/backward copies; 32x32 gives one
 *     payload and two scales), section 3.5.2.1 (unsupported block sizes
 *     raise an error).
 *
 * Number formats:
 *   payload  float8_e4m3fn: bias 7, no Inf, NaN = S.1111.111, max 448.
 *   scale    E8M0: code c in [0,254] means 2^(c-127); 0xFF is NaN.
 *   rule     e = ceil(log2(amax/448)) clamped to [-127,127]; amax 0 -> -127.
 *            q = round-to-nearest-even, saturating E4M3 of x * 2^-e.
 *            A group holding NaN or Inf gets scale 0xFF and payload
 *            0x7F | sign(x).
 *   GEMM     y = sum_k deq(a)[m,k] * deq(b)[n,k] with deq(q) = q * 2^e,
 *            accumulated in FP32 on the tensor cores, rounded once to BF16.
 *
 * Scale layouts (for an operand [R, C] quantized along C, scales [R, C/32]):
 *   MXQ_SCALE_ROWMAJOR   plain row-major [R][C/32] bytes.
 *   MXQ_SCALE_MMA_TILED  the layout the block-scaled tensor-core MMA reads:
 *                        R padded to a multiple of 128 and C/32 to a
 *                        multiple of 4; 512-byte atoms of 128 rows x 4
 *                        groups, atoms of one 128-row band consecutive;
 *                        inside an atom row r, group g sit at byte
 *                        16*(r%32) + 4*((r%128)/32) + (g%4).  Padding = 0.
 *   mxq_scale_bytes() gives the size of either.
 *
 * Conventions for every call:
 *   - Pointers named x, w, q*, s*, a*, b*, y, group_offsets are DEVICE
 *     pointers; the caller owns all memory (the library allocates nothing
 *     per call) and must keep it alive until the work on `stream` is done.
 *   - All device pointers must be 16-byte aligned; leading dimensions are
 *     in elements and must keep rows 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and run on the current CUDA device.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns a status and launches nothing.
 *   - Kernels bound every internal wait; a wait that runs out records
 *     MXQ_ERR_TIMEOUT in a device status word that mxq_get_device_status()
 *     reports.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXQ_ABI_VERSION 2

typedef struct CUstream_st* mxq_stream_t; /* the same type as cudaStream_t */

typedef enum {
    MXQ_OK = 0,
    MXQ_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum, misalignment */
    MXQ_ERR_UNSUPPORTED_SHAPE = 2,  /* a dimension that is not a supported multiple */
    MXQ_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 (GB300) */
    MXQ_ERR_CUDA = 4,               /* a CUDA runtime or driver call failed */
    MXQ_ERR_TIMEOUT = 5             /* a bounded device-side wait ran out */
} mxq_status;

typedef enum {
    MXQ_SCALE_ROWMAJOR = 0,
    MXQ_SCALE_MMA_TILED = 1
} mxq_scale_layout;

/* FP8 payload format (RFC section 3.5.2.3: dst_type E4M3 or E5M2).
 * E4M3 = float8_e4m3fn (max 448), the default of every call;
 * E5M2 = float8_e5m2 (bias 15, max 57344; rceil then uses 57344). */
typedef enum {
    MXQ_FP8_E4M3 = 0,
    MXQ_FP8_E5M2 = 1
} mxq_fp8_format;

/* Version of this ABI (MXQ_ABI_VERSION). */
int mxq_abi_version(void);

/* Static text for a status code. */
const char* mxq_status_string(mxq_status s);

/* Bytes of the scale matrix of an operand [rows, cols] quantized along cols
 * (cols % 32 == 0) in the given layout; 0 for invalid arguments. */
size_t mxq_scale_bytes(int64_t rows, int64_t cols, mxq_scale_layout layout);

/*
 * 1x32 dual-axis quantization (the "mxfp8" recipe; RFC section 3.3.3
 * "dual_axis_quant", tutorial "MXFP8_DUAL_AXIS_FORWARD").
 *
 * x      bf16 [rows, cols], row stride ld elements (ld >= cols, ld % 8 == 0).
 * q_row  u8 [rows, cols]       E4M3 payload, groups of 32 along cols.
 * s_row  u8 scales of q_row    ([rows, cols/32] in `layout`).
 * q_col  u8 [cols, rows]       E4M3 payload of x transposed: groups of 32
 *                              along rows; stored cols-major-first so that
 *                              every GEMM operand is K-major.
 * s_col  u8 scales of q_col    ([cols, rows/32] in `layout`).
 * Either pair may be NULL (row-only or column-only); not both.
 * Shapes: cols % 32 == 0; rows % 32 == 0 when the column pair is asked for;
 * rows >= 1 otherwise.  Output rows are dense (stride cols resp. rows).
 * Errors: MXQ_ERR_INVALID_ARG, MXQ_ERR_UNSUPPORTED_SHAPE,
 * MXQ_ERR_UNSUPPORTED_DEVICE, MXQ_ERR_CUDA (launch failure).
 */
mxq_status mxq_quant_1x32_dual(const void* x, int64_t rows, int64_t cols, int64_t ld,
                               void* q_row, void* s_row, void* q_col, void* s_col,
                               mxq_scale_layout layout, mxq_stream_t stream);

/*
 * Batched form of mxq_quant_1x32_dual: `batch` matrices [rows, cols] (row
 * stride ld, matrix b at x + b * batch_stride elements; batch_stride >=
 * rows * ld, a multiple of 8, ignored when batch == 1).  The outputs of
 * matrix b follow those of matrix b-1 with no gap: q_row + b*rows*cols,
 * s_row + b*mxq_scale_bytes(rows, cols, layout), q_col + b*cols*rows,
 * s_col + b*mxq_scale_bytes(cols, rows, layout).  Used for the stacked MoE
 * expert weights [G, N, K]: the row copies give the forward operand and the
 * column copies [G, K, N] the dgrad operand of mxq_grouped_gemm.  batch <= 65535.
 * fmt selects the payload format (mxq_quant_1x32_dual is fmt = MXQ_FP8_E4M3).
 */
mxq_status mxq_quant_1x32_dual_batched(const void* x, int64_t batch, int64_t rows, int64_t cols,
                                       int64_t ld, int64_t batch_stride, void* q_row, void* s_row,
                                       void* q_col, void* s_col, mxq_scale_layout layout,
                                       mxq_fp8_format fmt, mxq_stream_t stream);

/*
 * Token-axis (column) 1x32 quantization inside each MoE expert, the operand
 * form of the expert weight gradient (dW_g = dY_g^T X_g contracts over the
 * expert's tokens).  Rows of x [rows, cols] (row stride ld) are tokens sorted
 * by expert; group_offsets is the DEVICE int64 [G+1] of mxq_grouped_gemm.
 *
 * Expert g (m_g = off[g+1] - off[g] tokens) gets the slot [P_g, P_g + L_g) of
 * the token axis, L_g = m_g rounded up to a multiple of 128, P_g = sum of L_h
 * for h < g.  Its 32-token groups start at its first token; a group that runs
 * past its last token is completed with zeros (the pages leave this open; this
 * is the reading taken), so no scale is shared between experts.
 *
 * q_col  u8 [cols, capacity]: column c, slot position p = token P_g + i of expert g.
 * s_col  u8 scales [cols, capacity/32] in `layout`.
 * Slot positions past an expert's tokens hold zero payload and scale code 0;
 * positions past the last slot are not written.
 * capacity: a multiple of 128, >= rows + 127*G (enough for any offsets).
 * Shapes: cols % 32 == 0; 1 <= G <= 1024.  rows == 0 writes nothing.
 */
mxq_status mxq_quant_1x32_cols_grouped(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                       const int64_t* group_offsets, int32_t G, int64_t capacity,
                                       void* q_col, void* s_col, mxq_scale_layout layout,
                                       mxq_stream_t stream);

/* mxq_quant_1x32_cols_grouped with the payload format (E4M3 or E5M2: the RFC's
 * dst_type, section 3.5.2.3), e.g. E5M2 output gradients for the weight
 * gradient; the rceil rule uses the format's largest finite value. */
mxq_status mxq_quant_1x32_cols_grouped_fmt(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                           const int64_t* group_offsets, int32_t G, int64_t capacity,
                                           void* q_col, void* s_col, mxq_scale_layout layout,
                                           mxq_fp8_format fmt, mxq_stream_t stream);

/*
 * 32x32 block quantization (the "mxfp8-32x32" recipe; RFC sections 3.1 and
 * 3.3.3 "block_mx_quant": one payload, forward and backward scales).
 *
 * w      bf16 weight [n, k] (output_dim x input_dim), row stride ld.
 * q      u8 [n, k]  the single E4M3 payload used by forward and backward.
 * s_fwd  u8 scales for contraction over k: [n, k/32] in `layout`,
 *        s_fwd[r][j] = t[r/32][j].
 * s_bwd  u8 scales for contraction over n: [k, n/32] in `layout`,
 *        s_bwd[c][i] = t[i][c/32].
 * where t[i][j] is the E8M0 code of 32x32 tile (i, j) (tiles start at 0,0).
 * s_fwd or s_bwd may be NULL.  Shapes: n % 32 == 0, k % 32 == 0.
 * Errors: MXQ_ERR_INVALID_ARG (null w or q, bad ld or layout, misalignment),
 * MXQ_ERR_UNSUPPORTED_SHAPE, MXQ_ERR_UNSUPPORTED_DEVICE, MXQ_ERR_CUDA.
 */
mxq_status mxq_quant_32x32(const void* w, int64_t n, int64_t k, int64_t ld,
                           void* q, void* s_fwd, void* s_bwd,
                           mxq_scale_layout layout, mxq_stream_t stream);

/* mxq_quant_32x32 with the payload format (RFC section 3.5.2.3: the
 * quantizer of both recipes takes dst_type E4M3 or E5M2).  With E5M2 the tile
 * exponent is ceil(log2(amax / 57344)) and the payload float8_e5m2 (RNE,
 * saturating to +-57344); the scales and their layouts are as for E4M3.
 * mxq_quant_32x32 is fmt = MXQ_FP8_E4M3.  A bad fmt: MXQ_ERR_INVALID_ARG. */
mxq_status mxq_quant_32x32_fmt(const void* w, int64_t n, int64_t k, int64_t ld,
                               void* q, void* s_fwd, void* s_bwd,
                               mxq_scale_layout layout, mxq_fp8_format fmt, mxq_stream_t stream);

/*
 * Block-scaled FP8 GEMM with BF16 output: forward Y = X W^T, dgrad and
 * wgrad (tutorial: "前向用 npu_quant_matmul 执行 FP8 矩阵乘, 输出恢复为 BF16").
 *
 *   y[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k]        (0 <= m < M, 0 <= n < N)
 *
 * a_q   u8 [M, K] K-major E4M3 payload; a_s its scales [M, K/32], MMA-tiled.
 * b_q   b_mn_major == 0: u8 [N, K] K-major; b_s scales [N, K/32], MMA-tiled.
 *       b_mn_major == 1: u8 [K, N] (N contiguous) -- the single 32x32 weight
 *       payload read for dgrad -- with b_s = its backward scales [N, K/32]
 *       MMA-tiled (s_bwd of mxq_quant_32x32).
 * y     bf16 [M, N], row stride ldy (ldy >= N, ldy % 8 == 0).
 * layout  the layout of a_s and b_s: must be MXQ_SCALE_MMA_TILED, the layout
 *       the tensor cores read (every quantizer of this library writes it);
 *       MXQ_SCALE_ROWMAJOR scales are refused with MXQ_ERR_INVALID_ARG (an
 *       unsupported configuration, as the RFC's section 3.5.2.1 refuses one).
 * Shapes: M >= 0; N % 16 == 0 (N % 128 == 0 when b_mn_major); K % 32 == 0
 * (K % 128 == 0 when b_mn_major).  M == 0 or N == 0 writes nothing; K == 0
 * writes zeros.
 * Errors: MXQ_ERR_INVALID_ARG (null pointers, ldy, misalignment, layout),
 * MXQ_ERR_UNSUPPORTED_SHAPE, MXQ_ERR_UNSUPPORTED_DEVICE, MXQ_ERR_CUDA.
 * Operand pairing for training (contraction axis quantized in groups of 32):
 *   forward  A = X row copy,   B = W row copy           (M tokens, N out, K in)
 *   dgrad    A = dY row copy,  B = W column copy        (N = in, K = out)
 *            or, 32x32, B = W payload MN-major with s_bwd
 *   wgrad    A = dY column copy, B = X column copy      (M = out, N = in, K = tokens)
 * Schedule: launches of 1536 or more 256 x 256 output tiles (this call's and
 * mxq_gemm_bf16out_multi's, counted over all its GEMMs) run on clusters of two
 * SM pairs that share each B tile; smaller ones on single pairs.  The results
 * are bit-identical either way.  The environment variable MXQ_GEMM_CLUSTER,
 * read at each call, fixes the choice: "2" single pairs, "4" clusters of two
 * pairs (where the device holds them).
 */
mxq_status mxq_gemm_bf16out(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                            int64_t M, int64_t N, int64_t K, int b_mn_major,
                            void* y, int64_t ldy, mxq_scale_layout layout, mxq_stream_t stream);

/* mxq_gemm_bf16out with the payload format of each operand (E4M3 or E5M2,
 * e.g. E5M2 gradients against E4M3 weights); scales MMA-tiled.
 * mxq_gemm_bf16out is E4M3 x E4M3. */
mxq_status mxq_gemm_bf16out_fmt(const void* a_q, const void* a_s, mxq_fp8_format a_fmt,
                                const void* b_q, const void* b_s, mxq_fp8_format b_fmt,
                                int64_t M, int64_t N, int64_t K, int b_mn_major,
                                void* y, int64_t ldy, mxq_stream_t stream);

/* One GEMM of mxq_gemm_bf16out_multi: y = deq(A) deq(B)^T with the fields of
 * mxq_gemm_bf16out_fmt (caller-owned device buffers). */
typedef struct {
    const void* a_q;
    const void* a_s;
    const void* b_q;
    const void* b_s;
    int64_t M, N, K;
    void* y;
    int64_t ldy;
    mxq_fp8_format a_fmt, b_fmt;
} mxq_gemm_desc;

/*
 * 1 to 4 independent dense GEMMs (e.g. the dgrad and the wgrad of one linear
 * layer's backward pass, torchtitan-npu tutorial "MXFP8 与 HiF8 架构原理速览":
 * the backward matmuls of the MXFP8 recipe) computed by ONE persistent launch
 * over all their output tiles.  The results are those of mxq_gemm_bf16out_fmt
 * on each GEMM, bit for bit; only the scheduling differs: run back to back,
 * every GEMM ends in a partly filled last wave of 128 x 256 tiles, while one
 * launch (longest K first, the rounds alternating direction over the SMs)
 * shares a single last wave between them.  The pages run these GEMMs as
 * separate matmuls; this call has no counterpart there.
 *
 * gemms[i]    host array of count descriptors (read during the call only).
 * b_mn_major  the B orientation of every GEMM (0 K-major, 1 MN-major).
 * Every descriptor is checked as mxq_gemm_bf16out_fmt checks its arguments
 * before anything is launched; the first failing one decides the status and
 * nothing runs.  M == 0 or N == 0 GEMMs are skipped, K == 0 GEMMs write zeros.
 * Outputs must not overlap one another or any input (not checked).
 * count == 0 returns MXQ_OK; count > 4 or a NULL array: MXQ_ERR_INVALID_ARG.
 */
mxq_status mxq_gemm_bf16out_multi(const mxq_gemm_desc* gemms, int32_t count, int b_mn_major,
                                  mxq_stream_t stream);

/*
 * Block-scaled FP8 GEMM whose epilogue also quantizes its output: the BF16
 * result y (as mxq_gemm_bf16out computes it) is rounded to BF16 and each run
 * of 32 consecutive columns of a row gets the 1x32 rceil E8M0 scale and E4M3
 * payload, written straight from the accumulator registers.  This removes the
 * HBM round trip of quantizing y in a separate pass (DeepSeek-V4 Ascend
 * training write-up, "AutoFuse 收益分析": fused kernels keep intermediates on
 * chip instead of re-reading HBM); the bytes equal those of
 * mxq_quant_1x32_dual's row copy of y with the MMA-tiled layout.
 *
 * a_q, a_s, b_q, b_s, M, N, K, b_mn_major  as for mxq_gemm_bf16out (E4M3 x E4M3).
 * y     optional bf16 [M, N], row stride ldy (ldy >= N, ldy % 8 == 0); NULL to
 *       keep only the quantized output (ldy then ignored).
 * y_q   u8 [M, N] E4M3 payload, row stride N (required, 16-byte aligned).
 * y_s   u8 scales [M, N/32], MMA-tiled (mxq_scale_bytes(M, N, MXQ_SCALE_MMA_TILED)
 *       bytes, padding rows and groups written as zero).
 * Shapes: N % 32 == 0 (N % 128 == 0 when b_mn_major); K % 32 == 0 and K >= 32.
 * M == 0 or N == 0 writes nothing.  Errors: as mxq_gemm_bf16out.
 */
mxq_status mxq_gemm_mxfp8out(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                             int64_t M, int64_t N, int64_t K, int b_mn_major,
                             void* y, int64_t ldy, void* y_q, void* y_s, mxq_stream_t stream);

/*
 * Pre-quantized weight all-gather for fully sharded data parallelism
 * (MindSpeed RFC "Add MXFP8-32x32 quantization support to FSDP", section
 * 3.3.2: before the all-gather each rank quantizes its shard; the mxfp8
 * recipe gathers (weight_fwd, scale_fwd, weight_bwd, scale_bwd), the
 * mxfp8-32x32 recipe (weight, scale_fwd, scale_bwd), one weight tensor fewer;
 * after the gather the full tensors are rebuilt).
 *
 * A weight W [n, k] (bf16) is split into `world` shards of n_s = n / world
 * consecutive rows.  Rank r's payload is one contiguous byte buffer holding
 * its shard's quantized tensors at the offsets mxq_fsdp_payload_layout gives:
 *   MXQ_FSDP_1X32_DUAL  offsets[0] row payload [n_s, k]
 *                       offsets[1] row scales  tiled [n_s, k/32]
 *                       offsets[2] col payload [k, n_s]
 *                       offsets[3] col scales  tiled [k, n_s/32]
 *                       (= mxq_quant_1x32_dual of the shard, MMA-tiled)
 *   MXQ_FSDP_32X32      offsets[0] payload [n_s, k], offsets[1] s_fwd tiled
 *                       [n_s, k/32], offsets[2] = -1, offsets[3] s_bwd tiled
 *                       [k, n_s/32]  (= mxq_quant_32x32 of the shard)
 * so packing is the quantizer call itself with those output pointers.  The
 * gathered buffer is the world payloads back to back (rank r at
 * r * payload_bytes), as an all-gather into one buffer leaves them.
 * Shapes: n % (128 * world) == 0 (no scale atom spans two ranks), k % 32 == 0.
 */
typedef enum {
    MXQ_FSDP_1X32_DUAL = 0,
    MXQ_FSDP_32X32 = 1
} mxq_fsdp_recipe;

/* Host only.  offsets: 4 host int64 slots (offsets[2] = -1 for 32x32);
 * payload_bytes: one rank's payload size (a multiple of 512).  Returns
 * MXQ_ERR_UNSUPPORTED_SHAPE for unsupported n, k, world, MXQ_ERR_INVALID_ARG
 * for a bad recipe or NULL outputs. */
mxq_status mxq_fsdp_payload_layout(mxq_fsdp_recipe recipe, int64_t n, int64_t k, int32_t world,
                                   int64_t* offsets, int64_t* payload_bytes);

/*
 * Rebuilds the full-weight GEMM operands from the gathered buffer
 * (world * payload_bytes bytes, device).  Outputs (device):
 *   q_fwd  u8 [n, k]          row payload (32x32: the single payload)
 *   s_fwd  u8 tiled [n, k/32] mxq_scale_bytes(n, k, MXQ_SCALE_MMA_TILED) bytes
 *   q_bwd  u8 [k, n]          column payload (1x32 only; must be NULL for 32x32)
 *   s_bwd  u8 tiled [k, n/32]
 * The bytes equal those of quantizing the whole of W in one call.  One
 * kernel, HBM-bound: reads and writes world * payload_bytes bytes.
 */
mxq_status mxq_fsdp_unpack(mxq_fsdp_recipe recipe, int64_t n, int64_t k, int32_t world,
                           const void* gathered, void* q_fwd, void* s_fwd, void* q_bwd, void* s_bwd,
                           mxq_stream_t stream);

/*
 * Grouped block-scaled GEMM for MoE experts (tutorial: "MoE 专家层 (Grouped
 * MM)"; RFC section 2.2: gate_up_proj and down_proj).  Tokens are already
 * sorted by expert.  For each expert g and row r with
 * group_offsets[g] <= r < group_offsets[g+1]:
 *
 *   y[r, n] = sum_k deq(A)[r, k] * deq(B_g)[n, k]
 *
 * a_q            u8 [M_total, K] K-major; a_s scales [M_total, K/32] MMA-tiled.
 * b_q            u8 [G, N, K] K-major; b_s scales of the [G*N, K] stack, MMA-tiled.
 * group_offsets  DEVICE int64 [G+1]: 0 = off[0] <= off[1] <= ... <= off[G] = M_total.
 *                Empty experts are allowed.  Offsets are read on the device, so
 *                the call does not synchronize with the host; offsets that break
 *                the rule above give unspecified rows (never out-of-bounds access).
 * y              bf16 [M_total, N], dense (row stride N).
 * workspace      optional DEVICE scratch owned by the caller, 16-byte aligned,
 *                of workspace_bytes >= mxq_grouped_gemm_workspace_size(G,
 *                M_total, N, K) bytes.  With it the call first copies A's scales
 *                into the workspace tiled per expert (mxq_scale_regroup_rows),
 *                so that every 128-row tile starts at an expert's first row and
 *                no tile spans two experts; without it (workspace NULL and
 *                workspace_bytes 0) the tiles lie on the 128-row grid of all
 *                rows and tiles at expert boundaries are computed for each
 *                expert they touch.  The results are bit-identical either way.
 *                The workspace must not be used by other work until this call's
 *                work on `stream` has finished; its contents afterwards are
 *                unspecified.
 * Shapes: 1 <= G <= 1024; N % 128 == 0; K % 32 == 0, K > 0; M_total >= 0
 * (M_total == 0 writes nothing).
 * Errors: MXQ_ERR_INVALID_ARG (null pointers, misalignment, a workspace that
 * is too small, or only one of workspace / workspace_bytes given),
 * MXQ_ERR_UNSUPPORTED_SHAPE, MXQ_ERR_UNSUPPORTED_DEVICE, MXQ_ERR_CUDA.
 */
mxq_status mxq_grouped_gemm(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                            const int64_t* group_offsets, int32_t G, int64_t M_total,
                            int64_t N, int64_t K, void* y, void* workspace, size_t workspace_bytes,
                            mxq_stream_t stream);

/* Bytes of the workspace that lets mxq_grouped_gemm (and _fmt) tile A's
 * scales per expert, for any offsets of M_total rows over G experts:
 * (ceil(M_total/128) + G) * ceil(K/128) * 512.  N does not enter.  0 for
 * arguments mxq_grouped_gemm would refuse.  Host only. */
size_t mxq_grouped_gemm_workspace_size(int32_t G, int64_t M_total, int64_t N, int64_t K);

/* mxq_grouped_gemm with the payload format of each operand (E4M3 or E5M2),
 * e.g. E5M2 gradients against E4M3 weights in the MoE dgrad, and an output
 * row stride ldy (ldy >= N, ldy % 8 == 0). */
mxq_status mxq_grouped_gemm_fmt(const void* a_q, const void* a_s, mxq_fp8_format a_fmt,
                                const void* b_q, const void* b_s, mxq_fp8_format b_fmt,
                                const int64_t* group_offsets, int32_t G, int64_t M_total,
                                int64_t N, int64_t K, void* y, int64_t ldy, void* workspace,
                                size_t workspace_bytes, mxq_stream_t stream);

/*
 * Group-tiled A scales for mxq_grouped_gemm_group_tiled.  The rows of expert g,
 * [group_offsets[g], group_offsets[g+1]), are tiled on their own: the
 * MXQ_SCALE_MMA_TILED layout of that expert's [n_g, cols/32] scales (n_g rows
 * padded to a multiple of 128 with zeros), the experts' layouts one after the
 * other in expert order.  Expert g's first 128-row band is therefore band
 * B_g = sum over g' < g of ceil(n_g' / 128); band b occupies bytes
 * [b * A, (b+1) * A) with A = ceil(cols / 128) * 512.  The pages do not define
 * this layout (nor any scale layout for the tensor cores): it exists so that
 * a grouped GEMM's row tiles can start at every expert's first row.
 *
 * s_tiled    u8 MXQ_SCALE_MMA_TILED scales of a row quantization [rows, cols]
 *            (mxq_quant_1x32_dual's s_row).
 * group_offsets  DEVICE int64 [G+1], as for mxq_grouped_gemm (off[G] = rows).
 * bands_cap  bands of s_out; must be >= ceil(rows/128) + G, which holds every
 *            expert's bands for any offsets.  s_out has bands_cap * A bytes;
 *            bands after the last expert's are not written.  Offsets that break
 *            mxq_grouped_gemm's rule are clamped and never cause an access out of
 *            bounds (the scales are then unspecified).
 * Shapes: 1 <= G <= 1024; cols % 32 == 0.  One HBM-bound kernel: reads and
 * writes about rows * cols / 32 bytes.
 */
mxq_status mxq_scale_regroup_rows(const void* s_tiled, int64_t rows, int64_t cols,
                                  const int64_t* group_offsets, int32_t G, int64_t bands_cap, void* s_out,
                                  mxq_stream_t stream);

/*
 * mxq_grouped_gemm_fmt with A's scales group-tiled (mxq_scale_regroup_rows on
 * the same group_offsets and bands_cap = a_bands_cap).  Each expert's 128-row
 * tiles start at its first row, so no tile spans two experts: an expert with
 * n_g rows costs ceil(n_g / 128) row tiles instead of the up to ceil(n_g / 128)
 * + 1 of the 128-row grid over all rows.  Results are bit-identical to
 * mxq_grouped_gemm_fmt on the same payloads.  Arguments and errors as for
 * mxq_grouped_gemm_fmt, plus a_bands_cap >= ceil(M_total/128) + G
 * (MXQ_ERR_INVALID_ARG otherwise).
 */
mxq_status mxq_grouped_gemm_group_tiled(const void* a_q, const void* a_s, mxq_fp8_format a_fmt,
                                        const void* b_q, const void* b_s, mxq_fp8_format b_fmt,
                                        const int64_t* group_offsets, int32_t G, int64_t M_total, int64_t N,
                                        int64_t K, int64_t a_bands_cap, void* y, int64_t ldy,
                                        mxq_stream_t stream);

/*
 * Grouped weight-gradient GEMM for MoE experts: for every expert g
 *
 *   y[g][m, n] = sum over the slot positions p of expert g of deq(A)[m, p] * deq(B)[n, p]
 *
 * i.e. dW_g = dY_g^T X_g with A = dY's token-axis quantization [M, capacity]
 * and B = X's [N, capacity] (both from mxq_quant_1x32_cols_grouped with the
 * same group_offsets and capacity; scales MMA-tiled).  The slots are
 * recomputed from group_offsets on the device, exactly as the quantizer does.
 * y: bf16 [G, M, N], row stride ldy, expert g at y + g*M*ldy; an empty
 * expert gets zeros.  Shapes: N % 16 == 0, capacity % 128 == 0 and
 * capacity >= M_total + 127*G, 1 <= G <= 1024.
 */
mxq_status mxq_grouped_gemm_wgrad(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                                  const int64_t* group_offsets, int32_t G, int64_t M_total,
                                  int64_t capacity, int64_t M, int64_t N, void* y, int64_t ldy,
                                  mxq_stream_t stream);

/* mxq_grouped_gemm_wgrad with the payload format of each operand (E4M3 or E5M2). */
mxq_status mxq_grouped_gemm_wgrad_fmt(const void* a_q, const void* a_s, mxq_fp8_format a_fmt,
                                      const void* b_q, const void* b_s, mxq_fp8_format b_fmt,
                                      const int64_t* group_offsets, int32_t G, int64_t M_total,
                                      int64_t capacity, int64_t M, int64_t N, void* y, int64_t ldy,
                                      mxq_stream_t stream);

/*
 * mxq_grouped_gemm for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a convenience of this library.
 *
 * Who needs it: code that receives only its input and output buffers (for
 * instance an operator plugged into a host framework or a serving runtime
 * whose allocator owns all device memory and hands out nothing else), and
 * code that must not call cudaMalloc or cudaFree, which can synchronize the
 * whole device.  Such a caller cannot supply mxq_grouped_gemm's workspace.
 *
 * What it does: exactly mxq_grouped_gemm with a workspace (E4M3 x E4M3, y
 * dense [M_total, N]; same arguments, shapes and errors), except that the
 * workspace is a fixed array of MXQ_GROUPED_NOALLOC_MAX_WORKSPACE bytes that
 * the library keeps in device memory.  The call itself allocates nothing.
 *   - Limit: mxq_grouped_gemm_workspace_size(G, M_total, N, K) must not exceed
 *     MXQ_GROUPED_NOALLOC_MAX_WORKSPACE (e.g. 131072 rows, 128 experts and
 *     K up to 7168 fit); larger problems return MXQ_ERR_UNSUPPORTED_SHAPE
 *     and launch nothing.
 *   - Memory: every GPU that loads this library holds the array until the
 *     process exits, whether or not this call is used.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (with that device current); make that first call before any
 *     stream capture.
 *   - Sharing: all calls in the process use the same array, which keeps what
 *     the last call wrote.  Nothing in it needs to start at zero: each call
 *     rewrites every byte it later reads.  Calls whose work can overlap on the
 *     GPU (different streams, or several host threads) race on the array and
 *     give wrong results; order them on one stream or with events.
 */
#define MXQ_GROUPED_NOALLOC_MAX_WORKSPACE ((size_t)32 << 20)
mxq_status mxq_grouped_gemm_noalloc(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                                    const int64_t* group_offsets, int32_t G, int64_t M_total,
                                    int64_t N, int64_t K, void* y, mxq_stream_t stream);

/* Waits for the work queued on `stream` (synchronizes the host with it), then
 * returns MXQ_ERR_TIMEOUT if any kernel of this library on the current device
 * recorded a bounded wait that ran out since the last call, MXQ_ERR_CUDA if
 * the device reports an error, MXQ_OK otherwise.  The record is read and
 * cleared in one atomic exchange on the device, so a timeout recorded by a
 * kernel on another stream at the same moment is never lost: it is reported
 * by this call or by the next one.  Calls from several host threads take
 * turns. */
mxq_status mxq_get_device_status(mxq_stream_t stream);

/* Test hook for the bounded-wait machinery: launches one small kernel that
 * waits on a barrier no thread ever completes, giving up after timeout_us
 * microseconds (1..1000000) and recording MXQ_ERR_TIMEOUT the way every
 * kernel of the library does.  Returns the launch status. */
mxq_status mxq_debug_wait_timeout(uint32_t timeout_us, mxq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
