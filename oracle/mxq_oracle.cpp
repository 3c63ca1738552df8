// mxq_oracle.cpp -- the CPU oracle for MXFP8 microscaled quantization and
// block-scaled GEMM.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
// load or call this file.  Its only users are the tests, the smoke check and
// the timed CPU baseline of the benchmark.  It shares no code, header, table
// or constant with the CUDA library: everything here is re-derived from the
// definitions below, in plain loops, in the order the method states them.
//
// What the method computes (sources, by page and section):
//  * "torchtitan-npu MXFP8/HiF8 low-precision training tutorial", section
//    "MXFP8 与 HiF8 架构原理速览": MXFP8 is per-block dynamic quantization in
//    which every 32 consecutive elements share one E8M0 scale; the FP8 matmul
//    returns BF16.  Section "第 3 步 验证 converter 生效" names the scale rule
//    "mxfp8_rceil" (scale exponent rounded up).
//  * MindSpeed RFC "Add MXFP8-32x32 quantization support to FSDP" (issue 175):
//    section 3.1 (block size [1,32,32]: blocks of 32 on input_dim and
//    output_dim, token_dim not blocked; forward and backward share one
//    weight payload), section 3.3.1 (element type E4M3, dynamic scaling),
//    section 3.3.3 (mxfp8 uses a dual-axis quantizer that gives separate
//    forward and backward copies; mxfp8-32x32 gives one payload, and only
//    the scales differ), section 3.5.2.3 (process_quant_result_fn serves
//    both recipes; its dst_type is float8_e4m3fn or float8_e5m2).
//
// Readings taken where the pages are silent:
//  * E4M3 is the OCP "fn" variant (float8_e4m3fn): bias 7, no infinities,
//    NaN = S.1111.111, largest finite 448.  Conversion is round to nearest,
//    ties to even, saturating to +-448; the sign of zero is kept.
//  * E8M0 code c in [0,254] means 2^(c-127); 0xFF is NaN.
//  * The RFC also allows dst_type E5M2 (section 3.5.2.3): OCP float8_e5m2,
//    bias 15, max finite 57344, RNE saturating; rceil then uses 57344.  The
//    same function serves the 32x32 recipe, so both the 1x32 and the 32x32
//    quantizers take either format.
//  * rceil: e = ceil(log2(amax / 448)), clamped to [-127, 127]; amax == 0
//    gives e = -127.  Evaluated exactly: with amax = f * 2^k, f in [0.5,1),
//    448 = 0.875 * 2^9, so e = k - 9 + (f > 0.875).
//  * A group (or 32x32 tile) holding any NaN or Inf gets scale code 0xFF and
//    every payload byte 0x7F | sign(x).
//  * GEMM: exact products of the dequantized operands summed in FP64 in
//    increasing contraction index, rounded once to BF16 (ties to even).
//
// Build: g++ -O2 -std=c++17 -fopenmp -shared -fPIC (see oracle.py).

#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>

namespace {

// ---- BF16 <-> double ------------------------------------------------------

double bf16_bits_to_double(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

// Round a double to the nearest BF16 value (ties to even) in one step.
// BF16 has 8 significant bits and the float32 exponent range: normal
// numbers from 2^-126, subnormal spacing 2^-133, largest finite
// (2 - 2^-7) * 2^127.
uint16_t double_to_bf16_bits(double v) {
    if (std::isnan(v)) return 0x7FC0;
    uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    double a = std::fabs(v);
    if (std::isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int k;
    std::frexp(a, &k);  // a = f * 2^k, f in [0.5, 1): leading bit has weight 2^(k-1)
    int lead = k - 1;
    if (lead < -126) lead = -126;            // subnormal range: fixed spacing
    double quantum = std::ldexp(1.0, lead - 7);
    double n = std::nearbyint(a / quantum);  // exact division; FE_TONEAREST = ties to even
    double r = n * quantum;
    const double bf16_max = std::ldexp(255.0, 120);  // (2 - 2^-7) * 2^127
    if (r > bf16_max) return sign | 0x7F80;          // rounded past the largest finite
    float f = static_cast<float>(r);                 // r is exactly representable
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>(sign | ((u >> 16) & 0x7FFF));
}

// ---- E4M3 (float8_e4m3fn) ---------------------------------------------------

double e4m3_decode(uint8_t c) {
    int s = c >> 7, E = (c >> 3) & 0xF, m = c & 0x7;
    if (E == 0xF && m == 0x7) return std::nan("");
    double mag = (E == 0) ? std::ldexp(static_cast<double>(m), -9)        // m/8 * 2^-6
                          : std::ldexp(static_cast<double>(8 + m), E - 10); // (1+m/8) * 2^(E-7)
    return s ? -mag : mag;
}

// Round-to-nearest-even, saturating encode of an exact double.
uint8_t e4m3_encode(double v) {
    uint8_t sign = std::signbit(v) ? 0x80 : 0;
    if (std::isnan(v)) return sign | 0x7F;
    double a = std::fabs(v);
    if (a >= 448.0) return sign | 0x7E;  // saturate (also +-inf)
    if (a == 0.0) return sign;
    int k;
    std::frexp(a, &k);
    int lead = k - 1;               // exponent of the leading bit
    if (lead < -6) lead = -6;       // below 2^-6 the spacing is fixed (subnormals)
    double quantum = std::ldexp(1.0, lead - 3);  // 3 mantissa bits
    double n = std::nearbyint(a / quantum);      // integer in [0, 16]
    // Rebuild the code from the rounded value n * quantum.
    if (lead == -6 && n < 8) return sign | static_cast<uint8_t>(n);  // subnormal (or zero)
    if (n == 16) { n = 8; lead += 1; }                               // carried into next binade
    int E = lead + 7;
    int m = static_cast<int>(n) - 8;
    // a < 448 rounds at most to 448 = code 0x7E, so E <= 15 and (E,m) != (15,7).
    return sign | static_cast<uint8_t>((E << 3) | m);
}

// ---- E5M2 (float8_e5m2) ---------------------------------------------------------
// Bias 15, 2 mantissa bits; S.11111.00 = Inf, S.11111.xx (xx != 0) = NaN;
// largest finite 57344 = 1.75 * 2^15, smallest normal 2^-14, subnormal spacing 2^-16.

double e5m2_decode(uint8_t c) {
    int s = c >> 7, E = (c >> 2) & 0x1F, m = c & 0x3;
    double mag;
    if (E == 0x1F) mag = m == 0 ? HUGE_VAL : std::nan("");
    else if (E == 0) mag = std::ldexp(static_cast<double>(m), -16);
    else mag = std::ldexp(static_cast<double>(4 + m), E - 17);
    return s ? -mag : mag;
}

// Round-to-nearest-even, saturating (to +-57344) encode of an exact double.
uint8_t e5m2_encode(double v) {
    uint8_t sign = std::signbit(v) ? 0x80 : 0;
    if (std::isnan(v)) return sign | 0x7F;
    double a = std::fabs(v);
    if (a >= 57344.0) return sign | 0x7B;
    if (a == 0.0) return sign;
    int k;
    std::frexp(a, &k);
    int lead = k - 1;
    if (lead < -14) lead = -14;
    double quantum = std::ldexp(1.0, lead - 2);  // 2 mantissa bits
    double n = std::nearbyint(a / quantum);      // integer in [0, 8]
    if (lead == -14 && n < 4) return sign | static_cast<uint8_t>(n);
    if (n == 8) { n = 4; lead += 1; }
    // a < 57344 rounds at most to 57344 (E = 30, m = 3).
    return sign | static_cast<uint8_t>(((lead + 15) << 2) | (static_cast<int>(n) - 4));
}

double e8m0_decode(uint8_t c) {
    if (c == 0xFF) return std::nan("");
    return std::ldexp(1.0, static_cast<int>(c) - 127);
}

// rceil scale exponent of a finite, non-negative amax: ceil(log2(amax / max))
// with max = 448 = 0.875 * 2^9 (E4M3) or 57344 = 0.875 * 2^16 (E5M2).
int rceil_exponent(double amax, int fmt = 0) {
    if (amax == 0.0) return -127;
    int k;
    double f = std::frexp(amax, &k);
    int e = k - (fmt == 0 ? 9 : 16) + (f > 0.875 ? 1 : 0);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

// Quantize a set of n values that share one scale.  Writes the payload bytes
// via `put(i, byte)` and returns the E8M0 scale code.
template <class Get, class Put>
uint8_t quant_shared_scale(int64_t n, Get get, Put put, int fmt = 0) {
    double amax = 0.0;
    bool nonfinite = false;
    for (int64_t i = 0; i < n; ++i) {
        double x = get(i);
        if (!std::isfinite(x)) nonfinite = true;
        else if (std::fabs(x) > amax) amax = std::fabs(x);
    }
    if (nonfinite) {
        for (int64_t i = 0; i < n; ++i) put(i, static_cast<uint8_t>((std::signbit(get(i)) ? 0x80 : 0) | 0x7F));
        return 0xFF;
    }
    int e = rceil_exponent(amax, fmt);
    for (int64_t i = 0; i < n; ++i) {  // x * 2^-e is exact
        const double v = std::ldexp(get(i), -e);
        put(i, fmt == 0 ? e4m3_encode(v) : e5m2_encode(v));
    }
    return static_cast<uint8_t>(e + 127);
}

}  // namespace

extern "C" {

// ---- scalar entry points (exposed for the pins) ----------------------------

double orc_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
uint8_t orc_e4m3_encode(double v) { return e4m3_encode(v); }
double orc_e8m0_decode(uint8_t c) { return e8m0_decode(c); }
int orc_rceil_exponent(double amax) { return rceil_exponent(amax); }
double orc_e5m2_decode(uint8_t c) { return e5m2_decode(c); }
int orc_rceil_exponent_fmt(double amax, int fmt) { return rceil_exponent(amax, fmt); }

void orc_e5m2_encode_array(const double* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = e5m2_encode(v[i]);
}
uint16_t orc_bf16_from_double(double v) { return double_to_bf16_bits(v); }
double orc_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

void orc_e4m3_encode_array(const double* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(v[i]);
}

void orc_bf16_from_double_array(const double* v, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_bits(v[i]);
}

// ---- 1x32 quantization -----------------------------------------------------
// x: bf16 bits [rows, cols] with row stride ld (elements); cols % 32 == 0.
// q: [rows, cols] payload; s: [rows, cols/32] scale codes (plain row-major).
// Each group is 32 consecutive elements of one row.
void orc_quant_rows_fmt(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                        uint8_t* q, uint8_t* s, int fmt) {
    const int64_t groups = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            const uint16_t* src = x + r * ld + g * 32;
            uint8_t* dst = q + r * cols + g * 32;
            s[r * groups + g] = quant_shared_scale(
                32, [&](int64_t i) { return bf16_bits_to_double(src[i]); },
                [&](int64_t i, uint8_t b) { dst[i] = b; }, fmt);
        }
    }
}

void orc_quant_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                    uint8_t* q, uint8_t* s) {
    orc_quant_rows_fmt(x, rows, cols, ld, q, s, 0);
}

// Dual-axis 1x32 quantization: the row copy is orc_quant_rows(x); the column
// copy is the row quantization of x transposed, stored [cols, rows] with
// scales [cols, rows/32].  Either pair of outputs may be null.
void orc_quant_dual(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                    uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col) {
    if (q_row && s_row) orc_quant_rows(x, rows, cols, ld, q_row, s_row);
    if (q_col && s_col) {
        uint16_t* xt = new uint16_t[static_cast<size_t>(rows) * cols];
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c)
            for (int64_t r = 0; r < rows; ++r) xt[c * rows + r] = x[r * ld + c];
        orc_quant_rows(xt, cols, rows, rows, q_col, s_col);
        delete[] xt;
    }
}

// ---- 32x32 block quantization ----------------------------------------------
// w: bf16 bits [n, k] (row stride ld), n % 32 == 0, k % 32 == 0.  Tiles of
// 32 x 32 start at (0,0).  One payload q [n, k] in format fmt (0 E4M3,
// 1 E5M2).  The tile exponent t[i][j] (tile row i, tile column j) is written
// twice:
//   s_fwd [n, k/32]:  s_fwd[r][j] = t[r/32][j]   (forward, contraction over k)
//   s_bwd [k, n/32]:  s_bwd[c][i] = t[i][c/32]   (backward, contraction over n)
void orc_quant_32x32_fmt(const uint16_t* w, int64_t n, int64_t k, int64_t ld,
                         uint8_t* q, uint8_t* s_fwd, uint8_t* s_bwd, int fmt) {
    const int64_t tn = n / 32, tk = k / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < tn; ++i) {
        for (int64_t j = 0; j < tk; ++j) {
            uint8_t code = quant_shared_scale(
                32 * 32,
                [&](int64_t e) { return bf16_bits_to_double(w[(i * 32 + e / 32) * ld + j * 32 + e % 32]); },
                [&](int64_t e, uint8_t b) { q[(i * 32 + e / 32) * k + j * 32 + e % 32] = b; }, fmt);
            for (int64_t r = 0; r < 32; ++r) {
                if (s_fwd) s_fwd[(i * 32 + r) * tk + j] = code;
                if (s_bwd) s_bwd[(j * 32 + r) * tn + i] = code;
            }
        }
    }
}

void orc_quant_32x32(const uint16_t* w, int64_t n, int64_t k, int64_t ld,
                     uint8_t* q, uint8_t* s_fwd, uint8_t* s_bwd) {
    orc_quant_32x32_fmt(w, n, k, ld, q, s_fwd, s_bwd, 0);
}

// ---- grouped column quantization (MoE weight gradient) ----------------------
// x: bf16 bits [rows, cols] (row stride ld) with rows sorted by expert;
// off: [G+1] expert row offsets.  Expert g's tokens are quantized along the
// token axis in groups of 32 that start at the expert's first token; a group
// that runs past the expert's last token is completed with zeros (reading of
// the unstated padding rule).  Output layout: expert g occupies the column
// slot [P_g, P_g + L_g) of q_col [cols, capacity] with L_g = m_g rounded up
// to a multiple of 128 and P_g = sum of L_h over h < g; everything in the slot
// past the expert's groups is zero payload with scale code 0.  s_col holds the
// plain scales [cols, capacity/32].  Columns past P_G are left untouched.
void orc_quant_cols_grouped_fmt(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                const int64_t* off, int32_t G, int64_t capacity,
                                uint8_t* q_col, uint8_t* s_col, int fmt) {
    (void)rows;
    const int64_t cgroups = capacity / 32;
    int64_t P = 0;
    for (int32_t g = 0; g < G; ++g) {
        const int64_t lo = off[g], m = off[g + 1] - off[g];
        const int64_t L = (m + 127) / 128 * 128;
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c) {
            for (int64_t j = 0; j < L / 32; ++j) {
                uint8_t* dst = q_col + c * capacity + P + 32 * j;
                s_col[c * cgroups + P / 32 + j] = quant_shared_scale(
                    32,
                    [&](int64_t i) {
                        const int64_t t = 32 * j + i;
                        return t < m ? bf16_bits_to_double(x[(lo + t) * ld + c]) : 0.0;
                    },
                    [&](int64_t i, uint8_t b) { dst[i] = b; }, fmt);
            }
        }
        P += L;
    }
}

void orc_quant_cols_grouped(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                            const int64_t* off, int32_t G, int64_t capacity,
                            uint8_t* q_col, uint8_t* s_col) {
    orc_quant_cols_grouped_fmt(x, rows, cols, ld, off, G, capacity, q_col, s_col, 0);
}

// ---- scale layout: plain -> MMA-tiled ---------------------------------------
// s: plain [rows, groups].  out: tiled, sized roundup(rows,128) *
// roundup(groups,4) bytes.  Atoms of 128 rows x 4 groups (512 bytes) are
// stored atom-row-major (the 4-group atoms of one 128-row band are
// consecutive); inside an atom, row r and group g sit at byte
// 16*(r%32) + 4*((r%128)/32) + (g%4).  Padding bytes are zero.
void orc_scale_tiled(const uint8_t* s, int64_t rows, int64_t groups, uint8_t* out) {
    const int64_t rows_p = (rows + 127) / 128 * 128;
    const int64_t groups_p = (groups + 3) / 4 * 4;
    const int64_t atoms_per_band = groups_p / 4;
    std::memset(out, 0, static_cast<size_t>(rows_p * groups_p));
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            int64_t atom = (r / 128) * atoms_per_band + g / 4;
            int64_t inner = 16 * (r % 32) + 4 * ((r % 128) / 32) + (g % 4);
            out[atom * 512 + inner] = s[r * groups + g];
        }
    }
}

// ---- dequantization ----------------------------------------------------------
// out[r][c] = fp8(q[r][c]) * 2^(s[r][c/32] - 127)   (plain scales)
void orc_dequant_rows_fmt(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols, double* out,
                          int fmt) {
    const int64_t groups = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = (fmt == 0 ? e4m3_decode(q[r * cols + c]) : e5m2_decode(q[r * cols + c])) *
                                e8m0_decode(s[r * groups + c / 32]);
}

void orc_dequant_rows(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols, double* out) {
    const int64_t groups = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = e4m3_decode(q[r * cols + c]) * e8m0_decode(s[r * groups + c / 32]);
}

// ---- GEMM ------------------------------------------------------------------------
// y[i][n] = bf16( sum_{k=0..K-1} a[row_i][k] * b[n][k] ), FP64, increasing k.
// a: [M, K] dequantized, b: [N, K] dequantized.  rows: nrows indices into a
// (null -> all M rows in order).  y: [nrows, N] bf16 bits.
void orc_gemm(const double* a, const double* b, int64_t M, int64_t N, int64_t K,
              const int64_t* rows, int64_t nrows, uint16_t* y) {
    if (!rows) nrows = M;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        for (int64_t n = 0; n < N; ++n) {
            const double* ar = a + (rows ? rows[i] : i) * K;
            const double* br = b + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += ar[k] * br[k];
            y[i * N + n] = double_to_bf16_bits(acc);
        }
    }
}

// Grouped GEMM: for expert g the rows off[g] <= r < off[g+1] use weight
// b[g] ([N, K]).  y[i][n] for the sampled rows (null -> all rows).
void orc_grouped_gemm(const double* a, const double* b, const int64_t* off, int32_t G,
                      int64_t N, int64_t K, const int64_t* rows, int64_t nrows, uint16_t* y) {
    const int64_t M = off[G];
    if (!rows) nrows = M;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        for (int64_t n = 0; n < N; ++n) {
            const int64_t r = rows ? rows[i] : i;
            int32_t g = 0;
            while (g + 1 < G && !(off[g] <= r && r < off[g + 1])) ++g;  // the expert that owns row r
            const double* ar = a + r * K;
            const double* br = b + (static_cast<int64_t>(g) * N + n) * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += ar[k] * br[k];
            y[i * N + n] = double_to_bf16_bits(acc);
        }
    }
}

}  // extern "C"
