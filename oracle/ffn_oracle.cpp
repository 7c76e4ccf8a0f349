// CPU oracle for the FP8 SwiGLU FFN block: prefill chain, its recompute form,
// the attention projections' quantise-then-matmul, the FP8 backward of the FFN
// and the single-token decode FFN.
//
// TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
// entry point and the benchmark's CPU-baseline / reference legs load this
// library.  It shares no code, header, table or constant with the CUDA
// library: plain C++17, the C and C++ standard libraries and OpenMP only.
//
// Sources (page title, function):
//  [llmq-model]  IST-DASLab/llmq "src/models/llama_model.cpp":
//     LLamaModel::_forward_block, FFN half (fused_residual_rmsnorm_forward ->
//     forward_qmm on the up projection -> swiglu_forward -> forward_qmm on the
//     down projection); forward_qmm (quantise with the recorded abs-max, then a
//     matmul multiplied by the weight and activation scales);
//     _recompute_block (swiglu_forward_quant); _backward_block and
//     backward_qmm (FP8 branch); fill_block_shapes (UP_W [2H, C],
//     DOWN_W [C, H]); LLamaModel::forward (fill_zero(AbsMaxes) first).
//  [llmq-state]  IST-DASLab/llmq "src/models/llama_run_state.cpp":
//     buffer dtypes (ln2, mlp_up, swiglu, mlp_down bf16; their quantised
//     copies FP8) and the stats block, two floats per tensor (abs-max, scale).
//  [metrale-decode]  metrale "layers/dense_ffn_decode.rs",
//     DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual (gate and up GEMVs of
//     one input, fp32 scale per output row), silu_mul back into the gate
//     buffer, w8a16_gemv for down.
//
// The pages call these kernels without defining their arithmetic.  The
// readings taken where they leave a step open (each applied where it is
// used below):
//  R1  gate = rows/columns [0, H) of the fused up projection, up = [H, 2H).
//  R2  scale = abs_max / 448 is the dequantisation multiplier (448 is the
//      largest finite E4M3 value).
//  R3  the norm reads the stored, bf16-rounded residual sum.
//  R4  y = bf16(r * rstd * g), one rounding; rstd is returned as fp32.
//  R5  the abs-max is taken over the bf16 values that are quantised.
//  R6  each element is e4m3(float(v) * (448f / abs_max)), the product
//      rounded to fp32, then to E4M3 (nearest even, saturating at +-448).
//  R7  abs_max == 0: scale 1, every code 0.
//  R9  GEMM: exact sum times both scales, one rounding to bf16; SwiGLU reads
//      those bf16 values.
//  R10 silu(z) = z / (1 + exp(-z)).
//  R11 SwiGLU with quantisation = swiglu recording the abs-max of bf16 h,
//      then quantisation of that same bf16 h.
//  R14 decode g, u, h are bf16; the row scale multiplies the finished sum.
//  R15 the decode input is already normalised.
//  R19 a matmul bias is added to the scaled sum before its one rounding.
//  R20 backward gradients are bf16, their FP8 copies E4M3.
//  R21 dg = dh * u * s * (1 + g * (1 - s)), du = dh * silu(g), s = sigmoid(g),
//      each rounded once; gate gradient in columns [0, H).
//  R22 gradient accumulation: bf16(old + scaled product), one rounding.
//
// Precision.  bf16 and E4M3 are decoded from their bit fields and encoded by
// rounding to nearest (ties to even) on the format's grid: a value is
// divided by the spacing of its binade with ldexp, rounded with rint (the
// default rounding mode, ties to even) and multiplied back.  The FP8 GEMM is
// exact: every E4M3 value is an integer multiple of 2^-9 of magnitude at most
// 229376 = 448 * 2^9, so each product of two is an integer below 2^36 and the
// int64 sum of up to 2^27 of them is exact; the sum times 2^-18 and the two
// fp32 scales (in fp64) is rounded once to bf16.  RMSNorm's sum of squares
// and the GEMV dot products are fp64 sums with a running compensation term
// (Neumaier's variant of Kahan summation): every term is exact in fp64, and
// the compensated sum is within a few units of 2^-100 of the exact sum, so
// the one final rounding to bf16 is that of the exact value except within
// about 2^-50 of a rounding midpoint.  The library must be compiled without
// floating-point contraction (-ffp-contract=off), so no product and sum are
// fused into a single rounding.
//
// Output rows are distributed over OpenMP threads; each result is computed
// by one thread in a fixed order, so results do not depend on the thread
// count.

#include <omp.h>

#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// Deliberate mistakes that the pin tests plant to show that they can fail.
// 0 = none.  Never set outside those tests.
enum Plant : int {
    PLANT_NONE = 0,
    PLANT_GATE_UP_SWAPPED = 1,     // SwiGLU reads up as the gate and gate as up
    PLANT_E4M3_TIES_AWAY = 2,      // E4M3 rounding ties go away from zero
    PLANT_E4M3_NO_SATURATION = 3,  // E4M3 overflow becomes the NaN code
    PLANT_NORM_UNROUNDED_SUM = 4,  // RMSNorm reads res + x before its bf16 rounding
    PLANT_GEMM_DROPS_LAST_K = 5,   // the GEMM sum misses its last term
    PLANT_SILU_SIGN = 6,           // silu(z) = z / (1 + exp(+z))
    PLANT_BF16_TRUNCATES = 7,      // bf16 rounding truncates instead of rounding
    PLANT_QUANT_DIVIDES = 8,       // elements scaled as v / scale instead of v * (448 / amax)
    PLANT_DSILU_NO_CORRECTION = 9, // swiglu_backward drops the g * (1 - s) term
    PLANT_GEMV_SCALE_BY_FIRST = 10 // every decode row uses the first row's scale
};
int g_plant = PLANT_NONE;

constexpr float kE4M3Max = 448.0f;

// ------------------------------------------------------------------ bf16
// bf16: binary32 with the low 16 mantissa bits dropped (1 sign bit,
// 8 exponent bits with bias 127, 7 stored mantissa bits).
double bf16_value(uint16_t bits) {
    uint32_t w = uint32_t(bits) << 16;
    float f;
    std::memcpy(&f, &w, 4);
    return double(f);
}

// Round an fp64 value to bf16, nearest with ties to even, in one step.  In
// the binade [2^(e-1), 2^e) (frexp exponent e) a normal bf16 has spacing
// 2^(e-8); below the smallest normal 2^-126 the spacing stays at the
// subnormal quantum 2^-133.  Values that round past the largest finite bf16
// become infinity.
uint16_t bf16_round(double x) {
    double q;
    if (std::isnan(x)) {
        q = x;
    } else {
        int e = 0;
        std::frexp(x, &e);
        int q_exp = e - 8 < -133 ? -133 : e - 8;
        double scaled = std::ldexp(x, -q_exp);
        double n = g_plant == PLANT_BF16_TRUNCATES ? std::trunc(scaled) : std::rint(scaled);
        q = std::ldexp(n, q_exp);
    }
    float f = float(q);   // exact: q has at most 8 significant bits (or overflows to inf)
    uint32_t w;
    std::memcpy(&w, &f, 4);
    return uint16_t(w >> 16);
}

// ------------------------------------------------------------------ e4m3
// OCP FP8 E4M3 ("fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
// bits.  Exponent field 0 holds subnormals m * 2^-9; S.1111.111 is NaN; there
// is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
double e4m3_value(uint8_t code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 0xF, m = code & 7;
    double mag;
    if (e == 15 && m == 7) mag = NAN;
    else if (e == 0) mag = std::ldexp(double(m), -9);
    else mag = std::ldexp(double(8 + m), e - 10);   // (1 + m/8) * 2^(e-7)
    return s ? -mag : mag;
}

// The value times 2^9 as an integer (|v| <= 229376); 0 for the NaN codes,
// which the GEMMs never receive.
int32_t e4m3_scaled_int(uint8_t code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 0xF, m = code & 7;
    if (e == 15 && m == 7) return 0;
    int32_t mag = e == 0 ? m : (8 + m) << (e - 1);      // (8 + m) * 2^(e-10) * 2^9
    return s ? -mag : mag;
}

// Round to E4M3: nearest on the E4M3 grid with ties to even, saturating at
// +-448.  In the binade [2^E, 2^(E+1)) with E >= -6 the spacing is 2^(E-3);
// below the smallest normal 2^-6 it is the subnormal quantum 2^-9.  NaN gives
// the NaN code with the input's sign.
uint8_t e4m3_round(double v) {
    bool neg = std::signbit(v);
    double a = std::fabs(v);
    if (std::isnan(a)) return neg ? 0xFF : 0x7F;
    int e = 0;
    std::frexp(a, &e);                      // a = f * 2^e, f in [0.5, 1): E = e - 1
    int E = e - 1 < -6 ? -6 : e - 1;
    int q_exp = E - 3;
    double scaled = std::ldexp(a, -q_exp);
    double n;
    if (g_plant == PLANT_E4M3_TIES_AWAY) n = std::floor(scaled + 0.5);
    else n = std::rint(scaled);
    double q = std::ldexp(n, q_exp);
    uint8_t code;
    if (q > kE4M3Max) {
        if (g_plant == PLANT_E4M3_NO_SATURATION) return neg ? 0xFF : 0x7F;
        q = kE4M3Max;
    }
    if (q < std::ldexp(1.0, -6)) {
        code = uint8_t(std::ldexp(q, 9));                  // subnormal: m * 2^-9, m in 0..7
    } else {
        int e2 = 0;
        std::frexp(q, &e2);
        int E2 = e2 - 1;
        int mant = int(std::ldexp(q, -E2) * 8.0) - 8;      // 0..7
        code = uint8_t((E2 + 7) * 8 + mant);
    }
    return neg ? uint8_t(code | 0x80) : code;
}

// ------------------------------------------------------------------ compensated fp64 sum
// Neumaier's running compensation: s + c carries the sum to about twice the
// precision of fp64; the result is rounded once at the end.
struct CompSum {
    double s = 0.0, c = 0.0;
    void add(double x) {
        double t = s + x;
        if (std::fabs(s) >= std::fabs(x)) c += (s - t) + x;
        else c += (x - t) + s;
        s = t;
    }
    double value() const { return s + c; }
};

double silu(double z) {
    // R10
    if (g_plant == PLANT_SILU_SIGN) return z / (1.0 + std::exp(z));
    return z / (1.0 + std::exp(-z));
}

float absmax_bf16(const uint16_t* v, int64_t n) {
    double m = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double a = std::fabs(bf16_value(v[i]));
        if (a > m) m = a;
    }
    return float(m);   // exact: a bf16 value
}

// A2 (quantize_with_abs_max) on fp32 inputs: R2, R6, R7.
void quantize_f32(const float* v, int64_t n, float amax, uint8_t* codes, float* scale) {
    if (amax == 0.0f) {
        for (int64_t i = 0; i < n; ++i) codes[i] = 0;
        *scale = 1.0f;
        return;
    }
    *scale = amax / kE4M3Max;
    float inv = kE4M3Max / amax;      // an fp32 division
    float s = *scale;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float p = g_plant == PLANT_QUANT_DIVIDES ? v[i] / s : v[i] * inv;   // fp32 product
        codes[i] = e4m3_round(double(p));
    }
}

// R1, R9, R10: h = bf16(silu(bf16 g) * bf16 u) for one row of the gate|up output.
void swiglu_row(const uint16_t* gu, int64_t H, uint16_t* h) {
    const uint16_t* gp = gu;
    const uint16_t* up = gu + H;
    if (g_plant == PLANT_GATE_UP_SWAPPED) std::swap(gp, up);
    for (int64_t j = 0; j < H; ++j) h[j] = bf16_round(silu(bf16_value(gp[j])) * bf16_value(up[j]));
}

// Scaled-integer copy of an E4M3 operand, K contiguous: dst[r][k] = int(src(r, k)),
// src(r, k) = src[r * rs + k * ks].
std::vector<int32_t> decode_operand(const uint8_t* src, int64_t rows, int64_t K, int64_t rs, int64_t ks) {
    std::vector<int32_t> dst(static_cast<size_t>(rows * K));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) dst[size_t(r) * K + k] = e4m3_scaled_int(src[r * rs + k * ks]);
    return dst;
}

}  // namespace

extern "C" {

// ------------------------------------------------------------------ control
void orc_set_plant(int which) { g_plant = which; }
int orc_get_plant() { return g_plant; }
void orc_set_threads(int n) { omp_set_num_threads(n > 0 ? n : omp_get_num_procs()); }
int orc_max_threads() { return omp_get_max_threads(); }

// ------------------------------------------------------------------ codecs
void orc_bf16_decode(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(in[i]);
}
void orc_bf16_round(const double* in, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static) if (n > (1 << 16))
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_round(in[i]);
}
void orc_e4m3_decode(const uint8_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
}
void orc_e4m3_scaled_int(const uint8_t* in, int32_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_scaled_int(in[i]);
}
void orc_e4m3_round(const double* in, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static) if (n > (1 << 16))
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_round(in[i]);
}
void orc_silu(const double* z, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = silu(z[i]);
}

// ------------------------------------------------------------------ A1
// Unrounded RMSNorm of bf16 rows r [N, C] with gain g [C]: y64 = r * rstd * g,
// rstd = 1 / sqrt(mean_C(r^2) + eps) in fp64 [llmq-model,
// fused_residual_rmsnorm_forward / rmsnorm_forward with Config.RmsNormEps].
void orc_rmsnorm_f64(const uint16_t* r, const uint16_t* gain, float eps, int64_t N, int64_t C,
                     double* y64, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i) {
        CompSum ss;
        for (int64_t k = 0; k < C; ++k) {
            double v = bf16_value(r[i * C + k]);
            ss.add(v * v);                               // exact square of a bf16 value
        }
        double ms = ss.value() / double(C);
        double rs = 1.0 / std::sqrt(ms + double(eps));
        rstd[i] = rs;
        for (int64_t k = 0; k < C; ++k) y64[i * C + k] = bf16_value(r[i * C + k]) * rs * bf16_value(gain[k]);
    }
}

// Step A1: fused residual add + RMSNorm + abs-max [llmq-model _forward_block:
// fused_residual_rmsnorm_forward(ResidualAtt, LN2.Value, LN2_Rstd, residual,
// AttO, LN2_w, LN2.Quant.abs_max(), eps, B*T, C)].  res == NULL is
// rmsnorm_forward: r is x.  Writes r, y [N, C] bf16, rstd [N] fp32 and the
// abs-max of y (R3, R4, R5).
void orc_residual_rmsnorm_absmax(const uint16_t* res, const uint16_t* x, const uint16_t* gain, float eps,
                                 int64_t N, int64_t C, uint16_t* r, uint16_t* y, float* rstd, float* amax) {
    double m = 0.0;
#pragma omp parallel for schedule(static) reduction(max : m)
    for (int64_t i = 0; i < N; ++i) {
        const int64_t o = i * C;
        std::vector<double> rv(static_cast<size_t>(C));
        for (int64_t k = 0; k < C; ++k) {
            if (res == nullptr) {
                r[o + k] = x[o + k];
                rv[k] = bf16_value(x[o + k]);
            } else {
                double sum = bf16_value(res[o + k]) + bf16_value(x[o + k]);   // exact in fp64
                r[o + k] = bf16_round(sum);                                    // stored ResidualAtt
                rv[k] = g_plant == PLANT_NORM_UNROUNDED_SUM ? sum : bf16_value(r[o + k]);   // R3
            }
        }
        CompSum ss;
        for (int64_t k = 0; k < C; ++k) ss.add(rv[k] * rv[k]);
        double rs = 1.0 / std::sqrt(ss.value() / double(C) + double(eps));
        rstd[i] = float(rs);
        for (int64_t k = 0; k < C; ++k) {
            uint16_t b = bf16_round(rv[k] * rs * bf16_value(gain[k]));   // R4: one rounding
            y[o + k] = b;
            double a = std::fabs(bf16_value(b));
            if (a > m) m = a;
        }
    }
    *amax = float(m);
}

float orc_absmax_bf16(const uint16_t* v, int64_t n) { return absmax_bf16(v, n); }

// ------------------------------------------------------------------ A2
// quantize_with_abs_max [llmq-model forward_qmm: quantize_with_abs_max(
// inp.Quant, inp.Quant.scale(), inp.Value, inp.Quant.abs_max(), B*T*C)]:
// codes = e4m3(float(v) * (448f / amax)), scale = amax / 448f (R2, R6, R7).
void orc_quantize_with_abs_max(const uint16_t* v, int64_t n, float amax, uint8_t* codes, float* scale) {
    std::vector<float> f(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) f[i] = float(bf16_value(v[i]));   // exact
    quantize_f32(f.data(), n, amax, codes, scale);
}

// Per-output-row E4M3 records of the decode weights [metrale-decode: the FP8
// weights carry one fp32 row_scale per output row]: each row quantised by
// A2's rule with its own abs-max.
void orc_quantize_rows(const uint16_t* w, int64_t R, int64_t K, uint8_t* codes, float* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        float amax = absmax_bf16(w + r * K, K);
        if (amax == 0.0f) {
            for (int64_t k = 0; k < K; ++k) codes[r * K + k] = 0;
            scales[r] = 1.0f;
            continue;
        }
        scales[r] = amax / kE4M3Max;
        float inv = kE4M3Max / amax;
        for (int64_t k = 0; k < K; ++k) {
            float p = float(bf16_value(w[r * K + k])) * inv;
            codes[r * K + k] = e4m3_round(double(p));
        }
    }
}

// ------------------------------------------------------------------ A3 / A5
// Scaled FP8 matmul [llmq-model forward_qmm -> matmul(out, weight, inp.Quant,
// bias, weight.scale(), inp.Quant.scale(), ..., TN)]:
//   out[m, n] = bf16( old[m, n] + (sum_k A(m, k) * B(n, k)) * sa * sb + bias[n] )
// with A(m, k) = A[m * a_ms + k * a_ks], B(n, k) = B[n * b_ns + k * b_ks]
// (strides in elements, so transposed operands need no copy); old (R22) and
// bias (R19) may be NULL.  The sum is exact (int64 over the codes' scaled
// integers, then times 2^-18); the scaled value is formed in fp64, the one
// rounding is to bf16 (R9).
int orc_fp8_gemm(const uint8_t* A, int64_t a_ms, int64_t a_ks, float sa, const uint8_t* B, int64_t b_ns,
                 int64_t b_ks, float sb, int64_t M, int64_t N, int64_t K, const uint16_t* bias,
                 const uint16_t* old, uint16_t* out) {
    if (K >= (int64_t(1) << 27)) return 1;                // int64 exactness bound
    std::vector<int32_t> a = decode_operand(A, M, K, a_ms, a_ks);
    std::vector<int32_t> b = decode_operand(B, N, K, b_ns, b_ks);
    const int64_t Kd = g_plant == PLANT_GEMM_DROPS_LAST_K ? K - 1 : K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        const int32_t* ar = a.data() + size_t(m) * K;
        for (int64_t n = 0; n < N; ++n) {
            const int32_t* br = b.data() + size_t(n) * K;
            int64_t acc = 0;
            for (int64_t k = 0; k < Kd; ++k) acc += int64_t(ar[k]) * int64_t(br[k]);
            double v = std::ldexp(double(acc), -18) * double(sa) * double(sb);
            if (bias != nullptr) v = v + bf16_value(bias[n]);
            if (old != nullptr) v = bf16_value(old[m * N + n]) + v;
            out[m * N + n] = bf16_round(v);
        }
    }
    return 0;
}

// The unrounded value of the scaled FP8 matmul above (no bias, no old):
// exact[m, n] = (sum_k A(m, k) * B(n, k)) * 2^-18 * sa * sb in fp64.  Tests
// use it to bound how far a result computed with another summation order
// may lie from the exact value.
int orc_fp8_gemm_exact(const uint8_t* A, int64_t a_ms, int64_t a_ks, float sa, const uint8_t* B,
                       int64_t b_ns, int64_t b_ks, float sb, int64_t M, int64_t N, int64_t K, double* out) {
    if (K >= (int64_t(1) << 27)) return 1;
    std::vector<int32_t> a = decode_operand(A, M, K, a_ms, a_ks);
    std::vector<int32_t> b = decode_operand(B, N, K, b_ns, b_ks);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        const int32_t* ar = a.data() + size_t(m) * K;
        for (int64_t n = 0; n < N; ++n) {
            const int32_t* br = b.data() + size_t(n) * K;
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k) acc += int64_t(ar[k]) * int64_t(br[k]);
            out[m * N + n] = std::ldexp(double(acc), -18) * double(sa) * double(sb);
        }
    }
    return 0;
}

// ------------------------------------------------------------------ A4
// swiglu_forward [llmq-model: swiglu_forward(SwiGLu.Value, MlpUp,
// SwiGLu.Quant.abs_max(), B, T, D)]: h [N, H] from gu [N, 2H] (R1, R9, R10)
// and the abs-max of h.
void orc_swiglu(const uint16_t* gu, int64_t N, int64_t H, uint16_t* h, float* amax) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i) swiglu_row(gu + i * 2 * H, H, h + i * H);
    *amax = absmax_bf16(h, N * H);
}

// silu_mul [metrale-decode]: h = bf16(silu(g) * u).
void orc_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h) {
    for (int64_t j = 0; j < n; ++j) h[j] = bf16_round(silu(bf16_value(g[j])) * bf16_value(u[j]));
}

// swiglu_backward [llmq-model _backward_block: swiglu_backward(DMlpUp.Value,
// DSwiGLU, MlpUp, DMlpUp.Quant.abs_max(), B, T, D)], R21: d_gu [N, 2H] and
// its abs-max.
void orc_swiglu_backward(const uint16_t* dh, const uint16_t* gu, int64_t N, int64_t H, uint16_t* dgu,
                         float* amax) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i) {
        for (int64_t j = 0; j < H; ++j) {
            double g = bf16_value(gu[i * 2 * H + j]);
            double u = bf16_value(gu[i * 2 * H + H + j]);
            double d = bf16_value(dh[i * H + j]);
            double s = 1.0 / (1.0 + std::exp(-g));
            double corr = g_plant == PLANT_DSILU_NO_CORRECTION ? 1.0 : 1.0 + g * (1.0 - s);
            dgu[i * 2 * H + j] = bf16_round(d * u * s * corr);
            dgu[i * 2 * H + H + j] = bf16_round(d * (g * s));
        }
    }
    *amax = absmax_bf16(dgu, N * 2 * H);
}

// ------------------------------------------------------------------ A1..A5
// The prefill chain [llmq-model _forward_block, FFN half], the stats zeroed
// first (fill_zero(AbsMaxes)), so each abs-max is that of the tensor just
// produced.  w1 [2H, C], w2 [C, H] E4M3 with per-tensor scales.  Every
// intermediate is an output: r, y [N, C]; rstd [N]; stats_y[2]; yq [N, C];
// gu [N, 2H]; h [N, H]; stats_h[2]; hq [N, H]; out [N, C].  res may be NULL.
// *seconds (if not NULL) receives the steady-clock time of the whole chain.
int orc_ffn_forward(const uint16_t* res, const uint16_t* x, const uint16_t* gain, float eps,
                    const uint8_t* w1, float w1_scale, const uint8_t* w2, float w2_scale, int64_t N,
                    int64_t C, int64_t H, uint16_t* r, uint16_t* y, float* rstd, float* stats_y, uint8_t* yq,
                    uint16_t* gu, uint16_t* h, float* stats_h, uint8_t* hq, uint16_t* out, double* seconds) {
    auto t0 = std::chrono::steady_clock::now();
    orc_residual_rmsnorm_absmax(res, x, gain, eps, N, C, r, y, rstd, &stats_y[0]);
    orc_quantize_with_abs_max(y, N * C, stats_y[0], yq, &stats_y[1]);
    int rc = orc_fp8_gemm(yq, C, 1, stats_y[1], w1, C, 1, w1_scale, N, 2 * H, C, nullptr, nullptr, gu);
    orc_swiglu(gu, N, H, h, &stats_h[0]);
    orc_quantize_with_abs_max(h, N * H, stats_h[0], hq, &stats_h[1]);
    rc |= orc_fp8_gemm(hq, H, 1, stats_h[1], w2, H, 1, w2_scale, N, C, H, nullptr, nullptr, out);
    if (seconds) *seconds = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    return rc;
}

// The chain with both activation abs-maxes given [llmq-model _recompute_block,
// FFN half]: the norm re-run without recording, LN2 quantised with its stored
// abs-max, swiglu_forward_quant quantising h with the stored SwiGLU abs-max
// (values beyond it saturate, R8), then the forward's down projection.  Writes
// r, y, rstd, stats_y = {amax_y, scale}, yq, gu, hq, stats_h = {amax_h,
// scale}, out.
int orc_ffn_forward_recompute(const uint16_t* res, const uint16_t* x, const uint16_t* gain, float eps,
                              const uint8_t* w1, float w1_scale, const uint8_t* w2, float w2_scale,
                              int64_t N, int64_t C, int64_t H, float amax_y, float amax_h, uint16_t* r,
                              uint16_t* y, float* rstd, float* stats_y, uint8_t* yq, uint16_t* gu,
                              uint8_t* hq, float* stats_h, uint16_t* out) {
    float unused = 0.0f;
    orc_residual_rmsnorm_absmax(res, x, gain, eps, N, C, r, y, rstd, &unused);
    stats_y[0] = amax_y;
    orc_quantize_with_abs_max(y, N * C, amax_y, yq, &stats_y[1]);
    int rc = orc_fp8_gemm(yq, C, 1, stats_y[1], w1, C, 1, w1_scale, N, 2 * H, C, nullptr, nullptr, gu);
    std::vector<uint16_t> h(static_cast<size_t>(N * H));
    orc_swiglu(gu, N, H, h.data(), &unused);
    stats_h[0] = amax_h;
    orc_quantize_with_abs_max(h.data(), N * H, amax_h, hq, &stats_h[1]);
    rc |= orc_fp8_gemm(hq, H, 1, stats_h[1], w2, H, 1, w2_scale, N, C, H, nullptr, nullptr, out);
    return rc;
}

// The FP8 branch of backward_qmm [llmq-model] for one projection
// out = inp @ W^T, with dout [N, OC], inp_q [N, IC], W [OC, IC]:
// dout quantised with its recorded abs-max; dinp = dout_q @ W (reduction
// over the output channels) with dout.scale * W.scale; dW (+)= dout_q^T @
// inp_q (reduction over the tokens) with dout.scale * inp.scale.  dw_old may
// be NULL (no accumulation).  Writes dinp [N, IC], dw [OC, IC], dout_q and
// its scale.
int orc_backward_qmm(const uint16_t* dout, float dout_amax, const uint8_t* inp_q, float inp_scale,
                     const uint8_t* w, float w_scale, int64_t N, int64_t OC, int64_t IC,
                     const uint16_t* dw_old, uint16_t* dinp, uint16_t* dw, uint8_t* dout_q, float* dout_scale) {
    orc_quantize_with_abs_max(dout, N * OC, dout_amax, dout_q, dout_scale);
    // dinp(n, ic) = sum_oc dq(n, oc) * W(oc, ic): A = dq rows, B(ic, oc) = W[oc * IC + ic]
    int rc = orc_fp8_gemm(dout_q, OC, 1, *dout_scale, w, 1, IC, w_scale, N, IC, OC, nullptr, nullptr, dinp);
    // dW(oc, ic) = sum_n dq(n, oc) * inp(n, ic): A(oc, n) = dq[n * OC + oc], B(ic, n) = inp[n * IC + ic]
    rc |= orc_fp8_gemm(dout_q, 1, OC, *dout_scale, inp_q, 1, IC, inp_scale, OC, IC, N, nullptr, dw_old, dw);
    return rc;
}

// Backward of the FFN after the norm [llmq-model _backward_block, FFN half]:
// the down projection's backward_qmm (inp = the quantised SwiGLU output),
// the up projection's output recomputed from yq (as _recompute_block does),
// swiglu_backward, the up projection's backward_qmm (dout = d_gu with the
// abs-max swiglu_backward recorded, inp = the quantised LN2 output).
int orc_ffn_backward(const uint16_t* dout, float dout_amax, const uint8_t* yq, float y_scale,
                     const uint8_t* hq, float h_scale, const uint8_t* w1, float w1_scale, const uint8_t* w2,
                     float w2_scale, int64_t N, int64_t C, int64_t H, const uint16_t* dw1_old,
                     const uint16_t* dw2_old, uint16_t* dh, uint16_t* dw2, uint8_t* dout_q, float* stats_dout,
                     uint16_t* gu, uint16_t* d_gu, uint8_t* d_gu_q, float* stats_dgu, uint16_t* d_ln2,
                     uint16_t* dw1) {
    stats_dout[0] = dout_amax;
    int rc = orc_backward_qmm(dout, dout_amax, hq, h_scale, w2, w2_scale, N, C, H, dw2_old, dh, dw2, dout_q,
                              &stats_dout[1]);
    rc |= orc_fp8_gemm(yq, C, 1, y_scale, w1, C, 1, w1_scale, N, 2 * H, C, nullptr, nullptr, gu);
    orc_swiglu_backward(dh, gu, N, H, d_gu, &stats_dgu[0]);
    rc |= orc_backward_qmm(d_gu, stats_dgu[0], yq, y_scale, w1, w1_scale, N, 2 * H, C, dw1_old, d_ln2, dw1,
                           d_gu_q, &stats_dgu[1]);
    return rc;
}

// ------------------------------------------------------------------ A6..A8
// w8a16_gemv [metrale-decode]: out[r] = bf16(row_scale[r] * sum_k W[r, k] * x[k]),
// FP8 weight rows, bf16 input; the sum in fp64 (every product of an E4M3 and
// a bf16 value is exact in fp64) with compensation, the row scale applied to
// the finished sum (R14), one rounding.
void orc_gemv_row_scaled(const uint16_t* x, const uint8_t* w, const float* row_scale, int64_t R, int64_t K,
                         uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        CompSum acc;
        for (int64_t k = 0; k < K; ++k) acc.add(e4m3_value(w[r * K + k]) * bf16_value(x[k]));
        float s = g_plant == PLANT_GEMV_SCALE_BY_FIRST ? row_scale[0] : row_scale[r];
        out[r] = bf16_round(double(s) * acc.value());
    }
}

// The unrounded value of w8a16_gemv: row_scale[r] * sum_k W[r, k] * x[k] in
// fp64 (compensated sum), for the tests' error bounds.
void orc_gemv_exact(const uint16_t* x, const uint8_t* w, const float* row_scale, int64_t R, int64_t K,
                    double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        CompSum acc;
        for (int64_t k = 0; k < K; ++k) acc.add(e4m3_value(w[r * K + k]) * bf16_value(x[k]));
        out[r] = double(row_scale[r]) * acc.value();
    }
}

// The single-token FP8 decode FFN, split-SiLU arm [metrale-decode
// DenseFfnLayer::forward]: w8a16_gemv_dual (gate and up rows over the same
// x), silu_mul, w8a16_gemv of the down projection.  g, u, h [H], out [C].
void orc_decode_forward(const uint16_t* x, const uint8_t* wg, const float* sg, const uint8_t* wu,
                        const float* su, const uint8_t* wd, const float* sd, int64_t C, int64_t H, uint16_t* g,
                        uint16_t* u, uint16_t* h, uint16_t* out) {
    orc_gemv_row_scaled(x, wg, sg, H, C, g);
    orc_gemv_row_scaled(x, wu, su, H, C, u);
    orc_silu_mul(g, u, H, h);
    orc_gemv_row_scaled(h, wd, sd, C, H, out);
}

}  // extern "C"
