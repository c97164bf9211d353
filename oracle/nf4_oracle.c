/*
 * nf4_oracle.c -- plain CPU oracle for NF4 weight-only quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file.  It may be used by the tests, by the smoke check and by
 * the benchmark's CPU-baseline leg, and by nothing else.  It shares no code,
 * header, table or constant with the CUDA library: the codebook below is typed
 * here a second time on purpose.
 *
 * What it computes (the source page is the diffuseR pull request "Gemma3 NF4
 * on GPU: quantized encoder, batch encoding, byte-LUT eager dequant", #39,
 * Summary paragraph): the seven projection weights of every Gemma3 layer are
 * packed to NF4 while activations stay at the compute dtype (bf16), and the
 * eager forward dequantizes them and runs a dense matmul.  The page prints
 * neither the codebook, the block size, the scale dtype nor the nibble order.
 * The readings used here:
 *
 *   - codebook: the 16-value NormalFloat-4 table of QLoRA (Dettmers et al.
 *     2023, arXiv:2305.14314, appendix), stored as fp32 constants;
 *   - blocks of 64 consecutive elements of the row-major flattened weight,
 *     one fp32 absmax per block, no double quantization; a partial last block
 *     uses the elements it has;
 *   - code = the codebook index nearest to w / absmax (fp32 IEEE division),
 *     distances compared in fp64, ties to the lower index; an all-zero block
 *     gets absmax +0 and code 7 (value 0) everywhere;
 *   - packing: element 2j in the high nibble of byte j, element 2j+1 in the
 *     low nibble;
 *   - dequant by nibble unpack (not a lookup table):
 *     y = bf16_rne( float(bf16_rne(C[code])) * absmax ), one fp32 multiply;
 *   - other compute dtypes (the unquantized tensors stay in the compute dtype):
 *     fp16 the same with binary16 in place of bf16; fp32 without roundings,
 *     y = C[code] * absmax in fp32; quantize reads the dtype's values exactly;
 *   - linear: Y[m][n] = sum_k X[m][k] * Wdeq[n][k], accumulated in fp64;
 *   - gate/up pair (the Gemma3 MLP): gelu_tanh(gate) * up of two linears
 *     whose weights are stacked into one [2F, K] tensor, in fp64.
 *
 * Every loop below is the definition written out, one element at a time.
 * OpenMP splits only the outermost independent loop (blocks or rows); it
 * changes no arithmetic and no summation order.
 *
 * Parity pins for every exported function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* NormalFloat-4 codebook, QLoRA appendix, ascending. */
static const float ORACLE_NF4[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

/* ---- bf16 <-> fp32 from the IEEE bit layout ----------------------------- */

/* A bf16 value is the upper 16 bits of the fp32 with the same value. */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 to the nearest bf16, ties to even.  NaN maps to a quiet NaN
 * with the sign kept.  Overflow rounds to infinity as IEEE prescribes. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* ---- fp16 <-> fp32 from the IEEE binary16 layout ------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 * exponent 0 holds zero and the subnormals (fraction * 2^-24), exponent 31
 * infinity and NaN. */
static float f16_to_f32(uint16_t h) {
    int e = (h >> 10) & 0x1f, m = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m | 0x400), e - 25);
    return (h & 0x8000u) ? -v : v;
}

/* Round an fp32 to the nearest binary16, ties to even: the value's quantum is
 * 2^-24 below 2^-14 (subnormals) and 2^(e - 10) in [2^e, 2^(e+1)) above;
 * rint() rounds the scaled value (exact in fp64) to an integer with ties to
 * even; 65520 and above round to infinity; NaN maps to a quiet NaN. */
static uint16_t f32_to_f16_rne(float f) {
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return sign | 0x7e00u;
    if (isinf(f)) return sign | 0x7c00u;
    double v = fabs((double)f);
    if (v == 0.0) return sign;
    int e2;
    frexp(v, &e2);                                  /* v in [2^(e2-1), 2^e2) */
    int qexp = (e2 - 1 < -14) ? -24 : (e2 - 1) - 10;
    double n = rint(ldexp(v, -qexp));
    double r = ldexp(n, qexp);
    if (r >= 65536.0) return sign | 0x7c00u;
    if (r < ldexp(1.0, -14)) return sign | (uint16_t)n;   /* subnormal: the fraction is n */
    frexp(r, &e2);
    int e = e2 - 1;
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)(ldexp(r, 10 - e) - 1024.0);
}

/* ---- element types ------------------------------------------------------ */

/* The compute dtype of weights, activations and outputs.  The page keeps the
 * tensors it does not quantize in the compute dtype, bf16 in its encoder
 * runs; fp16 and fp32 are the other floating types that dtype can take. */
enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F32 = 2 };

static float load_f32(const void* p, int dt, int64_t i) {
    if (dt == ORACLE_BF16) return bf16_to_f32(((const uint16_t*)p)[i]);
    if (dt == ORACLE_F16) return f16_to_f32(((const uint16_t*)p)[i]);
    return ((const float*)p)[i];
}

/* Store v rounded to nearest even in the element type. */
static void store_rne(void* p, int dt, int64_t i, float v) {
    if (dt == ORACLE_BF16)
        ((uint16_t*)p)[i] = f32_to_bf16_rne(v);
    else if (dt == ORACLE_F16)
        ((uint16_t*)p)[i] = f32_to_f16_rne(v);
    else
        ((float*)p)[i] = v;
}

/* Codebook value k as held in the element type (the lookup table holds
 * output-dtype values), widened back to fp32. */
static float code_value(int dt, int k) {
    if (dt == ORACLE_BF16) return bf16_to_f32(f32_to_bf16_rne(ORACLE_NF4[k]));
    if (dt == ORACLE_F16) return f16_to_f32(f32_to_f16_rne(ORACLE_NF4[k]));
    return ORACLE_NF4[k];
}

static size_t elem_size(int dt) { return dt == ORACLE_F32 ? 4 : 2; }

/* ---- exported ----------------------------------------------------------- */

const float* oracle_codebook(void) { return ORACLE_NF4; }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
uint16_t oracle_f32_to_f16(float f) { return f32_to_f16_rne(f); }
float oracle_f16_to_f32(uint16_t h) { return f16_to_f32(h); }

void oracle_f32_to_f16_array(const float* f, int64_t count, uint16_t* h) {
    for (int64_t i = 0; i < count; ++i) h[i] = f32_to_f16_rne(f[i]);
}

void oracle_f16_to_f32_array(const uint16_t* h, int64_t count, float* f) {
    for (int64_t i = 0; i < count; ++i) f[i] = f16_to_f32(h[i]);
}

/* Index of the codebook value nearest to n; fp64 distances, the first
 * (lowest) index wins a tie. */
static int nearest_code(float n) {
    int best = 0;
    double best_d = fabs((double)n - (double)ORACLE_NF4[0]);
    for (int k = 1; k < 16; ++k) {
        double d = fabs((double)n - (double)ORACLE_NF4[k]);
        if (d < best_d) {
            best_d = d;
            best = k;
        }
    }
    return best;
}

/* Code selection alone, exposed so that the tests can sweep normalised
 * values directly. */
void oracle_nearest_code(const float* n, int64_t count, uint8_t* code) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) code[i] = (uint8_t)nearest_code(n[i]);
}

/* Blockwise absmax quantization of a tensor of `numel` elements of type dt
 * (numel even) into numel/2 packed bytes and ceil(numel/block) fp32 scales. */
void oracle_quantize_dt(const void* w, int dt, int64_t numel, int32_t block, uint8_t* packed,
                        float* absmax) {
    int64_t nblocks = (numel + block - 1) / block;
    uint8_t* codes = (uint8_t*)malloc((size_t)numel);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        int64_t lo = b * block;
        int64_t hi = lo + block < numel ? lo + block : numel;
        float am = 0.0f;
        for (int64_t i = lo; i < hi; ++i) {
            float a = fabsf(load_f32(w, dt, i));
            if (a > am) am = a;
        }
        absmax[b] = am;
        for (int64_t i = lo; i < hi; ++i) {
            if (am == 0.0f) {
                codes[i] = 7;
            } else {
                float n = load_f32(w, dt, i) / am;
                codes[i] = (uint8_t)nearest_code(n);
            }
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < numel / 2; ++j)
        packed[j] = (uint8_t)((codes[2 * j] << 4) | codes[2 * j + 1]);
    free(codes);
}

void oracle_quantize(const uint16_t* w, int64_t numel, int32_t block, uint8_t* packed,
                     float* absmax) {
    oracle_quantize_dt(w, ORACLE_BF16, numel, block, packed, absmax);
}

/* Dequantize by unpacking each nibble and scaling its codebook value (as held
 * in the output type dt) by the block absmax with one fp32 multiply, then
 * rounding once to dt. */
void oracle_dequantize_dt(const uint8_t* packed, const float* absmax, int64_t numel, int32_t block,
                          int dt, void* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < numel; ++i) {
        uint8_t byte = packed[i / 2];
        int code = (i % 2 == 0) ? (byte >> 4) : (byte & 0x0f);
        float y = code_value(dt, code) * absmax[i / block];
        store_rne(out, dt, i, y);
    }
}

void oracle_dequantize(const uint8_t* packed, const float* absmax, int64_t numel, int32_t block,
                       uint16_t* out) {
    oracle_dequantize_dt(packed, absmax, numel, block, ORACLE_BF16, out);
}

/* Y[M][N] = X[M][K] . Wdeq[N][K]^T in fp64, W given as NF4 (packed, absmax)
 * over the flattened [N][K] weight and dequantized to dt; X is dt,
 * row-major. */
void oracle_linear_dt(const void* x, int dt, int64_t M, int64_t K, const uint8_t* packed,
                      const float* absmax, int64_t N, int32_t block, double* y) {
    void* wq = malloc((size_t)(N * K) * elem_size(dt));
    oracle_dequantize_dt(packed, absmax, N * K, block, dt, wq);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)load_f32(x, dt, m * K + k) * (double)load_f32(wq, dt, n * K + k);
            y[m * N + n] = acc;
        }
    }
    free(wq);
}

void oracle_linear(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                   const float* absmax, int64_t N, int32_t block, double* y) {
    oracle_linear_dt(x, ORACLE_BF16, M, K, packed, absmax, N, block, y);
}

/* ---- gate/up projection pair with the GELU gate ------------------------- */

/* GELU in its tanh form (Hendrycks and Gimpel, "Gaussian Error Linear Units
 * (GELUs)", arXiv:1606.08415, section 2), the activation between the gate and
 * up projections of the Gemma3 MLP:
 *   gelu(x) = x/2 * (1 + tanh( sqrt(2/pi) * (x + 0.044715 x^3) )),
 * evaluated in fp64. */
static double gelu_tanh(double x) {
    const double k = sqrt(2.0 / acos(-1.0));
    return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
}

void oracle_gelu_tanh(const double* x, int64_t count, double* y) {
    for (int64_t i = 0; i < count; ++i) y[i] = gelu_tanh(x[i]);
}

/* GeGLU of the gate and up projections held as ONE weight: W [2F][K] is the
 * gate weight (rows 0 .. F-1) followed by the up weight (rows F .. 2F-1),
 * quantized as one tensor.  With G = X . Wdeq^T [M][2F] from oracle_linear,
 *   out[m][n] = gelu(G[m][n]) * G[m][F + n],   n < F,
 * all in fp64. */
void oracle_linear_geglu_dt(const void* x, int dt, int64_t M, int64_t K, const uint8_t* packed,
                            const float* absmax, int64_t F, int32_t block, double* out) {
    double* g = (double*)malloc((size_t)(M * 2 * F) * sizeof(double));
    oracle_linear_dt(x, dt, M, K, packed, absmax, 2 * F, block, g);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < F; ++n)
            out[m * F + n] = gelu_tanh(g[m * 2 * F + n]) * g[m * 2 * F + F + n];
    free(g);
}

void oracle_linear_geglu(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                         const float* absmax, int64_t F, int32_t block, double* out) {
    oracle_linear_geglu_dt(x, ORACLE_BF16, M, K, packed, absmax, F, block, out);
}
