// CPU oracle for the group-wise affine-quantized multi-row matmul (qmm).
//
// TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
// CPU-baseline leg may load this library. The product path never calls it;
// it shares no code, header, table or helper with the CUDA library.
//
// What it computes (the plain definition, in float64):
//   W[n,k]  = s[n, k/group] * q[n,k] + b[n, k/group]
//   y[m,n]  = sum_k x[m,k] * W[n,k]          (k ascending)
// The method on the pages reaches the same value through the dequant-after-dot
// form  y = sum_g ( s*P + b*XS ),  P = sum_{k in g} x*q,  XS = sum_{k in g} x
// (vmlx-swift PR #565 "Enable bundle-aware Qwen speculation and dense mixed
// JANGH loading", LaneQMM commit: "C += s*P + b*XS"); that form is provided
// separately (oracle_qmm_spbxs_f64) so the tests can check the identity.
//
// Storage conventions the pages leave open (the plainest readings, shared by the workloads):
//   * codes q[n,k] are an LSB-first bit stream per row: bit j of code k is
//     bit (k*bits+j) mod 32 of word (k*bits+j) / 32 of that row; a row spans
//     K*bits/32 uint32 words and starts on a word boundary.
//   * scales / biases are IEEE binary16, row-major [N, K/group].
//   * activations are bfloat16 (the upper half of an IEEE binary32).
//
// Decoding is done twice, independently: a bit-at-a-time reader
// (oracle_decode_bitwise) and a word-wise shift/mask reader
// (oracle_decode_wordwise). The matmul uses the bit-at-a-time reader.
//
// Build: g++ -O2 -fopenmp -shared -fPIC (no -ffast-math: every sum is done in
// the written order).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// ---------------------------------------------------------------------------
// Scalar conversions, from the IEEE-754 format definitions.
// ---------------------------------------------------------------------------

// binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double oracle_f16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = std::ldexp((double)f, -24);               // subnormal: f * 2^-24
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = std::ldexp((double)(1024 + f), e - 25);   // (1 + f/1024) * 2^(e-15)
    }
    return sign ? -v : v;
}

// bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
double oracle_bf16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 7) & 0xFF;
    const int f = h & 0x7F;
    double v;
    if (e == 0) {
        v = std::ldexp((double)f, -133);              // subnormal: f * 2^-133
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = std::ldexp((double)(128 + f), e - 134);   // (1 + f/128) * 2^(e-127)
    }
    return sign ? -v : v;
}

void oracle_f16_to_f64_array(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(h[i]);
}

void oracle_bf16_to_f64_array(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(h[i]);
}

// ---------------------------------------------------------------------------
// Argument checks shared by every entry point of this file.
// ---------------------------------------------------------------------------
static int check_shape(int64_t K, int64_t N, int bits) {
    if (K <= 0 || N < 0) return 1;
    if (bits < 1 || bits > 8) return 1;
    if ((K * bits) % 32 != 0) return 1;   // every row starts on a word boundary
    return 0;
}

// ---------------------------------------------------------------------------
// Decoders.
// ---------------------------------------------------------------------------

// Bit-at-a-time reference reader: code k of row n collects stream bits
// k*bits .. k*bits+bits-1, least significant first.
static void decode_row_bitwise(const uint32_t* row, int64_t K, int bits, uint8_t* codes) {
    for (int64_t k = 0; k < K; ++k) {
        unsigned code = 0;
        for (int j = 0; j < bits; ++j) {
            const int64_t p = k * bits + j;             // absolute bit position
            const unsigned bit = (row[p / 32] >> (p % 32)) & 1u;
            code |= bit << j;
        }
        codes[k] = (uint8_t)code;
    }
}

int oracle_decode_bitwise(const uint32_t* words, int64_t N, int64_t K, int bits, uint8_t* codes) {
    if (check_shape(K, N, bits)) return 1;
    const int64_t wpr = K * bits / 32;
    for (int64_t n = 0; n < N; ++n) decode_row_bitwise(words + n * wpr, K, bits, codes + n * K);
    return 0;
}

// Word-wise reader: take the word holding the first bit, shift, and splice in
// the next word when the code straddles a word boundary.
int oracle_decode_wordwise(const uint32_t* words, int64_t N, int64_t K, int bits, uint8_t* codes) {
    if (check_shape(K, N, bits)) return 1;
    const int64_t wpr = K * bits / 32;
    const uint32_t mask = (bits == 32) ? 0xFFFFFFFFu : ((1u << bits) - 1u);
    for (int64_t n = 0; n < N; ++n) {
        const uint32_t* row = words + n * wpr;
        for (int64_t k = 0; k < K; ++k) {
            const int64_t p = k * bits;
            const int64_t w = p / 32;
            const int o = (int)(p % 32);
            uint32_t v = row[w] >> o;
            if (o + bits > 32) v |= row[w + 1] << (32 - o);
            codes[n * K + k] = (uint8_t)(v & mask);
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Dequantization:  W[n,k] = s[n,g] * q[n,k] + b[n,g],  g = k / group.
// ---------------------------------------------------------------------------
static int check_qmm(int64_t M, int64_t K, int64_t N, int bits, int group) {
    if (M < 0) return 1;
    if (check_shape(K, N, bits)) return 1;
    if (group <= 0 || K % group != 0) return 1;
    return 0;
}

static void dequant_row(const uint32_t* row, const uint16_t* srow, const uint16_t* brow,
                        int64_t K, int bits, int group, uint8_t* codes, double* w) {
    decode_row_bitwise(row, K, bits, codes);
    for (int64_t k = 0; k < K; ++k) {
        const int64_t g = k / group;
        const double s = oracle_f16_to_f64(srow[g]);
        const double b = oracle_f16_to_f64(brow[g]);
        w[k] = s * (double)codes[k] + b;
    }
}

int oracle_dequant_f64(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                       int64_t K, int64_t N, int bits, int group, double* W) {
    if (check_qmm(0, K, N, bits, group)) return 1;
    const int64_t wpr = K * bits / 32;
    const int64_t G = K / group;
    std::vector<uint8_t> codes((size_t)K);
    for (int64_t n = 0; n < N; ++n)
        dequant_row(words + n * wpr, scales + n * G, biases + n * G, K, bits, group,
                    codes.data(), W + n * K);
    return 0;
}

// ---------------------------------------------------------------------------
// The oracle proper: dequantize row n in float64, then a naive dot product with
// every x row, k ascending. Columns listed in `cols` (ncols of them) are
// computed; cols == nullptr means all N columns. y is [M, ncols] row-major.
// Parallel over columns only; every column's arithmetic is sequential.
// ---------------------------------------------------------------------------
int oracle_qmm_f64_cols(const uint16_t* x_bf16, int64_t M, const uint32_t* words,
                        const uint16_t* scales, const uint16_t* biases, int64_t K, int64_t N,
                        int bits, int group, const int64_t* cols, int64_t ncols, double* y) {
    if (check_qmm(M, K, N, bits, group)) return 1;
    if (cols == nullptr) ncols = N;
    for (int64_t c = 0; cols && c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N) return 1;
    const int64_t wpr = K * bits / 32;
    const int64_t G = K / group;

    std::vector<double> xd((size_t)(M * K));
    for (int64_t i = 0; i < M * K; ++i) xd[(size_t)i] = oracle_bf16_to_f64(x_bf16[i]);

#pragma omp parallel
    {
        std::vector<uint8_t> codes((size_t)K);
        std::vector<double> w((size_t)K);
        std::vector<double> acc((size_t)(M > 0 ? M : 1));
#pragma omp for schedule(static)
        for (int64_t c = 0; c < ncols; ++c) {
            const int64_t n = cols ? cols[c] : c;
            dequant_row(words + n * wpr, scales + n * G, biases + n * G, K, bits, group,
                        codes.data(), w.data());
            for (int64_t m = 0; m < M; ++m) acc[(size_t)m] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double wk = w[(size_t)k];
                for (int64_t m = 0; m < M; ++m) acc[(size_t)m] += xd[(size_t)(m * K + k)] * wk;
            }
            for (int64_t m = 0; m < M; ++m) y[m * ncols + c] = acc[(size_t)m];
        }
    }
    return 0;
}

int oracle_qmm_f64(const uint16_t* x_bf16, int64_t M, const uint32_t* words,
                   const uint16_t* scales, const uint16_t* biases, int64_t K, int64_t N,
                   int bits, int group, double* y) {
    return oracle_qmm_f64_cols(x_bf16, M, words, scales, biases, K, N, bits, group, nullptr, N, y);
}

// ---------------------------------------------------------------------------
// The pages' dequant-after-dot form, in float64:
//   P[m,n,g]  = sum_{k in g} x[m,k] * q[n,k]
//   XS[m,g]   = sum_{k in g} x[m,k]
//   y[m,n]    = sum_g ( s[n,g] * P[m,n,g] + b[n,g] * XS[m,g] )
// Used only to check that this form and the definition above agree.
// ---------------------------------------------------------------------------
int oracle_qmm_spbxs_f64(const uint16_t* x_bf16, int64_t M, const uint32_t* words,
                         const uint16_t* scales, const uint16_t* biases, int64_t K, int64_t N,
                         int bits, int group, double* y) {
    if (check_qmm(M, K, N, bits, group)) return 1;
    const int64_t wpr = K * bits / 32;
    const int64_t G = K / group;

    std::vector<double> xd((size_t)(M * K));
    for (int64_t i = 0; i < M * K; ++i) xd[(size_t)i] = oracle_bf16_to_f64(x_bf16[i]);
    std::vector<double> XS((size_t)(M * G), 0.0);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t g = 0; g < G; ++g) {
            double s = 0.0;
            for (int64_t k = g * group; k < (g + 1) * group; ++k) s += xd[(size_t)(m * K + k)];
            XS[(size_t)(m * G + g)] = s;
        }

#pragma omp parallel
    {
        std::vector<uint8_t> codes((size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            decode_row_bitwise(words + n * wpr, K, bits, codes.data());
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0;
                for (int64_t g = 0; g < G; ++g) {
                    double P = 0.0;
                    for (int64_t k = g * group; k < (g + 1) * group; ++k)
                        P += xd[(size_t)(m * K + k)] * (double)codes[(size_t)k];
                    const double s = oracle_f16_to_f64(scales[n * G + g]);
                    const double b = oracle_f16_to_f64(biases[n * G + g]);
                    acc += s * P + b * XS[(size_t)(m * G + g)];
                }
                y[m * N + n] = acc;
            }
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Fused gate/up projection with a SwiGLU epilogue ("Qwen3.8 Flash Next
// performance and parity receipt": the exact fused projection promoted over
// separate gate and up projections):
//   y[m,n] = silu(g[m,n]) * u[m,n],   silu(v) = v / (1 + exp(-v)),
// g and u being the plain-definition results above for the gate weights and
// the up weights on the same x.
// ---------------------------------------------------------------------------
int oracle_qmm_swiglu_f64(const uint16_t* x_bf16, int64_t M, const uint32_t* words_gate,
                          const uint16_t* scales_gate, const uint16_t* biases_gate, const uint32_t* words_up,
                          const uint16_t* scales_up, const uint16_t* biases_up, int64_t K, int64_t N, int bits,
                          int group, double* y) {
    if (check_qmm(M, K, N, bits, group)) return 1;
    std::vector<double> g((size_t)(M * N)), u((size_t)(M * N));
    if (oracle_qmm_f64(x_bf16, M, words_gate, scales_gate, biases_gate, K, N, bits, group, g.data())) return 1;
    if (oracle_qmm_f64(x_bf16, M, words_up, scales_up, biases_up, K, N, bits, group, u.data())) return 1;
    for (int64_t i = 0; i < M * N; ++i) {
        const double v = g[(size_t)i];
        y[i] = v / (1.0 + std::exp(-v)) * u[(size_t)i];
    }
    return 0;
}

// The same for the listed output columns only (ncols of them; y is [M, ncols]),
// from the column-subset form of the plain definition.
int oracle_qmm_swiglu_f64_cols(const uint16_t* x_bf16, int64_t M, const uint32_t* words_gate,
                               const uint16_t* scales_gate, const uint16_t* biases_gate,
                               const uint32_t* words_up, const uint16_t* scales_up, const uint16_t* biases_up,
                               int64_t K, int64_t N, int bits, int group, const int64_t* cols, int64_t ncols,
                               double* y) {
    if (check_qmm(M, K, N, bits, group) || cols == nullptr || ncols < 0) return 1;
    std::vector<double> g((size_t)(M * ncols)), u((size_t)(M * ncols));
    if (oracle_qmm_f64_cols(x_bf16, M, words_gate, scales_gate, biases_gate, K, N, bits, group, cols, ncols,
                            g.data()))
        return 1;
    if (oracle_qmm_f64_cols(x_bf16, M, words_up, scales_up, biases_up, K, N, bits, group, cols, ncols, u.data()))
        return 1;
    for (int64_t i = 0; i < M * ncols; ++i) {
        const double v = g[(size_t)i];
        y[i] = v / (1.0 + std::exp(-v)) * u[(size_t)i];
    }
    return 0;
}

// Number of threads the parallel regions above use (for reporting).
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

}  // extern "C"
