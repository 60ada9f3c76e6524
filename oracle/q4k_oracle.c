/*
 * CPU ORACLE for the Q4_K x M-row weight-streaming matmul -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may call this
 * code.  It shares no code, header, table or helper with the CUDA path.  It is the plain
 * definition of what that path computes, written for a reader to check by eye:
 *
 *   y[m, n] = sum_k w[n, k] * x[m, k],   w[n, k] = d * sc_j * q - dmin * m_j,
 *
 * where (d, dmin, sc_j, m_j, q) come from the 144-byte super-block that holds weight
 * (n, k).  Sources:
 *  - Page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for Qwen3.8-27B"
 *    (molayo1419.me), section "How parallel decoding works": the M stacked rows are each
 *    multiplied against every weight, so the result is an ordinary matmul y = x W^T.
 *  - Same page, section "Accuracy": outputs differ from other engines in the last bits
 *    because the arithmetic order differs, so parity is a tolerance, not byte equality.
 *  - The model file format the pages name, Q4_K_M: the GGUF Q4_K super-block.  Byte order
 *    and bit packing below are that format's convention (readings, listed with the design
 *    notes):  bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15 scales s[0..11], 16-143 qs[0..127].
 *      j = 0..3:  sc_j = s[j] & 63,                       m_j = s[j+4] & 63
 *      j = 4..7:  sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),
 *                 m_j  = (s[j+4] >> 4) | ((s[j] >> 6) << 4)
 *      weight i of the block (i = 0..255): chunk c = i / 64, r = i % 64;
 *                 q = low nibble of qs[32c + r] if r < 32, else high nibble of qs[32c + r - 32];
 *                 its sub-block is j = i / 32.
 *
 * Precision: dequantisation in fp32 (d*sc and dmin*m are exact in fp32; a*q - c rounds
 * once), accumulation in double in increasing k.  The abs-sum S[m, n] = sum_k |w x| is
 * returned alongside for the tolerance |y_gpu - y| <= 2e-3 * S + 1e-6.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE binary16 bit pattern -> double (exact: every fp16 value is a double). */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* The 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes. */
void oracle_scale_min(const uint8_t s[12], int j, int* sc, int* mn) {
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* The 4-bit quant of weight i (0..255) of a block. */
int oracle_quant(const uint8_t qs[128], int i) {
    int c = i / 64, r = i % 64;
    return r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
}

/* Dequantise one 144-byte super-block to 256 fp32 weights. */
void oracle_dequant_block(const uint8_t* blk, float* w) {
    float d = (float)oracle_f16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    float dmin = (float)oracle_f16_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t* s = blk + 4;
    const uint8_t* qs = blk + 16;
    for (int j = 0; j < 8; ++j) {
        int sc, mn;
        oracle_scale_min(s, j, &sc, &mn);
        float a = d * (float)sc;      /* exact in fp32 */
        float c = dmin * (float)mn;   /* exact in fp32 */
        for (int i = 32 * j; i < 32 * j + 32; ++i) {
            float q = (float)oracle_quant(qs, i);
            w[i] = a * q - c;
        }
    }
}

/*
 * y[m*N + n] = sum_k w[n,k] x[m,k] (double), s_abs[m*N + n] = sum_k |w[n,k] x[m,k]|.
 * blocks: N rows of K/256 blocks (row-major, GGUF order); x: M*K fp16 bit patterns.
 * s_abs may be NULL.  nthreads <= 0 uses the OpenMP default.  Returns 0, or -1 on a
 * bad shape or allocation failure.
 */
int oracle_qmm(const uint8_t* blocks, int64_t N, int64_t K, const uint16_t* x, int64_t M,
               double* y, double* s_abs, int nthreads) {
    if (N < 0 || M < 0 || K < 0 || K % 256 != 0) return -1;
    int64_t kb = K / 256;
    double* xd = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -1;
    for (int64_t i = 0; i < M * K; ++i) xd[i] = oracle_f16_to_double(x[i]);
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        float* w = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
        if (!w) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
            for (int64_t n = 0; n < N; ++n) {
                for (int64_t b = 0; b < kb; ++b)
                    oracle_dequant_block(blocks + (n * kb + b) * 144, w + b * 256);
                for (int64_t m = 0; m < M; ++m) {
                    const double* xr = xd + m * K;
                    double acc = 0.0, sabs = 0.0;
                    for (int64_t k = 0; k < K; ++k) {
                        double p = (double)w[k] * xr[k];
                        acc += p;
                        sabs += fabs(p);
                    }
                    y[m * N + n] = acc;
                    if (s_abs) s_abs[m * N + n] = sabs;
                }
            }
            free(w);
        }
    }
    free(xd);
    return failed ? -1 : 0;
}

/*
 * Other block formats of a mixed-quant model file (page "Running 4 coding agents on one RTX
 * 3090", the note on mixed-quant builds; page "Breaking the limits of Qwen3.8-27B again",
 * the int8 weights of its lm_head).  Their byte layouts are the GGUF conventions (readings,
 * listed with the design notes); each weight is computed exactly in double:
 *
 * Q8_0: 34-byte blocks of 32 weights: bytes 0-1 d (fp16), 2-33 q[0..31] (int8);
 *       weight i = d * q[i].
 * Q6_K: 210-byte super-blocks of 256 weights: bytes 0-127 ql, 128-191 qh, 192-207 sc[0..15]
 *       (int8), 208-209 d (fp16).  Weight i: h = i / 128, c = (i % 128) / 32, l = i % 32;
 *       low 4 bits = (ql[64h + l + 32 (c & 1)] >> (4 (c >> 1))) & 15, high 2 bits =
 *       (qh[32h + l] >> (2c)) & 3, q = low | high << 4 (0..63), sub-block j = i / 16;
 *       weight i = d * sc[j] * (q - 32).
 */
enum { ORACLE_Q4_K = 0, ORACLE_Q6_K = 1, ORACLE_Q8_0 = 2 };

static void dequant_q8_0(const uint8_t* blk, double* w) {
    double d = oracle_f16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int i = 0; i < 32; ++i) w[i] = d * (double)(int8_t)blk[2 + i];
}

/* The 6-bit quant of weight i (0..255) of a Q6_K block. */
int oracle_q6k_quant(const uint8_t* blk, int i) {
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    int h = i / 128, c = (i % 128) / 32, l = i % 32;
    int lo = (ql[64 * h + l + 32 * (c & 1)] >> (4 * (c >> 1))) & 15;
    int hi = (qh[32 * h + l] >> (2 * c)) & 3;
    return lo | (hi << 4);
}

static void dequant_q6_k(const uint8_t* blk, double* w) {
    double d = oracle_f16_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
    const int8_t* sc = (const int8_t*)(blk + 192);
    for (int i = 0; i < 256; ++i) w[i] = d * (double)sc[i / 16] * (double)(oracle_q6k_quant(blk, i) - 32);
}

/*
 * oracle_qmm for any of the three formats.  blocks: N rows of K / (weights per block)
 * blocks in GGUF order (Q4_K 144 B / 256 weights, Q6_K 210 B / 256, Q8_0 34 B / 32).
 * Q4_K goes through oracle_qmm above; the others dequantise a row in double and
 * accumulate in double in increasing k.
 */
int oracle_qmm_fmt(int fmt, const uint8_t* blocks, int64_t N, int64_t K, const uint16_t* x, int64_t M,
                   double* y, double* s_abs, int nthreads) {
    if (fmt == ORACLE_Q4_K) return oracle_qmm(blocks, N, K, x, M, y, s_abs, nthreads);
    int per = fmt == ORACLE_Q6_K ? 256 : fmt == ORACLE_Q8_0 ? 32 : 0;
    int bytes = fmt == ORACLE_Q6_K ? 210 : 34;
    if (!per || N < 0 || M < 0 || K < 0 || K % per != 0) return -1;
    int64_t nb = K / per;
    double* xd = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -1;
    for (int64_t i = 0; i < M * K; ++i) xd[i] = oracle_f16_to_double(x[i]);
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!w) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
            for (int64_t n = 0; n < N; ++n) {
                for (int64_t b = 0; b < nb; ++b) {
                    const uint8_t* blk = blocks + (n * nb + b) * bytes;
                    if (fmt == ORACLE_Q6_K) dequant_q6_k(blk, w + b * per);
                    else dequant_q8_0(blk, w + b * per);
                }
                for (int64_t m = 0; m < M; ++m) {
                    const double* xrow = xd + m * K;
                    double sum = 0.0, sum_abs = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) {
                        double prod = w[kk] * xrow[kk];
                        sum += prod;
                        sum_abs += fabs(prod);
                    }
                    y[m * N + n] = sum;
                    if (s_abs) s_abs[m * N + n] = sum_abs;
                }
            }
            free(w);
        }
    }
    free(xd);
    return failed ? -1 : 0;
}

/* Dequantise one block of format fmt (256 weights for Q4_K / Q6_K, 32 for Q8_0) to double. */
int oracle_dequant_fmt(int fmt, const uint8_t* blk, double* w) {
    if (fmt == ORACLE_Q4_K) {
        float wf[256];
        oracle_dequant_block(blk, wf);
        for (int i = 0; i < 256; ++i) w[i] = wf[i];
        return 256;
    }
    if (fmt == ORACLE_Q6_K) {
        dequant_q6_k(blk, w);
        return 256;
    }
    if (fmt == ORACLE_Q8_0) {
        dequant_q8_0(blk, w);
        return 32;
    }
    return -1;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
