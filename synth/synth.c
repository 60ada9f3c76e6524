/*
 * Seeded synthetic inputs for the Q4_K x M-row weight-streaming matmul.
 *
 * This module only draws random bytes and rounds random reals to fp16.  It holds
 * none of the matmul's arithmetic (no scale unpacking, no dequantisation, no dot
 * products), so that the CPU oracle and the CUDA path can both be fed from it
 * without sharing any of the method's code.
 *
 * Generator: a counter-based SplitMix64.  Value number i of stream `key` is
 * mix64(key + (i + 1) * 0x9E3779B97F4A7C15), where mix64 is the SplitMix64
 * finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014).  Every output is a pure function of
 * (seed, tensor_id, index), so any block or row can be regenerated on its own.
 *
 * Workload value distributions (a single projection in the Q4_K-style layout):
 *   quants uniform on 0..15, 6-bit scales and mins uniform on 0..63,
 *   d and dmin = fp16(|N(0,1)| * 1e-3), activations fp16(N(0,1)),
 *   optional outliers: each activation independently, with probability p,
 *   is multiplied by a factor before the fp16 rounding.
 * The 12 scale bytes pack 16 six-bit values into 96 bits with every bit used once,
 * so uniform random bytes give uniform, independent scales and mins; likewise
 * uniform quant bytes give uniform 4-bit quants.  The generator therefore draws
 * raw bytes for bytes 4..143 of each 144-byte super-block.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Stream key for one tensor of one seed. */
uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(mix64(seed + GOLDEN) ^ (tensor_id * 0xD1B54A32D192ED03ULL + 0x8CB92BA72F3D8DD7ULL));
}

static inline uint64_t ctr_rand(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* Uniform double in the open interval (0, 1): 53 random bits, centred in their cell. */
static inline double u01(uint64_t r) { return ((double)(r >> 11) + 0.5) * 0x1p-53; }

/* Round a double to IEEE binary16, round-to-nearest-even, with subnormals and
 * overflow to infinity.  Returns the 16-bit pattern. */
uint16_t synth_f16_from_double(double v) {
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(a)) return (uint16_t)(sign | 0x7E00u);
    /* 65520 is the midpoint between 65504 (largest finite) and 65536; ties go to even (inf). */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < 0x1p-14) {
        /* subnormal range: value = m * 2^-24 with m in [0, 1024]; m = 1024 is the smallest normal */
        double m = nearbyint(a * 0x1p24);
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e;
    double f = frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    double m = nearbyint((2.0 * f - 1.0) * 1024.0);
    int e16 = e - 1 + 15;
    if (m == 1024.0) { m = 0.0; e16 += 1; }
    if (e16 >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint16_t)e16 << 10) | (uint16_t)m);
}

/* Two standard normals from two uniforms (Box-Muller, 1958). */
static inline void box_muller(uint64_t r0, uint64_t r1, double* z0, double* z1) {
    double rad = sqrt(-2.0 * log(u01(r0)));
    double th = 6.283185307179586476925286766559 * u01(r1);
    *z0 = rad * cos(th);
    *z1 = rad * sin(th);
}

#define WORDS_PER_BLOCK 20   /* 18 words -> 144 raw bytes (140 used), 2 words -> d, dmin */

/*
 * Fill `nblocks` 144-byte super-blocks, blocks first_block .. first_block+nblocks-1 of
 * tensor (seed, tensor_id).  Layout of each block: bytes 0-1 d (fp16, little-endian),
 * 2-3 dmin, 4-15 packed scales/mins, 16-143 quants.
 * scale_mul multiplies |N(0,1)| before rounding d and dmin (1e-3 for the workloads).
 */
void synth_q4k_blocks(uint8_t* out, int64_t nblocks, uint64_t seed, uint64_t tensor_id,
                      int64_t first_block, double scale_mul) {
    uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(first_block + b) * WORDS_PER_BLOCK;
        uint8_t raw[144];
        for (int w = 0; w < 18; ++w) {
            uint64_t r = ctr_rand(key, base + (uint64_t)w);
            for (int i = 0; i < 8; ++i) raw[8 * w + i] = (uint8_t)(r >> (8 * i));
        }
        double z0, z1;
        box_muller(ctr_rand(key, base + 18), ctr_rand(key, base + 19), &z0, &z1);
        uint16_t d = synth_f16_from_double(fabs(z0) * scale_mul);
        uint16_t dmin = synth_f16_from_double(fabs(z1) * scale_mul);
        uint8_t* blk = out + 144 * b;
        blk[0] = (uint8_t)(d & 0xFF);
        blk[1] = (uint8_t)(d >> 8);
        blk[2] = (uint8_t)(dmin & 0xFF);
        blk[3] = (uint8_t)(dmin >> 8);
        memcpy(blk + 4, raw, 140);
    }
}

/*
 * Fill `nblocks` blocks of another GGUF block type, blocks first_block ..
 * first_block+nblocks-1 of tensor (seed, tensor_id): every byte random from the counter
 * stream, then the fp16 scale field(s) overwritten with fp16(|N(0,1)| * scale_mul).
 *   bytes = 34  (Q8_0): d at bytes 0-1, 32 int8 quants.
 *   bytes = 210 (Q6_K): d at bytes 208-209; ql, qh and the 16 int8 scales random.
 * Each block draws from its own range of 32 counter values.
 */
void synth_blocks(uint8_t* out, int64_t nblocks, int64_t bytes, uint64_t seed, uint64_t tensor_id,
                  int64_t first_block, double scale_mul) {
    uint64_t key = synth_key(seed, tensor_id);
    const int d_off = bytes == 34 ? 0 : (int)bytes - 2;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(first_block + b) * 32;
        uint8_t* blk = out + bytes * b;
        for (int64_t i = 0; i < bytes; i += 8) {
            uint64_t r = ctr_rand(key, base + (uint64_t)(i / 8));
            for (int64_t j = 0; j < 8 && i + j < bytes; ++j) blk[i + j] = (uint8_t)(r >> (8 * j));
        }
        double z0, z1;
        box_muller(ctr_rand(key, base + 30), ctr_rand(key, base + 31), &z0, &z1);
        uint16_t d = synth_f16_from_double(fabs(z0) * scale_mul);
        blk[d_off] = (uint8_t)(d & 0xFF);
        blk[d_off + 1] = (uint8_t)(d >> 8);
    }
}

/*
 * Fill `nrecords` KV records of 17,408 bytes (records first .. first+nrecords-1 of tensor
 * (seed, tensor_id)): K quants (8192 random bytes), 256 K scales, V quants (8192 random
 * bytes), 256 V scales; each scale fp16(|N(0,1)| * scale_mul).  Record r draws from its own
 * range of 4096 counter values.
 */
void synth_kv_records(uint8_t* out, int64_t nrecords, uint64_t seed, uint64_t tensor_id, int64_t first,
                      double scale_mul) {
    uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t rr = 0; rr < nrecords; ++rr) {
        uint64_t base = (uint64_t)(first + rr) * 4096;
        uint8_t* rec = out + 17408 * rr;
        for (int part = 0; part < 2; ++part) {
            uint8_t* qs = rec + part * 8704;
            for (int i = 0; i < 8192; i += 8) {
                uint64_t r = ctr_rand(key, base + (uint64_t)(part * 2048 + i / 8));
                for (int j = 0; j < 8; ++j) qs[i + j] = (uint8_t)(r >> (8 * j));
            }
            uint8_t* sc = qs + 8192;
            for (int i = 0; i < 256; i += 2) {
                double z0, z1;
                uint64_t c = base + 1024 + (uint64_t)(part * 256 + i);
                box_muller(ctr_rand(key, c), ctr_rand(key, c + 1), &z0, &z1);
                uint16_t h0 = synth_f16_from_double(fabs(z0) * scale_mul);
                uint16_t h1 = synth_f16_from_double(fabs(z1) * scale_mul);
                sc[2 * i] = (uint8_t)(h0 & 0xFF);
                sc[2 * i + 1] = (uint8_t)(h0 >> 8);
                sc[2 * i + 2] = (uint8_t)(h1 & 0xFF);
                sc[2 * i + 3] = (uint8_t)(h1 >> 8);
            }
        }
    }
}

/*
 * Fill n fp16 activations, elements first .. first+n-1 of tensor (seed, tensor_id),
 * as N(0,1); with probability outlier_p an element is multiplied by outlier_mul before
 * rounding.  Element i uses normal number i of the pair stream (pairs from Box-Muller)
 * and an independent uniform from a disjoint counter range for the outlier draw.
 */
void synth_x_f16(uint16_t* out, int64_t n, uint64_t seed, uint64_t tensor_id, int64_t first,
                 double outlier_p, double outlier_mul) {
    uint64_t key = synth_key(seed, tensor_id);
    const uint64_t outlier_base = 1ULL << 62;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t e = (uint64_t)(first + i);
        uint64_t pair = e >> 1;
        double z0, z1;
        box_muller(ctr_rand(key, 2 * pair), ctr_rand(key, 2 * pair + 1), &z0, &z1);
        double z = (e & 1) ? z1 : z0;
        if (outlier_p > 0.0 && u01(ctr_rand(key, outlier_base + e)) < outlier_p) z *= outlier_mul;
        out[i] = synth_f16_from_double(z);
    }
}

/* Raw counter stream, exposed for the generator's own tests. */
void synth_raw(uint64_t* out, int64_t n, uint64_t key, uint64_t first) {
    for (int64_t i = 0; i < n; ++i) out[i] = ctr_rand(key, first + (uint64_t)i);
}
