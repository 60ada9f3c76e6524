/*
 * CPU ORACLE for stacked-row decode attention over a paged q8_0 KV pool -- TEST
 * INFRASTRUCTURE ONLY (only the tests, the smoke check and the benchmark's CPU leg call it;
 * it shares nothing with the CUDA path).
 *
 * Sources: page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
 * Qwen3.8-27B", section "How parallel decoding works": every step stacks each active agent's
 * next token and its drafts into one batch of rows, and what grows with the number of agents
 * is attention, each agent reading its own KV cache; and the same page's shared KV pool: one
 * pool of q8_0 entries in pages, so that one agent may hold most of it.
 *
 * The plain definition, in double:
 *
 *   out[r][h][:] = sum_t p_t v_t,   p = softmax over t of s_t,   s_t = (q[r][h] . k_t) / sqrt(D)
 *
 * over the tokens t = 0 .. len[r] - 1 of the agent of row r (a row attends to its agent's
 * cache and to the step's earlier rows of the same agent, whose K and V are in the pool
 * already), with k_t, v_t from KV head g = h / (H / Hkv) (grouped-query attention).
 * Also returned: S[r][h][d] = sum_t p_t |v_t[d]|, for the tolerance of the GPU result.
 *
 * Pool layout (a reading; the pages give none): a page holds 64 consecutive tokens of one
 * agent for every KV head; (page P, head g) is the 17,408-byte record at (P * Hkv + g) * 17408:
 *   bytes     0 ..  8191  K quants, int8: token t's 128 dims in a 128-byte row, dim d at
 *                         t * 128 + 16 * ((d / 16) XOR key(t)) + d % 16, key(t) =
 *                         2 * (t % 4) + (t / 4) % 2 (16-byte pieces of a row permuted by the
 *                         token, so that the pieces that four consecutive tokens read together,
 *                         two neighbouring pieces each, lie in different shared-memory banks)
 *   bytes  8192 ..  8703  K scales, fp16 [token 64][dim block 4]
 *   bytes  8704 .. 16895  V quants, int8 [dim 128][token 64]   (dim-major)
 *   bytes 16896 .. 17407  V scales, fp16 [dim block 4][token 64]
 * A K or V element is scale * quant, with the scale of its 32-dim block (q8_0).  Token t of
 * agent a is slot t % 64 of page page_table[a * max_pages + t / 64].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ATTN_D 128
#define ATTN_PT 64
#define ATTN_REC 17408

double oracle_f16_to_double(uint16_t h);

/* Element d of K (which = 0) or V (which = 1) of token `slot` in the record `rec`. */
double oracle_kv(const uint8_t* rec, int which, int slot, int d) {
    const uint8_t* base = rec + which * 8704;
    int8_t q;
    const uint8_t* sc;
    if (which == 0) {
        q = (int8_t)base[slot * ATTN_D + 16 * ((d / 16) ^ (2 * (slot % 4) + (slot / 4) % 2)) + d % 16];
        sc = base + 8192 + 2 * (slot * 4 + d / 32);
    } else {
        q = (int8_t)base[d * ATTN_PT + slot];
        sc = base + 8192 + 2 * ((d / 32) * ATTN_PT + slot);
    }
    return oracle_f16_to_double((uint16_t)(sc[0] | (sc[1] << 8))) * (double)q;
}

/*
 * q: fp16 bit patterns [rows][H][D]; row_agent, row_len: [rows]; page_table: [agents][max_pages].
 * out, s_abs: [rows][H][D] (s_abs may be NULL).  Returns 0, or -1 on a bad argument.
 */
int oracle_attn(const uint8_t* pool, const int32_t* page_table, int max_pages, const uint16_t* q,
                const int32_t* row_agent, const int32_t* row_len, int rows, int H, int Hkv, double* out,
                double* s_abs, int nthreads) {
    if (rows < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0) return -1;
    for (int r = 0; r < rows; ++r)
        if (row_len[r] < 1 || row_len[r] > max_pages * ATTN_PT) return -1;
    const int group = H / Hkv;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(nthreads) reduction(| : failed)
#endif
    for (int r = 0; r < rows; ++r)
        for (int h = 0; h < H; ++h) {
            const int g = h / group, len = row_len[r], a = row_agent[r];
            double* s = (double*)malloc(sizeof(double) * (size_t)len);
            if (!s) {
                failed = 1;
                continue;
            }
            double qd[ATTN_D];
            for (int d = 0; d < ATTN_D; ++d) qd[d] = oracle_f16_to_double(q[((size_t)r * H + h) * ATTN_D + d]);
            double mx = -INFINITY;
            for (int t = 0; t < len; ++t) {
                const uint8_t* rec = pool + ((size_t)page_table[a * max_pages + t / ATTN_PT] * Hkv + g) * ATTN_REC;
                double dot = 0.0;
                for (int d = 0; d < ATTN_D; ++d) dot += qd[d] * oracle_kv(rec, 0, t % ATTN_PT, d);
                s[t] = dot / sqrt((double)ATTN_D);
                if (s[t] > mx) mx = s[t];
            }
            double z = 0.0;
            for (int t = 0; t < len; ++t) {
                s[t] = exp(s[t] - mx);
                z += s[t];
            }
            double o[ATTN_D] = {0}, sa[ATTN_D] = {0};
            for (int t = 0; t < len; ++t) {
                const uint8_t* rec = pool + ((size_t)page_table[a * max_pages + t / ATTN_PT] * Hkv + g) * ATTN_REC;
                const double p = s[t] / z;
                for (int d = 0; d < ATTN_D; ++d) {
                    const double v = oracle_kv(rec, 1, t % ATTN_PT, d);
                    o[d] += p * v;
                    sa[d] += p * fabs(v);
                }
            }
            for (int d = 0; d < ATTN_D; ++d) {
                out[((size_t)r * H + h) * ATTN_D + d] = o[d];
                if (s_abs) s_abs[((size_t)r * H + h) * ATTN_D + d] = sa[d];
            }
            free(s);
        }
    return failed ? -1 : 0;
}
