/*
 * Oracle-side synthetic weight generator (TEST INFRASTRUCTURE ONLY).
 *
 * Plain C restatement of the seeded "N(0, std)" weights of the synthetic
 * decoder: element e of tensor t is an Irwin-Hall(4) sum over the four words
 * of one Philox4x32-10 call (Salmon et al., SC'11), counter
 * (e mod 2^32, e div 2^32, t, 1), key (seed mod 2^32, seed div 2^32):
 *
 *     s = sum_j (word_j >> 9)                  (integer, < 2^25)
 *     w = fp32(s - 2^24) * fp32(std * sqrt(3) / 2^23)
 *
 * which has mean 0 and variance std^2 (each 23-bit uniform has variance
 * ~1/12).  The value is then rounded to bfloat16 (round to nearest even) and
 * returned as the fp32 number it represents.  Built with -ffp-contract=off.
 *
 * It exists in C only for speed (a 30-layer model has ~2.5e10 elements); the
 * Python oracle calls it through ctypes.  It shares nothing with the GPU
 * library.
 */
#include <math.h>
#include <stdint.h>

static void philox_round(uint32_t c[4], const uint32_t k[2]) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k[0];
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k[1];
    uint32_t n3 = (uint32_t)p0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
}

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        philox_round(c, k);
        k[0] += 0x9E3779B9u;
        k[1] += 0xBB67AE85u;
    }
    out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

static float round_to_bf16(float x) {
    union { float f; uint32_t u; } v;
    v.f = x;
    uint32_t lsb = (v.u >> 16) & 1u;
    v.u = (v.u + 0x7FFFu + lsb) & 0xFFFF0000u;
    return v.f;
}

/* out[j] = weight element (e0 + j) of tensor `tid`, j < n. */
void oracle_weights(uint64_t seed, uint32_t tid, uint64_t e0, uint64_t n, float std_dev,
                    float *out) {
    const float scale = (float)((double)std_dev * sqrt(3.0) / 8388608.0);
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < (int64_t)n; ++j) {
        uint64_t e = e0 + (uint64_t)j;
        uint32_t ctr[4] = {(uint32_t)e, (uint32_t)(e >> 32), tid, 1u};
        uint32_t w[4];
        oracle_philox4x32_10(ctr, key, w);
        int32_t s = (int32_t)(w[0] >> 9) + (int32_t)(w[1] >> 9) + (int32_t)(w[2] >> 9) +
                    (int32_t)(w[3] >> 9);
        float v = (float)(s - (1 << 24)) * scale;
        out[j] = round_to_bf16(v);
    }
}
