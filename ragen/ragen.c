/*
 * Seeded, counter-based input generator for the attention workloads.
 *
 * This file holds no attention arithmetic: it only turns (seed, tensor id,
 * element index) into a standard-normal sample, so that the CPU oracle and the
 * GPU path can both be fed the very same inputs, and so that any subset of a
 * tensor (for example a few sampled query rows of a 1M-token sequence) can be
 * regenerated without materialising the rest.
 *
 * Bit source: Philox-4x32-10, as published by Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3" (SC'11): a 10-round
 * multiply-xor network on a 128-bit counter under a 64-bit key, with the
 * round multipliers 0xD2511F53 / 0xCD9E8D57 and the Weyl key increments
 * 0x9E3779B9 / 0xBB67AE85.
 *
 * Stream layout (this generator's own convention):
 *   key     = (low 32 bits of seed, tensor id)
 *   counter = (block index low word, block index high word, 0, 0)
 *   element e of a tensor comes from block e / 4, output word e % 4.
 * Normal samples: Box-Muller on the word pairs (w0, w1) and (w2, w3):
 *   u1 = (w_even + 1) * 2^-32  in (0, 1],  u2 = w_odd * 2^-32  in [0, 1)
 *   r  = sqrt(-2 ln u1);  z_even = r cos(2 pi u2),  z_odd = r sin(2 pi u2)
 * evaluated in double precision, rounded to float32 (round to nearest even),
 * and, for bf16 output, rounded again from float32 to bfloat16 (round to
 * nearest even on the upper 16 bits).
 */
#include <math.h>
#include <stdint.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static inline void philox_round(uint32_t c[4], const uint32_t k[2]) {
    uint64_t p0 = (uint64_t)PHILOX_M0 * c[0];
    uint64_t p1 = (uint64_t)PHILOX_M1 * c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k[0];
    uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

/* Philox-4x32-10 block function: ctr (in/out) is replaced by the output. */
void ragen_philox4x32_10(uint32_t ctr[4], const uint32_t key_in[2]) {
    uint32_t k[2] = {key_in[0], key_in[1]};
    for (int r = 0; r < 10; ++r) {
        philox_round(ctr, k);
        k[0] += PHILOX_W0;
        k[1] += PHILOX_W1;
    }
}

static inline void block_normals(uint64_t seed, uint32_t tensor_id, uint64_t blk,
                                 float out[4]) {
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    uint32_t c[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
    ragen_philox4x32_10(c, key);
    const double two_pi = 6.283185307179586476925286766559;
    const double inv32 = 1.0 / 4294967296.0;
    for (int p = 0; p < 2; ++p) {
        double u1 = ((double)c[2 * p] + 1.0) * inv32;
        double u2 = (double)c[2 * p + 1] * inv32;
        double r = sqrt(-2.0 * log(u1));
        double th = two_pi * u2;
        out[2 * p] = (float)(r * cos(th));
        out[2 * p + 1] = (float)(r * sin(th));
    }
}

static inline uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } x;
    x.f = f;
    uint32_t u = x.u;
    if ((u & 0x7f800000u) == 0x7f800000u) /* inf / nan: keep, quiet nan */
        return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* Elements [start, start + n) of tensor (seed, tensor_id), as float32. */
void ragen_normal_f32(uint64_t seed, uint32_t tensor_id, int64_t start, int64_t n,
                      float* out) {
    if (n <= 0) return;
    int64_t b0 = start / 4, b1 = (start + n - 1) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t b = b0; b <= b1; ++b) {
        float z[4];
        block_normals(seed, tensor_id, (uint64_t)b, z);
        for (int w = 0; w < 4; ++w) {
            int64_t e = b * 4 + w;
            if (e >= start && e < start + n) out[e - start] = z[w];
        }
    }
}

/* Same elements as ragen_normal_f32, rounded to bfloat16 (raw 16-bit words). */
void ragen_normal_bf16(uint64_t seed, uint32_t tensor_id, int64_t start, int64_t n,
                       uint16_t* out) {
    if (n <= 0) return;
    int64_t b0 = start / 4, b1 = (start + n - 1) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t b = b0; b <= b1; ++b) {
        float z[4];
        block_normals(seed, tensor_id, (uint64_t)b, z);
        for (int w = 0; w < 4; ++w) {
            int64_t e = b * 4 + w;
            if (e >= start && e < start + n) out[e - start] = f32_to_bf16_rne(z[w]);
        }
    }
}

/* Gather rows: for each of n_rows row indices, elements [row*row_len, +row_len). */
void ragen_normal_bf16_rows(uint64_t seed, uint32_t tensor_id, const int64_t* rows,
                            int64_t n_rows, int64_t row_len, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_rows; ++i)
        ragen_normal_bf16(seed, tensor_id, rows[i] * row_len, row_len, out + i * row_len);
}
