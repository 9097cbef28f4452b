/*
 * Seeded synthetic inputs for the lookahead-decoding step: model weights drawn
 * N(0, std) and uniform token ids.  This file holds generators only -- none of
 * the decoding arithmetic -- and serves both the CPU oracle and the CUDA path.
 *
 * Counter-based generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11), written from that
 * paper's definition.  Normal deviates use the Box-Muller transform in double
 * precision.  Each value depends only on (seed, stream, index), so any thread
 * split gives the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

static void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

/* Exposed so the tests can check the generator against published answers. */
void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    philox4x32_10(c, key[0], key[1]);
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/* Two normals from counter (pair index, stream). */
static void normal_pair(uint64_t seed, uint32_t stream, uint64_t pair, double *z0, double *z1) {
    uint32_t c[4] = {(uint32_t)pair, (uint32_t)(pair >> 32), stream, 0x6e6f726du};
    philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
    uint64_t a = ((uint64_t)c[0] << 32) | c[1];
    uint64_t b = ((uint64_t)c[2] << 32) | c[3];
    double u1 = ((double)(a >> 11) + 0.5) * (1.0 / 9007199254740992.0); /* (0,1) */
    double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);         /* [0,1) */
    double r = sqrt(-2.0 * log(u1));
    double t = 6.283185307179586476925286766559 * u2;
    *z0 = r * cos(t);
    *z1 = r * sin(t);
}

static uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } v; v.f = f;
    uint32_t u = v.u;
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* NaN stays NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[i] = (float)(std * z_i) for i in [0, n). */
void synth_normal_f32(uint64_t seed, uint32_t stream, double std, float *out, int64_t n) {
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npair; ++p) {
        double z0, z1;
        normal_pair(seed, stream, (uint64_t)p, &z0, &z1);
        out[2 * p] = (float)(std * z0);
        if (2 * p + 1 < n) out[2 * p + 1] = (float)(std * z1);
    }
}

/* Same values as synth_normal_f32, rounded to bfloat16 (round to nearest even). */
void synth_normal_bf16(uint64_t seed, uint32_t stream, double std, uint16_t *out, int64_t n) {
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npair; ++p) {
        double z0, z1;
        normal_pair(seed, stream, (uint64_t)p, &z0, &z1);
        out[2 * p] = f32_to_bf16_rne((float)(std * z0));
        if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16_rne((float)(std * z1));
    }
}

/* Token ids uniform in [0, vocab): multiply-shift of one 32-bit Philox word. */
void synth_uniform_tokens(uint64_t seed, uint32_t stream, int32_t vocab, int32_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t c[4] = {(uint32_t)i, (uint32_t)((uint64_t)i >> 32), stream, 0x746f6b6eu};
        philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
        out[i] = (int32_t)(((uint64_t)c[0] * (uint64_t)(uint32_t)vocab) >> 32);
    }
}
