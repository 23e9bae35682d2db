/*
 * synth.c - seeded synthetic inputs for the MXFP4 routed-expert layer.
 *
 * This module only draws numbers.  It holds none of the layer's arithmetic:
 * no e2m1 or ue8m0 decoding, no routing, no activation.  Both the CPU oracle
 * (through the tests) and the CUDA path (through the tests and the bench)
 * receive their inputs from here, so the two sides see identical bytes.
 *
 * Generator: counter-based.  Element i of stream s under seed k is
 *     mix64(key(k, s) + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the SplitMix64 output function (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) and
 * key(k, s) = mix64(k ^ mix64(s + 0x632BE59BD9B4E019)).  Any element of any
 * stream can be drawn on its own, so a single expert of the 896 can be
 * produced without producing the others.
 *
 * Distributions (the recipe of the workloads in the routed-expert configs):
 *   bytes        : the 8 bytes of each 64-bit draw, little-endian order, so
 *                  both nibbles of every byte are uniform on 0..15;
 *   scale bytes  : lo + floor(u32 * (hi - lo + 1) / 2^32), the multiply-shift
 *                  map of the high 32 bits of a draw; with probability p (an
 *                  independent stream, u53 < p) the byte is set to 255;
 *   normal       : Box-Muller on two draws of 53 bits, in double, rounded to
 *                  fp32 once; mean + std * z;
 *   bf16         : round-to-nearest-even of the fp32 bit pattern.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

uint64_t synth_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t stream)
{
    return synth_mix64(seed ^ synth_mix64(stream + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i)
{
    return synth_mix64(key + (i + 1) * SYNTH_GOLDEN);
}

/* n uniform bytes */
void synth_bytes(uint8_t *out, size_t n, uint64_t seed, uint64_t stream)
{
    const uint64_t key = synth_key(seed, stream);
    const size_t nw = n / 8;
    #pragma omp parallel for schedule(static)
    for (long long w = 0; w < (long long)nw; w++) {
        uint64_t d = draw(key, (uint64_t)w);
        memcpy(out + (size_t)w * 8, &d, 8);   /* little-endian on both hosts */
    }
    if (n % 8) {
        uint64_t d = draw(key, (uint64_t)nw);
        for (size_t j = 0; j < n % 8; j++)
            out[nw * 8 + j] = (uint8_t)(d >> (8 * j));
    }
}

/* n bytes uniform on [lo, hi]; a fraction nan_frac (own stream) set to 255 */
void synth_scale_bytes(uint8_t *out, size_t n, uint64_t seed, uint64_t stream,
                       int lo, int hi, double nan_frac)
{
    const uint64_t key = synth_key(seed, stream);
    const uint64_t nkey = synth_key(seed, stream ^ 0x5A5A5A5A00000000ULL);
    const uint64_t span = (uint64_t)(hi - lo + 1);
    #pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; i++) {
        uint64_t d = draw(key, (uint64_t)i);
        int v = lo + (int)(((d >> 32) * span) >> 32);
        if (nan_frac > 0.0) {
            double u = (double)(draw(nkey, (uint64_t)i) >> 11) * 0x1.0p-53;
            if (u < nan_frac) v = 255;
        }
        out[i] = (uint8_t)v;
    }
}

/* n fp32 values mean + std * N(0,1) (Box-Muller in double, one rounding) */
void synth_normal_f32(float *out, size_t n, uint64_t seed, uint64_t stream,
                      double mean, double std)
{
    const uint64_t key = synth_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
    const size_t npair = (n + 1) / 2;
    #pragma omp parallel for schedule(static)
    for (long long p = 0; p < (long long)npair; p++) {
        double u1 = (double)((draw(key, 2 * (uint64_t)p) >> 11) + 1) * 0x1.0p-53; /* (0,1] */
        double u2 = (double)(draw(key, 2 * (uint64_t)p + 1) >> 11) * 0x1.0p-53;    /* [0,1) */
        double r = sqrt(-2.0 * log(u1));
        double z0 = r * cos(two_pi * u2), z1 = r * sin(two_pi * u2);
        out[2 * p] = (float)(mean + std * z0);
        if ((size_t)(2 * p + 1) < n) out[2 * p + 1] = (float)(mean + std * z1);
    }
}

/* fp32 -> bf16 bit patterns, round to nearest even (NaN kept quiet) */
void synth_f32_to_bf16(uint16_t *out, const float *in, size_t n)
{
    #pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; i++) {
        uint32_t b;
        memcpy(&b, &in[i], 4);
        if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) {
            out[i] = (uint16_t)((b >> 16) | 0x0040u);
        } else {
            uint32_t lsb = (b >> 16) & 1u;
            out[i] = (uint16_t)((b + 0x7FFFu + lsb) >> 16);
        }
    }
}

/* bf16 bit patterns -> fp32 (exact widening) */
void synth_bf16_to_f32(float *out, const uint16_t *in, size_t n)
{
    #pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; i++) {
        uint32_t b = (uint32_t)in[i] << 16;
        memcpy(&out[i], &b, 4);
    }
}

/*
 * One routed expert, written in arena order: w1 packed, w1 scales,
 * w3 packed, w3 scales, w2 packed, w2 scales.  w1 and w3 are [F x D],
 * w2 is [D x F], packed row-major with two columns per byte, scales
 * row-major with one byte per 32 columns.  Streams are numbered per
 * (expert, tensor) so any expert is drawn independently of the others.
 */
size_t synth_expert_bytes(int D, int F)
{
    size_t a = (size_t)F * D / 2, s = (size_t)F * D / 32;
    return 3 * (a + s);
}

void synth_expert(uint8_t *dst, uint64_t seed, int expert, int D, int F,
                  int lo, int hi, double nan_frac)
{
    const size_t a = (size_t)F * D / 2, s = (size_t)F * D / 32;
    const uint64_t base = 0x100000ULL + (uint64_t)expert * 8;
    uint8_t *p = dst;
    for (int t = 0; t < 3; t++) {
        synth_bytes(p, a, seed, base + 2 * t);
        p += a;
        synth_scale_bytes(p, s, seed, base + 2 * t + 1, lo, hi, nan_frac);
        p += s;
    }
}
