/*
 * synth.c -- seeded, counter-based generator of synthetic inputs (weights,
 * biases, activations).  It holds none of the MoE layer's arithmetic; both the
 * oracle's tests and the CUDA path's tests/benchmark draw their inputs here.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based
 * hash: draw i of stream s is mix64(key(seed, s) + (i + 1) * GAMMA).
 * Uniforms take the top 53 bits; normals come in Box-Muller pairs
 * (draws 2j and 2j+1 give normals 2j and 2j+1).  Value i of a stream does not
 * depend on how the stream is cut into calls or threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define GAMMA 0x9E3779B97F4A7C15ULL
#define TWO_PI 6.283185307179586476925286766559

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed + GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

/* (0, 1]: never zero, so log() below is finite */
static inline double unit_open0(uint64_t b) { return ((double)(b >> 11) + 1.0) * (1.0 / 9007199254740992.0); }
/* [0, 1) */
static inline double unit_closed0(uint64_t b) { return (double)(b >> 11) * (1.0 / 9007199254740992.0); }

static inline double normal_at(uint64_t key, uint64_t i)
{
    uint64_t j = i >> 1;
    double u1 = unit_open0(draw(key, 2 * j));
    double u2 = unit_closed0(draw(key, 2 * j + 1));
    double r = sqrt(-2.0 * log(u1));
    return (i & 1) ? r * sin(TWO_PI * u2) : r * cos(TWO_PI * u2);
}

/* Round-to-nearest-even binary32 -> bfloat16 bit pattern (finite inputs). */
static inline uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[i] = mean + std * N_i for i in [offset, offset + n) of the stream. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double mean, double std, float *out)
{
    uint64_t key = stream_key(seed, stream);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(mean + std * normal_at(key, offset + (uint64_t)i));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double mean, double std, uint16_t *out)
{
    uint64_t key = stream_key(seed, stream);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne((float)(mean + std * normal_at(key, offset + (uint64_t)i)));
}

/* out[i] = lo + (hi - lo) * U_i, U_i in [0, 1). */
void synth_uniform_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double lo, double hi, float *out)
{
    uint64_t key = stream_key(seed, stream);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(lo + (hi - lo) * unit_closed0(draw(key, offset + (uint64_t)i)));
}

void synth_uniform_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                        double lo, double hi, uint16_t *out)
{
    uint64_t key = stream_key(seed, stream);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne((float)(lo + (hi - lo) * unit_closed0(draw(key, offset + (uint64_t)i))));
}

/* Raw 64-bit draws (for permutations and other integer choices). */
void synth_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t *out)
{
    uint64_t key = stream_key(seed, stream);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i)
        out[i] = draw(key, offset + (uint64_t)i);
}

/* bf16 <-> f32 conversions for host-side staging of inputs. */
void synth_f32_to_bf16(const float *in, int64_t n, uint16_t *out)
{
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne(in[i]);
}

void synth_bf16_to_f32(const uint16_t *in, int64_t n, float *out)
{
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = ((uint32_t)in[i]) << 16;
        memcpy(&out[i], &u, sizeof u);
    }
}
