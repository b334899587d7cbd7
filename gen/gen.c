/*
 * Seeded synthetic inputs shared by the CPU oracle and the GPU library's tests
 * and benchmark.  Nothing in this file is part of the W8A8 method: it only
 * turns (seed, stream, index) into numbers.  Both sides read the bytes this
 * file writes, so they see identical inputs.
 *
 * Counter-based generator: draw(key, i) = splitmix64_finalizer(key + (i+1)*G),
 * with G = 0x9E3779B97F4A7C15 and the finalizer of Steele, Lea and Flood's
 * SplitMix64 (OOPSLA 2014), so any element can be produced independently of
 * the others and the result does not depend on the thread count.
 *
 * Approximate normals: Irwin-Hall sum of eight independent 32-bit uniforms,
 * centred and scaled to unit variance.  The sum is an exact integer; the
 * scaling is two IEEE double multiplies and one conversion to float, each
 * correctly rounded, so the value is the same on every machine.  Tails are
 * bounded at about +-4.9 sigma.
 */
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t gen_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL + 1));
}

uint64_t gen_draw(uint64_t key, uint64_t i)
{
    return mix64(key + (i + 1) * GOLDEN);
}

/* sqrt(3/8) * 2^-32: unit variance for (2*S - 8*(2^32-1)), S a sum of eight uint32 */
static const double NORM_SCALE = 0x1.3988e1409212ep-1 / 4294967296.0;

static inline double unit_normal(uint64_t key, uint64_t i)
{
    uint64_t s = 0;
    for (int j = 0; j < 4; ++j) {
        uint64_t d = gen_draw(key, 4 * i + (uint64_t)j);
        s += (d & 0xFFFFFFFFULL) + (d >> 32);
    }
    int64_t c = 2 * (int64_t)s - 8 * (int64_t)0xFFFFFFFFLL;
    return (double)c * NORM_SCALE;
}

/* out[j] = float(unit_normal(offset + j) * sigma), j in [0, count) */
void gen_normal_f32(uint64_t seed, uint64_t stream, int64_t offset, int64_t count,
                    double sigma, float *out)
{
    uint64_t key = gen_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < count; ++j) {
        double z = unit_normal(key, (uint64_t)(offset + j));
        out[j] = (float)(z * sigma);
    }
}

/* Raw 64-bit draws (used for index choices such as outlier channels). */
void gen_u64(uint64_t seed, uint64_t stream, int64_t offset, int64_t count, uint64_t *out)
{
    uint64_t key = gen_key(seed, stream);
    for (int64_t j = 0; j < count; ++j)
        out[j] = gen_draw(key, (uint64_t)(offset + j));
}

/*
 * bf16 activations, row-major [rows, cols] with row stride ld (elements):
 * x = unit_normal * sigma, times `outlier_gain` on the listed channels, then
 * narrowed to bf16 by dropping the low 16 bits (round toward zero).  Element
 * (r, c) uses normal index r*cols + c, so rows are independent of `rows`.
 */
void gen_act_bf16(uint64_t seed, uint64_t stream, int64_t row0, int64_t rows, int64_t cols,
                  int64_t ld, double sigma, const int64_t *outliers, int n_outliers,
                  double outlier_gain, uint16_t *out)
{
    uint64_t key = gen_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            double z = unit_normal(key, (uint64_t)((row0 + r) * cols + c)) * sigma;
            for (int o = 0; o < n_outliers; ++o)
                if (outliers[o] == c) z = z * outlier_gain;
            float f = (float)z;
            uint32_t bits;
            memcpy(&bits, &f, 4);
            out[r * ld + c] = (uint16_t)(bits >> 16);
        }
    }
}
