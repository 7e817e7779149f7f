/*
 * Seeded synthetic inputs shared by the oracle and the GPU path.
 *
 * This module holds no step of the quantize-and-multiply method: it only draws
 * numbers.  Element i of tensor (seed, tensor_id) is
 *
 *     value = (float)( sigma * Phi^-1(u_i) )          (f64 -> f32, RNE)
 *
 *     key  = mix64((seed + 1) * G) ^ mix64((tensor_id + 1) * H)
 *     u_i  = ((mix64(key + (i + 1) * G) >> 11) + 0.5) * 2^-53      in (0, 1)
 *
 * with G = 0x9E3779B97F4A7C15 (the SplitMix64 increment) and
 * H = 0xD1B54A32D192ED03 (an odd constant): u_i comes from output i+1 of the
 * SplitMix64 stream whose state starts at `key`.  mix64 is the SplitMix64
 * output finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014, with the constants Vigna published for it).
 *
 * Phi^-1 is the normal quantile function by Wichura's algorithm AS 241
 * (PPND16; M. J. Wichura, Applied Statistics 37(3), 1988, 477-484): a 7/7
 * rational function of (0.180625 - q^2) for |q| = |u - 1/2| <= 0.425, and
 * 7/7 rational functions of sqrt(-ln(min(u, 1-u))) in the two tail ranges.
 * Its relative accuracy is about 1e-16.  Every element is a pure function of
 * its index, so generation is parallel and independent of the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define SM_G 0x9E3779B97F4A7C15ULL
#define SM_H 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
    return mix64((seed + 1) * SM_G) ^ mix64((tensor_id + 1) * SM_H);
}

double synth_uniform(uint64_t key, uint64_t i) {
    uint64_t z = mix64(key + (i + 1) * SM_G);
    return ((double)(z >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Normal quantile, AS 241 (PPND16). p in (0, 1). */
double synth_ndtri(double p) {
    double q = p - 0.5;
    if (fabs(q) <= 0.425) {
        double r = 0.180625 - q * q;
        double num = ((((((2.5090809287301226727e+3 * r + 3.3430575583588128105e+4) * r
                      + 6.7265770927008700853e+4) * r + 4.5921953931549871457e+4) * r
                      + 1.3731693765509461125e+4) * r + 1.9715909503065514427e+3) * r
                      + 1.3314166789178437745e+2) * r + 3.3871328727963666080e+0;
        double den = ((((((5.2264952788528545610e+3 * r + 2.8729085735721942674e+4) * r
                      + 3.9307895800092710610e+4) * r + 2.1213794301586595867e+4) * r
                      + 5.3941960214247511077e+3) * r + 6.8718700749205790830e+2) * r
                      + 4.2313330701600911252e+1) * r + 1.0;
        return q * num / den;
    }
    double r = q < 0 ? p : 1.0 - p;
    r = sqrt(-log(r));
    double v;
    if (r <= 5.0) {
        r -= 1.6;
        double num = ((((((7.74545014278341407640e-4 * r + 2.27238449892691845833e-2) * r
                      + 2.41780725177450611770e-1) * r + 1.27045825245236838258e+0) * r
                      + 3.64784832476320460504e+0) * r + 5.76949722146069140550e+0) * r
                      + 4.63033784615654529590e+0) * r + 1.42343711074968357734e+0;
        double den = ((((((1.05075007164441684324e-9 * r + 5.47593808499534494600e-4) * r
                      + 1.51986665636164571966e-2) * r + 1.48103976427480074590e-1) * r
                      + 6.89767334985100004550e-1) * r + 1.67638483018380384940e+0) * r
                      + 2.05319162663775882187e+0) * r + 1.0;
        v = num / den;
    } else {
        r -= 5.0;
        double num = ((((((2.01033439929228813265e-7 * r + 2.71155556874348757815e-5) * r
                      + 1.24266094738807843860e-3) * r + 2.65321895265761230930e-2) * r
                      + 2.96560571828504891230e-1) * r + 1.78482653991729133580e+0) * r
                      + 5.46378491116411436990e+0) * r + 6.65790464350110377720e+0;
        double den = ((((((2.04426310338993978564e-15 * r + 1.42151175831644588870e-7) * r
                      + 1.84631831751005468180e-5) * r + 7.86869131145613259100e-4) * r
                      + 1.48753612908506148525e-2) * r + 1.36929880922735805310e-1) * r
                      + 5.99832206555887937690e-1) * r + 1.0;
        v = num / den;
    }
    return q < 0 ? -v : v;
}

/* out[t] = (float)(sigma * Phi^-1(u_{start+t})) for t in [0, count). */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count,
                      double sigma, float* out) {
    const uint64_t key = synth_key(seed, tensor_id);
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; t++)
        out[t] = (float)(sigma * synth_ndtri(synth_uniform(key, start + (uint64_t)t)));
}

/* out[t] = u_{start+t} (the raw uniforms, for checking the generator). */
void synth_uniform_f64(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count,
                       double* out) {
    const uint64_t key = synth_key(seed, tensor_id);
    for (uint64_t t = 0; t < count; t++) out[t] = synth_uniform(key, start + t);
}

/* float -> bfloat16 bits, round to nearest even (finite inputs). */
void synth_f32_to_bf16(const float* in, uint16_t* out, uint64_t count) {
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; t++) {
        union { float f; uint32_t u; } c;
        c.f = in[t];
        uint32_t u = c.u;
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7FFFu + lsb;
        out[t] = (uint16_t)(u >> 16);
    }
}
