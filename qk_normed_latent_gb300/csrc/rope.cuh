// Rotary position embedding (the original formulation on interleaved pairs):
// (x_2i, x_2i+1) is rotated by the angle pos * theta^(-2i/d).
//
// The angle is formed in fp32 without losing its low bits at long positions:
// f = theta^(-2i/d) is computed once in fp64 and kept as f_hi + f_lo (two fp32);
// pos * f_hi is split error-free with an fma (Dekker's product), then reduced
// modulo 2 pi with a two-part constant (Cody-Waite reduction), and only the
// reduced angle goes to sincosf.  An fp32 product alone would be off by up to
// pos * 2^-24 radians (0.016 at position 262144).
#pragma once

#include <cuda_runtime.h>

namespace qkmla {

struct RopeFreq {
    float hi, lo;
};

// theta^(-2i/d) as hi + lo (fp64 once; cheap next to the GEMM it feeds).
__device__ __forceinline__ RopeFreq rope_freq(float theta, int i, int d) {
    const double f = pow((double)theta, -(double)(2 * i) / (double)d);
    RopeFreq r;
    r.hi = (float)f;
    r.lo = (float)(f - (double)r.hi);
    return r;
}

// cos and sin of pos * f.  Kept out of line: sincosf carries a large slow path
// (for arguments far beyond this reduced range), and one copy per unrolled use
// would overflow the instruction cache of the kernels that rotate many pairs.
static __device__ __noinline__ void rope_cos_sin(int pos, RopeFreq f, float* c, float* s) {
    constexpr float kTwoPiHi = 6.2831854820251465f;      // 2 pi rounded to fp32
    constexpr float kTwoPiLo = -1.7484555314695172e-07f;  // 2 pi - kTwoPiHi
    constexpr float kInvTwoPi = 0.15915493667125702f;
    const float P = (float)pos;                          // exact below 2^24
    const float a = P * f.hi;
    const float ae = fmaf(P, f.hi, -a) + P * f.lo;       // a + ae = pos * f
    const float k = rintf(a * kInvTwoPi);
    float r = fmaf(-k, kTwoPiHi, a);
    r = fmaf(-k, kTwoPiLo, r);
    r += ae;
    sincosf(r, s, c);
}

// cos and sin of pos * f for four frequencies at once: four independent chains,
// so their latencies overlap (the kernels that rotate many pairs per thread call
// this instead of four rope_cos_sin).
static __device__ __noinline__ void rope_cos_sin4(int pos, const RopeFreq* f, float* c, float* s) {
    constexpr float kTwoPiHi = 6.2831854820251465f;
    constexpr float kTwoPiLo = -1.7484555314695172e-07f;
    constexpr float kInvTwoPi = 0.15915493667125702f;
    const float P = (float)pos;
    float r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = P * f[i].hi;
        const float ae = fmaf(P, f[i].hi, -a) + P * f[i].lo;
        const float k = rintf(a * kInvTwoPi);
        r[i] = fmaf(-k, kTwoPiLo, fmaf(-k, kTwoPiHi, a)) + ae;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sincosf(r[i], &s[i], &c[i]);
}

// One interleaved pair's rotation: element j (= 2i or 2i+1) of the rotated
// vector, from its own value v and its pair partner's value w.
__device__ __forceinline__ float rope_apply(int j, float v, float w, float c, float s) {
    return (j & 1) ? fmaf(w, s, v * c) : fmaf(-w, s, v * c);
}

}  // namespace qkmla
