// 19-tap WENO consumer arithmetic, shared by the resolver kernels
// (vbm_weno.cu: tree walk and cached table; vbm_brick.cu: bricks).
//
// Source (web page; cited by title and section):
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
//
// [2258] "A/B - decode" names a 19-tap WENO consumer without its formula.
// Here it is the Godunov upwind squared gradient norm of a level set phi at
// unit spacing, from fifth-order WENO one-sided derivatives (Jiang & Shu,
// J. Comput. Phys. 126, 1996; Jiang & Peng, SIAM J. Sci. Comput. 21, 2000),
// epsilon = 1e-6.  Taps j = 0..18: the centre and the voxels 1, 2, 3 steps
// away along each axis, in increasing (di,dj,dk) lexicographic order (the box
// order restricted):
//   j  0  1  2 | 3  4  5 | 6  7  8 | 9 | 10 11 12 | 13 14 15 | 16 17 18
//      x-3..x-1 | y-3..y-1 | z-3..z-1 | c | z+1..z+3 | y+1..y+3 | x+1..x+3
// An inactive tap reads phi[0], the background value's row.  Every operation
// is a separately rounded fp32 operation in a fixed order (no FMA), so the
// output is reproducible bit for bit.
#pragma once

#include "vbm_internal.h"

namespace vbm {

// Tap j = 0..18 <-> offset, lexicographic in (di,dj,dk).
__device__ __forceinline__ constexpr int weno_axis(int j) { return (j <= 2 || j >= 16) ? 0 : (j <= 5 || j >= 13) ? 1 : 2; }
__device__ __forceinline__ constexpr int weno_step(int j) {
    return j <= 2 ? j - 3 : j <= 5 ? j - 6 : j <= 8 ? j - 9 : j <= 12 ? j - 9 : j <= 15 ? j - 12 : j - 15;
}

// Fifth-order WENO one-sided derivative from five first differences, upwind
// side first; each operation rounded, in the order of the oracle's statement.
__device__ __forceinline__ float weno5(float a, float b, float c, float d, float e) {
    const float k13_12 = 13.0f / 12.0f;
    const float eps = 1.0e-6f;
    const float t1 = __fadd_rn(__fsub_rn(a, __fmul_rn(2.0f, b)), c);
    const float t2 = __fadd_rn(__fsub_rn(a, __fmul_rn(4.0f, b)), __fmul_rn(3.0f, c));
    const float s1 = __fadd_rn(__fmul_rn(k13_12, __fmul_rn(t1, t1)), __fmul_rn(0.25f, __fmul_rn(t2, t2)));
    const float u1 = __fadd_rn(__fsub_rn(b, __fmul_rn(2.0f, c)), d);
    const float u2 = __fsub_rn(b, d);
    const float s2 = __fadd_rn(__fmul_rn(k13_12, __fmul_rn(u1, u1)), __fmul_rn(0.25f, __fmul_rn(u2, u2)));
    const float v1 = __fadd_rn(__fsub_rn(c, __fmul_rn(2.0f, d)), e);
    const float v2 = __fadd_rn(__fsub_rn(__fmul_rn(3.0f, c), __fmul_rn(4.0f, d)), e);
    const float s3 = __fadd_rn(__fmul_rn(k13_12, __fmul_rn(v1, v1)), __fmul_rn(0.25f, __fmul_rn(v2, v2)));
    const float r1 = __fadd_rn(s1, eps), r2 = __fadd_rn(s2, eps), r3 = __fadd_rn(s3, eps);
    const float w1 = __fdiv_rn(0.1f, __fmul_rn(r1, r1));
    const float w2 = __fdiv_rn(0.6f, __fmul_rn(r2, r2));
    const float w3 = __fdiv_rn(0.3f, __fmul_rn(r3, r3));
    const float q1 = __fadd_rn(__fsub_rn(__fmul_rn(2.0f, a), __fmul_rn(7.0f, b)), __fmul_rn(11.0f, c));
    const float q2 = __fadd_rn(__fadd_rn(-b, __fmul_rn(5.0f, c)), __fmul_rn(2.0f, d));
    const float q3 = __fsub_rn(__fadd_rn(__fmul_rn(2.0f, c), __fmul_rn(5.0f, d)), e);
    const float num = __fadd_rn(__fadd_rn(__fmul_rn(w1, q1), __fmul_rn(w2, q2)), __fmul_rn(w3, q3));
    const float den = __fmul_rn(6.0f, __fadd_rn(__fadd_rn(w1, w2), w3));
    return __fdiv_rn(num, den);
}

// Godunov upwind square of the derivative along one axis from p[0..6] at
// offsets -3..+3 (p[3] the centre).
__device__ __forceinline__ float godunov_axis(const float (&p)[7], bool outside) {
    float d[6];
#pragma unroll
    for (int k = 0; k < 6; ++k) d[k] = __fsub_rn(p[k + 1], p[k]);
    const float minus = weno5(d[0], d[1], d[2], d[3], d[4]);
    const float plus = weno5(d[5], d[4], d[3], d[2], d[1]);
    float lo, hi;
    if (outside) {
        lo = minus > 0.0f ? minus : 0.0f;
        hi = plus < 0.0f ? plus : 0.0f;
    } else {
        lo = minus < 0.0f ? minus : 0.0f;
        hi = plus > 0.0f ? plus : 0.0f;
    }
    const float lo2 = __fmul_rn(lo, lo), hi2 = __fmul_rn(hi, hi);
    return lo2 > hi2 ? lo2 : hi2;
}

// The WENO value from the 19 tap values v[j] (tap order).
__device__ __forceinline__ float weno_value(const float (&v)[kWenoTaps], float iso) {
    const bool outside = v[9] > iso;
    const float px[7] = {v[0], v[1], v[2], v[9], v[16], v[17], v[18]};
    const float py[7] = {v[3], v[4], v[5], v[9], v[13], v[14], v[15]};
    const float pz[7] = {v[6], v[7], v[8], v[9], v[10], v[11], v[12]};
    float total = 0.0f;
    total = __fadd_rn(total, godunov_axis(px, outside));
    total = __fadd_rn(total, godunov_axis(py, outside));
    total = __fadd_rn(total, godunov_axis(pz, outside));
    return total;
}

}  // namespace vbm
