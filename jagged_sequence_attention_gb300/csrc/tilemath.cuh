// Element-wise pieces shared by the bf16 kernels: the relative-position bucket, the
// per-chunk constant-bias test, and the GDPA activations with their derivatives.
#pragma once

#include "ptx.cuh"

namespace jfa {

// bucket(r) = min(31, floor(log2((1+r)^2))) for r >= 0, in integer arithmetic:
// (1+r)^2 < 2^31 exactly when r < 46340, and then floor(log2(v)) = 31 - clz(v).
__device__ __forceinline__ int relpos_bucket(int r) {
    r = abs(r);
    const int rc = min(r, 46339);
    const uint32_t v = uint32_t(rc + 1) * uint32_t(rc + 1);
    const int b = 31 - __clz(v);
    return r >= 46340 ? 31 : b;
}

// The first relative position of bucket b or above: the smallest r >= 0 with
// (1 + r)^2 >= 2^b (b <= 31), by an exact integer search.
__host__ __device__ constexpr int relpos_bucket_start(int b) {
    long long lo = 0, hi = 46340;
    while (lo < hi) {
        const long long mid = (lo + hi) / 2;
        if ((1 + mid) * (1 + mid) >= (1LL << b))
            hi = mid;
        else
            lo = mid + 1;
    }
    return int(lo);
}

// Warp-level test of whether a 32-column chunk's bias is one value.  In the callers,
// the 32 lanes' windows for one chunk tile a range of 63 relative positions
// [lo, lo + 62] (consecutive rows or keys shift the window by one).  The bucket of |r| is monotone on a range that does not
// cross 0, so every lane's chunk is constant exactly when the whole range lies on one
// side of 0 and its two ends share a bucket; then all lanes share that bucket.  Each
// lane evaluates one chunk (the caller passes lane k the range of chunk k); returns the
// ballot of constant chunks, and the chunk's bucket in `bucket`.
__device__ __forceinline__ uint32_t warp_const_chunks(bool active, int lo, int& bucket) {
    bucket = relpos_bucket(lo + 62);
    const bool c = active && (lo >= 0 || lo + 62 <= 0) && relpos_bucket(lo) == bucket;
    return __ballot_sync(0xffffffffu, c);
}

// sigmoid(x) = 1 / (1 + exp(-x))
__device__ __forceinline__ float sigmoid_acc(float x) {
    return rcp_approx(1.f + ex2_approx(-1.4426950408889634f * x));
}

// GDPA activations and derivatives:
//   gelu(x)  = 0.5 x (1 + tanh(u)),  u = k0 x + k1 x^3,  k0 = sqrt(2/pi), k1 = 0.044715 k0
//            = x s,  s = sigmoid(2u) = 1 / (1 + 2^z),  z = -2 log2(e) u   (since 0.5 (1 + tanh u)
//              = sigmoid(2u)); the sigmoid form saturates to 0 and 1 without the cancellation
//              of 1 + tanh(u) for large negative x, in two fewer operations
//   gelu'(x) = s + 2 x s (1 - s) (k0 + 3 k1 x^2)
//   silu(x)  = x s(x),  silu'(x) = s(x) (1 + x (1 - s(x)))
__device__ __forceinline__ float gelu_sigmoid_arg(float x, float x2) {
    // z = -2 log2(e) (k0 x + k1 x^3)
    const float c0 = -2.3022082f, c1 = -0.10294324f;  // -2 log2(e) k0, -2 log2(e) k1
    return x * fmaf(c1, x2, c0);
}

__device__ __forceinline__ float gdpa_act(bool gelu, float x) {
    if (gelu) return x * rcp_approx(1.f + ex2_approx(gelu_sigmoid_arg(x, x * x)));
    return x * sigmoid_acc(x);
}

// gdpa_act on two elements (s0, s1) of the raw score, x = scale * s, with the products and
// sums on the paired fp32 pipe (one instruction per pair); the exponents and reciprocals
// stay per element.
template <bool GELU>
__device__ __forceinline__ float2 gdpa_act2(float2 s, float scale) {
    const float2 x = mul2(s, make_float2(scale, scale));
    float2 z;
    if (GELU) {
        const float2 t = fma2(mul2(x, x), make_float2(-0.10294324f, -0.10294324f), make_float2(-2.3022082f, -2.3022082f));
        z = mul2(x, t);  // gelu_sigmoid_arg of each element
    } else {
        z = mul2(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    }
    const float2 d = add2(make_float2(ex2_approx(z.x), ex2_approx(z.y)), make_float2(1.f, 1.f));
    return mul2(x, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// gdpa_act_grad on two elements of the raw score (x = scale * s), paired as gdpa_act2.
template <bool GELU>
__device__ __forceinline__ void gdpa_act_grad2(float2 s, float scale, float2& a, float2& da) {
    const float2 x = mul2(s, make_float2(scale, scale));
    if (GELU) {
        const float2 x2 = mul2(x, x);
        const float2 z = mul2(x, fma2(x2, make_float2(-0.10294324f, -0.10294324f), make_float2(-2.3022082f, -2.3022082f)));
        const float2 d = add2(make_float2(ex2_approx(z.x), ex2_approx(z.y)), make_float2(1.f, 1.f));
        const float2 sg = make_float2(rcp_approx(d.x), rcp_approx(d.y));
        a = mul2(x, sg);
        // gelu' = s + 2 a (1 - s) (k0 + 3 k1 x^2)
        const float2 oms = add2(make_float2(1.f, 1.f), make_float2(-sg.x, -sg.y));
        const float2 poly = fma2(x2, make_float2(3.f * 0.035677408136300125f, 3.f * 0.035677408136300125f),
                                 make_float2(0.7978845608028654f, 0.7978845608028654f));
        da = fma2(mul2(add2(a, a), oms), poly, sg);
    } else {
        const float2 z = mul2(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
        const float2 d = add2(make_float2(ex2_approx(z.x), ex2_approx(z.y)), make_float2(1.f, 1.f));
        const float2 sg = make_float2(rcp_approx(d.x), rcp_approx(d.y));
        a = mul2(x, sg);
        // silu' = s (1 + x (1 - s))
        const float2 oms = add2(make_float2(1.f, 1.f), make_float2(-sg.x, -sg.y));
        da = mul2(sg, fma2(x, oms, make_float2(1.f, 1.f)));
    }
}

__device__ __forceinline__ void gdpa_act_grad(bool gelu, float x, float& a, float& da) {
    if (gelu) {
        const float k0 = 0.7978845608028654f, k1 = 0.035677408136300125f;
        const float x2 = x * x;
        const float s = rcp_approx(1.f + ex2_approx(gelu_sigmoid_arg(x, x2)));
        a = x * s;
        da = fmaf(2.f * a * (1.f - s), fmaf(3.f * k1, x2, k0), s);
    } else {
        const float sg = sigmoid_acc(x);
        a = x * sg;
        da = sg * fmaf(x, 1.f - sg, 1.f);
    }
}

}  // namespace jfa
