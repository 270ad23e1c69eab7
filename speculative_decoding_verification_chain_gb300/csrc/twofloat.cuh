// Two-float arithmetic: a value is hi + lo with |lo| below half an ulp of hi
// (about 44 significant bits), built from fp32 operations only.  The kernels
// use it wherever a sum or a prefix must be carried beyond one thread: FP64
// issue is scarce on this part, and a chain of dependent fp64 operations on a
// latency-bound path costs microseconds.
#pragma once

namespace sv {

struct tf {
    float h, l;
};

// s + e == a + b exactly (Knuth's TwoSum; no multiplication, so no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ tf tf_of(float h) { return tf{h, 0.0f}; }

__device__ __forceinline__ tf tf_add(tf a, tf b) {
    float s, e;
    two_sum(a.h, b.h, s, e);
    e += a.l + b.l;
    tf r;
    r.h = s + e;
    r.l = e - (r.h - s);
    return r;
}

__device__ __forceinline__ tf tf_neg(tf a) { return tf{-a.h, -a.l}; }

// a * f for a two-float a and a float f.
__device__ __forceinline__ tf tf_mulf(tf a, float f) {
    const float p = a.h * f;
    const float e = fmaf(a.h, f, -p) + a.l * f;
    tf r;
    r.h = p + e;
    r.l = e - (r.h - p);
    return r;
}

// a * b exactly, as a two-float.
__device__ __forceinline__ tf tf_prod(float a, float b) {
    const float p = a * b;
    return tf{p, fmaf(a, b, -p)};
}

// a > b, decided on the two-float difference.
__device__ __forceinline__ bool tf_gt(tf a, tf b) { return (a.h - b.h) + (a.l - b.l) > 0.0f; }

__device__ __forceinline__ tf tf_shfl_xor(tf a, int o) {
    return tf{__shfl_xor_sync(0xffffffffu, a.h, o), __shfl_xor_sync(0xffffffffu, a.l, o)};
}

__device__ __forceinline__ tf tf_shfl(tf a, int src) {
    return tf{__shfl_sync(0xffffffffu, a.h, src), __shfl_sync(0xffffffffu, a.l, src)};
}

__device__ __forceinline__ tf warp_sum_tf(tf a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = tf_add(a, tf_shfl_xor(a, o));
    return a;
}

// Inclusive prefix over the lanes in lane order.
__device__ __forceinline__ tf warp_incl_scan_tf(tf a, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const tf y{__shfl_up_sync(0xffffffffu, a.h, o), __shfl_up_sync(0xffffffffu, a.l, o)};
        if (lane >= o) a = tf_add(y, a);
    }
    return a;
}

}  // namespace sv
