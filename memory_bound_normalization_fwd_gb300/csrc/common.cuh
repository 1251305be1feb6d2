// Shared device helpers for the RMSNorm forward kernels (sm_103a).
//
// The arithmetic every kernel performs per row follows the kernel listing of
// "Why cutile's rmsnorm required full register" (TileGym issue #169): widen to
// fp32, sum of squares, divide by N, add eps, rsqrt, store rstd, multiply by
// rstd and then by (offset + w), one rounding to the activation dtype.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

enum DType : int { kBF16 = 0, kFP16 = 1, kFP32 = 2 };

// Element codecs. A 32-bit word holds two elements, element 0 in the low half
// (little-endian memory order).
template <int DT>
struct Codec;

template <>
struct Codec<kBF16> {
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        // bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float unpack1(uint16_t u) {
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    }
    static __device__ __forceinline__ uint16_t pack1(float a) {
        __nv_bfloat16 h = __float2bfloat16_rn(a);
        return *reinterpret_cast<uint16_t*>(&h);
    }
};

template <>
struct Codec<kFP16> {
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float unpack1(uint16_t u) {
        __half h = *reinterpret_cast<__half*>(&u);
        return __half2float(h);
    }
    static __device__ __forceinline__ uint16_t pack1(float a) {
        __half h = __float2half_rn(a);
        return *reinterpret_cast<uint16_t*>(&h);
    }
};

// 16-byte vector = 8 elements of a 16-bit format (the backward's kernels use
// this constant; the forward's use VecElems<DT>).
constexpr int kVecElems = 8;

// Elements per 16-byte vector: 8 for bf16/fp16, 4 for fp32.
template <int DT>
struct VecElems {
    static constexpr int value = DT == kFP32 ? 4 : 8;
};

// acc + lo^2 + hi^2 for the two bf16 elements of a word, in that order, with
// mixed-precision FMAs (fma.rn.f32.bf16, sm_100 and later): the inputs widen
// exactly and each product-and-sum is rounded once to fp32, the same result
// as widening first and calling fmaf, without the widening instructions.
// (GB300, same box, A/B: 16384x8192 bf16 6233 -> 6403 GB/s, 16384x512 bf16
// with early loads 5575 -> 5647. The fp16 form, fma.rn.f32.f16, measured 9%
// slower at 131072x4096, so fp16 keeps the widening; products of pairs taken
// with mul.rn.f32x2 in the scale step measured neutral to 7% slower.)
__device__ __forceinline__ float sumsq2_bf16(uint32_t u, float acc) {
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n"
        " fma.rn.f32.bf16 %0, lo, lo, %0;\n fma.rn.f32.bf16 %0, hi, hi, %0;\n}"
        : "+f"(acc) : "r"(u));
    return acc;
}

// Sum of squares of the 8 elements of a vector, accumulated into acc in
// element order.
template <int DT>
__device__ __forceinline__ float sumsq8(const uint4& v, float acc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (DT == kBF16) {
            acc = sumsq2_bf16(w[k], acc);
        } else {
            const float2 f = Codec<DT>::unpack2(w[k]);
            acc = fmaf(f.x, f.x, acc);
            acc = fmaf(f.y, f.y, acc);
        }
    }
    return acc;
}

// y = (x * r) * s for 8 elements; s holds offset + w in fp32.
template <int DT>
__device__ __forceinline__ uint4 scale8(const uint4& v, float r, const float* s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float2 f = Codec<DT>::unpack2(w[k]);
        o[k] = Codec<DT>::pack2((f.x * r) * s[2 * k], (f.y * r) * s[2 * k + 1]);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// offset + w for the 8 weights of a vector, in fp32.
template <int DT>
__device__ __forceinline__ void weights8(const uint4& v, float offset, float* s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float2 f = Codec<DT>::unpack2(w[k]);
        s[2 * k] = offset + f.x;
        s[2 * k + 1] = offset + f.y;
    }
}

// One element in memory, for the element-wise kernel: its storage type, the
// widening to fp32 and the single rounding back.
template <int DT>
struct Elem {
    using T = uint16_t;
    static __device__ __forceinline__ float load(T u) { return Codec<DT>::unpack1(u); }
    static __device__ __forceinline__ T store(float f) { return Codec<DT>::pack1(f); }
};

template <>
struct Elem<kFP32> {
    using T = float;
    static __device__ __forceinline__ float load(T u) { return u; }
    static __device__ __forceinline__ T store(float f) { return f; }
};

// The forward's per-vector steps for any dtype: fp32 vectors are four floats
// (no conversion); 16-bit vectors go through the codecs above.
template <int DT>
__device__ __forceinline__ float sumsq_vec(const uint4& v, float acc) {
    if constexpr (DT == kFP32) {
        const float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                            __uint_as_float(v.w)};
#pragma unroll
        for (int k = 0; k < 4; ++k) acc = fmaf(f[k], f[k], acc);
        return acc;
    } else {
        return sumsq8<DT>(v, acc);
    }
}

// The same sum for fp16 by mixed-precision FMAs (fma.rn.f32.f16, sm_100 and
// later), which widen each element exactly: the bits of widening first and
// calling fmaf, without keeping the widened values live until the scale step
// (used by the TMA kernel's short-row instances, where that live range cost
// a resident CTA per SM).
__device__ __forceinline__ float sumsq2_f16(uint32_t u, float acc) {
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n"
        " fma.rn.f32.f16 %0, lo, lo, %0;\n fma.rn.f32.f16 %0, hi, hi, %0;\n}"
        : "+f"(acc) : "r"(u));
    return acc;
}

template <int DT>
__device__ __forceinline__ float sumsq_vec_packed(const uint4& v, float acc) {
    if constexpr (DT == kFP16) {
        acc = sumsq2_f16(v.x, acc);
        acc = sumsq2_f16(v.y, acc);
        acc = sumsq2_f16(v.z, acc);
        return sumsq2_f16(v.w, acc);
    } else {
        return sumsq_vec<DT>(v, acc);
    }
}

template <int DT>
__device__ __forceinline__ uint4 scale_vec(const uint4& v, float r, const float* s) {
    if constexpr (DT == kFP32) {
        return make_uint4(__float_as_uint((__uint_as_float(v.x) * r) * s[0]),
                          __float_as_uint((__uint_as_float(v.y) * r) * s[1]),
                          __float_as_uint((__uint_as_float(v.z) * r) * s[2]),
                          __float_as_uint((__uint_as_float(v.w) * r) * s[3]));
    } else {
        return scale8<DT>(v, r, s);
    }
}

template <int DT>
__device__ __forceinline__ void weights_vec(const uint4& v, float offset, float* s) {
    if constexpr (DT == kFP32) {
        s[0] = offset + __uint_as_float(v.x);
        s[1] = offset + __uint_as_float(v.y);
        s[2] = offset + __uint_as_float(v.z);
        s[3] = offset + __uint_as_float(v.w);
    } else {
        weights8<DT>(v, offset, s);
    }
}

// (offset + w) of vector c kept in shared memory as VecElems floats (float4
// reads), and the scale step with those weights.
template <int DT>
__device__ __forceinline__ void weights_from_smem(const float4* sw, int c, float* s) {
    constexpr int kE = VecElems<DT>::value;
#pragma unroll
    for (int q = 0; q < kE / 4; ++q) {
        const float4 t = sw[c * (kE / 4) + q];
        s[4 * q] = t.x;
        s[4 * q + 1] = t.y;
        s[4 * q + 2] = t.z;
        s[4 * q + 3] = t.w;
    }
}

template <int DT>
__device__ __forceinline__ uint4 scale_vec_smem(const uint4& v, float r, const float4* sw, int c) {
    float s[VecElems<DT>::value];
    weights_from_smem<DT>(sw, c, s);
    return scale_vec<DT>(v, r, s);
}

// All elements of a 16-byte vector widened to fp32, and the single rounding of
// a vector's worth of fp32 values back to the dtype.
template <int DT>
__device__ __forceinline__ void unpack_vec(const uint4& v, float* f) {
    if constexpr (DT == kFP32) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 p = Codec<DT>::unpack2(w[k]);
            f[2 * k] = p.x;
            f[2 * k + 1] = p.y;
        }
    }
}

template <int DT>
__device__ __forceinline__ uint4 pack_vec(const float* f) {
    if constexpr (DT == kFP32) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    } else {
        return make_uint4(Codec<DT>::pack2(f[0], f[1]), Codec<DT>::pack2(f[2], f[3]),
                          Codec<DT>::pack2(f[4], f[5]), Codec<DT>::pack2(f[6], f[7]));
    }
}

template <int DT>
__device__ __forceinline__ void weights_vec_to_smem(const uint4& wv, float offset, float4* sw,
                                                    int c) {
    constexpr int kE = VecElems<DT>::value;
    float s[kE];
    weights_vec<DT>(wv, offset, s);
#pragma unroll
    for (int q = 0; q < kE / 4; ++q)
        sw[c * (kE / 4) + q] = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
}

// Streaming global accesses: x and y are touched once, so they are loaded and
// stored with the evict-first (.cs) policy and do not displace the weights.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }

// y = (x * r) * s for 8 elements, with the 8 scales read as two float4 (from
// shared memory).
template <int DT>
__device__ __forceinline__ uint4 scale8(const uint4& v, float r, const float4& s0,
                                        const float4& s1) {
    const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    return scale8<DT>(v, r, s);
}

// Programmatic dependent launch. Every kernel is launched with programmatic
// stream serialisation allowed, so it may be scheduled while the previous
// kernel on the stream is finishing. pdl_wait() blocks until that kernel has
// completed and its memory is visible; it comes before the first global
// memory access. pdl_launch_dependents() lets the next kernel be scheduled
// into SM slots as this one's CTAs retire. Without a programmatic dependency
// both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// The per-row scalar step: mean of squares, plus eps, rsqrt.
__device__ __forceinline__ float row_rstd(float sumsq, float n, float eps) {
    return rsqrtf(__fdiv_rn(sumsq, n) + eps);
}

}  // namespace rmsn
