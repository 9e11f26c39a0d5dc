// Device helpers shared by the library's kernels (not by the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

constexpr int kChunk = 64;  // chunk length of the chunked prefill

// ---- scalar conversions ----------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// ---- short vector loads / stores (N consecutive elements, converted) -------
// N * sizeof(T) must be 4, 8 or 16 bytes and the address aligned to that size.
template <typename T, int N> struct Vec;

template <> struct Vec<float, 4> {
    static __device__ __forceinline__ void load(const float* p, float* out) {
        float4 t = *reinterpret_cast<const float4*>(p);
        out[0] = t.x; out[1] = t.y; out[2] = t.z; out[3] = t.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* in) {
        *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
    // streaming store (evict-first): data this kernel never reads back
    static __device__ __forceinline__ void store_cs(float* p, const float* in) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(in[0], in[1], in[2], in[3]));
    }
};
template <> struct Vec<float, 2> {
    static __device__ __forceinline__ void load(const float* p, float* out) {
        float2 t = *reinterpret_cast<const float2*>(p);
        out[0] = t.x; out[1] = t.y;
    }
    static __device__ __forceinline__ void store(float* p, const float* in) {
        *reinterpret_cast<float2*>(p) = make_float2(in[0], in[1]);
    }
    static __device__ __forceinline__ void store_cs(float* p, const float* in) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(in[0], in[1]));
    }
};
template <> struct Vec<__nv_bfloat16, 4> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* out) {
        uint2 t = *reinterpret_cast<const uint2*>(p);
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&t.x);
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&t.y);
        float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        out[0] = fa.x; out[1] = fa.y; out[2] = fb.x; out[3] = fb.y;
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* in) {
        __nv_bfloat162 a = __floats2bfloat162_rn(in[0], in[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(in[2], in[3]);
        uint2 t;
        t.x = *reinterpret_cast<uint32_t*>(&a);
        t.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = t;
    }
    // streaming store (evict-first): data this kernel never reads back
    static __device__ __forceinline__ void store_cs(__nv_bfloat16* p, const float* in) {
        __nv_bfloat162 a = __floats2bfloat162_rn(in[0], in[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(in[2], in[3]);
        uint2 t;
        t.x = *reinterpret_cast<uint32_t*>(&a);
        t.y = *reinterpret_cast<uint32_t*>(&b);
        __stcs(reinterpret_cast<uint2*>(p), t);
    }
};
template <> struct Vec<__nv_bfloat16, 8> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* out) {
        uint4 t = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
};
template <> struct Vec<__nv_bfloat16, 2> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* out) {
        float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        out[0] = f.x; out[1] = f.y;
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* in) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(in[0], in[1]);
    }
    static __device__ __forceinline__ void store_cs(__nv_bfloat16* p, const float* in) {
        __nv_bfloat162 a = __floats2bfloat162_rn(in[0], in[1]);
        __stcs(reinterpret_cast<unsigned int*>(p), *reinterpret_cast<unsigned int*>(&a));
    }
};

// ---- warp reductions -------------------------------------------------------
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// One halving step of a multi-value warp reduction: H values per lane become
// H/2, pairing lane with lane ^ OFF.  The lane whose OFF bit is set keeps the
// upper half.  Five steps (16,16) (8,8) (4,4) (2,2) (1,1) reduce 32 values per
// lane to one, and lane l then holds the full sum of value l.
template <int H, int OFF>
__device__ __forceinline__ void halve(float* x, int lane) {
    const bool up = (lane & OFF) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float send = up ? x[i] : x[i + H];
        const float keep = up ? x[i + H] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
    }
}

__device__ __forceinline__ float reduce32_to_lane(float (&x)[32], int lane) {
    halve<16, 16>(x, lane);
    halve<8, 8>(x, lane);
    halve<4, 4>(x, lane);
    halve<2, 2>(x, lane);
    halve<1, 1>(x, lane);
    return x[0];
}

// The last four steps: 16 values per lane (value i on lane l stands for value
// i of the lane's half-warp, i.e. index 16 * (l >> 4) + i) become one, lane l
// holding the full sum of index l.
__device__ __forceinline__ float reduce16_to_lane(float (&x)[32], int lane) {
    halve<8, 8>(x, lane);
    halve<4, 4>(x, lane);
    halve<2, 2>(x, lane);
    halve<1, 1>(x, lane);
    return x[0];
}

}  // namespace gdr
