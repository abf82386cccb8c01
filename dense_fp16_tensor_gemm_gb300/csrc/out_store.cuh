// out_store.cuh -- typed stores of Out elements: fp32 as computed, or rounded
// to nearest even into fp16 / bf16.  Stores use the streaming hint (.cs): Out
// is written once and never read back by the product.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gnt {

enum OutType { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

template <int OT>
struct OutStore;

template <>
struct OutStore<kOutF32> {
    using T = float;
    static __device__ __forceinline__ void st1(T* p, float v) { __stcs(p, v); }
    static __device__ __forceinline__ void st2(T* p, float a, float b) { __stcs(reinterpret_cast<float2*>(p), make_float2(a, b)); }
    static __device__ __forceinline__ void st4(T* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }
    static __device__ __forceinline__ void add1(T* p, float v) { atomicAdd(p, v); }
};

template <>
struct OutStore<kOutF16> {
    using T = unsigned short;  // fp16 bit pattern
    static __device__ __forceinline__ void st1(T* p, float v) { __stcs(p, __half_as_ushort(__float2half_rn(v))); }
    static __device__ __forceinline__ unsigned pack(float a, float b)
    {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const unsigned*>(&h);
    }
    static __device__ __forceinline__ void st2(T* p, float a, float b) { __stcs(reinterpret_cast<unsigned*>(p), pack(a, b)); }
    static __device__ __forceinline__ void st4(T* p, float4 v)
    {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack(v.x, v.y), pack(v.z, v.w)));
    }
    // never used: partial sums are only accumulated into fp32 Out
    static __device__ __forceinline__ void add1(T* p, float v) { st1(p, v); }
};

template <>
struct OutStore<kOutBF16> {
    using T = unsigned short;  // bf16 bit pattern
    static __device__ __forceinline__ void st1(T* p, float v)
    {
        __stcs(p, __bfloat16_as_ushort(__float2bfloat16_rn(v)));
    }
    static __device__ __forceinline__ unsigned pack(float a, float b)
    {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const unsigned*>(&h);
    }
    static __device__ __forceinline__ void st2(T* p, float a, float b) { __stcs(reinterpret_cast<unsigned*>(p), pack(a, b)); }
    static __device__ __forceinline__ void st4(T* p, float4 v)
    {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack(v.x, v.y), pack(v.z, v.w)));
    }
    static __device__ __forceinline__ void add1(T* p, float v) { st1(p, v); }
};

}  // namespace gnt
