// op16.cuh -- the 16-bit MMA operand types of the tensor-core kernels and their conversions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gcl {

// The 16-bit operand types of the tensor-core paths: bf16 (every variant) and fp16 (GDN's
// forward, whose MMA operands and records are then all fp16: one kind::f16 instruction takes
// A and B of the same type).
template <typename T> struct Op16;
template <> struct Op16<__nv_bfloat16> {
    static constexpr uint32_t fmt = 1;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&t);
    }
    static __device__ __forceinline__ float2 unpack2(uint32_t w) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    }
    static __device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_float(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Op16<__half> {
    static constexpr uint32_t fmt = 0;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __half2 t = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&t);
    }
    static __device__ __forceinline__ float2 unpack2(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    static __device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_float(float x) { return __float2half_rn(x); }
};

template <typename T>
__device__ __forceinline__ uint4 pack8_as(const float *x) {
    uint4 pk;
    uint32_t *pw = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
    for (int e = 0; e < 4; ++e) pw[e] = Op16<T>::pack2(x[2 * e], x[2 * e + 1]);
    return pk;
}
// Eight 16-bit values of a uint4 as floats.
template <typename T>
__device__ __forceinline__ void unpack8_as(const uint4 &v, float *x) {
    const uint32_t *pw = reinterpret_cast<const uint32_t *>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = Op16<T>::unpack2(pw[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

}  // namespace gcl
