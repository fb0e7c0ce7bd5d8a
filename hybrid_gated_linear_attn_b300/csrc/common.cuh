// common.cuh -- element access and small math shared by the Lizard kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lizard {

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// log(sigmoid(x)) = min(x, 0) - log(1 + e^{-|x|}); the exp argument is never
// positive, so neither tail overflows.  Gate of the GLA branch (Lizard,
// gist.science/de section 2, item 1: Gamma = sigmoid(W x)).
__device__ __forceinline__ float log_sigmoid(float x) { return fminf(x, 0.f) - log1pf(expf(-fabsf(x))); }

// Four consecutive elements as fp32 (16-byte load for fp32, 8-byte for bf16).
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p)
{
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v)
{
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Grouped key/value heads: query head h of a batch row reads key/value head
// h / group of that row (group = H / Hkv; 1 when every head has its own).
__host__ __device__ __forceinline__ int kv_unit(int unit, int H, int group)
{
    return (unit / H) * (H / group) + (unit % H) / group;
}
// The anchor weight of head h: per head when alpha_h is given.
__device__ __forceinline__ float head_alpha(const float *alpha_h, float alpha, int h)
{
    return alpha_h ? alpha_h[h] : alpha;
}

// Library-wide device error word.  A kernel that abandons a bounded wait,
// or finds a state it cannot use, records a code here and skips the work;
// the host reads and clears it (lizard_check_device_status).  The library is
// compiled as one translation unit, so this is the only definition.
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_POS = 2 };
__device__ int g_device_error = DEV_OK;

}  // namespace lizard
