// Device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace moe {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// binary16 pair (low half = scale, high half = bias) -> float2
__device__ __forceinline__ float2 meta_to_f2(uint32_t m) {
    __half2 h = *reinterpret_cast<__half2*>(&m);
    return __half22float2(h);
}

// 4-bit code at bit offset `sh` of `w` as an exact float: the code is placed
// in the low mantissa bits of 2^23 and 2^23 is subtracted.
__device__ __forceinline__ float nib_f(uint32_t w, int sh) {
    return __uint_as_float(0x4B000000u | ((w >> sh) & 0xFu)) - 8388608.0f;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float load_act(const void* x, int is_bf16, size_t i) {
    if (is_bf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[i]);
    return static_cast<const float*>(x)[i];
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Row-record sizes (same definitions as the host side).
__host__ __device__ __forceinline__ size_t d_row_meta_bytes(int K) {
    return ((size_t)(K / 64) * 4 + 15) / 16 * 16;
}
__host__ __device__ __forceinline__ size_t d_row_bytes(int K) { return (size_t)K / 2 + d_row_meta_bytes(K); }

}  // namespace moe
