// Device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "moe.h"
#include "route_mode.h"

namespace moe {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// L2 policy for weights read exactly once per token: evict them first, so that
// data staged for later (prefetched rows, activations) stays resident.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ldg_stream_hint(const void* p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint32_t ldg_u32_hint(const void* p, uint64_t pol) {
    uint32_t r;
    asm volatile("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
    return r;
}
// Asynchronous prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2_hint(const void* p, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(pol)
                 : "memory");
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

namespace moe {

// ---- programmatic dependent launch ------------------------------------------------
// Wait until the preceding kernel in the stream has completed and its memory is
// visible (a no-op when the kernel was launched without the PDL attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to be scheduled (it still waits with pdl_wait).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- 4-bit x fp16-pair dot products ------------------------------------------------
//
// Codes: a 16-byte chunk holds the 32 nibbles of half a group (32 inputs),
// element k in byte k/2, low nibble for even k. One 32-bit word w holds the 8
// elements of a run. Two nibbles at a time become a pair of binary16 values by
// masking into the mantissa of 1024: bits 0..3 of each 16-bit half give
// 1024 + q (elements 0, 4 and, after w >> 8, elements 2, 6), bits 4..7 give
// 1024 + 16 q (elements 1, 5, 3, 7). Each half is multiplied by a binary16
// activation with one mixed-precision FMA (f16 x f16 + f32), exact in the
// product, accumulated in fp32.
//
// The activations are staged as x' = x * 2^e (e per vector, keeps
// |x * 2^e| < 2^11), times 16 at even k, in binary16 pairs {(x'0,x'4),
// (x'1,x'5), (x'2,x'6), (x'3,x'7)} per run. Then for a half-group
//   A = sum_k f_k x'_k = Z + 16 * 2^e * sum_k q_k x_k,  Z = 1024 * sum_k x'_k,
// and the affine sum is sum_k (q_k s + b) x_k = s (A - Z) / (16 * 2^e) + b X,
// X = sum_k x_k. Z and X are precomputed per half-group.

__device__ __forceinline__ float hfma_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %3;}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float hfma_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %3;}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void word_f16(uint32_t w, const uint4 xp, float& a0, float& a1) {
    const uint32_t w8 = w >> 8;
    const uint32_t p0 = (w & 0x000F000Fu) | 0x64006400u;
    const uint32_t p1 = (w & 0x00F000F0u) | 0x64006400u;
    const uint32_t p2 = (w8 & 0x000F000Fu) | 0x64006400u;
    const uint32_t p3 = (w8 & 0x00F000F0u) | 0x64006400u;
    a0 = hfma_lo(p0, xp.x, a0);
    a1 = hfma_hi(p0, xp.x, a1);
    a0 = hfma_lo(p1, xp.y, a0);
    a1 = hfma_hi(p1, xp.y, a1);
    a0 = hfma_lo(p2, xp.z, a0);
    a1 = hfma_hi(p2, xp.z, a1);
    a0 = hfma_lo(p3, xp.w, a0);
    a1 = hfma_hi(p3, xp.w, a1);
}

__device__ __forceinline__ uint32_t u4w(const uint4 c, int i) { return i == 0 ? c.x : i == 1 ? c.y : i == 2 ? c.z : c.w; }

// 2^e with |max_abs * 2^e| in [2^10, 2^11); 1 when max_abs is 0 or not finite
__device__ __forceinline__ float pow2_scale(float max_abs) {
    const uint32_t u = __float_as_uint(max_abs);
    const int ex = (int)((u >> 23) & 0xFF);
    if (ex == 0 || ex == 0xFF) return 1.0f;
    int e = 10 - (ex - 127);
    e = max(-126, min(127, e));
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

// Stage one 8-element run v[0..7] (already times the vector scale) as x'
// pairs; the run's share of Z (1024 * sum of staged values) and of X (sum of
// v / scale). HILO also produces the residual pairs fp16(v' - fp16(v')).
template <bool HILO>
__device__ __forceinline__ void stage_run(const float* v, float inv_scale, uint4& hi, uint4& lo, float& Z, float& X) {
    float vp[8], z = 0.f, x = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        vp[i] = (i & 1) ? v[i] : 16.0f * v[i];
        x += v[i];
    }
    uint32_t hw[4], lw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half h0 = __float2half_rn(vp[i]), h1 = __float2half_rn(vp[i + 4]);
        hw[i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
        const float r0 = __half2float(h0), r1 = __half2float(h1);
        z += r0 + r1;
        if (HILO) {
            const __half l0 = __float2half_rn(vp[i] - r0), l1 = __float2half_rn(vp[i + 4] - r1);
            lw[i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            z += __half2float(l0) + __half2float(l1);
        }
    }
    hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    Z = 1024.0f * z;
    X = x * inv_scale;
}

}  // namespace moe

namespace moe {

// ---- 4-bit x 16-bit fixed-point dot products (integer dp4a) -------------------------
//
// A code word w holds the 8 nibbles of a run (element k in byte k/2, low nibble
// for even k); w & 0x0F0F0F0F gives the even elements as bytes 0..3 and
// (w >> 4) & 0x0F0F0F0F the odd ones. Activations are staged per half-group of
// 32 inputs as 16-bit fixed point, X16 = rne(x * 2^f) with 2^f chosen so that
// max |x| of the half-group times 2^f lies in [2^13, 2^14), split exactly as
// X16 = 256 * hi + lo with hi, lo signed bytes. A run is stored as one uint4
// {hi of even k, hi of odd k, lo of even k, lo of odd k} (byte i = element
// 2i or 2i+1), so that four dp4a give sum_k q_k * hi_k and sum_k q_k * lo_k in
// exact int32 arithmetic. The half-group's sum_k q_k x_k is then
// (256 * acc_hi + acc_lo) * 2^-f (the int32 is below 2^24, exact in fp32), and
// the affine group sum is s * that + b * X with X = sum_k x_k (fp32).

__device__ __forceinline__ void word_dp4a(uint32_t w, const uint4 xs, int& ah, int& al) {
    const uint32_t e = w & 0x0F0F0F0Fu, o = (w >> 4) & 0x0F0F0F0Fu;
    ah = __dp4a((int)e, (int)xs.x, ah);
    ah = __dp4a((int)o, (int)xs.y, ah);
    al = __dp4a((int)e, (int)xs.z, al);
    al = __dp4a((int)o, (int)xs.w, al);
}

// 2^f with max_abs * 2^f in [2^13, 2^14); 1 when max_abs is 0 or not finite
__device__ __forceinline__ float q16_scale(float max_abs) {
    const uint32_t u = __float_as_uint(max_abs);
    const int ex = (int)((u >> 23) & 0xFF);
    if (ex == 0 || ex == 0xFF) return 1.0f;
    int f = 13 - (ex - 127);
    f = max(-126, min(127, f));
    return __uint_as_float((uint32_t)(f + 127) << 23);
}

// Quantise one run v[0..7] with scale sc into the staged uint4 layout. The
// rounding to the nearest integer (ties to even) is one fma with 1.5 * 2^23:
// the sum lies in [2^23, 2^24), where the unit in the last place is 1, so the
// fma's rounding is the rounding to an integer, and the integer is the low
// bits of the sum (sc is a power of two, so v * sc is exact).
__device__ __forceinline__ uint4 quant_run(const float* v, float sc) {
    uint32_t he = 0, ho = 0, le = 0, lo = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = __float_as_int(fmaf(v[i], sc, 12582912.0f)) - 0x4B400000;   // |q| <= 2^14
        const int h = (q + 128) >> 8;                  // floor((q + 128) / 256)
        const int l = q - 256 * h;                     // in [-128, 127]
        const uint32_t hb = (uint32_t)(h & 0xFF), lb = (uint32_t)(l & 0xFF);
        const int sh = 8 * (i >> 1);
        if (i & 1) { ho |= hb << sh; lo |= lb << sh; }
        else { he |= hb << sh; le |= lb << sh; }
    }
    return make_uint4(he, ho, le, lo);
}

// Stage runs of a vector: called by whole warps with a warp-uniform trip count;
// `v` holds this lane's run (8 values, zero when !valid), lanes 4h..4h+3 hold
// the runs of half-group h (requires the run index to be 4-aligned per warp).
// Writes xq[wi * KG + hg], inv[hg] = 2^-f, X[hg] = sum of the 32 values.
__device__ __forceinline__ void stage_q16_run(const float* v, bool valid, int r, int KG, uint4* xq, float* inv,
                                              float* X) {
    float m = 0.f, s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) { m = fmaxf(m, fabsf(v[i])); s += v[i]; }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    const float sc = q16_scale(m);
    const uint4 q = quant_run(v, sc);
    if (valid) {
        const int hg = r >> 2, wi = r & 3;
        xq[wi * KG + hg] = q;
        if (wi == 0) { inv[hg] = 1.0f / sc; X[hg] = s; }
    }
}

// Token scale: the exponent a with max_abs * 2^a in [1, 2) (0 when max_abs is
// 0, subnormal or not finite). Activations are staged as x * 2^a, so that the
// staged values and everything computed from them stay far from both ends of
// the fp32 range whatever the token's magnitude; results are scaled back by
// exact powers of two.
__device__ __forceinline__ int token_exp(float max_abs) {
    const int ex = (int)((__float_as_uint(max_abs) >> 23) & 0xFF);
    if (ex == 0 || ex == 0xFF) return 0;
    return max(-126, min(126, 127 - ex));
}
__device__ __forceinline__ float exp2i(int a) { return __uint_as_float((uint32_t)(a + 127) << 23); }   // |a| <= 126

// Prefill operands: the exponent e with max_abs * 2^e in [2^14, 2^15), so that
// values times 2^e lie well inside the binary16 range while keeping its full
// precision (0 for a zero, subnormal or non-finite maximum; |e| <= 126).
__device__ __forceinline__ int fp16_fit_exp(float max_abs) {
    const int ex = (int)((__float_as_uint(max_abs) >> 23) & 0xFF);
    if (ex == 0 || ex == 0xFF) return 0;
    return max(-126, min(126, 141 - ex));
}

}  // namespace moe

namespace moe {
// Phase stamp (global timer, ns) for the decode trace: thread 0 of CTA `cta`
// writes point `p` of its 4-entry record when tracing is on (tr != null).
__device__ __forceinline__ void ktrace(unsigned long long* tr, int cta, int p) {
    if (tr && threadIdx.x == 0 && cta < MOE_TRACE_MAX_CTAS) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        tr[(size_t)cta * 4 + p] = t;
    }
}
}  // namespace moe

namespace moe {

// ---- exact top-k + softmax over the selected keys, one CTA ----------------------------
//
// Selection is the first k of the experts ordered by (-key_e, e): the largest
// key first, the lower index on equal values; NaN keys count as -inf.

// Order-preserving unsigned image of a key (NaN as -inf, -0 as +0): a > b as
// floats iff img(a) > img(b), equal floats have equal images.
__device__ __forceinline__ uint32_t key_img(float v) {
    if (v != v) v = -INFINITY;
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Selection key of one expert from its logit l and bias b (b = 0 without a
// bias). softmax: the biased logit. sigmoid (DeepSeek-V3-style router of the
// Colibri README, "What's implemented"): the score s = 1 / (1 + e^-l), written
// to *score, plus the bias, which steers the selection only.
__device__ __forceinline__ float route_key(float l, float b, RouteMode m, float* score) {
    if (!m.sigmoid) return l + b;
    const float sc = 1.0f / (1.0f + expf(-l));
    *score = sc;
    return sc + b;
}

// Top k of the keys sl[0..E) (shared memory) by rank: every thread takes
// experts e = tid, tid + blockDim, ... and counts the experts that come before
// e in the order; the expert of rank r < k is selection r. The ranks are a
// permutation (the index breaks ties), so each r < k is written exactly once.
// su: shared scratch of round4(E) words. Weights, by thread 0 in selection
// order: the softmax over the selected keys (the first selected is the
// maximum), or, when `score` is given (sigmoid scoring), scale * score_j / sum
// over the selection of score. Ends with the block synchronised; E <= 1024.
__device__ __forceinline__ void block_topk_rank(const float* sl, uint32_t* su, int E, int k, int32_t* ids_out,
                                                float* w_out, const float* score = nullptr, float scale = 1.0f) {
    __shared__ float s_v[MOE_MAX_TOP_K];
    __shared__ int s_i[MOE_MAX_TOP_K];
    const int E4 = (E + 3) & ~3;
    for (int e = threadIdx.x; e < E4; e += blockDim.x) su[e] = e < E ? key_img(sl[e]) : key_img(-INFINITY);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const uint32_t ue = su[e];
        int rank = 0;
        for (int j0 = 0; j0 < E4; j0 += 4) {
            const uint4 q = *reinterpret_cast<const uint4*>(su + j0);
            // (j < e and u_j >= u_e) or (j > e and u_j > u_e); padding never
            // counts (it equals -inf and lies past every real index)
            rank += (q.x > ue) | ((q.x == ue) & (j0 + 0 < e));
            rank += (q.y > ue) | ((q.y == ue) & (j0 + 1 < e));
            rank += (q.z > ue) | ((q.z == ue) & (j0 + 2 < e));
            rank += (q.w > ue) | ((q.w == ue) & (j0 + 3 < e));
        }
        if (rank < k) {
            const float v = sl[e];
            s_v[rank] = (v != v) ? -INFINITY : v;
            s_i[rank] = e;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float ex[MOE_MAX_TOP_K], den = 0.f;
#pragma unroll
        for (int r = 0; r < MOE_MAX_TOP_K; ++r)
            if (r < k) {
                ex[r] = score ? score[s_i[r]] : expf(s_v[r] - s_v[0]);
                den += ex[r];
            }
        const float mul = score ? scale : 1.0f;
#pragma unroll
        for (int r = 0; r < MOE_MAX_TOP_K; ++r)
            if (r < k) { ids_out[r] = s_i[r]; w_out[r] = ex[r] / den * mul; }
    }
    __syncthreads();
}

}  // namespace moe
