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

// Quantise one run v[0..7] with scale sc into the staged uint4 layout.
__device__ __forceinline__ uint4 quant_run(const float* v, float sc) {
    uint32_t he = 0, ho = 0, le = 0, lo = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = __float2int_rn(v[i] * sc);       // |q| <= 2^14
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

// ---- exact top-k + softmax over the selected logits, one 256-thread CTA --------------
//
// Selection is the first k of the experts ordered by (-l_e, e): the largest
// logit first, the lower index on equal values; NaN logits count as -inf so
// every round selects a valid expert.
// The warp's largest (bv, lowest bi among equal bv), in two warp reductions:
// the key as an unsigned integer of the same order (-0 taken as +0, so that
// equal floats stay equal), its maximum, then the smallest index holding it.
// bv is never NaN here; bi is at most INT_MAX.
__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
    const uint32_t u = __float_as_uint(bv + 0.0f);
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
    const uint32_t mi = __reduce_min_sync(0xffffffffu, key == mk ? (uint32_t)bi : 0xffffffffu);
    bv = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk);
    bi = (int)mi;
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

// Two stages without block-wide rounds: every warp selects the top k of its
// contiguous range of experts (k rounds of a warp argmax), then warp 0 selects
// the top k of the <= 8 * k candidates. The union of the per-range top-k holds
// the global top-k, so the result is the same selection. E <= 1024, at least
// 8 warps (warps beyond the eighth only join the barriers).
// Weights: the softmax over the selected keys, or, when `score` is given
// (sigmoid scoring), scale * score_j / sum over the selection of score.
__device__ __forceinline__ void block_topk_softmax(const float* sl, int E, int k, int32_t* ids_out, float* w_out,
                                                   const float* score = nullptr, float scale = 1.0f) {
    __shared__ float c_v[8 * MOE_MAX_TOP_K];
    __shared__ int c_i[8 * MOE_MAX_TOP_K];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunk = (E + 8 - 1) / 8;   // <= 128
    const int e0 = warp * chunk, e1 = min(E, e0 + chunk);
    float v[4];
    bool live[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int e = e0 + lane + 32 * m;
        live[m] = e < e1 && lane + 32 * m < chunk;
        const float t = live[m] ? sl[e] : -INFINITY;
        v[m] = (t != t) ? -INFINITY : t;
    }
    for (int r = 0; r < k && warp < 8; ++r) {   // warps 8 and up (larger blocks) take no range
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int e = e0 + lane + 32 * m;
            if (live[m] && (v[m] > bv || (v[m] == bv && e < bi))) { bv = v[m]; bi = e; }
        }
        warp_argmax(bv, bi);
        if (lane == 0) { c_v[warp * MOE_MAX_TOP_K + r] = bv; c_i[warp * MOE_MAX_TOP_K + r] = bi; }
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (e0 + lane + 32 * m == bi) live[m] = false;
    }
    __syncthreads();
    if (warp == 0) {
        const int n = 8 * k;   // candidates, <= 64
        float cv[2];
        int ci[2];
        bool cl[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int c = lane + 32 * m;
            cl[m] = c < n;
            const int w = c / (cl[m] ? k : 1), rr = c - w * (cl[m] ? k : 1);
            cv[m] = cl[m] ? c_v[w * MOE_MAX_TOP_K + rr] : -INFINITY;
            ci[m] = cl[m] ? c_i[w * MOE_MAX_TOP_K + rr] : INT_MAX;
        }
        float sel_l[MOE_MAX_TOP_K];
        int sel_i[MOE_MAX_TOP_K];
#pragma unroll
        for (int r = 0; r < MOE_MAX_TOP_K; ++r) {
            if (r >= k) break;
            float bv = -INFINITY;
            int bi = INT_MAX;
#pragma unroll
            for (int m = 0; m < 2; ++m)
                if (cl[m] && (cv[m] > bv || (cv[m] == bv && ci[m] < bi))) { bv = cv[m]; bi = ci[m]; }
            warp_argmax(bv, bi);
            sel_l[r] = bv;
            sel_i[r] = bi;
#pragma unroll
            for (int m = 0; m < 2; ++m)
                if (cl[m] && ci[m] == bi) cl[m] = false;
        }
        if (lane == 0) {
            // softmax over the selected keys (the first selected is the
            // maximum), or the selected sigmoid scores renormalised and scaled
            float ex[MOE_MAX_TOP_K], den = 0.f;
#pragma unroll
            for (int r = 0; r < MOE_MAX_TOP_K; ++r)
                if (r < k) {
                    ex[r] = score ? score[sel_i[r]] : expf(sel_l[r] - sel_l[0]);
                    den += ex[r];
                }
            const float mul = score ? scale : 1.0f;
#pragma unroll
            for (int r = 0; r < MOE_MAX_TOP_K; ++r)
                if (r < k) { ids_out[r] = sel_i[r]; w_out[r] = ex[r] / den * mul; }
        }
    }
}


// Sum the router's partial logits part[s][e] (s < splits <= 8, fixed order),
// apply the layer's scoring and bias, and select: selection keys into sl[E]
// and, for sigmoid scoring, the scores into ss[E] (both shared), ids /
// weights into ids_out / w_out (shared or global). All 256 threads; E <= 1024.
__device__ __forceinline__ void block_select(const float* part, int splits, int E, const float* bias, int k,
                                             float* sl, int32_t* ids_out, float* w_out, RouteMode mode,
                                             float* ss) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float v[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) v[s] = (s < splits) ? __ldcg(part + (size_t)s * E + e) : 0.f;
        float l = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) l += v[s];
        sl[e] = route_key(l, bias ? __ldg(bias + e) : 0.f, mode, ss + e);
    }
    __syncthreads();
    block_topk_softmax(sl, E, k, ids_out, w_out, mode.sigmoid ? ss : nullptr, mode.scale);
    __syncthreads();
}

}  // namespace moe
