// Device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <climits>
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

// 2^f with max_abs * 2^f in [2^13, 2^14); 1 when max_abs is 0 or not finite.
// *inv gets 2^-f exactly (f <= 127, so 2^-f >= 2^-127, the one subnormal case).
__device__ __forceinline__ float q16_scale(float max_abs, float* inv) {
    const uint32_t u = __float_as_uint(max_abs);
    const int ex = (int)((u >> 23) & 0xFF);
    if (ex == 0 || ex == 0xFF) {
        *inv = 1.0f;
        return 1.0f;
    }
    int f = 13 - (ex - 127);
    f = max(-126, min(127, f));
    *inv = f == 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - f) << 23);
    return __uint_as_float((uint32_t)(f + 127) << 23);
}

// Quantise one run v[0..7] with scale sc into the staged uint4 layout. One
// fma with 1.5 * 2^23 + 128 per value: the sum lies in [2^23, 2^24), where the
// unit in the last place is 1, so the fma's rounding is the rounding of v * sc
// to the nearest integer q (ties to even: the added constant is even; sc is a
// power of two, so v * sc is exact), and the low 16 bits of the sum's bit
// pattern are t = q + 128 (|q| <= 2^14). Then hi = t >> 8 is byte 1 of t and
// lo = q - 256 hi = (t & 255) - 128 is byte 0 of t with its top bit flipped;
// byte permutes gather them.
__device__ __forceinline__ uint4 quant_run(const float* v, float sc) {
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = __float_as_uint(fmaf(v[i], sc, 12583040.0f));   // 1.5 * 2^23 + 128
    // pairs (i, i + 2): hi bytes (byte 1 of each), lo bytes (byte 0 of each)
    const uint32_t h02 = __byte_perm(t[0], t[2], 0x0051), h46 = __byte_perm(t[4], t[6], 0x0051);
    const uint32_t h13 = __byte_perm(t[1], t[3], 0x0051), h57 = __byte_perm(t[5], t[7], 0x0051);
    const uint32_t l02 = __byte_perm(t[0], t[2], 0x0040), l46 = __byte_perm(t[4], t[6], 0x0040);
    const uint32_t l13 = __byte_perm(t[1], t[3], 0x0040), l57 = __byte_perm(t[5], t[7], 0x0040);
    return make_uint4(__byte_perm(h02, h46, 0x5410), __byte_perm(h13, h57, 0x5410),
                      __byte_perm(l02, l46, 0x5410) ^ 0x80808080u, __byte_perm(l13, l57, 0x5410) ^ 0x80808080u);
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
    float isc;
    const float sc = q16_scale(m, &isc);
    const uint4 q = quant_run(v, sc);
    if (valid) {
        const int hg = r >> 2, wi = r & 3;
        xq[wi * KG + hg] = q;
        if (wi == 0) { inv[hg] = isc; X[hg] = s; }
    }
}

// Tag of one decode token's router partials: odd, so that a zeroed word
// never carries a valid tag; seq counts the layer's decodes on the device.
__device__ __forceinline__ unsigned decode_tag(unsigned seq) { return (seq << 1) | 1u; }

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

// Top k of the keys sl[0..E) (shared memory): the first k experts in the
// order by (-key, e), NaN keys counted as -inf. Each expert gets a unique
// 64-bit sort key, (order-preserving image of its key) << 32 | ~e, so that the
// order is plain integer order. Two levels of ranking by counting: warp w
// ranks each expert of chunk w (E / warps contiguous experts) among the chunk,
// and those of chunk rank < k become candidates; each candidate is then
// ranked among all candidates, and the candidate of rank r < k is selection
// r. This is exact: an expert that comes before one of the first k is itself
// among the first k and comes before it in their common chunk too, so all of
// the first k are candidates and their rank among candidates is their rank
// among all experts. The counting loops have fixed trip counts (chunks of at
// most 32 experts, at most 64 candidates) so that their shared-memory reads
// are all in flight together. Weights (one warp, each lane one selection; the
// hardware exponential and division, ~1e-6 relative): the softmax over the
// selected keys (the first selected is the maximum), or,
// when `score` is given (sigmoid scoring), scale * score_j / sum over the
// selection of score; the sum runs in selection order. Ends with the block
// synchronised. blockDim.x = 256 (8 warps), E <= 1024.
__device__ __forceinline__ void block_topk(const float* sl, int E, int k, int32_t* ids_out, float* w_out,
                                           const float* score = nullptr, float scale = 1.0f) {
    constexpr int NW = 8, NC = NW * MOE_MAX_TOP_K;   // warps, candidate places
    __shared__ __align__(16) unsigned long long s_key[1024];
    __shared__ __align__(16) unsigned long long s_cand[NC];   // 0: no candidate
    __shared__ int s_sel[MOE_MAX_TOP_K];
    __shared__ int s_rank[NC];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        s_key[e] = ((unsigned long long)key_img(sl[e]) << 32) | (uint32_t)~(uint32_t)e;
    if (threadIdx.x < NC) {
        s_cand[threadIdx.x] = 0ull;
        s_rank[threadIdx.x] = 0;
    }
    __syncthreads();
    const int C = (E + NW - 1) / NW;
    const int c0 = min(E, warp * C), c1 = min(E, c0 + C);
    if (C <= 32) {
        // one expert per lane, ranked against the 32 places of the chunk
        // (places past the chunk's end count as absent)
        const int e = c0 + lane;
        const unsigned long long me = e < c1 ? s_key[e] : 0ull;
        int rank = 0;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const ulonglong2 q = *reinterpret_cast<const ulonglong2*>(s_key + (c0 & ~1) + j);
            const int ja = (c0 & ~1) + j;
            rank += (ja >= c0 && ja < c1 && q.x > me) + (ja + 1 >= c0 && ja + 1 < c1 && q.y > me);
        }
        if (e < c1 && rank < k) s_cand[warp * k + rank] = me;
    } else {
        for (int e = c0 + lane; e < c1; e += 32) {
            const unsigned long long me = s_key[e];
            int rank = 0;
            for (int j = c0; j < c1; ++j) rank += s_key[j] > me;
            if (rank < k) s_cand[warp * k + rank] = me;
        }
    }
    __syncthreads();
    {
        // thread t counts the candidates of quarter t / NC that come before
        // candidate t % NC; the four counts add up in shared memory
        const int c = threadIdx.x % NC, q4 = threadIdx.x / NC;
        const unsigned long long me = s_cand[c];
        int rank = 0;
#pragma unroll
        for (int i = 0; i < NC / 8; ++i) {
            const ulonglong2 q = *reinterpret_cast<const ulonglong2*>(s_cand + q4 * (NC / 4) + 2 * i);
            rank += (q.x > me) + (q.y > me);
        }
        if (rank) atomicAdd(&s_rank[c], rank);
    }
    __syncthreads();
    if (threadIdx.x < NC) {
        const unsigned long long me = s_cand[threadIdx.x];
        const int rank = s_rank[threadIdx.x];
        if (me != 0ull && rank < k) s_sel[rank] = (int)~(uint32_t)me;
    }
    __syncthreads();
    if (warp == 0) {
        // lane r computes term r; the sum runs in selection order (gathered by
        // shuffles); lane r writes selection r
        const int r = lane < k ? lane : 0;
        const int e = s_sel[r], e0 = s_sel[0];
        float v = sl[e], v0 = sl[e0];
        v = (v != v) ? -INFINITY : v;
        v0 = (v0 != v0) ? -INFINITY : v0;
        // the hardware exponential: relative error ~1e-6 here (v - v0 <= 0)
        const float ex = score ? score[e] : __expf(v - v0);
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOP_K; ++j) {
            const float t = __shfl_sync(0xffffffffu, ex, j);
            if (j < k) den += t;
        }
        if (lane < k) {
            ids_out[lane] = e;
            w_out[lane] = __fdividef(ex, den) * (score ? scale : 1.0f);   // den in (0, k]: within 2 ulp
        }
    }
    __syncthreads();
}

}  // namespace moe
