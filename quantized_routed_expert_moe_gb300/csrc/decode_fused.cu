// Fused decode step: one persistent, cooperative kernel per token.
//
// Every CTA (one per SM) streams its share of the token's weight bytes through
// a shared-memory ring filled by one producer lane with bulk asynchronous
// copies (cp.async.bulk, completion counted on an mbarrier), while eight
// consumer warps dequantise and multiply. The CTA's work list is, in order:
//   P0  router rows (fp32 or 8-bit), partial logits to global memory;
//   P1  shared-expert gate/up rows (need no routing);
//   P2  routed-expert gate/up rows (the producer waits for the expert IDs);
//   P3  the CTA's block of output rows: down rows of every selected expert,
//       one (row block, slot) item at a time, then the weighted combine (the
//       consumers wait until every CTA has written its SwiGLU outputs; the
//       producer keeps prefetching down rows meanwhile).
// A control warp per CTA detects, through a global counter, the last router
// chunk of the grid and runs the exact top-k + softmax there, then publishes
// the IDs with a release flag. Every wait is bounded; a wait that runs out
// sets a sticky error bit, raises the CTA's abort flag and the CTA drains out.
// The last CTA to exit resets the grid counters, so the kernel can be
// relaunched (or replayed from a CUDA graph) without host bookkeeping.
//
// Router, exact top-8, shared expert overlapped with routing, combine:
// TurboFieldfare article, "token generation"; 4-bit/8-bit affine group-64
// weights: same article, "execution architecture".
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace fused {

constexpr int NCW = 8;                    // consumer warps
constexpr int PRODUCER = NCW;             // warp index of the producer
constexpr int CONTROL = NCW + 1;          // warp index of the control warp
constexpr int NT = (NCW + 2) * 32;
constexpr int STAGE = 16384;              // bytes per ring stage
constexpr int MAX_STAGES = 12;
constexpr int CTRL_BYTES = 8192;          // barriers, flags, logits scratch
constexpr int MAX_OWN_ROWS = 128;         // output rows one CTA owns in the down phase
constexpr uint32_t SPIN_LIMIT = 1u << 22; // ~0.5 s of polling with back-off

// grid counters (device, zero between launches)
enum { C_ROUTER = 0, C_IDS = 1, C_H = 2, C_EXIT = 3, C_ERR = 4, C_HMAX = 8 /* [k + 1] */ };
enum { ERR_IDS = 1, ERR_H = 2, ERR_STAGE = 4, ERR_CTRL = 8 };

struct Params {
    const uint8_t* const* rec_tab;
    const void* router;
    const float* router_bias;
    const void* x;
    void* y;
    float* y32;
    float* part;      // [E][nsr]
    float* h;         // [k + 1][I]
    float* logits;    // [E]
    int32_t* ids;     // [k]
    float* wts;       // [k]
    unsigned* ctr;    // grid counters
    int act_bf16;
    int H, I, E, k, n_shared, q8;
    int R, nsr;       // router K chunk and splits per row
    int p;            // gate/up row pairs per chunk
    int n_gu;         // gate/up chunks per slot
    int rbm;          // down rows per item (one slot)
    int stages;
    size_t rbH, rbI, gu_block;
    int union_bytes;
    int test_no_publish;  // test hook: never publish the IDs, so every wait on them runs out
    unsigned long long* trace;  // [grid][MOE_TRACE_POINTS] global-timer stamps, or null
};

__device__ __forceinline__ void tstamp(const Params& P, int point) {
    if (P.trace) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        P.trace[(size_t)blockIdx.x * MOE_TRACE_POINTS + point] = t;
    }
}

// ---- PTX helpers --------------------------------------------------------------
__device__ __forceinline__ uint32_t s_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t cnt) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(cnt) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
        : "=r"(ok) : "r"(b), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Bounded wait on an mbarrier phase. Returns false on timeout or abort.
__device__ __forceinline__ bool mbar_wait(uint32_t b, uint32_t parity, volatile int* abort) {
    for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
        if (mbar_try(b, parity)) return true;
        if (*abort) return false;
        if (i > 16) __nanosleep(64);
    }
    return false;
}

// ---- nibble dot products ---------------------------------------------------------
//
// Codes: a 16-byte chunk holds the 32 nibbles of half a group, element k in
// byte k/2, low nibble for even k. One 32-bit word w holds elements 0..7 of an
// 8-element run. Two nibbles at a time become a pair of binary16 values by
// masking into the mantissa of 1024: bits 0..3 of each half give 1024 + q
// (elements 0, 4 and, after w >> 8, 2, 6), bits 4..7 give 1024 + 16 q
// (elements 1, 5, 3, 7). Each half is multiplied by a binary16 activation and
// accumulated in fp32 with one mixed-precision FMA (f16 x f16 + f32), which
// is exact in the product.
//
// The staged activations x' are x * 2^e (e per token, keeps |x'| < 2^11) and
// additionally * 16 at even k, so that every product is 16 q x' / 16 ... more
// precisely A = sum_k f_k x'_k = Z + 16 * 2^e * sum_k q_k x_k, with
// Z = 1024 * sum_k x'_k precomputed per half-group. The affine group sum is
// then sum_k (q_k s + b) x_k = s (A - Z) / (16 * 2^e) + b X, X = sum_k x_k.

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

// x' pairs for one code word: {(x'0,x'4), (x'1,x'5), (x'2,x'6), (x'3,x'7)}
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

__device__ __forceinline__ uint32_t cw(const uint4 c, int i) { return i == 0 ? c.x : i == 1 ? c.y : i == 2 ? c.z : c.w; }

// R rows (R <= 4) of one half-group against single-precision pairs xq[4][stride]
template <int R>
__device__ __forceinline__ void hg_rows(const uint4* c, const uint4* xq, int stride, float* A) {
    float a0[R], a1[R];
#pragma unroll
    for (int r = 0; r < R; ++r) a0[r] = a1[r] = 0.f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint4 xp = xq[wi * stride];
#pragma unroll
        for (int r = 0; r < R; ++r) word_f16(cw(c[r], wi), xp, a0[r], a1[r]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) A[r] = a0[r] + a1[r];
}

// same with hi/lo pairs (two products per weight; ~22 bits of the activation)
template <int R>
__device__ __forceinline__ void hg_rows_hilo(const uint4* c, const uint4* xh, const uint4* xl, int stride, float* A) {
    float a0[R], a1[R];
#pragma unroll
    for (int r = 0; r < R; ++r) a0[r] = a1[r] = 0.f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint4 ph = xh[wi * stride], pl = xl[wi * stride];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            word_f16(cw(c[r], wi), ph, a0[r], a1[r]);
            word_f16(cw(c[r], wi), pl, a0[r], a1[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) A[r] = a0[r] + a1[r];
}

// Load 8 consecutive activations (bf16 or fp32) starting at element 8*ch.
__device__ __forceinline__ void load8_act(const void* src, int is_bf16, int ch, float* v) {
    if (is_bf16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(src) + ch);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4*>(src) + 2 * ch);
        const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 2 * ch + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// 2^e with |max_abs * 2^e| in [2^10, 2^11); 1 when max_abs is 0 or not finite
__device__ __forceinline__ float pow2_scale(float max_abs) {
    const uint32_t u = __float_as_uint(max_abs);
    const int ex = (int)((u >> 23) & 0xFF);
    if (ex == 0 || ex == 0xFF) return 1.0f;
    int e = 10 - (ex - 127);
    e = max(-126, min(127, e));
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const uint32_t a = __half_as_ushort(__float2half_rn(lo)), b = __half_as_ushort(__float2half_rn(hi));
    return a | (b << 16);
}

// Stage one half-group (32 values v[0..31], already multiplied by the token
// scale) as x' pairs; returns (Z, X-part) contributions through refs.
// Element order of v: v[8*wi + i]. hi/lo: lo pairs hold fp16(v' - fp16(v')).
template <bool HILO>
__device__ __forceinline__ void stage_hg(const float* v, float inv_scale, uint4* xh, uint4* xl, int stride,
                                         float& Z, float& X) {
    float z = 0.f, x = 0.f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        float vp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            vp[i] = (i & 1) ? v[8 * wi + i] : 16.0f * v[8 * wi + i];
            x += v[8 * wi + i];
        }
        uint32_t hw[4], lw[4];
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
        xh[wi * stride] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if (HILO) xl[wi * stride] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    Z = 1024.0f * z;
    X = x * inv_scale;
}

struct Work {
    int beg[3], cnt[4], tot;
    int own0, own1, nblk;   // down phase: owned output rows [own0, own1), row blocks
};

__device__ __forceinline__ void work_ranges(const Params& P, int c, int G, Work& w) {
    const int n[3] = {P.E * P.nsr, P.n_shared ? P.n_gu : 0, P.k * P.n_gu};
    w.tot = 0;
#pragma unroll
    for (int ph = 0; ph < 3; ++ph) {
        const int b = (int)((long long)n[ph] * c / G), e = (int)((long long)n[ph] * (c + 1) / G);
        w.beg[ph] = b;
        w.cnt[ph] = e - b;
        w.tot += e - b;
    }
    w.own0 = (int)((long long)P.H * c / G);
    w.own1 = (int)((long long)P.H * (c + 1) / G);
    w.nblk = (w.own1 - w.own0 + P.rbm - 1) / P.rbm;
    w.cnt[3] = w.nblk * (P.k + P.n_shared);
    w.tot += w.cnt[3];
}

// local chunk index -> (phase, item); phase-3 items are (block, slot) = (item / ns, item % ns)
__device__ __forceinline__ void locate(const Work& w, int lc, int& ph, int& item) {
    if (lc < w.cnt[0]) { ph = 0; item = w.beg[0] + lc; return; }
    lc -= w.cnt[0];
    if (lc < w.cnt[1]) { ph = 1; item = w.beg[1] + lc; return; }
    lc -= w.cnt[1];
    if (lc < w.cnt[2]) { ph = 2; item = w.beg[2] + lc; return; }
    ph = 3;
    item = lc - w.cnt[2];
}

// ---- the kernel -----------------------------------------------------------------

__global__ void __launch_bounds__(NT, 1) k_decode_fused(const Params P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + MAX_STAGES;
    volatile int* s_abort = reinterpret_cast<volatile int*>(empty + MAX_STAGES);
    volatile int* s_rdone = s_abort + 1;
    volatile int* s_last = s_abort + 2;
    volatile int* s_go = s_abort + 3;
    int* s_rows = const_cast<int*>(s_abort) + 4;                              // GU rows done by this CTA
    unsigned* s_hmax = reinterpret_cast<unsigned*>(const_cast<int*>(s_abort) + 8);   // [k + 1] |h| max bits
    float* s_w = reinterpret_cast<float*>(const_cast<int*>(s_abort) + 24);         // [k + 1] weight per down slot
    float* s_hsc = s_w + 16;                                                 // [k + 1] inverse h scale per slot
    const uint8_t** s_rec = reinterpret_cast<const uint8_t**>(smem + 512);  // [k + 1] record per slot
    float* s_logit = reinterpret_cast<float*>(smem + 1024);                 // [E] (control warp)
    uint8_t* s_taken = smem + 1024 + 4 * 1024;                              // [E]
    uint8_t* uni = smem + CTRL_BYTES;
    uint8_t* ring = uni + P.union_bytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int H = P.H, I = P.I, k = P.k;
    const int HG = H / 32, IG = I / 32;
    const int ns = k + P.n_shared;
    Work W;
    work_ranges(P, blockIdx.x, G, W);

    if (threadIdx.x == 0) {
        if (P.trace)
            for (int i = 1; i < MOE_TRACE_POINTS; ++i) P.trace[(size_t)blockIdx.x * MOE_TRACE_POINTS + i] = 0ull;
        tstamp(P, 0);
        for (int s = 0; s < P.stages; ++s) {
            mbar_init(s_addr(&full[s]), 1);
            mbar_init(s_addr(&empty[s]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
        *s_rdone = 0;
        *s_last = 0;
        *s_go = 0;
        *s_rows = 0;
    }
    if (threadIdx.x < MOE_MAX_TOP_K + 1) s_hmax[threadIdx.x] = 0u;
    __syncthreads();

    if (warp == PRODUCER) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool have_ids = false;
            // record base per slot (routed slots in selection order, then the
            // shared expert at slot k), read from global memory once per token
            if (P.n_shared) s_rec[k] = P.rec_tab[P.E];
            for (int lc = 0; lc < W.tot; ++lc) {
                if (*s_abort) break;
                int ph, item;
                locate(W, lc, ph, item);
                const int st = lc % P.stages;
                if (lc >= P.stages && !mbar_wait(s_addr(&empty[st]), ((lc / P.stages) - 1) & 1, s_abort)) {
                    atomicOr(&P.ctr[C_ERR], ERR_STAGE);
                    *s_abort = 1;
                    break;
                }
                if (ph >= 2 && !have_ids) {
                    bool ok = false;
                    for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
                        if (ld_acquire(&P.ctr[C_IDS]) != 0u) { ok = true; break; }
                        if (*s_abort) break;
                        __nanosleep(64);
                    }
                    if (!ok) {
                        atomicOr(&P.ctr[C_ERR], ERR_IDS);
                        *s_abort = 1;
                        break;
                    }
                    int ev[MOE_MAX_TOP_K];
#pragma unroll
                    for (int j = 0; j < MOE_MAX_TOP_K; ++j) ev[j] = (j < k) ? __ldcg(P.ids + j) : 0;
                    const uint8_t* rp[MOE_MAX_TOP_K];
#pragma unroll
                    for (int j = 0; j < MOE_MAX_TOP_K; ++j) {
                        const int e = ((unsigned)ev[j] < (unsigned)P.E) ? ev[j] : 0;
                        rp[j] = (j < k) ? P.rec_tab[e] : nullptr;
                    }
#pragma unroll
                    for (int j = 0; j < MOE_MAX_TOP_K; ++j)
                        if (j < k) s_rec[j] = rp[j];
                    have_ids = true;
                    tstamp(P, 4);
                }
                const uint32_t bar = s_addr(&full[st]);
                const uint32_t dst = s_addr(ring + (size_t)st * STAGE);
                if (ph == 0) {
                    const int e = item / P.nsr, sr = item - e * P.nsr;
                    if (!P.q8) {
                        const float* src = static_cast<const float*>(P.router) + (size_t)e * H + (size_t)sr * P.R;
                        mbar_expect_tx(bar, P.R * 4);
                        bulk_g2s(dst, src, P.R * 4, bar);
                    } else {
                        // codes only; the consumers read the small metadata directly
                        const uint8_t* codes = static_cast<const uint8_t*>(P.router) + (size_t)e * H + (size_t)sr * P.R;
                        mbar_expect_tx(bar, P.R);
                        bulk_g2s(dst, codes, P.R, bar);
                    }
                } else if (ph <= 2) {
                    const int j = (ph == 1) ? k : item / P.n_gu;
                    const int u = (ph == 1) ? item : item - j * P.n_gu;
                    const int i0 = u * P.p, i1 = min(I, i0 + P.p);
                    const uint8_t* src = s_rec[j] + (size_t)(2 * i0) * P.rbH;
                    const uint32_t bytes = (uint32_t)(2 * (i1 - i0) * P.rbH);
                    mbar_expect_tx(bar, bytes);
                    bulk_g2s(dst, src, bytes, bar);
                } else {
                    const int b = item / ns, s = item - b * ns;
                    const int n0 = W.own0 + b * P.rbm, n1 = min(W.own1, n0 + P.rbm);
                    const int j = (P.n_shared && s == 0) ? k : s - P.n_shared;
                    const uint8_t* src = s_rec[j] + P.gu_block + (size_t)n0 * P.rbI;
                    const uint32_t bytes = (uint32_t)((n1 - n0) * P.rbI);
                    mbar_expect_tx(bar, bytes);
                    bulk_g2s(dst, src, bytes, bar);
                }
            }
        }
    } else if (warp == CONTROL) {
        // ------------------------------------------------------------- control
        // Once this CTA's router chunks are all done, the consumer that
        // finished the grid's last router chunk (if it is in this CTA) has set
        // s_last: reduce the logits, select, publish.
        bool ok = W.cnt[0] == 0;
        for (uint32_t i = 0; !ok && i < SPIN_LIMIT; ++i) {
            if (*s_abort) break;
            if (*s_rdone >= W.cnt[0]) { ok = true; break; }
            __nanosleep(64);
        }
        if (lane == 0) tstamp(P, 2);
        if (!ok && !*s_abort && lane == 0) atomicOr(&P.ctr[C_ERR], ERR_CTRL);
        if (ok && W.cnt[0] > 0 && *s_last == 1 && !*s_abort && !P.test_no_publish) {
            __threadfence();
            const int E = P.E;
            for (int e0 = 0; e0 < E; e0 += 8 * 32) {
                float l[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {   // 8 logits per lane in flight
                    const int e = e0 + u * 32 + lane;
                    l[u] = 0.f;
                    if (e < E) {
                        for (int s = 0; s < P.nsr; ++s) l[u] += __ldcg(P.part + (size_t)e * P.nsr + s);
                        if (P.router_bias) l[u] += __ldg(P.router_bias + e);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = e0 + u * 32 + lane;
                    if (e < E) {
                        s_logit[e] = (l[u] != l[u]) ? -INFINITY : l[u];
                        s_taken[e] = 0;
                        P.logits[e] = l[u];
                    }
                }
            }
            __syncwarp();
            float sel_l[MOE_MAX_TOP_K];
            int sel_i[MOE_MAX_TOP_K];
#pragma unroll
            for (int r = 0; r < MOE_MAX_TOP_K; ++r) {
                if (r >= k) break;
                float bv = -INFINITY;
                int bi = INT_MAX;
                for (int e = lane; e < E; e += 32) {
                    const float v = s_logit[e];
                    if (!s_taken[e] && (v > bv || (v == bv && e < bi))) { bv = v; bi = e; }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
                }
                sel_l[r] = bv;
                sel_i[r] = bi;
                if (lane == 0) s_taken[bi] = 1;
                __syncwarp();
            }
            if (lane == 0) {
                float ex[MOE_MAX_TOP_K], den = 0.f;
#pragma unroll
                for (int r = 0; r < MOE_MAX_TOP_K; ++r)
                    if (r < k) { ex[r] = expf(sel_l[r] - sel_l[0]); den += ex[r]; }
#pragma unroll
                for (int r = 0; r < MOE_MAX_TOP_K; ++r)
                    if (r < k) { P.ids[r] = sel_i[r]; P.wts[r] = ex[r] / den; }
                __threadfence();
                st_release(&P.ctr[C_IDS], 1u);
                tstamp(P, 3);
            }
        }
    } else {
        // ----------------------------------------------------------- consumers
        const int ct = threadIdx.x;  // 0 .. NCW*32-1
        float* xf = reinterpret_cast<float*>(uni);                          // [H] plain x (router)
        uint4* xq = reinterpret_cast<uint4*>(uni + (size_t)H * 4);          // [4][HG] x' pairs
        float* Zx = reinterpret_cast<float*>(uni + (size_t)H * 6);          // [HG]
        float* Xx = Zx + HG;                                                // [HG]
        float* s_red = Xx + HG;                                             // [NCW] scratch
        // token scale: max |x| over H, every CTA computes the same value
        float mx = 0.f;
        {
            // 8 activations per thread per step, 4 steps of loads in flight
            const int nch = H / 8;
            for (int base = ct; base < nch; base += 4 * NCW * 32) {
                float v[4][8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int ch = base + u * NCW * 32;
                    if (ch < nch) load8_act(P.x, P.act_bf16, ch, v[u]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int ch = base + u * NCW * 32;
                    if (ch < nch) {
                        reinterpret_cast<float4*>(xf + 8 * ch)[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
                        reinterpret_cast<float4*>(xf + 8 * ch)[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[u][i]));
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_red[warp] = mx;
        named_sync(1, NCW * 32);
        mx = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) mx = fmaxf(mx, s_red[w]);
        const float xsc = pow2_scale(mx), inv_xsc = 1.0f / xsc;
        for (int hg = ct; hg < HG; hg += NCW * 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = xf[32 * hg + i] * xsc;
            stage_hg<false>(v, inv_xsc, xq + hg, nullptr, HG, Zx[hg], Xx[hg]);
        }
        named_sync(1, NCW * 32);
        const float gu_c = inv_xsc * 0.0625f;  // 1 / (16 * 2^e)
        if (ct == 0) tstamp(P, 1);

        const int nA = W.cnt[0] + W.cnt[1] + W.cnt[2];
        int rows_done = 0;
        for (int lc = warp; lc < nA; lc += NCW) {
            int ph, item;
            locate(W, lc, ph, item);
            const int st = lc % P.stages;
            if (!mbar_wait(s_addr(&full[st]), (lc / P.stages) & 1, s_abort)) {
                if (lane == 0) { atomicOr(&P.ctr[C_ERR], ERR_STAGE); *s_abort = 1; }
                break;
            }
            const uint8_t* buf = ring + (size_t)st * STAGE;
            if (ph == 0) {
                const int e = item / P.nsr, sr = item - e * P.nsr;
                const int k0 = sr * P.R;
                float acc = 0.f;
                if (!P.q8) {
                    const float4* w4 = reinterpret_cast<const float4*>(buf);
                    const float4* xv = reinterpret_cast<const float4*>(xf + k0);
                    for (int c = lane; c < P.R / 4; c += 32) {
                        const float4 a = w4[c], b = xv[c];
                        acc = fmaf(a.x, b.x, acc);
                        acc = fmaf(a.y, b.y, acc);
                        acc = fmaf(a.z, b.z, acc);
                        acc = fmaf(a.w, b.w, acc);
                    }
                } else {
                    const uint32_t* meta = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(P.router) +
                                                                             (size_t)P.E * H) +
                                           (size_t)e * (H / 64) + k0 / 64;
                    for (int c = lane; c < P.R / 16; c += 32) {
                        const uint4 q = *reinterpret_cast<const uint4*>(buf + 16 * c);
                        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
                        float aq = 0.f, ax = 0.f;
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const float xv = xf[k0 + 16 * c + t];
                            const float cv = __uint_as_float(0x4B000000u | ((qw[t >> 2] >> (8 * (t & 3))) & 0xFFu)) -
                                             8388608.0f;
                            aq = fmaf(cv, xv, aq);
                            ax += xv;
                        }
                        const float2 sb = meta_to_f2(__ldg(meta + (c >> 2)));
                        acc = fmaf(sb.x, aq, fmaf(sb.y, ax, acc));
                    }
                }
                acc = warp_sum(acc);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s_addr(&empty[st]));
                    P.part[(size_t)e * P.nsr + sr] = acc;
                    __threadfence();
                    const unsigned old = atomicAdd(&P.ctr[C_ROUTER], 1u);
                    if (old + 1 == (unsigned)(P.E * P.nsr)) *s_last = 1;
                    __threadfence_block();
                    atomicAdd(const_cast<int*>(s_rdone), 1);
                }
            } else {
                const int j = (ph == 1) ? k : item / P.n_gu;
                const int u = (ph == 1) ? item : item - j * P.n_gu;
                const int i0 = u * P.p, i1 = min(I, i0 + P.p);
                float hmax = 0.f;
                // two gate/up row pairs at a time: rows (gate i, up i, gate i+1, up i+1)
                for (int i = i0; i < i1; i += 2) {
                    const bool two = i + 1 < i1;
                    const uint8_t* r0 = buf + (size_t)(2 * (i - i0)) * P.rbH;
                    const uint8_t* rr[4] = {r0, r0 + P.rbH, two ? r0 + 2 * P.rbH : r0, two ? r0 + 3 * P.rbH : r0 + P.rbH};
                    float as[4] = {0.f, 0.f, 0.f, 0.f}, ab[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int hg = lane; hg < HG; hg += 32) {
                        uint4 c[4];
                        float2 sb[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            c[r] = *reinterpret_cast<const uint4*>(rr[r] + 16 * hg);
                            sb[r] = meta_to_f2(*reinterpret_cast<const uint32_t*>(rr[r] + H / 2 + 4 * (hg >> 1)));
                        }
                        float A[4];
                        hg_rows<4>(c, xq + hg, HG, A);
                        const float z = Zx[hg], xs = Xx[hg];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            as[r] = fmaf(sb[r].x, A[r] - z, as[r]);
                            ab[r] = fmaf(sb[r].y, xs, ab[r]);
                        }
                    }
                    float g[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) g[r] = warp_sum(fmaf(as[r], gu_c, ab[r]));
                    if (lane == 0) {
                        const float h0 = silu_f(g[0]) * g[1];
                        P.h[(size_t)j * I + i] = h0;
                        hmax = fmaxf(hmax, fabsf(h0));
                        if (two) {
                            const float h1 = silu_f(g[2]) * g[3];
                            P.h[(size_t)j * I + i + 1] = h1;
                            hmax = fmaxf(hmax, fabsf(h1));
                        }
                    }
                }
                rows_done += i1 - i0;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s_addr(&empty[st]));
                    if (hmax == hmax) atomicMax(&s_hmax[j], __float_as_uint(hmax));  // |h| >= 0: bits order as floats
                }
            }
        }

        // ------------------------------------------------ SwiGLU outputs barrier
        if (lane == 0 && rows_done) {
            __threadfence();
            atomicAdd(s_rows, rows_done);
        }
        named_sync(1, NCW * 32);
        if (ct == 0) {
            tstamp(P, 5);
            // publish this CTA's |h| maxima and row count, then wait for all rows
            for (int j = 0; j < ns; ++j) {
                const int jj = (j < k) ? j : k;
                if (s_hmax[jj]) atomicMax(&P.ctr[C_HMAX + jj], s_hmax[jj]);
            }
            __threadfence();
            if (*s_rows) atomicAdd(&P.ctr[C_H], (unsigned)*s_rows);
            const unsigned target = (unsigned)(ns * I);
            bool ok = false;
            for (uint32_t i = 0; !*s_abort && i < SPIN_LIMIT; ++i) {
                if (ld_acquire(&P.ctr[C_H]) >= target && ld_acquire(&P.ctr[C_IDS]) != 0u) { ok = true; break; }
                __nanosleep(128);
            }
            if (!ok && !*s_abort) { atomicOr(&P.ctr[C_ERR], ERR_H); *s_abort = 1; }
            *s_go = (!*s_abort && W.cnt[3] > 0) ? 1 : 0;
            tstamp(P, 6);
        }
        named_sync(1, NCW * 32);
        if (*s_go) {
            // stage h of every slot (shared first, then routed in selection order)
            // as hi/lo x' pairs with a per-slot power-of-two scale
            uint4* hh = reinterpret_cast<uint4*>(uni);                               // [ns][4][IG]
            uint4* hl = hh + (size_t)ns * 4 * IG;                                    // [ns][4][IG]
            float* Zh = reinterpret_cast<float*>(hl + (size_t)ns * 4 * IG);          // [ns][IG]
            float* Xh = Zh + ns * IG;                                                // [ns][IG]
            float* ypart = Xh + ns * IG;                                             // [ns][MAX_OWN_ROWS]
            if (ct < ns) {
                const bool sh = P.n_shared && ct == 0;
                const int j = sh ? k : ct - P.n_shared;
                s_w[ct] = sh ? 1.0f : __ldcg(P.wts + j);
                const float hm = __uint_as_float(ld_acquire(&P.ctr[C_HMAX + j]));
                s_hsc[ct] = pow2_scale(hm);
            }
            named_sync(1, NCW * 32);
            for (int idx = ct; idx < ns * IG; idx += NCW * 32) {
                const int s = idx / IG, hg = idx - s * IG;
                const int j = (P.n_shared && s == 0) ? k : s - P.n_shared;
                const float sc = s_hsc[s];
                const float4* src = reinterpret_cast<const float4*>(P.h + (size_t)j * I + 32 * hg);
                float v[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 t = __ldcg(src + q);
                    v[4 * q] = t.x * sc;
                    v[4 * q + 1] = t.y * sc;
                    v[4 * q + 2] = t.z * sc;
                    v[4 * q + 3] = t.w * sc;
                }
                stage_hg<true>(v, 1.0f / sc, hh + (size_t)s * 4 * IG + hg, hl + (size_t)s * 4 * IG + hg, IG,
                               Zh[idx], Xh[idx]);
            }
            named_sync(1, NCW * 32);

            if (ct == 0) tstamp(P, 7);
            const int nB = W.tot;
            const int first = nA + ((warp - nA % NCW) + NCW) % NCW;  // keep the round-robin of chunks
            for (int lc = first; lc < nB; lc += NCW) {
                const int item = lc - nA;
                const int b = item / ns, s = item - b * ns;
                const int st = lc % P.stages;
                if (!mbar_wait(s_addr(&full[st]), (lc / P.stages) & 1, s_abort)) {
                    if (lane == 0) { atomicOr(&P.ctr[C_ERR], ERR_STAGE); *s_abort = 1; }
                    break;
                }
                const uint8_t* buf = ring + (size_t)st * STAGE;
                const int n0 = W.own0 + b * P.rbm, n1 = min(W.own1, n0 + P.rbm);
                const uint4* xh = hh + (size_t)s * 4 * IG;
                const uint4* xl = hl + (size_t)s * 4 * IG;
                const float* zs = Zh + s * IG;
                const float* xs = Xh + s * IG;
                const float dc = 0.0625f / s_hsc[s];
                for (int n = n0; n < n1; n += 4) {
                    const int nr = min(4, n1 - n);
                    const uint8_t* rr[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) rr[r] = buf + (size_t)(n - n0 + min(r, nr - 1)) * P.rbI;
                    float as[4] = {0.f, 0.f, 0.f, 0.f}, ab[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int hg = lane; hg < IG; hg += 32) {
                        uint4 c[4];
                        float2 sb[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            c[r] = *reinterpret_cast<const uint4*>(rr[r] + 16 * hg);
                            sb[r] = meta_to_f2(*reinterpret_cast<const uint32_t*>(rr[r] + I / 2 + 4 * (hg >> 1)));
                        }
                        float A[4];
                        hg_rows_hilo<4>(c, xh + hg, xl + hg, IG, A);
                        const float z = zs[hg], xx = xs[hg];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            as[r] = fmaf(sb[r].x, A[r] - z, as[r]);
                            ab[r] = fmaf(sb[r].y, xx, ab[r]);
                        }
                    }
                    float d[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) d[r] = warp_sum(fmaf(as[r], dc, ab[r]));
                    if (lane < nr) {
                        const float dv = lane == 0 ? d[0] : lane == 1 ? d[1] : lane == 2 ? d[2] : d[3];
                        ypart[s * MAX_OWN_ROWS + (n - W.own0) + lane] = dv;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(s_addr(&empty[st]));
            }
            // combine in a fixed order: shared expert first, then routed slots
            named_sync(1, NCW * 32);
            if (!*s_abort) {
                for (int n = W.own0 + ct; n < W.own1; n += NCW * 32) {
                    float acc = 0.f;
                    for (int s = 0; s < ns; ++s) acc = fmaf(s_w[s], ypart[s * MAX_OWN_ROWS + (n - W.own0)], acc);
                    if (P.y32) P.y32[n] = acc;
                    if (P.y) {
                        if (P.act_bf16) static_cast<__nv_bfloat16*>(P.y)[n] = __float2bfloat16_rn(acc);
                        else static_cast<float*>(P.y)[n] = acc;
                    }
                }
            }
            if (ct == 0) tstamp(P, 8);
        }
    }

    // ------------------------------------------------------------------ exit
    __syncthreads();
    if (threadIdx.x == 0) {
        tstamp(P, 9);
        __threadfence();
        const unsigned old = atomicAdd(&P.ctr[C_EXIT], 1u);
        if (old + 1 == (unsigned)G) {
            P.ctr[C_ROUTER] = 0;
            P.ctr[C_IDS] = 0;
            P.ctr[C_H] = 0;
            for (int j = 0; j <= MOE_MAX_TOP_K; ++j) P.ctr[C_HMAX + j] = 0;
            __threadfence();
            P.ctr[C_EXIT] = 0;
        }
    }
}

}  // namespace fused

// ---- host side ------------------------------------------------------------------------

static int pick_router_chunk(int H, bool q8) {
    // largest R dividing H with R % 64 == 0 whose codes fit one stage
    for (int R = H; R >= 64; R -= 64) {
        if (H % R) continue;
        const int bytes = q8 ? R : R * 4;
        if (bytes <= fused::STAGE) return R;
    }
    return 0;
}

bool fused_setup(Layer& L) {
    using namespace fused;
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter, k = d.top_k, ns = k + d.n_shared;
    static_assert(sizeof(Params) <= sizeof(L.fused_params), "fused_params storage too small");
    Params& P = *reinterpret_cast<Params*>(L.fused_params);
    P = Params{};
    const bool q8 = d.router_fmt == MOE_W_Q8G64;
    P.R = pick_router_chunk(H, q8);
    if (!P.R) return false;
    P.nsr = H / P.R;
    P.rbH = row_bytes(H);
    P.rbI = row_bytes(I);
    P.gu_block = gu_block_bytes(H, I);
    if (2 * P.rbH > (size_t)STAGE || P.rbI > (size_t)STAGE) return false;
    P.p = std::min<int>(I, (int)(STAGE / (2 * P.rbH)));
    P.n_gu = (I + P.p - 1) / P.p;
    const int own_max = (H + L.num_sms - 1) / L.num_sms;
    if (own_max > MAX_OWN_ROWS) return false;
    P.rbm = std::max(1, std::min<int>(own_max, (int)(STAGE / P.rbI)));
    const size_t uA = (size_t)H * 6 + (size_t)(H / 32) * 8 + NCW * 4;
    const size_t uC = (size_t)ns * I * 4 + (size_t)ns * (I / 32) * 8 + (size_t)ns * MAX_OWN_ROWS * 4;
    const size_t uni = (std::max(uA, uC) + 1023) / 1024 * 1024;
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, L.device);
    const long avail = (long)max_smem - CTRL_BYTES - (long)uni;
    int stages = (int)std::min<long>(MAX_STAGES, avail / STAGE);
    if (stages < 4) return false;
    if (d.n_experts > 1024) return false;
    P.stages = stages;
    P.union_bytes = (int)uni;
    L.fused_smem = CTRL_BYTES + uni + (size_t)stages * STAGE;
    if (cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.fused_smem) !=
        cudaSuccess)
        return false;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_decode_fused, NT, L.fused_smem) != cudaSuccess ||
        occ < 1)
        return false;
    P.rec_tab = L.rec_table;
    P.router = L.router;
    P.router_bias = L.router_bias;
    P.part = L.logits_part;
    P.h = L.h;
    P.logits = L.logits;
    P.ids = L.ids;
    P.wts = L.wts;
    P.ctr = L.counters + 16;
    P.act_bf16 = d.act_dtype == MOE_BF16;
    P.H = H;
    P.I = I;
    P.E = d.n_experts;
    P.k = k;
    P.n_shared = d.n_shared;
    P.q8 = q8;
    return true;
}

cudaError_t launch_decode_fused(Layer& L, const void* x, void* y, float* y_f32, cudaStream_t s) {
    using namespace fused;
    Params P = *reinterpret_cast<const Params*>(L.fused_params);
    P.x = x;
    P.y = y;
    P.y32 = y_f32;
    P.test_no_publish = L.test_no_publish;
    P.trace = L.trace_on ? L.trace : nullptr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = L.fused_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_begin(L, K_DECODE_FUSED, s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_decode_fused, P);
    prof_end(L, s);
    return e;
}

unsigned* fused_error_word(Layer& L) { return L.counters + 16 + fused::C_ERR; }

}  // namespace moe
