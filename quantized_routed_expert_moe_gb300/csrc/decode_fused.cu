// Fused decode step: one persistent, cooperative kernel per token.
//
// One CTA per SM. Eight consumer warps each run their own copy pipeline: lane
// 0 issues bulk asynchronous copies (cp.async.bulk, completion counted on an
// mbarrier) of the warp's next chunks of weight bytes into the warp's three
// shared-memory buffers while the warp dequantises and multiplies the current
// one, so about two chunks per warp are always in flight. The CTA's work, in
// order:
//   P0  router rows (fp32 or 8-bit) -> partial logits in global memory;
//   P1  shared-expert gate/up rows (need no routing);
//   P2  routed-expert gate/up rows (their addresses need the expert IDs);
//   P3  the CTA's block of output rows: for each slot (shared expert first,
//       then the routed experts in selection order), the down rows of that
//       expert, then the weighted combine. P3 copies are issued as soon as the
//       IDs are known; their compute waits until every CTA has written its
//       SwiGLU outputs.
// A control warp per CTA does all waiting on other CTAs: it reduces the router
// logits and selects the experts if this CTA finished the grid's last router
// chunk, publishes or receives the IDs, and runs the grid-wide barrier on the
// SwiGLU outputs. Every wait is bounded; a wait that runs out sets a sticky
// error bit and the CTA drains out. The last CTA to exit resets the grid
// counters, so the kernel can be relaunched (or replayed from a CUDA graph)
// without host bookkeeping.
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
constexpr int CONTROL = NCW;              // warp index of the control warp
constexpr int NT = (NCW + 1) * 32;
constexpr int DEPTH = 3;                  // copy buffers per consumer warp
constexpr int MAX_STAGE = 16384;          // bytes per buffer (upper bound)
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
    float* part;      // [nsr][E] router partial logits
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
    int stage;        // bytes per copy buffer
    size_t rbH, rbI, gu_block;
    int union_bytes;
    int test_no_publish;        // test hook: never publish the IDs, so every wait on them runs out
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
        if (i > 64) __nanosleep(32);
    }
    return false;
}

// Bounded wait until a shared flag is nonzero. Returns false on timeout or abort.
__device__ __forceinline__ bool flag_wait(volatile int* f, volatile int* abort) {
    for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
        if (*f) return true;
        if (*abort) return false;
        if (i > 64) __nanosleep(32);
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
// accumulated in fp32 with one mixed-precision FMA (f16 x f16 + f32), exact in
// the product.
//
// The staged activations are x' = x * 2^e (e per token and vector, keeps
// |x * 2^e| in [2^10, 2^11)), times 16 at even k. Then
//   A = sum_k f_k x'_k = Z + 16 * 2^e * sum_k q_k x_k,   Z = 1024 * sum_k x'_k,
// and the affine group sum is sum_k (q_k s + b) x_k = s (A - Z) / (16 * 2^e) + b X
// with X = sum_k x_k; Z and X are precomputed per half-group.

__device__ __forceinline__ uint32_t cw(const uint4 c, int i) { return i == 0 ? c.x : i == 1 ? c.y : i == 2 ? c.z : c.w; }

// R rows of one half-group against pairs xq[4][stride] (x' pairs per code word)
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

// the same with hi/lo pairs (two products per weight; ~22 bits of the activation)
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

// element k of a staged vector (pairs layout [4][KG]) back as fp32 x'
__device__ __forceinline__ float staged_elem(const uint4* xq, int KG, int k) {
    const int hg = k >> 5, wi = (k >> 3) & 3, i = k & 7;
    const uint4 q = xq[wi * KG + hg];
    const uint32_t w = cw(q, i & 3);
    const uint16_t bits = (i < 4) ? (uint16_t)(w & 0xFFFFu) : (uint16_t)(w >> 16);
    return __half2float(__ushort_as_half(bits));
}

// ---- work lists -------------------------------------------------------------------

struct Work {
    int beg[3], cnt[3];     // P0..P2 item ranges of this CTA (router, shared GU, routed GU)
    int nA;                 // P0..P2 chunks of this CTA
    int own0, own1;         // P3: output rows of this CTA
    int r0, r1;             // P3: rows of this warp
    int sub_rows, nsub;     // P3: rows per item and items per slot for this warp
};

__device__ __forceinline__ void work_ranges(const Params& P, int c, int G, int warp, Work& w) {
    const int n[3] = {P.E * P.nsr, P.n_shared ? P.n_gu : 0, P.k * P.n_gu};
    w.nA = 0;
#pragma unroll
    for (int ph = 0; ph < 3; ++ph) {
        const int b = (int)((long long)n[ph] * c / G), e = (int)((long long)n[ph] * (c + 1) / G);
        w.beg[ph] = b;
        w.cnt[ph] = e - b;
        w.nA += e - b;
    }
    w.own0 = (int)((long long)P.H * c / G);
    w.own1 = (int)((long long)P.H * (c + 1) / G);
    const int own = w.own1 - w.own0;
    const int rpw = (own + NCW - 1) / NCW;
    w.r0 = min(w.own1, w.own0 + warp * rpw);
    w.r1 = min(w.own1, w.r0 + rpw);
    w.sub_rows = max(1, min(rpw, (int)(P.stage / P.rbI)));
    w.nsub = (w.r1 - w.r0 + w.sub_rows - 1) / w.sub_rows;
}

// P0..P2 local chunk index -> (phase, item)
__device__ __forceinline__ void locate(const Work& w, int lc, int& ph, int& item) {
    if (lc < w.cnt[0]) { ph = 0; item = w.beg[0] + lc; return; }
    lc -= w.cnt[0];
    if (lc < w.cnt[1]) { ph = 1; item = w.beg[1] + lc; return; }
    lc -= w.cnt[1];
    ph = 2;
    item = w.beg[2] + lc;
}

// ---- the kernel -----------------------------------------------------------------

__global__ void __launch_bounds__(NT, 1) k_decode_fused(const Params P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);                     // [NCW][DEPTH]
    volatile int* s_flags = reinterpret_cast<volatile int*>(smem + 192);
    volatile int* s_abort = s_flags + 0;
    volatile int* s_rdone = s_flags + 1;      // router chunks done in this CTA
    volatile int* s_last = s_flags + 2;       // this CTA finished the grid's last router chunk
    volatile int* s_ids = s_flags + 3;        // expert IDs and record bases are in s_rec
    volatile int* s_hok = s_flags + 4;        // all SwiGLU outputs visible; s_w / s_hsc set
    volatile int* s_gudone = s_flags + 5;     // consumer warps done with P0..P2
    int* s_rows = const_cast<int*>(s_flags) + 6;                          // gate/up rows done
    unsigned* s_hmax = reinterpret_cast<unsigned*>(smem + 256);            // [k + 1] |h| max bits
    float* s_w = reinterpret_cast<float*>(smem + 320);                    // [k + 1] weight per down slot
    float* s_hsc = reinterpret_cast<float*>(smem + 384);                  // [k + 1] h scale per down slot
    const uint8_t** s_rec = reinterpret_cast<const uint8_t**>(smem + 512);  // [k + 1] record per slot j
    float* s_logit = reinterpret_cast<float*>(smem + 1024);                // [E] (control warp)
    uint8_t* s_taken = smem + 1024 + 4 * 1024;                             // [E]
    uint8_t* uni = smem + CTRL_BYTES;
    uint8_t* bufs = uni + P.union_bytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int H = P.H, I = P.I, k = P.k;
    const int HG = H / 32, IG = I / 32;
    const int ns = k + P.n_shared;
    Work W;
    work_ranges(P, blockIdx.x, G, warp < NCW ? warp : 0, W);

    if (threadIdx.x == 0) {
        if (P.trace)
            for (int i = 1; i < MOE_TRACE_POINTS; ++i) P.trace[(size_t)blockIdx.x * MOE_TRACE_POINTS + i] = 0ull;
        tstamp(P, 0);
        for (int s = 0; s < NCW * DEPTH; ++s) mbar_init(s_addr(&full[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int i = 0; i < 8; ++i) const_cast<int*>(s_flags)[i] = 0;
        if (P.n_shared) s_rec[k] = P.rec_tab[P.E];
    }
    if (threadIdx.x < MOE_MAX_TOP_K + 1) s_hmax[threadIdx.x] = 0u;
    __syncthreads();

    if (warp == CONTROL) {
        // ================================================================ control
        bool ok = true;
        // (1) select, if this CTA holds the grid's last router chunk
        if (W.cnt[0] > 0) {
            ok = false;
            for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
                if (*s_abort) break;
                if (*s_rdone >= W.cnt[0]) { ok = true; break; }
                if (i > 64) __nanosleep(32);
            }
            if (lane == 0) tstamp(P, 2);
            if (ok && *s_last == 1 && !P.test_no_publish) {
                __threadfence();
                const int E = P.E;
                for (int e0 = 0; e0 < E; e0 += 8 * 32) {
                    float l[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) l[u] = 0.f;
                    for (int s = 0; s < P.nsr; ++s) {
                        float v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {   // 8 independent loads in flight
                            const int e = e0 + u * 32 + lane;
                            v[u] = (e < E) ? __ldcg(P.part + (size_t)s * E + e) : 0.f;
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) l[u] += v[u];
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = e0 + u * 32 + lane;
                        if (e < E) {
                            if (P.router_bias) l[u] += __ldg(P.router_bias + e);
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
            if (!ok && !*s_abort && lane == 0) { atomicOr(&P.ctr[C_ERR], ERR_CTRL); *s_abort = 1; }
        }
        // (2) receive the IDs; record bases for the copies
        if (lane == 0 && !*s_abort) {
            bool got = false;
            for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
                if (ld_acquire(&P.ctr[C_IDS]) != 0u) { got = true; break; }
                if (*s_abort) break;
                if (i > 64) __nanosleep(32);
            }
            if (got) {
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
                __threadfence_block();
                *s_ids = 1;
                tstamp(P, 4);
            } else if (!*s_abort) {
                atomicOr(&P.ctr[C_ERR], ERR_IDS);
                *s_abort = 1;
            }
        }
        // (3) SwiGLU outputs barrier across the grid
        if (lane == 0 && !*s_abort) {
            bool ok3 = false;
            for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
                if (*s_gudone >= NCW) { ok3 = true; break; }
                if (*s_abort) break;
                if (i > 64) __nanosleep(32);
            }
            if (ok3) {
                tstamp(P, 5);
                for (int j = 0; j < ns; ++j) {
                    const int jj = (j < k) ? j : k;
                    if (s_hmax[jj]) atomicMax(&P.ctr[C_HMAX + jj], s_hmax[jj]);
                }
                __threadfence();
                if (*s_rows) atomicAdd(&P.ctr[C_H], (unsigned)*s_rows);
                const unsigned target = (unsigned)(ns * I);
                ok3 = false;
                for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
                    if (ld_acquire(&P.ctr[C_H]) >= target) { ok3 = true; break; }
                    if (*s_abort) break;
                    if (i > 64) __nanosleep(32);
                }
            }
            if (ok3) {
                for (int s = 0; s < ns; ++s) {
                    const bool sh = P.n_shared && s == 0;
                    const int j = sh ? k : s - P.n_shared;
                    s_w[s] = sh ? 1.0f : __ldcg(P.wts + j);
                    s_hsc[s] = pow2_scale(__uint_as_float(ld_acquire(&P.ctr[C_HMAX + j])));
                }
                __threadfence_block();
                *s_hok = 1;
                tstamp(P, 6);
            } else if (!*s_abort) {
                atomicOr(&P.ctr[C_ERR], ERR_H);
                *s_abort = 1;
            }
        }
    } else {
        // ============================================================== consumers
        const int ct = threadIdx.x;  // 0 .. NCW*32-1
        uint4* xq = reinterpret_cast<uint4*>(uni);                                 // [4][HG] x' pairs
        float* Zx = reinterpret_cast<float*>(uni + (size_t)H * 2);                // [HG]
        float* Xx = Zx + HG;                                                      // [HG]
        float* s_red = Xx + HG;                                                   // [NCW]
        uint8_t* mybuf = bufs + (size_t)warp * DEPTH * P.stage;
        uint64_t* myfull = full + warp * DEPTH;

        // ---- the warp's copy pipeline over its chunk list
        // chunks [0, nAw): P0..P2 chunks lc = warp + NCW * i; chunks [nAw, nAw + ns * nsub): P3 (slot, sub)
        const int nAw = (W.nA > warp) ? (W.nA - warp + NCW - 1) / NCW : 0;
        const int nCw = ns * W.nsub;
        const int nw = nAw + nCw;
        int issued = 0;  // uniform across the warp
        auto issue_upto = [&](int limit, bool must) {
            int n = issued;
            if (lane == 0) {
                while (n < min(limit, nw)) {
                    const int b = n % DEPTH;
                    const uint32_t bar = s_addr(&myfull[b]);
                    const uint32_t dst = s_addr(mybuf + (size_t)b * P.stage);
                    const uint8_t* src = nullptr;
                    uint32_t bytes = 0;
                    if (n < nAw) {
                        int ph, item;
                        locate(W, warp + NCW * n, ph, item);
                        if (ph == 0) {
                            const int e = item / P.nsr, sr = item - e * P.nsr;
                            if (!P.q8) {
                                src = reinterpret_cast<const uint8_t*>(static_cast<const float*>(P.router) +
                                                                       (size_t)e * H + (size_t)sr * P.R);
                                bytes = P.R * 4;
                            } else {
                                src = static_cast<const uint8_t*>(P.router) + (size_t)e * H + (size_t)sr * P.R;
                                bytes = P.R;
                            }
                        } else {
                            if (ph == 2 && !*s_ids) {
                                if (!must || !flag_wait(s_ids, s_abort)) break;
                            }
                            const int j = (ph == 1) ? k : item / P.n_gu;
                            const int u = (ph == 1) ? item : item - j * P.n_gu;
                            const int i0 = u * P.p, i1 = min(I, i0 + P.p);
                            src = s_rec[j] + (size_t)(2 * i0) * P.rbH;
                            bytes = (uint32_t)(2 * (i1 - i0) * P.rbH);
                        }
                    } else {
                        if (!*s_ids) {
                            if (!must || !flag_wait(s_ids, s_abort)) break;
                        }
                        const int c = n - nAw, s = c / W.nsub, sub = c - s * W.nsub;
                        const int j = (P.n_shared && s == 0) ? k : s - P.n_shared;
                        const int n0 = W.r0 + sub * W.sub_rows, n1 = min(W.r1, n0 + W.sub_rows);
                        src = s_rec[j] + P.gu_block + (size_t)n0 * P.rbI;
                        bytes = (uint32_t)((n1 - n0) * P.rbI);
                    }
                    // the buffer's previous contents were read by generic loads
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(bar, bytes);
                    bulk_g2s(dst, src, bytes, bar);
                    ++n;
                }
            }
            issued = __shfl_sync(0xffffffffu, n, 0);
        };
        // returns the buffer of chunk i once its bytes have landed (nullptr on abort)
        auto acquire = [&](int i) -> const uint8_t* {
            issue_upto(i + DEPTH, false);
            if (issued <= i) issue_upto(i + 1, true);
            if (issued <= i) return nullptr;
            if (!mbar_wait(s_addr(&myfull[i % DEPTH]), (i / DEPTH) & 1, s_abort)) {
                if (lane == 0 && !*s_abort) { atomicOr(&P.ctr[C_ERR], ERR_STAGE); *s_abort = 1; }
                return nullptr;
            }
            return mybuf + (size_t)(i % DEPTH) * P.stage;
        };
        issue_upto(DEPTH, false);   // start the router / shared-expert copies right away

        // ---- stage the activations: x' pairs and per-half-group Z, X (token scale)
        {
            const int nrun = H / 8;
            float v[4][8];
            float mx = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = ct + u * NCW * 32;
#pragma unroll
                for (int i = 0; i < 8; ++i) v[u][i] = 0.f;
                if (r < nrun) {
                    if (P.act_bf16) {
                        const uint4 q = __ldg(reinterpret_cast<const uint4*>(P.x) + r);
                        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            v[u][2 * i] = __uint_as_float(w4[i] << 16);
                            v[u][2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
                        }
                    } else {
                        const float4 a = __ldg(reinterpret_cast<const float4*>(P.x) + 2 * r);
                        const float4 b = __ldg(reinterpret_cast<const float4*>(P.x) + 2 * r + 1);
                        v[u][0] = a.x; v[u][1] = a.y; v[u][2] = a.z; v[u][3] = a.w;
                        v[u][4] = b.x; v[u][5] = b.y; v[u][6] = b.z; v[u][7] = b.w;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[u][i]));
                }
            }
            for (int r = ct + 4 * NCW * 32; r < nrun; r += NCW * 32) {   // H > 8192: rare, plain loop
                for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(load_act(P.x, P.act_bf16, (size_t)8 * r + i)));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) s_red[warp] = mx;
            named_sync(1, NCW * 32);
            mx = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) mx = fmaxf(mx, s_red[w]);
            const float sc = pow2_scale(mx), inv = 1.0f / sc;
            // warp-uniform trip count: every lane takes part in the shuffles
            for (int rb = warp * 32; rb < nrun; rb += NCW * 32) {
                const int r = rb + lane;
                const bool valid = r < nrun;
                float vv[8];
                const int u = (rb - warp * 32) / (NCW * 32);
                if (u < 4) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) vv[i] = (u == 0 ? v[0][i] : u == 1 ? v[1][i] : u == 2 ? v[2][i] : v[3][i]) * sc;
                } else {
                    for (int i = 0; i < 8; ++i) vv[i] = valid ? load_act(P.x, P.act_bf16, (size_t)8 * r + i) * sc : 0.f;
                }
                uint4 hi, lo;
                float z, xs;
                stage_run<false>(vv, inv, hi, lo, z, xs);
                const int hg = r >> 2, wi = r & 3;
                // the four runs of a half-group sit in four consecutive lanes (nrun % 4 == 0)
                z += __shfl_xor_sync(0xffffffffu, z, 1);
                z += __shfl_xor_sync(0xffffffffu, z, 2);
                xs += __shfl_xor_sync(0xffffffffu, xs, 1);
                xs += __shfl_xor_sync(0xffffffffu, xs, 2);
                if (valid) {
                    xq[wi * HG + hg] = hi;
                    if (wi == 0) { Zx[hg] = z; Xx[hg] = xs; }
                }
            }
            s_red[NCW] = inv;   // written identically by every thread
        }
        named_sync(1, NCW * 32);
        const float xinv = s_red[NCW];
        const float gu_c = xinv * 0.0625f;  // 1 / (16 * 2^e)
        if (ct == 0) tstamp(P, 1);

        // ---- P0..P2
        int rows_done = 0;
        float hmax[MOE_MAX_TOP_K + 1];
#pragma unroll
        for (int j = 0; j <= MOE_MAX_TOP_K; ++j) hmax[j] = 0.f;
        for (int i = 0; i < nAw; ++i) {
            const uint8_t* buf = acquire(i);
            if (!buf) break;
            int ph, item;
            locate(W, warp + NCW * i, ph, item);
            if (ph == 0) {
                const int e = item / P.nsr, sr = item - e * P.nsr;
                const int k0 = sr * P.R;
                float acc = 0.f;
                if (!P.q8) {
                    const float4* w4 = reinterpret_cast<const float4*>(buf);
                    for (int c = lane; c < P.R / 4; c += 32) {
                        const float4 a = w4[c];
                        const int kk = k0 + 4 * c;
                        const uint4 q = xq[((kk >> 3) & 3) * HG + (kk >> 5)];
                        const uint32_t wa = (kk & 4) ? (q.x >> 16) | (q.y & 0xFFFF0000u) : (q.x & 0xFFFFu) | (q.y << 16);
                        const uint32_t wb = (kk & 4) ? (q.z >> 16) | (q.w & 0xFFFF0000u) : (q.z & 0xFFFFu) | (q.w << 16);
                        const float2 xa = __half22float2(*reinterpret_cast<const __half2*>(&wa));
                        const float2 xb = __half22float2(*reinterpret_cast<const __half2*>(&wb));
                        // staged x' = 16 x * 2^e at even k, x * 2^e at odd k
                        acc = fmaf(a.x, xa.x * 0.0625f, acc);
                        acc = fmaf(a.y, xa.y, acc);
                        acc = fmaf(a.z, xb.x * 0.0625f, acc);
                        acc = fmaf(a.w, xb.y, acc);
                    }
                    acc *= xinv;
                } else {
                    const uint32_t* meta = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(P.router) +
                                                                             (size_t)P.E * H) +
                                           (size_t)e * (H / 64) + k0 / 64;
                    for (int c = lane; c < P.R / 16; c += 32) {
                        const uint4 q = *reinterpret_cast<const uint4*>(buf + 16 * c);
                        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
                        const uint32_t mw = __ldg(meta + (c >> 2));
                        float aq = 0.f, ax = 0.f;
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const int kk = k0 + 16 * c + t;
                            const float xv = staged_elem(xq, HG, kk) * ((t & 1) ? 1.0f : 0.0625f);
                            const float cv = __uint_as_float(0x4B000000u | ((qw[t >> 2] >> (8 * (t & 3))) & 0xFFu)) -
                                             8388608.0f;
                            aq = fmaf(cv, xv, aq);
                            ax += xv;
                        }
                        const float2 sb = meta_to_f2(mw);
                        acc = fmaf(sb.x, aq, fmaf(sb.y, ax, acc));
                    }
                    acc *= xinv;
                }
                acc = warp_sum(acc);
                if (lane == 0) {
                    P.part[(size_t)sr * P.E + e] = acc;
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
                // two gate/up row pairs at a time: rows (gate i, up i, gate i+1, up i+1)
                for (int ii = i0; ii < i1; ii += 2) {
                    const bool two = ii + 1 < i1;
                    const uint8_t* r0 = buf + (size_t)(2 * (ii - i0)) * P.rbH;
                    float g[4];
                    if (two) {
                        const uint8_t* rr[4] = {r0, r0 + P.rbH, r0 + 2 * P.rbH, r0 + 3 * P.rbH};
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
#pragma unroll
                        for (int r = 0; r < 4; ++r) g[r] = warp_sum(fmaf(as[r], gu_c, ab[r]));
                    } else {
                        const uint8_t* rr[2] = {r0, r0 + P.rbH};
                        float as[2] = {0.f, 0.f}, ab[2] = {0.f, 0.f};
                        for (int hg = lane; hg < HG; hg += 32) {
                            uint4 c[2];
                            float2 sb[2];
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                c[r] = *reinterpret_cast<const uint4*>(rr[r] + 16 * hg);
                                sb[r] = meta_to_f2(*reinterpret_cast<const uint32_t*>(rr[r] + H / 2 + 4 * (hg >> 1)));
                            }
                            float A[2];
                            hg_rows<2>(c, xq + hg, HG, A);
                            const float z = Zx[hg], xs = Xx[hg];
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                as[r] = fmaf(sb[r].x, A[r] - z, as[r]);
                                ab[r] = fmaf(sb[r].y, xs, ab[r]);
                            }
                        }
#pragma unroll
                        for (int r = 0; r < 2; ++r) g[r] = warp_sum(fmaf(as[r], gu_c, ab[r]));
                        g[2] = g[3] = 0.f;
                    }
                    if (lane == 0) {
                        const float h0 = silu_f(g[0]) * g[1];
                        P.h[(size_t)j * I + ii] = h0;
                        float m = fabsf(h0);
                        if (two) {
                            const float h1 = silu_f(g[2]) * g[3];
                            P.h[(size_t)j * I + ii + 1] = h1;
                            m = fmaxf(m, fabsf(h1));
                        }
#pragma unroll
                        for (int jj = 0; jj <= MOE_MAX_TOP_K; ++jj)
                            if (jj == j) hmax[jj] = fmaxf(hmax[jj], m);
                    }
                }
                rows_done += i1 - i0;
            }
            __syncwarp();
        }
        // this warp is done with P0..P2
        if (lane == 0) {
#pragma unroll
            for (int jj = 0; jj <= MOE_MAX_TOP_K; ++jj)
                if (hmax[jj] > 0.f) atomicMax(&s_hmax[jj], __float_as_uint(hmax[jj]));   // |h| >= 0: bits order as floats
            if (rows_done) {
                __threadfence();
                atomicAdd(s_rows, rows_done);
            }
            __threadfence_block();
            atomicAdd(const_cast<int*>(s_gudone), 1);
        }

        // ---- P3: wait for every SwiGLU output, then slot by slot
        const bool go = __shfl_sync(0xffffffffu, lane == 0 ? (int)flag_wait(s_hok, s_abort) : 0, 0) != 0;
        // h staging buffers (double-buffered by slot parity)
        uint4* hb[2][2];     // [buffer][hi/lo] -> [4][IG]
        float* Zh[2];
        float* Xh[2];
        {
            uint8_t* p = uni;
            for (int b = 0; b < 2; ++b) {
                hb[b][0] = reinterpret_cast<uint4*>(p); p += (size_t)I * 2;
                hb[b][1] = reinterpret_cast<uint4*>(p); p += (size_t)I * 2;
            }
            for (int b = 0; b < 2; ++b) { Zh[b] = reinterpret_cast<float*>(p); p += (size_t)IG * 4; }
            for (int b = 0; b < 2; ++b) { Xh[b] = reinterpret_cast<float*>(p); p += (size_t)IG * 4; }
        }
        float* ypart = reinterpret_cast<float*>(uni + (size_t)I * 8 + (size_t)IG * 16);  // [ns][MAX_OWN_ROWS]
        // every consumer thread stages runs of slot s into buffer b
        auto stage_h = [&](int s, int b) {
            const int j = (P.n_shared && s == 0) ? k : s - P.n_shared;
            const float sc = s_hsc[s], inv = 1.0f / sc;
            const int nrun = I / 8;
            for (int rb = warp * 32; rb < nrun; rb += NCW * 32) {   // warp-uniform trip count
                const int r = rb + lane;
                const bool valid = r < nrun;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
                if (valid) {
                    const float4* src = reinterpret_cast<const float4*>(P.h + (size_t)j * I + 8 * (size_t)r);
                    a = __ldcg(src);
                    c = __ldcg(src + 1);
                }
                const float vv[8] = {a.x * sc, a.y * sc, a.z * sc, a.w * sc, c.x * sc, c.y * sc, c.z * sc, c.w * sc};
                uint4 hi, lo;
                float z, xs;
                stage_run<true>(vv, inv, hi, lo, z, xs);
                const int hg = r >> 2, wi = r & 3;
                z += __shfl_xor_sync(0xffffffffu, z, 1);
                z += __shfl_xor_sync(0xffffffffu, z, 2);
                xs += __shfl_xor_sync(0xffffffffu, xs, 1);
                xs += __shfl_xor_sync(0xffffffffu, xs, 2);
                if (valid) {
                    hb[b][0][wi * IG + hg] = hi;
                    hb[b][1][wi * IG + hg] = lo;
                    if (wi == 0) { Zh[b][hg] = z; Xh[b][hg] = xs; }
                }
            }
        };
        if (go) stage_h(0, 0);
        named_sync(1, NCW * 32);
        if (ct == 0) tstamp(P, 7);
        bool alive = go;
        for (int s = 0; s < ns; ++s) {
            const int b = s & 1;
            if (go && s + 1 < ns) stage_h(s + 1, b ^ 1);
            const float dc = 0.0625f / s_hsc[s];
            for (int sub = 0; sub < W.nsub && alive; ++sub) {
                const int i = nAw + s * W.nsub + sub;
                const uint8_t* buf = acquire(i);
                if (!buf) { alive = false; break; }
                const int n0 = W.r0 + sub * W.sub_rows, n1 = min(W.r1, n0 + W.sub_rows);
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
                        hg_rows_hilo<4>(c, hb[b][0] + hg, hb[b][1] + hg, IG, A);
                        const float z = Zh[b][hg], xx = Xh[b][hg];
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
            }
            named_sync(1, NCW * 32);   // slot s done everywhere; buffer b free for slot s + 2
        }
        // combine in a fixed order: shared expert first, then routed slots
        if (go && !*s_abort) {
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
        // drain: copies issued but never consumed (after an abort) must land
        // before the CTA exits; consumed ones return at once
        for (int i = max(0, issued - DEPTH); i < issued; ++i) {
            const uint32_t bar = s_addr(&myfull[i % DEPTH]);
            for (uint32_t t = 0; t < SPIN_LIMIT && !mbar_try(bar, (i / DEPTH) & 1); ++t) __nanosleep(32);
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

bool fused_setup(Layer& L) {
    using namespace fused;
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter, k = d.top_k, ns = k + d.n_shared;
    static_assert(sizeof(Params) <= sizeof(L.fused_params), "fused_params storage too small");
    Params& P = *reinterpret_cast<Params*>(L.fused_params);
    P = Params{};
    const bool q8 = d.router_fmt == MOE_W_Q8G64;
    if (d.n_experts > 1024) return false;
    P.rbH = row_bytes(H);
    P.rbI = row_bytes(I);
    P.gu_block = gu_block_bytes(H, I);
    const int own_max = (H + L.num_sms - 1) / L.num_sms;
    if (own_max > MAX_OWN_ROWS) return false;
    // shared memory: control + union (staged activations / staged h + partial outputs) + buffers
    const size_t uA = (size_t)H * 2 + (size_t)(H / 32) * 8 + (NCW + 1) * 4;
    const size_t uC = (size_t)I * 8 + (size_t)(I / 32) * 16 + (size_t)ns * MAX_OWN_ROWS * 4;
    const size_t uni = (std::max(uA, uC) + 127) / 128 * 128;
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, L.device);
    long stage = ((long)max_smem - CTRL_BYTES - (long)uni) / (NCW * DEPTH);
    stage = std::min<long>(stage, MAX_STAGE) / 128 * 128;
    if (stage < (long)(2 * P.rbH) || stage < (long)P.rbI || stage < 256) return false;
    // router chunk: largest R dividing H, R % 64 == 0, whose codes fit one buffer
    P.R = 0;
    for (int R = H; R >= 64; R -= 64) {
        if (H % R) continue;
        if ((long)(q8 ? R : R * 4) <= stage) { P.R = R; break; }
    }
    if (!P.R) return false;
    P.nsr = H / P.R;
    if (P.nsr > L.router_splits * std::max(1, d.max_tokens)) return false;  // partial-logit scratch size
    P.stage = (int)stage;
    P.p = std::min<int>(I, (int)(stage / (2 * P.rbH)));
    P.n_gu = (I + P.p - 1) / P.p;
    P.union_bytes = (int)uni;
    L.fused_smem = CTRL_BYTES + uni + (size_t)NCW * DEPTH * stage;
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
