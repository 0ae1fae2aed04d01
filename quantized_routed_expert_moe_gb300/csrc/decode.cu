// Decode path: router GEMV + exact top-k + softmax, gate/up dequant-GEMV with
// SwiGLU, down dequant-GEMV with the weighted combine.
//
// Router, exact top-8, shared expert and combine: TurboFieldfare article,
// "token generation"; weight format: same article, "execution architecture";
// exact routing: Inferno README "Current Scope", Colibri report section 3.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// exact top-k + softmax over the selected logits, one CTA
// ---------------------------------------------------------------------------
//
// Selection is the first k of the experts ordered by (-l_e, e): each round
// takes the largest remaining logit, the lower index on equal values. NaN
// logits are treated as -inf so that every round selects a valid expert.
__device__ void block_topk_softmax(const float* sl, int E, int k, int32_t* ids_out, float* w_out) {
    __shared__ float s_v[32];
    __shared__ int s_i[32];
    __shared__ int s_sel[MOE_MAX_TOP_K];
    __shared__ float s_lv[MOE_MAX_TOP_K];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    constexpr int M = 1024 / kThreads;
    float v[M];
    bool taken[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const int e = tid + m * blockDim.x;
        float t = (e < E) ? sl[e] : -INFINITY;
        v[m] = (t != t) ? -INFINITY : t;
        taken[m] = (e >= E);
    }
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int e = tid + m * blockDim.x;
            if (!taken[m] && (v[m] > bv || (v[m] == bv && e < bi))) { bv = v[m]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { s_v[warp] = bv; s_i[warp] = bi; }
        __syncthreads();
        if (warp == 0) {
            bv = (lane < nw) ? s_v[lane] : -INFINITY;
            bi = (lane < nw) ? s_i[lane] : INT_MAX;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (lane == 0) { s_sel[r] = bi; s_lv[r] = bv; }
        }
        __syncthreads();
        const int win = s_sel[r];
#pragma unroll
        for (int m = 0; m < M; ++m)
            if (tid + m * (int)blockDim.x == win) taken[m] = true;
    }
    if (tid == 0) {
        // softmax over the selected logits; the first selected is the maximum
        const float mx = s_lv[0];
        float ex[MOE_MAX_TOP_K];
        float den = 0.f;
        for (int r = 0; r < k; ++r) { ex[r] = expf(s_lv[r] - mx); den += ex[r]; }
        for (int r = 0; r < k; ++r) { ids_out[r] = s_sel[r]; w_out[r] = ex[r] / den; }
    }
}

// ---------------------------------------------------------------------------
// router GEMV for one token: split over H, last CTA reduces and selects
// ---------------------------------------------------------------------------
template <bool Q8>
__global__ void __launch_bounds__(kThreads) k_router_decode(
    const void* __restrict__ W, const void* __restrict__ x, int x_bf16, int H, int E, int splits,
    const float* __restrict__ bias, float* __restrict__ part, float* __restrict__ logits,
    int32_t* __restrict__ ids, float* __restrict__ wts, int k, unsigned* __restrict__ counter) {
    extern __shared__ float sm[];
    __shared__ unsigned s_last;
    const int Ls = H / splits;
    const int k0 = blockIdx.y * Ls;
    for (int i = threadIdx.x; i < Ls; i += blockDim.x) sm[i] = load_act(x, x_bf16, (size_t)k0 + i);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kWarps + warp;
    if (e < E) {
        float acc = 0.f;
        if (!Q8) {
            const float4* row = reinterpret_cast<const float4*>(static_cast<const float*>(W) + (size_t)e * H + k0);
            const float4* xs = reinterpret_cast<const float4*>(sm);
            for (int c = lane; c < Ls / 4; c += 32) {
                const float4 w = __ldg(row + c);
                const float4 xv = xs[c];
                acc = fmaf(w.x, xv.x, acc);
                acc = fmaf(w.y, xv.y, acc);
                acc = fmaf(w.z, xv.z, acc);
                acc = fmaf(w.w, xv.w, acc);
            }
        } else {
            const uint8_t* codes = static_cast<const uint8_t*>(W) + (size_t)e * H + k0;
            const uint32_t* meta = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(W) + (size_t)E * H) +
                                   (size_t)e * (H / 64) + k0 / 64;
            for (int c = lane; c < Ls / 16; c += 32) {
                const uint4 q = ldg_stream(codes + 16 * c);
                const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
                float aq = 0.f, ax = 0.f;
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const float xv = sm[16 * c + t];
                    aq = fmaf((float)((qw[t >> 2] >> (8 * (t & 3))) & 0xFFu), xv, aq);
                    ax += xv;
                }
                const float2 sb = meta_to_f2(meta[c >> 2]);
                acc = fmaf(sb.x, aq, fmaf(sb.y, ax, acc));
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) part[(size_t)blockIdx.y * E + e] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(counter, 1u);
        s_last = (prev == gridDim.x * gridDim.y - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int e2 = threadIdx.x; e2 < E; e2 += blockDim.x) {
        float l = 0.f;
        for (int s = 0; s < splits; ++s) l += __ldcg(part + (size_t)s * E + e2);
        if (bias) l += bias[e2];
        sm[e2] = l;
        logits[e2] = l;
    }
    __syncthreads();
    block_topk_softmax(sm, E, k, ids, wts);
    if (threadIdx.x == 0) *counter = 0u;
}

// ---------------------------------------------------------------------------
// router for T tokens: split-K tiles (16 tokens x 64 experts), then per-token top-k
// ---------------------------------------------------------------------------
constexpr int RT_T = 16, RT_E = 64, RT_K = 64;

template <bool Q8>
__global__ void __launch_bounds__(kThreads) k_router_tokens(const void* __restrict__ W, const void* __restrict__ x,
                                                            int x_bf16, int T, int H, int E, int splits,
                                                            float* __restrict__ part) {
    __shared__ float xs[RT_T][RT_K + 1];
    __shared__ __align__(16) float ws[RT_K][RT_E];
    const int e0 = blockIdx.x * RT_E, t0 = blockIdx.y * RT_T;
    const int Ls = H / splits, kb = blockIdx.z * Ls;
    const int tid = threadIdx.x, tt = tid >> 4, te = (tid & 15) * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kc = kb; kc < kb + Ls; kc += RT_K) {
        for (int i = tid; i < RT_T * RT_K; i += kThreads) {
            const int r = i / RT_K, c = i % RT_K;
            xs[r][c] = (t0 + r < T) ? load_act(x, x_bf16, (size_t)(t0 + r) * H + kc + c) : 0.f;
        }
        for (int i = tid; i < RT_E * RT_K; i += kThreads) {
            const int r = i / RT_K, c = i % RT_K;  // r: expert in tile, c: k in chunk
            float w = 0.f;
            if (e0 + r < E) {
                if (!Q8) {
                    w = __ldg(static_cast<const float*>(W) + (size_t)(e0 + r) * H + kc + c);
                } else {
                    const uint8_t* base = static_cast<const uint8_t*>(W);
                    const uint32_t m = __ldg(reinterpret_cast<const uint32_t*>(base + (size_t)E * H) +
                                             (size_t)(e0 + r) * (H / 64) + (kc / 64));
                    const float2 sb = meta_to_f2(m);
                    w = fmaf((float)base[(size_t)(e0 + r) * H + kc + c], sb.x, sb.y);
                }
            }
            ws[c][r] = w;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < RT_K; ++c) {
            const float a = xs[tt][c];
            const float4 w4 = *reinterpret_cast<const float4*>(&ws[c][te]);
            acc[0] = fmaf(a, w4.x, acc[0]);
            acc[1] = fmaf(a, w4.y, acc[1]);
            acc[2] = fmaf(a, w4.z, acc[2]);
            acc[3] = fmaf(a, w4.w, acc[3]);
        }
        __syncthreads();
    }
    const int t = t0 + tt;
    if (t < T)
        for (int j = 0; j < 4; ++j)
            if (e0 + te + j < E) part[((size_t)blockIdx.z * T + t) * E + e0 + te + j] = acc[j];
}

__global__ void __launch_bounds__(kThreads) k_topk_tokens(const float* __restrict__ part, int splits, int T, int E,
                                                          const float* __restrict__ bias, float* __restrict__ logits,
                                                          int32_t* __restrict__ ids, float* __restrict__ wts, int k) {
    extern __shared__ float sl[];
    const int t = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float l = 0.f;
        for (int s = 0; s < splits; ++s) l += part[((size_t)s * T + t) * E + e];
        if (bias) l += bias[e];
        sl[e] = l;
        logits[(size_t)t * E + e] = l;
    }
    __syncthreads();
    block_topk_softmax(sl, E, k, ids + (size_t)t * k, wts + (size_t)t * k);
}

// ---------------------------------------------------------------------------
// expert GEMVs
// ---------------------------------------------------------------------------
//
// Activations sit in shared memory as float4 [8][H/32]: element
// (c, hg) holds x[32*hg + 4*c .. 32*hg + 4*c + 3], so lane `hg` reads its 32
// inputs with 8 conflict-free 16-byte loads. A lane handles 32 inputs of a row
// per step: 16 bytes of codes (one 16-byte load) and the (scale, bias) pair of
// their group. For the group the sum is
//   sum_k (q_k s + b) x_k = s * sum_k q_k x_k + b * sum_k x_k,
// with the half-group sums of x precomputed once per CTA.

__device__ __forceinline__ float dot32(const uint4 q, const float4* xs, int stride) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 xv = xs[c * stride];
        const uint32_t word = w[c >> 1];
        const int sh = (c & 1) * 16;
        a0 = fmaf(nib_f(word, sh + 0), xv.x, a0);
        a1 = fmaf(nib_f(word, sh + 4), xv.y, a1);
        a0 = fmaf(nib_f(word, sh + 8), xv.z, a0);
        a1 = fmaf(nib_f(word, sh + 12), xv.w, a1);
    }
    return a0 + a1;
}

__device__ __forceinline__ void stage_vector_t(float4* dst, float* sums, int K, int nvec, const float* const* src,
                                               const void* xsrc, int x_bf16) {
    // dst: nvec blocks of [8][K/32] float4; sums: nvec x [K/32]
    const int KG = K / 32;
    // 4 consecutive values per item, 4 items per thread in flight
    const int nq = K / 4, nitems = nvec * nq;
    for (int base = threadIdx.x; base < nitems; base += 4 * blockDim.x) {
        float4 val[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            if (idx < nitems) {
                const int v = idx / nq, i4 = idx - v * nq;
                if (src) {
                    val[u] = __ldcg(reinterpret_cast<const float4*>(src[v]) + i4);
                } else if (x_bf16) {
                    const uint2 w = __ldg(reinterpret_cast<const uint2*>(xsrc) + i4);
                    val[u] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                                         __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
                } else {
                    val[u] = __ldg(reinterpret_cast<const float4*>(xsrc) + i4);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            if (idx < nitems) {
                const int v = idx / nq, i4 = idx - v * nq;
                const int i = 4 * i4, hg = i >> 5, c = (i & 31) >> 2;
                dst[(size_t)v * 8 * KG + c * KG + hg] = val[u];
            }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nvec * KG; idx += blockDim.x) {
        const int v = idx / KG, hg = idx - v * KG;
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 t = dst[(size_t)v * 8 * KG + c * KG + hg];
            s += (t.x + t.y) + (t.z + t.w);
        }
        sums[idx] = s;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) k_gateup_decode(const uint8_t* const* __restrict__ rec_tab,
                                                            const int32_t* __restrict__ ids, int k, int E,
                                                            int slot0, int nslots, const void* __restrict__ x,
                                                            int x_bf16, int H, int I, float* __restrict__ h) {
    extern __shared__ float4 smx[];
    const int HG = H / 32;
    float* xsum = reinterpret_cast<float*>(smx + 8 * HG);
    stage_vector_t(smx, xsum, H, 1, nullptr, x, x_bf16);
    const size_t rb = d_row_bytes(H);
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
    const int nrows = nslots * I;
    for (int r = gw; r < nrows; r += nw) {
        const int jj = r / I, i = r - jj * I, j = slot0 + jj;
        const int e = (j < k) ? ids[j] : E;
        if ((unsigned)e > (unsigned)E) {  // cannot happen for a valid selection
            if (lane == 0) h[(size_t)j * I + i] = __int_as_float(0x7fc00000);
            continue;
        }
        const uint8_t* g = rec_tab[e] + (size_t)(2 * i) * rb;
        const uint8_t* u = g + rb;
        float ga = 0.f, ua = 0.f;
        for (int hg = lane; hg < HG; hg += 32) {
            const uint4 gc = ldg_stream(g + 16 * hg);
            const uint4 uc = ldg_stream(u + 16 * hg);
            const uint32_t gm = ldg_u32(g + H / 2 + 4 * (hg >> 1));
            const uint32_t um = ldg_u32(u + H / 2 + 4 * (hg >> 1));
            const float dg = dot32(gc, smx + hg, HG);
            const float du = dot32(uc, smx + hg, HG);
            const float2 sg = meta_to_f2(gm), su = meta_to_f2(um);
            const float xs = xsum[hg];
            ga = fmaf(sg.x, dg, fmaf(sg.y, xs, ga));
            ua = fmaf(su.x, du, fmaf(su.y, xs, ua));
        }
        ga = warp_sum(ga);
        ua = warp_sum(ua);
        if (lane == 0) h[(size_t)j * I + i] = silu_f(ga) * ua;
    }
}

// Slot order in the down kernel: the shared expert first (weight 1), then the
// routed experts in selection order. h holds routed slot j at j*I and the
// shared expert at k*I.
__global__ void __launch_bounds__(kThreads) k_down_decode(const uint8_t* const* __restrict__ rec_tab,
                                                          const int32_t* __restrict__ ids,
                                                          const float* __restrict__ wts, int k, int E,
                                                          int n_shared, int H, int I, const float* __restrict__ h,
                                                          void* __restrict__ y, int y_bf16,
                                                          float* __restrict__ y32) {
    extern __shared__ float4 smh[];
    const int IG = I / 32, ns = k + n_shared;
    float* hsum = reinterpret_cast<float*>(smh + (size_t)ns * 8 * IG);
    __shared__ const float* srcs[MOE_MAX_TOP_K + 1];
    __shared__ const uint8_t* rows0[MOE_MAX_TOP_K + 1];
    __shared__ float wsl[MOE_MAX_TOP_K + 1];
    if (threadIdx.x < ns) {
        const int s = threadIdx.x;
        const bool sh = n_shared && s == 0;
        const int j = sh ? k : s - n_shared;
        srcs[s] = h + (size_t)j * I;
        int e = sh ? E : ids[j];
        if ((unsigned)e > (unsigned)E) e = E;  // guarded; a valid selection never hits this
        rows0[s] = rec_tab[e] + 2 * (size_t)I * d_row_bytes(H);
        wsl[s] = sh ? 1.0f : wts[j];
    }
    __syncthreads();
    stage_vector_t(smh, hsum, I, ns, srcs, nullptr, 0);
    const size_t rb = d_row_bytes(I);
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
    for (int n = gw; n < H; n += nw) {
        float acc = 0.f;
        for (int s = 0; s < ns; ++s) {
            const uint8_t* row = rows0[s] + (size_t)n * rb;
            const float4* hv = smh + (size_t)s * 8 * IG;
            float part = 0.f;
            for (int hg = lane; hg < IG; hg += 32) {
                const uint4 c = ldg_stream(row + 16 * hg);
                const uint32_t m = ldg_u32(row + I / 2 + 4 * (hg >> 1));
                const float d = dot32(c, hv + hg, IG);
                const float2 sb = meta_to_f2(m);
                part = fmaf(sb.x, d, fmaf(sb.y, hsum[s * IG + hg], part));
            }
            acc = fmaf(wsl[s], part, acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) {
            if (y32) y32[n] = acc;
            if (y) {
                if (y_bf16) static_cast<__nv_bfloat16*>(y)[n] = __float2bfloat16_rn(acc);
                else static_cast<float*>(y)[n] = acc;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

static size_t gu_smem(int H) { return (size_t)H * 4 + (size_t)(H / 32) * 4; }
static size_t down_smem(int I, int ns) { return (size_t)ns * ((size_t)I * 4 + (size_t)(I / 32) * 4); }
static size_t router_smem(const Layer& L) {
    return (size_t)std::max(L.d.hidden / L.router_splits, L.d.n_experts) * 4;
}

cudaError_t decode_kernel_setup(Layer& L) {
    const int H = L.d.hidden, I = L.d.inter, ns = L.d.top_k + L.d.n_shared;
    cudaError_t e;
    e = cudaFuncSetAttribute(k_gateup_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu_smem(H));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_down_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)down_smem(I, ns));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_router_decode<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)router_smem(L));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_router_decode<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)router_smem(L));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_topk_tokens, cudaFuncAttributeMaxDynamicSharedMemorySize, L.d.n_experts * 4);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_gu, k_gateup_decode, kThreads, gu_smem(H));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_down, k_down_decode, kThreads, down_smem(I, ns));
    if (e != cudaSuccess) return e;
    if (L.occ_gu < 1 || L.occ_down < 1) return cudaErrorInvalidConfiguration;
    return cudaSuccess;
}

cudaError_t launch_route_decode(Layer& L, const void* x, cudaStream_t s) {
    const auto& d = L.d;
    dim3 grid((d.n_experts + kWarps - 1) / kWarps, L.router_splits);
    const int xb = d.act_dtype == MOE_BF16;
    prof_begin(L, K_ROUTER_DECODE, s);
    if (d.router_fmt == MOE_W_F32)
        k_router_decode<false><<<grid, kThreads, router_smem(L), s>>>(L.router, x, xb, d.hidden, d.n_experts,
                                                                      L.router_splits, L.router_bias, L.logits_part,
                                                                      L.logits, L.ids, L.wts, d.top_k, L.counters);
    else
        k_router_decode<true><<<grid, kThreads, router_smem(L), s>>>(L.router, x, xb, d.hidden, d.n_experts,
                                                                     L.router_splits, L.router_bias, L.logits_part,
                                                                     L.logits, L.ids, L.wts, d.top_k, L.counters);
    prof_end(L, s);
    return cudaGetLastError();
}

cudaError_t launch_route_tokens(Layer& L, const void* x, int T, cudaStream_t s) {
    const auto& d = L.d;
    const int xb = d.act_dtype == MOE_BF16;
    const int splits = L.router_splits;
    dim3 grid((d.n_experts + RT_E - 1) / RT_E, (T + RT_T - 1) / RT_T, splits);
    if ((d.hidden / splits) % RT_K) return cudaErrorInvalidValue;
    prof_begin(L, K_ROUTER_TOKENS, s);
    if (d.router_fmt == MOE_W_F32)
        k_router_tokens<false><<<grid, kThreads, 0, s>>>(L.router, x, xb, T, d.hidden, d.n_experts, splits,
                                                         L.logits_part);
    else
        k_router_tokens<true><<<grid, kThreads, 0, s>>>(L.router, x, xb, T, d.hidden, d.n_experts, splits,
                                                        L.logits_part);
    prof_end(L, s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prof_begin(L, K_TOPK_TOKENS, s);
    k_topk_tokens<<<T, kThreads, d.n_experts * 4, s>>>(L.logits_part, splits, T, d.n_experts, L.router_bias,
                                                       L.logits, L.ids, L.wts, d.top_k);
    prof_end(L, s);
    return cudaGetLastError();
}

cudaError_t launch_experts_decode(Layer& L, const void* x, void* y, float* y_f32, int which, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter, k = d.top_k, E = d.n_experts;
    const int xb = d.act_dtype == MOE_BF16;
    int slot0 = -1, nslots = 0;
    if ((which & RUN_ROUTED_GU) && (which & RUN_SHARED_GU)) { slot0 = 0; nslots = k + d.n_shared; }
    else if (which & RUN_ROUTED_GU) { slot0 = 0; nslots = k; }
    else if ((which & RUN_SHARED_GU) && d.n_shared) { slot0 = k; nslots = 1; }
    if (nslots > 0) {
        const int need = (nslots * I + kWarps - 1) / kWarps;
        const int grid = std::min(need, L.num_sms * L.occ_gu);
        prof_begin(L, K_GATEUP_DECODE, s);
        k_gateup_decode<<<grid, kThreads, gu_smem(H), s>>>(L.rec_table, L.ids, k, E, slot0, nslots, x, xb, H, I,
                                                           L.h);
        prof_end(L, s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (which & RUN_DOWN) {
        const int ns = k + d.n_shared;
        const int need = (H + kWarps - 1) / kWarps;
        const int grid = std::min(need, L.num_sms * L.occ_down);
        prof_begin(L, K_DOWN_DECODE, s);
        k_down_decode<<<grid, kThreads, down_smem(I, ns), s>>>(L.rec_table, L.ids, L.wts, k, E, d.n_shared, H, I,
                                                               L.h, y, xb, y_f32);
        prof_end(L, s);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace moe
