// Routing: router GEMV/GEMM, exact top-k selection, softmax over the selected
// experts.
//
// Router and exact top-8 selection: TurboFieldfare article, "token
// generation"; Inferno README, "Current Scope"; Colibri report, section 3.
// 8-bit router weights: TurboFieldfare article, "execution architecture".
#include <cfloat>
#include <climits>

#include <algorithm>

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
// ---------------------------------------------------------------------------
// router GEMV for one token: split over H, last CTA reduces and selects
// ---------------------------------------------------------------------------
//
// Grid (ceil(E/8), splits); warp w of CTA (bx, by) computes the partial logit
// of expert 8*bx + w over inputs [by*Ls, (by+1)*Ls). With programmatic
// dependent launch, the weight slice is prefetched into L2 before waiting for
// the preceding kernel (the activations may come from it); the partials are
// then reduced in split order by the last CTA to finish, which selects and
// writes ids, weights and logits.
//
// One token's access to a device-managed cache (thread 0, on the slot state
// the block staged in shared memory: se expert, sc count, sl last use). The
// policy is the host's (cache.cu) step for step, with the counts and last uses
// kept per slot:
//   * a pinned expert (the learning cache) is a hit that leaves the state alone;
//   * hits first, in selection order: count + 1, last use = this token;
//   * then each miss in selection order takes the lowest free slot, else the
//     slot of the resident with the smallest count that this token does not
//     need (ties: the least recently used, then the lower expert id), and
//     enters with count 1;
//   * the record table points each admitted expert at its slot and forgets the
//     evicted one; the fill list and the statistics are written for the copy
//     kernel and the host.
__device__ void dev_lfu_access(const DevCacheArgs& dc, const int32_t* ids_g, int n, int32_t* se, uint32_t* sc,
                               uint32_t* sl) {
    int32_t ids[MOE_MAX_TOP_K];
    for (int i = 0; i < n; ++i) ids[i] = ids_g[i];
    const int S = dc.slots;
    const uint32_t clk = *dc.clock + 1u;
    *dc.clock = clk;
    int hits = 0, nf = 0;
    bool pin[MOE_MAX_TOP_K];
    for (int i = 0; i < n; ++i) {
        dc.usage[ids[i]] += 1ull;
        pin[i] = dc.pinned[ids[i]] != 0;
        hits += pin[i];   // pinned (learning cache): served outside the slots
    }
    for (int i = 0; i < n; ++i)
        for (int s = 0; s < S; ++s)
            if (se[s] == ids[i]) {
                ++hits;
                sc[s] += 1u;
                sl[s] = clk;
            }
    for (int i = 0; i < n; ++i) {
        const int e = ids[i];
        if (pin[i]) continue;
        bool resident = false;
        for (int s = 0; s < S; ++s) resident |= se[s] == e;
        if (resident) continue;
        int slot = -1;
        for (int s = 0; s < S && slot < 0; ++s)
            if (se[s] < 0) slot = s;
        if (slot < 0) {
            int vs = -1;
            for (int s = 0; s < S; ++s) {
                const int r = se[s];
                bool needed = false;
                for (int j = 0; j < n; ++j) needed |= ids[j] == r;
                if (needed) continue;
                if (vs < 0 || sc[s] < sc[vs] || (sc[s] == sc[vs] && (sl[s] < sl[vs] || (sl[s] == sl[vs] && r < se[vs]))))
                    vs = s;
            }
            if (vs < 0) {   // cannot happen while a token's ids fit the slots
                atomicOr(dc.err, 1u << 26);
                break;
            }
            dc.rec_table[se[vs]] = nullptr;
            slot = vs;
        }
        se[slot] = e;
        sc[slot] = 1u;
        sl[slot] = clk;
        dc.rec_table[e] = dc.slots_base + (size_t)slot * dc.rb;
        dc.fills[1 + 2 * nf] = e;
        dc.fills[2 + 2 * nf] = slot;
        ++nf;
    }
    dc.fills[0] = nf;
    dc.stats[0] += 1ull;
    dc.stats[1] += (unsigned long long)hits;
    dc.stats[2] += (unsigned long long)nf;
    dc.stats[3] += (unsigned long long)nf * dc.rb;
}

// Dot product of router row e with the activation slice [k0, k0 + Ls) staged
// as fp32 in xs_slice, by one warp; every lane returns the warp's sum. Fp32
// rows: 8 float4 loads in flight per lane. Q8 rows: 16 codes per load, each
// summed as scale * sum(q * x) + bias * sum(x) per 16 inputs of a group of 64.
template <bool Q8>
__device__ __forceinline__ float router_warp_dot(const void* __restrict__ W, const float* xs_slice, int H, int E,
                                                 int e, int k0, int Ls) {
    const int lane = threadIdx.x & 31;
    float acc = 0.f;
    if (!Q8) {
        const float4* row = reinterpret_cast<const float4*>(static_cast<const float*>(W) + (size_t)e * H + k0);
        const float4* xs = reinterpret_cast<const float4*>(xs_slice);
        for (int c0 = lane; c0 < Ls / 4; c0 += 32 * 8) {
            float4 wv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {   // 8 loads in flight per lane
                const int c = c0 + 32 * u;
                wv[u] = (c < Ls / 4) ? __ldg(row + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + 32 * u;
                if (c < Ls / 4) {
                    const float4 xv = xs[c];
                    acc = fmaf(wv[u].x, xv.x, acc);
                    acc = fmaf(wv[u].y, xv.y, acc);
                    acc = fmaf(wv[u].z, xv.z, acc);
                    acc = fmaf(wv[u].w, xv.w, acc);
                }
            }
        }
    } else {
        const uint8_t* codes = static_cast<const uint8_t*>(W) + (size_t)e * H + k0;
        const uint32_t* meta = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(W) + (size_t)E * H) +
                               (size_t)e * (H / 64) + k0 / 64;
        for (int c0 = lane; c0 < Ls / 16; c0 += 32 * 4) {
            uint4 qv[4];
            uint32_t mv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 32 * u;
                qv[u] = (c < Ls / 16) ? ldg_stream(codes + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
                mv[u] = (c < Ls / 16) ? __ldg(meta + (c >> 2)) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 32 * u;
                if (c < Ls / 16) {
                    const uint32_t qw[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
                    float aq = 0.f, ax = 0.f;
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const float xv = xs_slice[16 * c + t];
                        aq = fmaf(__uint_as_float(0x4B000000u | ((qw[t >> 2] >> (8 * (t & 3))) & 0xFFu)) - 8388608.0f,
                                  xv, aq);
                        ax += xv;
                    }
                    const float2 sb = meta_to_f2(mv[u]);
                    acc = fmaf(sb.x, aq, fmaf(sb.y, ax, acc));
                }
            }
        }
    }
    return warp_sum(acc);
}

template <bool Q8>
__global__ void __launch_bounds__(kThreads) k_router_decode(
    const void* __restrict__ W, const void* __restrict__ x, int x_bf16, int H, int E, int splits,
    const float* __restrict__ bias, float* __restrict__ part, float* __restrict__ logits,
    int32_t* __restrict__ ids, float* __restrict__ wts, int k, unsigned* __restrict__ counter,
    int select, RouteMode mode, int32_t* ids_pub, unsigned* seq_pub, unsigned seq, DevCacheArgs dc,
    unsigned* ids_ready, unsigned long long* part_tag, const unsigned* seq_word,
    unsigned long long* __restrict__ tr) {
    extern __shared__ float sm[];
    __shared__ unsigned s_last;
    const int cta = blockIdx.y * gridDim.x + blockIdx.x;
    ktrace(tr, cta, 0);
    const int Ls = H / splits;
    const int k0 = blockIdx.y * Ls;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kWarps + warp;
    // prefetch this warp's weight slice into L2 (constant data)
    if (e < E && lane == 0) {
        const uint8_t* src = Q8 ? static_cast<const uint8_t*>(W) + (size_t)e * H + k0
                                : reinterpret_cast<const uint8_t*>(static_cast<const float*>(W) + (size_t)e * H + k0);
        const uint32_t bytes = Q8 ? (uint32_t)Ls : (uint32_t)Ls * 4;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
    }
    pdl_wait();
    pdl_trigger();
    ktrace(tr, cta, 1);
    for (int i4 = threadIdx.x; i4 < Ls / 4; i4 += blockDim.x) {
        float4 v;
        if (x_bf16) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + k0) + i4);
            v = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                            __uint_as_float(w.y & 0xFFFF0000u));
        } else {
            v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + k0) + i4);
        }
        reinterpret_cast<float4*>(sm)[i4] = v;
    }
    __syncthreads();
    if (e < E) {
        const float acc = router_warp_dot<Q8>(W, reinterpret_cast<const float*>(sm), H, E, e, k0, Ls);
        if (lane == 0) {
            if (part_tag) {
                // tagged partial: the token's tag beside the value in one
                // 64-bit store, which readers poll for (no fence, no counter)
                const unsigned long long w =
                    ((unsigned long long)decode_tag(__ldcg(seq_word)) << 32) | __float_as_uint(acc);
                asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(part_tag + (size_t)blockIdx.y * E + e),
                             "l"(w)
                             : "memory");
            } else {
                part[(size_t)blockIdx.y * E + e] = acc;
            }
        }
    }
    __syncthreads();
    ktrace(tr, cta, 2);
    if (!select) {   // partials only
        ktrace(tr, cta, 3);
        return;
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(counter, 1u);
        s_last = (prev == gridDim.x * gridDim.y - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) { ktrace(tr, cta, 3); return; }
    __threadfence();
    for (int e2 = threadIdx.x; e2 < E; e2 += blockDim.x) {
        float v[kMaxRouterSplits];
#pragma unroll
        for (int s = 0; s < kMaxRouterSplits; ++s) v[s] = (s < splits) ? __ldcg(part + (size_t)s * E + e2) : 0.f;
        float l = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxRouterSplits; ++s)
            if (s < splits) l += v[s];
        // keys in sm[0, E), sigmoid scores in sm[E, 2E)
        const float key = route_key(l, bias ? bias[e2] : 0.f, mode, sm + E + e2);
        sm[e2] = key;
        logits[e2] = key;
    }
    __syncthreads();
    block_topk(sm, E, k, ids, wts, mode.sigmoid ? sm + E : nullptr, mode.scale);
    // the decode's gate/up waits for this flag instead of the grid's end
    // (thread 0 wrote the ids and weights)
    if (threadIdx.x == 0 && ids_ready) {
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ids_ready), "r"(1u) : "memory");
    }
    // streamed layers: the selection straight into host-mapped memory, then
    // its sequence number (thread 0 wrote the ids itself)
    if (threadIdx.x == 0 && ids_pub) {
        for (int r = 0; r < k; ++r) ids_pub[r] = ids[r];
        __threadfence_system();
        *(volatile unsigned*)seq_pub = seq;
    }
    // device-managed cache: the LFU step for this token's ids (thread 0 wrote
    // them), on the slot state staged in shared memory and written back
    if (dc.slot_expert) {
        int32_t* se = reinterpret_cast<int32_t*>(sm);
        uint32_t* sc = reinterpret_cast<uint32_t*>(sm) + dc.slots;
        uint32_t* sl = sc + dc.slots;
        __syncthreads();   // the selection is done with sm
        for (int s2 = threadIdx.x; s2 < dc.slots; s2 += blockDim.x) {
            se[s2] = dc.slot_expert[s2];
            sc[s2] = dc.slot_count[s2];
            sl[s2] = dc.slot_last[s2];
        }
        __syncthreads();
        if (threadIdx.x == 0) dev_lfu_access(dc, ids, k, se, sc, sl);
        __syncthreads();
        for (int s2 = threadIdx.x; s2 < dc.slots; s2 += blockDim.x) {
            dc.slot_expert[s2] = se[s2];
            dc.slot_count[s2] = sc[s2];
            dc.slot_last[s2] = sl[s2];
        }
    }
    if (threadIdx.x == 0) *counter = 0u;
    __syncthreads();
    ktrace(tr, cta, 3);
}

// ---------------------------------------------------------------------------
// router for T tokens: split-K tiles (16 tokens x 64 experts), then per-token top-k
// ---------------------------------------------------------------------------
constexpr int RT_T = 32, RT_E = 128, RT_K = 64;

// Tile of 32 tokens x 128 experts over one split's K range, in chunks of 64:
// x and W are staged transposed (k-major) in shared memory; thread (ty, tx)
// keeps the fp32 sums of tokens 4ty..4ty+3 x experts 4tx..4tx+3 (the four x
// values are one broadcast read per warp), and the next chunk's global loads
// are in flight while the current chunk is multiplied.
template <bool Q8>
__global__ void __launch_bounds__(kThreads, 2) k_router_tokens(const void* __restrict__ W, const void* __restrict__ x,
                                                            int x_bf16, int T, int H, int E, int splits,
                                                            float* __restrict__ part) {
    constexpr int NX = RT_T * RT_K / kThreads, NW = RT_E * RT_K / kThreads;   // 8, 32
    __shared__ __align__(16) float xs[RT_K][RT_T + 4];
    __shared__ __align__(16) float ws[RT_K][RT_E + 4];
    const int e0 = blockIdx.y * RT_E, t0 = blockIdx.x * RT_T;
    const int Ls = H / splits, kb = blockIdx.z * Ls;
    const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
    const int c = tid & (RT_K - 1), r0 = tid / RT_K;   // staging: k within the chunk, first row
    constexpr int RS = kThreads / RT_K;                 // rows per staging pass (4)
    float acc[4][4] = {};
    float vx[NX], vw[NW];
    auto load = [&](int kc) {
#pragma unroll
        for (int j = 0; j < NX; ++j) {
            const int r = r0 + RS * j;
            vx[j] = (t0 + r < T) ? load_act(x, x_bf16, (size_t)(t0 + r) * H + kc + c) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const int r = r0 + RS * j;
            float w = 0.f;
            if (e0 + r < E) {
                if (!Q8) {
                    w = __ldg(static_cast<const float*>(W) + (size_t)(e0 + r) * H + kc + c);
                } else {
                    const uint8_t* base = static_cast<const uint8_t*>(W);
                    const uint32_t m = __ldg(reinterpret_cast<const uint32_t*>(base + (size_t)E * H) +
                                             (size_t)(e0 + r) * (H / 64) + (kc / 64));
                    const float2 sb = meta_to_f2(m);
                    w = fmaf((float)__ldg(base + (size_t)(e0 + r) * H + kc + c), sb.x, sb.y);
                }
            }
            vw[j] = w;
        }
    };
    load(kb);
    for (int kc = kb; kc < kb + Ls; kc += RT_K) {
        __syncthreads();   // the previous chunk's reads of xs / ws are done
#pragma unroll
        for (int j = 0; j < NX; ++j) xs[c][r0 + RS * j] = vx[j];
#pragma unroll
        for (int j = 0; j < NW; ++j) ws[c][r0 + RS * j] = vw[j];
        __syncthreads();
        if (kc + RT_K < kb + Ls) load(kc + RT_K);
#pragma unroll 8
        for (int q = 0; q < RT_K; ++q) {
            const float4 a = *reinterpret_cast<const float4*>(&xs[q][4 * ty]);
            const float4 w4 = *reinterpret_cast<const float4*>(&ws[q][4 * tx]);
            const float av[4] = {a.x, a.y, a.z, a.w}, wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + 4 * ty + i;
        if (t < T)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e0 + 4 * tx + j < E) part[((size_t)blockIdx.z * T + t) * E + e0 + 4 * tx + j] = acc[i][j];
    }
}

// Prefill chunks also need each token's activation exponent a_t (see
// fp16_fit_exp): the grouped GEMM's operands are x_t * 2^a_t in binary16.
__global__ void __launch_bounds__(kThreads) k_topk_tokens(const float* __restrict__ part, int splits, int T, int E,
                                                          const float* __restrict__ bias, float* __restrict__ logits,
                                                          int32_t* __restrict__ ids, float* __restrict__ wts, int k,
                                                          RouteMode mode, const void* __restrict__ x, int x_bf16,
                                                          int H, int32_t* __restrict__ xexp) {
    extern __shared__ float sl[];   // keys [E], then sigmoid scores [E]
    __shared__ float s_red[kWarps];
    const int t = blockIdx.x;
    if (xexp) {   // the token's activation exponent (prefill chunks)
        // 8 activations per 16-byte load (H is a multiple of 64)
        float m = 0.f;
        for (int r = threadIdx.x; r < H / 8; r += blockDim.x) {
            float v[8];
            if (x_bf16) {
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * H) + r);
                const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = __uint_as_float(w4[i] << 16);
                    v[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
                }
            } else {
                const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)t * H) + 2 * r;
                const float4 a = __ldg(p), b = __ldg(p + 1);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float r = 0.f;
            for (int w = 0; w < kWarps; ++w) r = fmaxf(r, s_red[w]);
            xexp[t] = fp16_fit_exp(r);
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float v[kMaxTokSplits];
#pragma unroll
        for (int s = 0; s < kMaxTokSplits; ++s) v[s] = (s < splits) ? __ldcg(part + ((size_t)s * T + t) * E + e) : 0.f;
        float l = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxTokSplits; ++s) l += v[s];
        const float key = route_key(l, bias ? bias[e] : 0.f, mode, sl + E + e);
        sl[e] = key;
        logits[(size_t)t * E + e] = key;
    }
    __syncthreads();
    block_topk(sl, E, k, ids + (size_t)t * k, wts + (size_t)t * k, mode.sigmoid ? sl + E : nullptr, mode.scale);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

// keys [E], then sigmoid scores [E]
static int select_smem_words(int E) { return 2 * E; }

static size_t router_smem(const Layer& L) {
    // x slice, or the selection's arrays, or a device-managed cache's slot state
    return (size_t)std::max({L.d.hidden / L.router_splits, select_smem_words(L.d.n_experts), 3 * L.d.cache_slots}) * 4;
}

cudaError_t router_kernel_setup(Layer& L) {
    cudaError_t e;
    e = cudaFuncSetAttribute(k_router_decode<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)router_smem(L));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_router_decode<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)router_smem(L));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_topk_tokens, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                select_smem_words(L.d.n_experts) * 4);
}

cudaError_t launch_route_decode(Layer& L, const void* x, cudaStream_t s, int select, int32_t* ids_pub,
                                unsigned* seq_pub, unsigned seq, const DevCacheArgs* dc, const DecodeScratch* out) {
    const DevCacheArgs dca = dc ? *dc : DevCacheArgs{};
    const auto& d = L.d;
    dim3 grid((d.n_experts + kWarps - 1) / kWarps, L.router_splits);
    const int xb = d.act_dtype == MOE_BF16;
    float* part = out ? out->part : L.logits_part;
    float* logits = out ? out->logits : L.logits;
    int32_t* ids = out ? out->ids : L.ids;
    float* wts = out ? out->wts : L.wts;
    unsigned* cnt = out ? out->router_cnt : L.counters + CNT_ROUTER;
    unsigned* ready = out ? out->ids_ready : nullptr;
    unsigned long long* ptag = out ? out->part_tag : nullptr;   // tagged partials, no selection here
    if (ptag) select = 0;
    auto kern = d.router_fmt == MOE_W_F32 ? k_router_decode<false> : k_router_decode<true>;
    prof_begin(L, K_ROUTER_DECODE, s);
    const cudaError_t e = launch_pdl(kern, grid, dim3(kThreads), router_smem(L), s, L.pdl, L.router, x, xb, d.hidden,
                                     d.n_experts, L.router_splits, (const float*)L.router_bias, part, logits, ids, wts,
                                     d.top_k, cnt, select, L.route_mode(), ids_pub, seq_pub, seq, dca, ready,
                                     ptag, out ? out->seq : nullptr, L.split_trace(0));
    prof_end(L, s);
    return e;
}

cudaError_t launch_route_tokens(Layer& L, const void* x, int T, cudaStream_t s, int32_t* xexp) {
    const auto& d = L.d;
    const int xb = d.act_dtype == MOE_BF16;
    const int splits = L.router_splits_tok;
    dim3 grid((T + RT_T - 1) / RT_T, (d.n_experts + RT_E - 1) / RT_E, splits);
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
    k_topk_tokens<<<T, kThreads, select_smem_words(d.n_experts) * 4, s>>>(L.logits_part, splits, T, d.n_experts, L.router_bias,
                                                           L.logits, L.ids, L.wts, d.top_k, L.route_mode(), x, xb,
                                                           d.hidden, xexp);
    prof_end(L, s);
    return cudaGetLastError();
}

}  // namespace moe
