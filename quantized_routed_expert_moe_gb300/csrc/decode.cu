// Three-kernel decode, expert part: gate/up dequant-GEMV with SwiGLU, then
// down dequant-GEMV with the weighted combine.
//
// The kernels are chained with programmatic dependent launch:
//   router   -- selects the experts (router.cu);
//   gate/up  -- starts early and stages the activations, waits for the router,
//               then computes the shared and the routed experts;
//   down     -- starts early: prefetches its weight rows into L2 while gate/up
//               finishes, waits for gate/up, then stages the SwiGLU outputs
//               and combines.
// Both expert kernels are persistent grids of many warps; each warp issues all
// of a row's weight loads (128-bit, streaming) before it computes, so enough
// bytes are in flight to run at the memory roofline. The 4-bit codes are
// multiplied with 16-bit fixed-point activations by integer dp4a (common.cuh),
// about one instruction per weight.
//
// Gated experts, shared expert, combine: Inferno README "Model"; TurboFieldfare
// article, "token generation"; weight format: same article, "execution
// architecture".
#include "common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGuBlock = 6;      // half-groups per lane whose loads are in flight together (gate/up)
constexpr int kDownRows = 4;     // output rows per down work item (share the staged activations)
constexpr int kDownMaxRows = 96; // output rows one CTA owns in the down kernel

// Stage a vector of K activations (global, bf16 or fp32; `cg` reads bypass L1)
// into 16-bit fixed-point runs xq[4][K/32] with per-half-group inverse scale and
// sum. Block-wide, warp-uniform trip counts.
__device__ void stage_vector_q16(const void* x, int x_bf16, bool cg, int K, uint4* xq, float* inv, float* X) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrun = K / 8, KG = K / 32;
    for (int rb = warp * 32; rb < ((nrun + 31) / 32) * 32; rb += blockDim.x) {
        const int r = rb + lane;
        const bool valid = r < nrun;
        float v[8];
        if (!valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        } else if (x_bf16) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + r);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w4[i] << 16);
                v[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
            }
        } else {
            const float4* p = reinterpret_cast<const float4*>(x) + 2 * r;
            const float4 a = cg ? __ldcg(p) : __ldg(p);
            const float4 b = cg ? __ldcg(p + 1) : __ldg(p + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
        stage_q16_run(v, valid, r, KG, xq, inv, X);
    }
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------
//
// h[j][i] = silu(gate_i . x) * (up_i . x) for slot j (routed slots 0..k-1 in
// selection order, the shared expert at slot k). One warp per (slot, row i);
// lane l takes half-groups l, l + 32, ... of both rows.
__global__ void __launch_bounds__(kThreads) k_gateup(const uint8_t* const* __restrict__ rec_tab,
                                                     const float* __restrict__ part, int splits,
                                                     const float* __restrict__ bias, int k, int E, int n_shared,
                                                     const void* __restrict__ x, int x_bf16, int H, int I,
                                                     float* __restrict__ h, size_t rbH,
                                                     int32_t* __restrict__ ids_out, float* __restrict__ wts_out,
                                                     float* __restrict__ logits_out,
                                                     const int32_t* __restrict__ sel_ids, int jj0, int jj1,
                                                     unsigned long long* __restrict__ tr) {
    extern __shared__ uint4 smq[];
    __shared__ float s_logit[1024];
    __shared__ int32_t s_ids[MOE_MAX_TOP_K];
    __shared__ float s_wts[MOE_MAX_TOP_K];
    ktrace(tr, blockIdx.x, 0);
    const int HG = H / 32;
    uint4* xq = smq;                                                   // [4][HG]
    float* Iv = reinterpret_cast<float*>(smq + 4 * HG);                // [HG] 2^-f
    float* Xx = Iv + HG;                                               // [HG]
    stage_vector_q16(x, x_bf16, false, H, xq, Iv, Xx);
    __syncthreads();
    ktrace(tr, blockIdx.x, 2);
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
    const int M = (HG + 31) / 32;
    const uint64_t stream_pol = policy_evict_first();
    const uint32_t pair_bytes = (uint32_t)(2 * rbH);

    // The router's last CTA is latency-bound (atomics, partial logits, top-k);
    // weight traffic started before it finishes slows it by more than it
    // hides, so the weight rows (shared and routed) are all read after it.
    pdl_wait();
    pdl_trigger();
    ktrace(tr, blockIdx.x, 1);
    if (sel_ids) {
        // the selection was made earlier (streamed layers: the host staged
        // those experts first)
        if (threadIdx.x < k) s_ids[threadIdx.x] = sel_ids[threadIdx.x];
        __syncthreads();
    } else {
        // every CTA reduces the router's partial logits and selects (same result
        // everywhere); no CTA has to wait for a single selecting CTA
        block_select(part, splits, E, bias, k, s_logit, s_ids, s_wts);
        if (blockIdx.x == 0) {   // publish the selection (read by the host and by later calls)
            for (int e = threadIdx.x; e < E; e += blockDim.x) logits_out[e] = s_logit[e];
            if (threadIdx.x < k) { ids_out[threadIdx.x] = s_ids[threadIdx.x]; wts_out[threadIdx.x] = s_wts[threadIdx.x]; }
        }
    }
    {
        // slots in row order: the shared expert (slot k) first, then routed
        // 0..k-1; this launch covers row-order slots jj0 .. jj1 - 1
        const int nrows = (jj1 - jj0) * I;
        for (int r0 = gw; r0 < nrows; r0 += nw) {
            const int r = r0 + jj0 * I;
            const int jj = r / I;
            const int j = n_shared ? (jj == 0 ? k : jj - 1) : jj;
            const int i = r - jj * I;
            int e = j == k ? E : s_ids[j];
            if ((unsigned)e >= (unsigned)E && j < k) e = 0;  // a valid selection never needs this
            const uint8_t* g = rec_tab[e] + (size_t)(2 * i) * rbH;
            const uint8_t* u = g + rbH;
            // keep HBM busy across this warp's compute: pull the row pair two
            // steps ahead into L2 (same slot; it is contiguous with this one)
            if (lane == 0) {
                const int r2 = r + 2 * nw;
                if (r2 < jj1 * I && r2 / I == jj)
                    prefetch_l2_hint(rec_tab[e] + (size_t)(2 * (r2 - jj * I)) * rbH, pair_bytes, stream_pol);
            }
            float acc_g = 0.f, acc_u = 0.f;
            for (int m0 = 0; m0 < M; m0 += kGuBlock) {
                uint4 cg[kGuBlock], cu[kGuBlock];
                uint32_t mg[kGuBlock], mu[kGuBlock];
#pragma unroll
                for (int mm = 0; mm < kGuBlock; ++mm) {
                    const int hg = lane + 32 * (m0 + mm);
                    if (m0 + mm < M && hg < HG) {
                        cg[mm] = ldg_stream_hint(g + 16 * hg, stream_pol);
                        cu[mm] = ldg_stream_hint(u + 16 * hg, stream_pol);
                        mg[mm] = ldg_u32_hint(g + H / 2 + 4 * (hg >> 1), stream_pol);
                        mu[mm] = ldg_u32_hint(u + H / 2 + 4 * (hg >> 1), stream_pol);
                    }
                }
#pragma unroll
                for (int mm = 0; mm < kGuBlock; ++mm) {
                    const int hg = lane + 32 * (m0 + mm);
                    if (m0 + mm < M && hg < HG) {
                        int gh = 0, gl = 0, uh = 0, ul = 0;
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            const uint4 xs = xq[wi * HG + hg];
                            word_dp4a(u4w(cg[mm], wi), xs, gh, gl);
                            word_dp4a(u4w(cu[mm], wi), xs, uh, ul);
                        }
                        const float iv = Iv[hg], xs = Xx[hg];
                        const float2 sg = meta_to_f2(mg[mm]), su = meta_to_f2(mu[mm]);
                        acc_g = fmaf(sg.x, (float)(gh * 256 + gl) * iv, fmaf(sg.y, xs, acc_g));
                        acc_u = fmaf(su.x, (float)(uh * 256 + ul) * iv, fmaf(su.y, xs, acc_u));
                    }
                }
            }
            const float gv = warp_sum(acc_g);
            const float uv = warp_sum(acc_u);
            if (lane == 0) h[(size_t)j * I + i] = silu_f(gv) * uv;
        }
    }
    __syncthreads();
    ktrace(tr, blockIdx.x, 3);
}

// ---------------------------------------------------------------------------
// down + combine
// ---------------------------------------------------------------------------
//
// CTA c owns output rows [c*H/G, (c+1)*H/G). Work items are (4 rows, slot);
// a warp computes the 4 rows' dot products with that slot's SwiGLU output
// (staged once per CTA in 16-bit fixed point per half-group), keeping the
// results per (slot, row); the rows are then combined in a fixed order:
// shared expert first (weight 1), then the routed slots in selection order.
__global__ void __launch_bounds__(kThreads) k_down(const uint8_t* const* __restrict__ rec_tab,
                                                   const float* __restrict__ part, int splits,
                                                   const float* __restrict__ bias,
                                                   int k, int E, int n_shared, int H, int I,
                                                   const float* __restrict__ h, void* __restrict__ y, int y_bf16,
                                                   float* __restrict__ y32, size_t rbI, size_t gu_block,
                                                   const int32_t* __restrict__ sel_ids,
                                                   const float* __restrict__ sel_wts,
                                                   unsigned long long* __restrict__ tr) {
    extern __shared__ uint4 smh[];
    ktrace(tr, blockIdx.x, 0);
    const int IG = I / 32, ns = k + n_shared;
    uint4* hq = smh;                                                     // [ns][4][IG]
    float* Iv = reinterpret_cast<float*>(hq + (size_t)ns * 4 * IG);     // [ns][IG]
    float* Xh = Iv + ns * IG;                                            // [ns][IG]
    float* ypart = Xh + ns * IG;                                         // [ns][kDownMaxRows]
    __shared__ const uint8_t* s_rows[MOE_MAX_TOP_K + 1];
    __shared__ float s_w[MOE_MAX_TOP_K + 1];
    __shared__ float s_logit[1024];
    __shared__ int32_t s_ids[MOE_MAX_TOP_K];
    __shared__ float s_wts[MOE_MAX_TOP_K];
    const int own0 = (int)((long long)H * blockIdx.x / gridDim.x);
    const int own1 = (int)((long long)H * (blockIdx.x + 1) / gridDim.x);
    // the router has completed when this kernel starts (gate/up waited for it
    // before allowing this launch): select from its partial logits and prefetch
    // this CTA's down rows of every slot into L2 while gate/up finishes
    if (sel_ids) {   // selection made earlier (streamed layers)
        if (threadIdx.x < k) { s_ids[threadIdx.x] = sel_ids[threadIdx.x]; s_wts[threadIdx.x] = sel_wts[threadIdx.x]; }
        __syncthreads();
    } else {
        block_select(part, splits, E, bias, k, s_logit, s_ids, s_wts);
    }
    if (threadIdx.x < ns) {
        const int s = threadIdx.x;
        const bool sh = n_shared && s == 0;
        const int j = sh ? k : s - n_shared;
        int e = sh ? E : s_ids[j];
        if ((unsigned)e > (unsigned)E) e = 0;
        const uint8_t* base = rec_tab[e] + gu_block;
        s_rows[s] = base;
        s_w[s] = sh ? 1.0f : s_wts[j];
        if (own1 > own0)
            prefetch_l2_hint(base + (size_t)own0 * rbI, (uint32_t)((own1 - own0) * rbI), policy_evict_last());
    }
    pdl_wait();     // gate/up complete: h is final
    pdl_trigger();  // the next token's router may start prefetching its weights
    ktrace(tr, blockIdx.x, 1);
    // stage every slot's h (shared first, then routed in selection order); all
    // of a thread's loads are issued before any is used (one L2 round trip)
    {
        const int warp0 = threadIdx.x >> 5, lane0 = threadIdx.x & 31;
        const int nrun = I / 8, total = ns * nrun;
        const int rounds = (total + blockDim.x - 1) / blockDim.x;   // warp-uniform
        for (int rb0 = 0; rb0 < rounds; rb0 += 4) {
            float v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = (rb0 + u) * blockDim.x + warp0 * 32 + lane0;
                const bool valid = rb0 + u < rounds && idx < total;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
                if (valid) {
                    const int s = idx / nrun, r = idx - s * nrun;
                    const int j = (n_shared && s == 0) ? k : s - n_shared;
                    const float4* src = reinterpret_cast<const float4*>(h + (size_t)j * I) + 2 * r;
                    a = __ldcg(src);
                    c = __ldcg(src + 1);
                }
                v[u][0] = a.x; v[u][1] = a.y; v[u][2] = a.z; v[u][3] = a.w;
                v[u][4] = c.x; v[u][5] = c.y; v[u][6] = c.z; v[u][7] = c.w;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (rb0 + u >= rounds) break;   // uniform across the block
                const int idx = (rb0 + u) * blockDim.x + warp0 * 32 + lane0;
                const bool valid = idx < total;
                const int s = valid ? idx / nrun : 0, r = valid ? idx - s * nrun : 0;
                // a half-group's four runs are in four consecutive lanes (nrun % 4 == 0)
                stage_q16_run(v[u], valid, r, IG, hq + (size_t)s * 4 * IG, Iv + s * IG, Xh + s * IG);
            }
        }
    }
    __syncthreads();
    ktrace(tr, blockIdx.x, 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int own = own1 - own0;
    const int nquad = (own + kDownRows - 1) / kDownRows;
    const int M = (IG + 31) / 32;
    for (int it = warp; it < nquad * ns; it += kWarps) {
        const int q = it / ns, s = it - q * ns;
        const int n0 = own0 + q * kDownRows, nr = min(kDownRows, own1 - n0);
        const uint8_t* rr[kDownRows];
#pragma unroll
        for (int r = 0; r < kDownRows; ++r) rr[r] = s_rows[s] + (size_t)(n0 + min(r, nr - 1)) * rbI;
        const uint4* xs = hq + (size_t)s * 4 * IG;
        const float* ivs = Iv + s * IG;
        const float* xsum = Xh + s * IG;
        float acc[kDownRows];
#pragma unroll
        for (int r = 0; r < kDownRows; ++r) acc[r] = 0.f;
        for (int m = 0; m < M; m += 2) {
            uint4 c[2][kDownRows];
            uint32_t mt[2][kDownRows];
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                const int hg = lane + 32 * (m + mm);
#pragma unroll
                for (int r = 0; r < kDownRows; ++r)
                    if (m + mm < M && hg < IG) {
                        c[mm][r] = ldg_stream(rr[r] + 16 * hg);
                        mt[mm][r] = ldg_u32(rr[r] + I / 2 + 4 * (hg >> 1));
                    }
            }
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                const int hg = lane + 32 * (m + mm);
                if (m + mm < M && hg < IG) {
                    int ah[kDownRows], al[kDownRows];
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r) ah[r] = al[r] = 0;
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint4 xv = xs[wi * IG + hg];
#pragma unroll
                        for (int r = 0; r < kDownRows; ++r) word_dp4a(u4w(c[mm][r], wi), xv, ah[r], al[r]);
                    }
                    const float iv = ivs[hg], xx = xsum[hg];
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r) {
                        const float2 sb = meta_to_f2(mt[mm][r]);
                        acc[r] = fmaf(sb.x, (float)(ah[r] * 256 + al[r]) * iv, fmaf(sb.y, xx, acc[r]));
                    }
                }
            }
        }
        float d[kDownRows];
#pragma unroll
        for (int r = 0; r < kDownRows; ++r) d[r] = warp_sum(acc[r]);
#pragma unroll
        for (int r = 0; r < kDownRows; ++r)
            if (lane == r && r < nr) ypart[s * kDownMaxRows + (n0 - own0) + r] = d[r];
    }
    __syncthreads();
    for (int n = own0 + threadIdx.x; n < own1; n += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < ns; ++s) acc = fmaf(s_w[s], ypart[s * kDownMaxRows + (n - own0)], acc);
        if (y32) y32[n] = acc;
        if (y) {
            if (y_bf16) static_cast<__nv_bfloat16*>(y)[n] = __float2bfloat16_rn(acc);
            else static_cast<float*>(y)[n] = acc;
        }
    }
    __syncthreads();
    ktrace(tr, blockIdx.x, 3);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

static size_t gu_smem(int H) { return (size_t)H * 2 + (size_t)(H / 32) * 8; }
static size_t down_smem(int I, int ns) {
    return (size_t)ns * I * 2 + (size_t)ns * (I / 32) * 8 + (size_t)ns * kDownMaxRows * 4;
}
static int down_grid(const Layer& L) { return L.num_sms * L.occ_down; }

cudaError_t decode_kernel_setup(Layer& L) {
    const int H = L.d.hidden, I = L.d.inter, ns = L.d.top_k + L.d.n_shared;
    cudaError_t e = router_kernel_setup(L);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu_smem(H));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)down_smem(I, ns));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_gu, k_gateup, kThreads, gu_smem(H));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_down, k_down, kThreads, down_smem(I, ns));
    if (e != cudaSuccess) return e;
    if (L.occ_gu < 1 || L.occ_down < 1) return cudaErrorInvalidConfiguration;
    // rows owned by one down CTA must fit its partial-sum buffer
    while ((H + down_grid(L) - 1) / down_grid(L) > kDownMaxRows) {
        if (L.occ_down >= 64) return cudaErrorInvalidConfiguration;
        ++L.occ_down;   // more (smaller) CTAs per SM are launched in waves
    }
    return cudaSuccess;
}

cudaError_t launch_experts_decode(Layer& L, const void* x, void* y, float* y_f32, int which, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter, k = d.top_k, E = d.n_experts;
    const int xb = d.act_dtype == MOE_BF16;
    cudaError_t e;
    if (which & (RUN_ROUTED_GU | RUN_SHARED_GU)) {
        const int need = ((k + d.n_shared) * I + kWarps - 1) / kWarps;
        const int grid = std::max(1, std::min(need, L.num_sms * L.occ_gu));
        prof_begin(L, K_GATEUP_DECODE, s);
        e = launch_pdl(k_gateup, dim3(grid), dim3(kThreads), gu_smem(H), s, L.pdl, (const uint8_t* const*)L.rec_table,
                       (const float*)L.logits_part, L.router_splits, (const float*)L.router_bias, k, E,
                       d.n_shared, x, xb, H, I, L.h, row_bytes(H), L.ids, L.wts, L.logits, (const int32_t*)nullptr, 0,
                       k + d.n_shared, L.split_trace(1));
        prof_end(L, s);
        if (e != cudaSuccess) return e;
    }
    if (which & RUN_DOWN) {
        const int ns = k + d.n_shared;
        prof_begin(L, K_DOWN_DECODE, s);
        e = launch_pdl(k_down, dim3(down_grid(L)), dim3(kThreads), down_smem(I, ns), s, L.pdl,
                       (const uint8_t* const*)L.rec_table, (const float*)L.logits_part, L.router_splits,
                       (const float*)L.router_bias, k, E,
                       d.n_shared, H, I, (const float*)L.h, y, xb, y_f32, row_bytes(I), gu_block_bytes(H, I),
                       (const int32_t*)nullptr, (const float*)nullptr, L.split_trace(2));
        prof_end(L, s);
        return e;
    }
    return cudaSuccess;
}

// The same two expert kernels over caller-given scratch: router partials
// `part` [splits][E] (already written on `s`), selection out (`logits` [E],
// `ids` [k], `wts` [k]) and SwiGLU outputs `h` [k + 1][I]. No profiling or tracing.
cudaError_t launch_experts_decode_scratch(Layer& L, const void* x, void* y, float* y_f32, const float* part,
                                          float* logits, int32_t* ids, float* wts, float* h, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter, k = d.top_k, E = d.n_experts, ns = k + d.n_shared;
    const int xb = d.act_dtype == MOE_BF16;
    const int need = (ns * I + kWarps - 1) / kWarps;
    const int grid = std::max(1, std::min(need, L.num_sms * L.occ_gu));
    cudaError_t e = launch_pdl(k_gateup, dim3(grid), dim3(kThreads), gu_smem(H), s, L.pdl,
                               (const uint8_t* const*)L.rec_table, part, L.router_splits,
                               (const float*)L.router_bias, k, E, d.n_shared, x, xb, H, I, h, row_bytes(H), ids, wts,
                               logits, (const int32_t*)nullptr, 0, ns, (unsigned long long*)nullptr);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_down, dim3(down_grid(L)), dim3(kThreads), down_smem(I, ns), s, L.pdl,
                      (const uint8_t* const*)L.rec_table, part, L.router_splits, (const float*)L.router_bias, k, E,
                      d.n_shared, H, I, (const float*)h, y, xb, y_f32, row_bytes(I), gu_block_bytes(H, I),
                      (const int32_t*)nullptr, (const float*)nullptr, (unsigned long long*)nullptr);
}

// Streamed layers: the selection (ids, wts of one token) is already on the
// device and the routed experts' records are resident. `jj0..jj1` are the
// row-order slots of gate/up to run (0 = the shared expert when there is one);
// `down` adds the down + combine kernel. Plain launches (no programmatic
// overlap): the caller orders them against the cache's copies with events.
cudaError_t launch_experts_decode_sel(Layer& L, const void* x, void* y, float* y_f32, const int32_t* ids,
                                      const float* wts, int jj0, int jj1, bool down, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter, k = d.top_k, E = d.n_experts, ns = k + d.n_shared;
    const int xb = d.act_dtype == MOE_BF16;
    cudaError_t e = cudaSuccess;
    if (jj1 > jj0) {
        const int need = ((jj1 - jj0) * I + kWarps - 1) / kWarps;
        const int grid = std::max(1, std::min(need, L.num_sms * L.occ_gu));
        prof_begin(L, K_GATEUP_DECODE, s);
        e = launch_pdl(k_gateup, dim3(grid), dim3(kThreads), gu_smem(H), s, false, (const uint8_t* const*)L.rec_table,
                       (const float*)nullptr, 0, (const float*)nullptr, k, E, d.n_shared, x, xb, H, I, L.h,
                       row_bytes(H), (int32_t*)nullptr, (float*)nullptr, (float*)nullptr, ids, jj0, jj1,
                       (unsigned long long*)nullptr);
        prof_end(L, s);
        if (e != cudaSuccess) return e;
    }
    if (down) {
        prof_begin(L, K_DOWN_DECODE, s);
        e = launch_pdl(k_down, dim3(down_grid(L)), dim3(kThreads), down_smem(I, ns), s, false,
                       (const uint8_t* const*)L.rec_table, (const float*)nullptr, 0, (const float*)nullptr, k, E,
                       d.n_shared, H, I, (const float*)L.h, y, xb, y_f32, row_bytes(I), gu_block_bytes(H, I), ids,
                       wts, (unsigned long long*)nullptr);
        prof_end(L, s);
    }
    return e;
}

}  // namespace moe
