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
#include "sm100.cuh"

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
// selection order, the shared expert at slot k). Rows are taken in "row order":
// the shared expert's rows first, then the routed slots, i ascending; CTA c owns
// rows [c R, (c + 1) R) of that order (R a multiple of 32), one or two
// contiguous runs of (gate row i, up row i) pairs in the weight records.
//
// One warp per row pair at a time: each lane issues all of its 128-bit loads of
// both rows (half-groups l, l + 32, ...) before it computes, so that HBM sees
// many independent requests (a burst of plain loads reaches the copy roofline;
// bulk copies through shared memory do not, for bursts this short, and bulk L2
// prefetches of the next pairs measured slower than none). The codes are multiplied with
// the 16-bit fixed-point activations by dp4a. The CTA ends by quantising its
// SwiGLU outputs into the down kernel's staged form, which the down kernel
// copies as it is.

constexpr int kGuThreads = 256;
constexpr int kGuWarps = kGuThreads / 32;

// The q16 SwiGLU output block (global, and the down kernel's shared-memory
// copy of it) for ns slots in row order: runs hq[ns][4][I/32] (uint4), then the
// inverse scales inv[ns][I/32], then the half-group sums X[ns][I/32].
__host__ __device__ inline size_t hq_block_bytes(int ns, int I) { return (size_t)ns * I * 2 + (size_t)ns * (I / 32) * 8; }

// expert (record index) of row-order slot jj
__device__ __forceinline__ int row_slot_expert(int jj, int k, int E, int n_shared, const int32_t* s_ids) {
    const int j = n_shared ? (jj == 0 ? k : jj - 1) : jj;
    if (j == k) return E;
    const int e = s_ids[j];
    return ((unsigned)e < (unsigned)E) ? e : 0;   // a valid selection never needs the clamp
}

// 16 two-bit codes of one kernel-layout word (two runs of 8: one code per byte
// in each of (w >> 2f) & 0x03030303) against the staged runs xa, xb.
__device__ __forceinline__ void word2_dp4a(uint32_t w, const uint4 xa, const uint4 xb, int& ah, int& al) {
    const uint32_t ea = w & 0x03030303u, oa = (w >> 2) & 0x03030303u;
    const uint32_t eb = (w >> 4) & 0x03030303u, ob = (w >> 6) & 0x03030303u;
    ah = __dp4a((int)ea, (int)xa.x, ah);
    ah = __dp4a((int)oa, (int)xa.y, ah);
    al = __dp4a((int)ea, (int)xa.z, al);
    al = __dp4a((int)oa, (int)xa.w, al);
    ah = __dp4a((int)eb, (int)xb.x, ah);
    ah = __dp4a((int)ob, (int)xb.y, ah);
    al = __dp4a((int)eb, (int)xb.z, al);
    al = __dp4a((int)ob, (int)xb.w, al);
}

// One 64-code group of 2-bit codes (16 bytes: words 0-1 are half-group 2G,
// words 2-3 half-group 2G + 1) against the staged activations: the group's
// contribution s * (D_0 + D_1) + b * (X_0 + X_1).
__device__ __forceinline__ float group2_dot(const uint4 c, uint32_t meta, const uint4* xq, int HG, int G,
                                            const float* Iv, const float* Xx, float acc) {
    int h0 = 0, l0 = 0, h1 = 0, l1 = 0;
    const int a = 2 * G, b = 2 * G + 1;
    word2_dp4a(c.x, xq[0 * HG + a], xq[1 * HG + a], h0, l0);
    word2_dp4a(c.y, xq[2 * HG + a], xq[3 * HG + a], h0, l0);
    word2_dp4a(c.z, xq[0 * HG + b], xq[1 * HG + b], h1, l1);
    word2_dp4a(c.w, xq[2 * HG + b], xq[3 * HG + b], h1, l1);
    const float2 sb = meta_to_f2(meta);
    const float d = (float)(h0 * 256 + l0) * Iv[a] + (float)(h1 * 256 + l1) * Iv[b];
    return fmaf(sb.x, d, fmaf(sb.y, Xx[a] + Xx[b], acc));
}

// The same for a gate row and an up row at once, sharing the staged activations.
__device__ __forceinline__ void group2_dot_gu(const uint4 cg, const uint4 cu, uint32_t mg, uint32_t mu,
                                              const uint4* xq, int HG, int G, const float* Iv, const float* Xx,
                                              float& acc_g, float& acc_u) {
    int gh0 = 0, gl0 = 0, gh1 = 0, gl1 = 0, uh0 = 0, ul0 = 0, uh1 = 0, ul1 = 0;
    const int a = 2 * G, b = 2 * G + 1;
    {
        const uint4 x0 = xq[0 * HG + a], x1 = xq[1 * HG + a], x2 = xq[2 * HG + a], x3 = xq[3 * HG + a];
        word2_dp4a(cg.x, x0, x1, gh0, gl0);
        word2_dp4a(cg.y, x2, x3, gh0, gl0);
        word2_dp4a(cu.x, x0, x1, uh0, ul0);
        word2_dp4a(cu.y, x2, x3, uh0, ul0);
    }
    {
        const uint4 x0 = xq[0 * HG + b], x1 = xq[1 * HG + b], x2 = xq[2 * HG + b], x3 = xq[3 * HG + b];
        word2_dp4a(cg.z, x0, x1, gh1, gl1);
        word2_dp4a(cg.w, x2, x3, gh1, gl1);
        word2_dp4a(cu.z, x0, x1, uh1, ul1);
        word2_dp4a(cu.w, x2, x3, uh1, ul1);
    }
    const float ia = Iv[a], ib = Iv[b], xs = Xx[a] + Xx[b];
    const float2 sg = meta_to_f2(mg), su = meta_to_f2(mu);
    acc_g = fmaf(sg.x, (float)(gh0 * 256 + gl0) * ia + (float)(gh1 * 256 + gl1) * ib, fmaf(sg.y, xs, acc_g));
    acc_u = fmaf(su.x, (float)(uh0 * 256 + ul0) * ia + (float)(uh1 * 256 + ul1) * ib, fmaf(su.y, xs, acc_u));
}

template <int BITS, int NQ = 1>
__global__ void __launch_bounds__(kGuThreads, 2) k_gateup(const uint8_t* const* __restrict__ rec_tab,
                                                         const float* __restrict__ part, int splits,
                                                         const float* __restrict__ bias, int k, int E, int n_shared,
                                                         const void* __restrict__ x, int x_bf16, int H, int I,
                                                         size_t rbH, int R, void* __restrict__ hout, int copies,
                                                         int32_t* __restrict__ ids_out, float* __restrict__ wts_out,
                                                         float* __restrict__ logits_out,
                                                         const int32_t* __restrict__ sel_ids, int jj0, int jj1,
                                                         RouteMode mode, const uint8_t* pf, size_t pf_bytes,
                                                         unsigned long long* __restrict__ tr) {
    extern __shared__ uint4 smq[];
    __shared__ float s_logit[1024];
    __shared__ float s_score[1024];
    __shared__ int32_t s_ids[MOE_MAX_TOP_K];
    __shared__ float s_wts[MOE_MAX_TOP_K];
    const int HG = H / 32, IG = I / 32, ns = k + n_shared;
    uint4* xq = smq;                                                   // [4][HG]
    float* Iv = reinterpret_cast<float*>(smq + 4 * HG);                // [HG] 2^-f
    float* Xx = Iv + HG;                                               // [HG]
    float* hbuf = Xx + HG;                                             // [R]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ktrace(tr, blockIdx.x, 0);
    if (pf && threadIdx.x == 0) {
        // the next layer's router weights into L2 (moe_layer_set_next): this
        // CTA's share, in 16-byte multiples, no later than 64 KB a request
        const size_t per = (pf_bytes / gridDim.x + 15) / 16 * 16;
        const size_t b0 = per * blockIdx.x, b1 = min(pf_bytes, b0 + per);
        for (size_t o = b0; o < b1; o += 65536)
            prefetch_l2(pf + o, (uint32_t)min((size_t)65536, b1 - o));
    }
    stage_vector_q16(x, x_bf16, false, H, xq, Iv, Xx);
    __syncthreads();
    ktrace(tr, blockIdx.x, 2);

    // no weight traffic before the selection is known
    pdl_wait();
    pdl_trigger();
    ktrace(tr, blockIdx.x, 1);
    if (sel_ids) {
        // the selection was made earlier (streamed layers: the host staged
        // those experts first)
        if (threadIdx.x < k) s_ids[threadIdx.x] = sel_ids[threadIdx.x];
        __syncthreads();
        // streamed layers: a launch made before the host has staged this
        // token's experts finds a missing expert's record null and does
        // nothing (the host launches again once every expert is resident)
        __shared__ int s_skip;
        if (threadIdx.x == 0) {
            int bad = 0;
            for (int jj = jj0; jj < jj1; ++jj) bad |= rec_tab[row_slot_expert(jj, k, E, n_shared, s_ids)] == nullptr;
            s_skip = bad;
        }
        __syncthreads();
        if (s_skip) return;
    } else {
        // every CTA reduces the router's partial logits and selects (same result
        // everywhere); no CTA has to wait for a single selecting CTA
        block_select(part, splits, E, bias, k, s_logit, s_ids, s_wts, mode, s_score);
        if (blockIdx.x == 0) {   // publish the selection (read by the host and by later calls)
            for (int e = threadIdx.x; e < E; e += blockDim.x) logits_out[e] = s_logit[e];
            if (threadIdx.x < k) { ids_out[threadIdx.x] = s_ids[threadIdx.x]; wts_out[threadIdx.x] = s_wts[threadIdx.x]; }
        }
    }

    const int NR = (jj1 - jj0) * I;
    const int rbeg = blockIdx.x * R;
    const int np = max(0, min(R, NR - rbeg));   // row pairs of this CTA
    const uint64_t pol = policy_evict_first();
    auto pair_ptr = [&](int p) {
        const int r = jj0 * I + rbeg + p;
        const int jj = r / I, i = r - jj * I;
        return rec_tab[row_slot_expert(jj, k, E, n_shared, s_ids)] + (size_t)2 * i * rbH;
    };
    if constexpr (BITS == 2) {
        // a lane takes whole groups of 64 codes (16 bytes each); a warp works
        // on two row pairs at a time, so that it keeps as many bytes in flight
        // as with 4-bit codes
        constexpr int B2 = kGuBlock / 2;
        const int GH = HG / 2, M2 = (GH + 31) / 32;
        for (int p0 = warp; p0 < np; p0 += 2 * kGuWarps) {
            const uint8_t* g[2];
            bool live[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int p = p0 + q * kGuWarps;
                live[q] = p < np;
                g[q] = pair_ptr(live[q] ? p : p0);
            }
            float acc_g[2] = {0.f, 0.f}, acc_u[2] = {0.f, 0.f};
            for (int m0 = 0; m0 < M2; m0 += B2) {
                uint4 cg[2][B2], cu[2][B2];
                uint32_t mg[2][B2], mu[2][B2];
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int mm = 0; mm < B2; ++mm) {
                        const int G = lane + 32 * (m0 + mm);
                        if (live[q] && m0 + mm < M2 && G < GH) {
                            cg[q][mm] = ldg_stream_hint(g[q] + 16 * G, pol);
                            cu[q][mm] = ldg_stream_hint(g[q] + rbH + 16 * G, pol);
                            mg[q][mm] = ldg_u32_hint(g[q] + H / 4 + 4 * G, pol);
                            mu[q][mm] = ldg_u32_hint(g[q] + rbH + H / 4 + 4 * G, pol);
                        }
                    }
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int mm = 0; mm < B2; ++mm) {
                        const int G = lane + 32 * (m0 + mm);
                        if (live[q] && m0 + mm < M2 && G < GH)
                            group2_dot_gu(cg[q][mm], cu[q][mm], mg[q][mm], mu[q][mm], xq, HG, G, Iv, Xx, acc_g[q],
                                          acc_u[q]);
                    }
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float gv = warp_sum(acc_g[q]);
                const float uv = warp_sum(acc_u[q]);
                if (live[q] && lane == 0) hbuf[p0 + q * kGuWarps] = silu_f(gv) * uv;
            }
        }
    } else {
        // 4-bit codes. A warp works on NQ row pairs at a time, and each lane
        // issues all loads of its kGuBlock / NQ half-groups of every row
        // before it computes. Short rows (at most kGuBlock / 2 half-groups
        // per lane) take two pairs at a time (NQ = 2), so that as many bytes
        // are in flight per warp as with long rows.
        {
            constexpr int BQ = kGuBlock / NQ;
            const int M = (HG + 31) / 32;
            for (int p0 = warp; p0 < np; p0 += NQ * kGuWarps) {
                const uint8_t* g[NQ];
                bool live[NQ];
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int p = p0 + q * kGuWarps;
                    live[q] = p < np;
                    g[q] = pair_ptr(live[q] ? p : p0);
                }
                float acc_g[NQ], acc_u[NQ];
#pragma unroll
                for (int q = 0; q < NQ; ++q) acc_g[q] = acc_u[q] = 0.f;
                for (int m0 = 0; m0 < M; m0 += BQ) {
                    uint4 cg[NQ][BQ], cu[NQ][BQ];
                    uint32_t mg[NQ][BQ], mu[NQ][BQ];
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
#pragma unroll
                        for (int mm = 0; mm < BQ; ++mm) {
                            const int hg = lane + 32 * (m0 + mm);
                            if (live[q] && m0 + mm < M && hg < HG) {
                                const uint8_t* u = g[q] + rbH;
                                cg[q][mm] = ldg_stream_hint(g[q] + 16 * hg, pol);
                                cu[q][mm] = ldg_stream_hint(u + 16 * hg, pol);
                                mg[q][mm] = ldg_u32_hint(g[q] + H / 2 + 4 * (hg >> 1), pol);
                                mu[q][mm] = ldg_u32_hint(u + H / 2 + 4 * (hg >> 1), pol);
                            }
                        }
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
#pragma unroll
                        for (int mm = 0; mm < BQ; ++mm) {
                            const int hg = lane + 32 * (m0 + mm);
                            if (live[q] && m0 + mm < M && hg < HG) {
                                int gh = 0, gl = 0, uh = 0, ul = 0;
#pragma unroll
                                for (int wi = 0; wi < 4; ++wi) {
                                    const uint4 xs = xq[wi * HG + hg];
                                    word_dp4a(u4w(cg[q][mm], wi), xs, gh, gl);
                                    word_dp4a(u4w(cu[q][mm], wi), xs, uh, ul);
                                }
                                const float iv = Iv[hg], xs = Xx[hg];
                                const float2 sg = meta_to_f2(mg[q][mm]), su = meta_to_f2(mu[q][mm]);
                                acc_g[q] = fmaf(sg.x, (float)(gh * 256 + gl) * iv, fmaf(sg.y, xs, acc_g[q]));
                                acc_u[q] = fmaf(su.x, (float)(uh * 256 + ul) * iv, fmaf(su.y, xs, acc_u[q]));
                            }
                        }
                }
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const float gv = warp_sum(acc_g[q]);
                    const float uv = warp_sum(acc_u[q]);
                    if (live[q] && lane == 0) hbuf[p0 + q * kGuWarps] = silu_f(gv) * uv;
                }
            }
        }
    }   // BITS == 4
    __syncthreads();
    ktrace(tr, blockIdx.x, 3);
    // the CTA's SwiGLU outputs in the down kernel's staged form; a half-group
    // (32 rows) never straddles CTAs or slots
    // (written `copies` times: the down kernel's CTAs all read the whole block,
    // and spreading them over several copies spreads the reads over L2)
    const int nrun = np / 8;
    const size_t blk = hq_block_bytes(ns, I);
    for (int rb = warp * 32; rb < ((nrun + 31) / 32) * 32; rb += blockDim.x) {
        const int rr = rb + lane;
        const bool valid = rr < nrun;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = valid ? hbuf[8 * rr + i] : 0.f;
        const int r0 = jj0 * I + rbeg + 8 * (valid ? rr : 0);
        const int jj = r0 / I, run = (r0 - jj * I) / 8;
        // quantise once (the run, its half-group's scale and sum) ...
        float m = 0.f, sum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) { m = fmaxf(m, fabsf(v[i])); sum += v[i]; }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        const float sc = q16_scale(m);
        const uint4 qv = quant_run(v, sc);
        // ... and store it into every replica
        if (valid) {
            const int hg = run >> 2, wi = run & 3;
            for (int c = 0; c < copies; ++c) {
                uint8_t* base = static_cast<uint8_t*>(hout) + (size_t)c * blk;
                uint4* hq = reinterpret_cast<uint4*>(base);
                float* hinv = reinterpret_cast<float*>(hq + (size_t)ns * 4 * IG);
                float* hX = hinv + ns * IG;
                hq[(size_t)jj * 4 * IG + wi * IG + hg] = qv;
                if (wi == 0) { hinv[jj * IG + hg] = 1.0f / sc; hX[jj * IG + hg] = sum; }
            }
        }
    }
    // the down kernel reads the block with a bulk copy (the async proxy)
    asm volatile("fence.proxy.async.global;" ::: "memory");
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
template <int BITS, int J = 1>
__global__ void __launch_bounds__(kThreads) k_down(const uint8_t* const* __restrict__ rec_tab,
                                                   const float* __restrict__ part, int splits,
                                                   const float* __restrict__ bias,
                                                   int k, int E, int n_shared, int H, int I,
                                                   const void* __restrict__ hblk, int copies, void* __restrict__ y,
                                                   int y_bf16,
                                                   float* __restrict__ y32, size_t rbI, size_t gu_block,
                                                   const int32_t* __restrict__ sel_ids,
                                                   const float* __restrict__ sel_wts, unsigned* __restrict__ err,
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
    __shared__ __align__(8) uint64_t s_hbar;
    __shared__ int s_abort, s_skip;
    if (threadIdx.x == 0) {
        bw::mbar_init(bw::saddr(&s_hbar), 1);
        s_abort = 0;
        s_skip = 0;
        bw::mbar_fence_init();
    }
    __shared__ int32_t s_ids[MOE_MAX_TOP_K];
    __shared__ float s_wts[MOE_MAX_TOP_K];
    // whole quads of rows per CTA (a partial quad costs a full work item)
    const int nquads_all = (H + kDownRows - 1) / kDownRows;
    const int own0 = kDownRows * (int)((long long)nquads_all * blockIdx.x / gridDim.x);
    const int own1 = min(H, kDownRows * (int)((long long)nquads_all * (blockIdx.x + 1) / gridDim.x));
    pdl_wait();     // gate/up complete: the selection it published and the staged SwiGLU outputs are final
    pdl_trigger();  // the next token's router may start prefetching its weights
    ktrace(tr, blockIdx.x, 1);
    // every slot's SwiGLU outputs, already in the staged form gate/up wrote:
    // one bulk copy into shared memory, in flight while the selection is read
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)hq_block_bytes(ns, I);
        bw::mbar_arrive_tx(bw::saddr(&s_hbar), bytes);
        const uint8_t* src = static_cast<const uint8_t*>(hblk) + (size_t)(blockIdx.x % copies) * bytes;
        bw::bulk_load(bw::saddr(smh), src, bytes, bw::saddr(&s_hbar), policy_evict_first());
    }
    if (threadIdx.x < k) {   // the selection (gate/up's CTA 0 published it; streamed layers pass their own)
        s_ids[threadIdx.x] = sel_ids[threadIdx.x];
        s_wts[threadIdx.x] = sel_wts[threadIdx.x];
    }
    __syncthreads();
    if (threadIdx.x < ns) {
        const int s = threadIdx.x;
        const bool sh = n_shared && s == 0;
        const int j = sh ? k : s - n_shared;
        int e = sh ? E : s_ids[j];
        if ((unsigned)e > (unsigned)E) e = 0;
        const uint8_t* rec = rec_tab[e];
        if (!rec) s_skip = 1;   // streamed layer, expert not resident yet: see below
        s_rows[s] = rec + gu_block;
        s_w[s] = sh ? 1.0f : s_wts[j];
    }
    bw::mbar_wait(bw::saddr(&s_hbar), 0, &s_abort, err, 1u << 27);
    __syncthreads();
    // a launch made before the host staged this token's experts (streamed
    // layers) does nothing once the staged copy has landed; the host launches
    // again when every expert is resident
    if (s_skip) return;
    ktrace(tr, blockIdx.x, 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int own = own1 - own0;
    const int nquad = (own + kDownRows - 1) / kDownRows;
    const int M = (IG + 31) / 32;
    if constexpr (BITS == 2) {
        // a lane takes whole groups of 64 codes (16 bytes each); a warp works
        // on two items at a time, so that it keeps as many bytes in flight as
        // with 4-bit codes
        const int GI = IG / 2, nit = nquad * ns;
        for (int it0 = warp; it0 < nit; it0 += 2 * kWarps) {
            const uint8_t* rr[2][kDownRows];
            int s2[2], n0s[2], nrs[2];
            bool live[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int it = it0 + j * kWarps;
                live[j] = it < nit;
                const int itv = live[j] ? it : it0;
                const int q = itv / ns;
                s2[j] = itv - q * ns;
                n0s[j] = own0 + q * kDownRows;
                nrs[j] = min(kDownRows, own1 - n0s[j]);
#pragma unroll
                for (int r = 0; r < kDownRows; ++r) rr[j][r] = s_rows[s2[j]] + (size_t)(n0s[j] + min(r, nrs[j] - 1)) * rbI;
            }
            float acc[2][kDownRows];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int r = 0; r < kDownRows; ++r) acc[j][r] = 0.f;
            for (int G = lane; G < GI; G += 32) {
                uint4 c[2][kDownRows];
                uint32_t mt[2][kDownRows];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r)
                        if (live[j]) {
                            c[j][r] = ldg_stream(rr[j][r] + 16 * G);
                            mt[j][r] = ldg_u32(rr[j][r] + I / 4 + 4 * G);
                        }
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (live[j]) {
                        const uint4* xs = hq + (size_t)s2[j] * 4 * IG;
#pragma unroll
                        for (int r = 0; r < kDownRows; ++r)
                            acc[j][r] = group2_dot(c[j][r], mt[j][r], xs, IG, G, Iv + s2[j] * IG, Xh + s2[j] * IG,
                                                   acc[j][r]);
                    }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float d[kDownRows];
#pragma unroll
                for (int r = 0; r < kDownRows; ++r) d[r] = warp_sum(acc[j][r]);
#pragma unroll
                for (int r = 0; r < kDownRows; ++r)
                    if (live[j] && lane == r && r < nrs[j]) ypart[s2[j] * kDownMaxRows + (n0s[j] - own0) + r] = d[r];
            }
        }
    } else {
        // 4-bit codes. A warp works on J items at a time, and each lane issues
        // the loads of MB half-groups of every row of them before it computes.
        // Short rows (one half-group per lane) take two items at a time
        // (J = 2), so that as many bytes are in flight per warp as with long
        // rows.
        {
            constexpr int MB = 2 / J;
            const int nit = nquad * ns;
            for (int it0 = warp; it0 < nit; it0 += J * kWarps) {
                const uint8_t* rr[J][kDownRows];
                int s2[J], n0s[J], nrs[J];
                bool live[J];
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int it = it0 + j * kWarps;
                    live[j] = it < nit;
                    const int itv = live[j] ? it : it0;
                    const int q = itv / ns;
                    s2[j] = itv - q * ns;
                    n0s[j] = own0 + q * kDownRows;
                    nrs[j] = min(kDownRows, own1 - n0s[j]);
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r)
                        rr[j][r] = s_rows[s2[j]] + (size_t)(n0s[j] + min(r, nrs[j] - 1)) * rbI;
                }
                float acc[J][kDownRows];
#pragma unroll
                for (int j = 0; j < J; ++j)
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r) acc[j][r] = 0.f;
                for (int m = 0; m < M; m += MB) {
                    uint4 c[J][MB][kDownRows];
                    uint32_t mt[J][MB][kDownRows];
#pragma unroll
                    for (int j = 0; j < J; ++j)
#pragma unroll
                        for (int mm = 0; mm < MB; ++mm) {
                            const int hg = lane + 32 * (m + mm);
#pragma unroll
                            for (int r = 0; r < kDownRows; ++r)
                                if (live[j] && m + mm < M && hg < IG) {
                                    c[j][mm][r] = ldg_stream(rr[j][r] + 16 * hg);
                                    mt[j][mm][r] = ldg_u32(rr[j][r] + I / 2 + 4 * (hg >> 1));
                                }
                        }
#pragma unroll
                    for (int j = 0; j < J; ++j)
#pragma unroll
                        for (int mm = 0; mm < MB; ++mm) {
                            const int hg = lane + 32 * (m + mm);
                            if (live[j] && m + mm < M && hg < IG) {
                                const uint4* xs = hq + (size_t)s2[j] * 4 * IG;
                                int ah[kDownRows], al[kDownRows];
#pragma unroll
                                for (int r = 0; r < kDownRows; ++r) ah[r] = al[r] = 0;
#pragma unroll
                                for (int wi = 0; wi < 4; ++wi) {
                                    const uint4 xv = xs[wi * IG + hg];
#pragma unroll
                                    for (int r = 0; r < kDownRows; ++r)
                                        word_dp4a(u4w(c[j][mm][r], wi), xv, ah[r], al[r]);
                                }
                                const float iv = Iv[s2[j] * IG + hg], xx = Xh[s2[j] * IG + hg];
#pragma unroll
                                for (int r = 0; r < kDownRows; ++r) {
                                    const float2 sb = meta_to_f2(mt[j][mm][r]);
                                    acc[j][r] = fmaf(sb.x, (float)(ah[r] * 256 + al[r]) * iv, fmaf(sb.y, xx, acc[j][r]));
                                }
                            }
                        }
                }
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    float d[kDownRows];
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r) d[r] = warp_sum(acc[j][r]);
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r)
                        if (live[j] && lane == r && r < nrs[j]) ypart[s2[j] * kDownMaxRows + (n0s[j] - own0) + r] = d[r];
                }
            }
        }
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

static int round32(int v) { return (v + 31) / 32 * 32; }
// rows one gate/up CTA owns for NR rows: a multiple of 32, spread over every resident CTA
static int gu_rows(const Layer& L, int NR) {
    return std::max(32, round32((NR + L.num_sms * L.occ_gu - 1) / (L.num_sms * L.occ_gu)));
}
static size_t gu_smem_for(const Layer& L, int R) {
    const int H = L.d.hidden;
    return (size_t)H * 2 + (size_t)(H / 32) * 8 + (size_t)R * 4;
}
static size_t down_smem(int I, int ns) {
    return (size_t)ns * I * 2 + (size_t)ns * (I / 32) * 8 + (size_t)ns * kDownMaxRows * 4;
}
static int down_grid(const Layer& L) { return L.num_sms * L.occ_down; }

using GuKernel = decltype(&k_gateup<4, 1>);
using DownKernel = decltype(&k_down<4, 1>);
// 4-bit rows of at most kGuBlock / 2 half-groups per lane (H <= 3072): two
// row pairs per warp at a time; down rows of one half-group per lane
// (I <= 1024): two items per warp at a time
static GuKernel gu_kernel(const Layer& L) {
    if (L.wbits == 2) return k_gateup<2, 1>;
    return (L.d.hidden / 32 + 31) / 32 <= kGuBlock / 2 ? k_gateup<4, 2> : k_gateup<4, 1>;
}
static DownKernel down_kernel(const Layer& L) {
    if (L.wbits == 2) return k_down<2, 1>;
    return (L.d.inter / 32 + 31) / 32 == 1 ? k_down<4, 2> : k_down<4, 1>;
}

cudaError_t decode_kernel_setup(Layer& L) {
    const int H = L.d.hidden, I = L.d.inter, ns = L.d.top_k + L.d.n_shared;
    cudaError_t e = router_kernel_setup(L);
    if (e != cudaSuccess) return e;
    const int R1 = round32((ns * I + L.num_sms - 1) / L.num_sms);   // rows per CTA at one CTA per SM (upper bound)
    L.gu_smem = gu_smem_for(L, R1);
    const void* gu = (const void*)gu_kernel(L);
    const void* dn = (const void*)down_kernel(L);
    e = cudaFuncSetAttribute(gu, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.gu_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)down_smem(I, ns));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_gu, gu, kGuThreads, L.gu_smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_down, dn, kThreads, down_smem(I, ns));
    if (e != cudaSuccess) return e;
    if (L.occ_gu < 1 || L.occ_down < 1) return cudaErrorInvalidConfiguration;
    // rows owned by one down CTA must fit its partial-sum buffer
    while (kDownRows * (((H + kDownRows - 1) / kDownRows + down_grid(L) - 1) / down_grid(L)) > kDownMaxRows) {
        if (L.occ_down >= 64) return cudaErrorInvalidConfiguration;
        ++L.occ_down;   // more (smaller) CTAs per SM are launched in waves
    }
    return cudaSuccess;
}

// gate/up over row-order slots jj0..jj1-1 (sel_ids null: select from `part`)
static cudaError_t launch_gateup(Layer& L, const void* x, const float* part, void* hblk, int copies, int32_t* ids_out,
                                 float* wts_out, float* logits_out, const int32_t* sel_ids, int jj0, int jj1,
                                 bool pdl, unsigned long long* tr, cudaStream_t s) {
    const auto& d = L.d;
    const int NR = (jj1 - jj0) * d.inter;
    const int R = gu_rows(L, NR);
    const int grid = (NR + R - 1) / R;
    return launch_pdl(gu_kernel(L), dim3(grid), dim3(kGuThreads), gu_smem_for(L, R), s,
                      pdl, (const uint8_t* const*)L.rec_table, part, L.router_splits, (const float*)L.router_bias,
                      d.top_k, d.n_experts, d.n_shared, x, d.act_dtype == MOE_BF16 ? 1 : 0, d.hidden, d.inter,
                      row_bytes(d.hidden, L.wbits), R, hblk, copies, ids_out, wts_out, logits_out, sel_ids, jj0, jj1,
                      L.route_mode(), (const uint8_t*)L.next_router, L.next_router_bytes, tr);
}

static cudaError_t launch_down(Layer& L, const float* part, const void* hblk, int copies, void* y, float* y_f32,
                               const int32_t* sel_ids, const float* sel_wts, bool pdl, unsigned long long* tr,
                               cudaStream_t s) {
    const auto& d = L.d;
    const int ns = d.top_k + d.n_shared;
    return launch_pdl(down_kernel(L), dim3(down_grid(L)), dim3(kThreads),
                      down_smem(d.inter, ns), s, pdl, (const uint8_t* const*)L.rec_table, part, L.router_splits,
                      (const float*)L.router_bias, d.top_k, d.n_experts, d.n_shared, d.hidden, d.inter, hblk, copies,
                      y, d.act_dtype == MOE_BF16 ? 1 : 0, y_f32, row_bytes(d.inter, L.wbits),
                      gu_block_bytes(d.hidden, d.inter, L.wbits), sel_ids, sel_wts, fused_error_word(L), tr);
}

cudaError_t launch_experts_decode(Layer& L, const void* x, void* y, float* y_f32, int which, cudaStream_t s) {
    const int ns = L.d.top_k + L.d.n_shared;
    cudaError_t e;
    if (which & (RUN_ROUTED_GU | RUN_SHARED_GU)) {
        prof_begin(L, K_GATEUP_DECODE, s);
        e = launch_gateup(L, x, L.logits_part, L.h, L.h_copies, L.ids, L.wts, L.logits, nullptr, 0, ns, L.pdl,
                          L.split_trace(1), s);
        prof_end(L, s);
        if (e != cudaSuccess) return e;
    }
    if (which & RUN_DOWN) {
        prof_begin(L, K_DOWN_DECODE, s);
        e = launch_down(L, L.logits_part, L.h, L.h_copies, y, y_f32, L.ids, L.wts, L.pdl, L.split_trace(2), s);
        prof_end(L, s);
        return e;
    }
    return cudaSuccess;
}

// The same two expert kernels over caller-given scratch: router partials
// `part` [splits][E] (already written on `s`), selection out (`logits` [E],
// `ids` [k], `wts` [k]) and the staged SwiGLU outputs `h` (at least
// hq_block_bytes(k + n_shared, I) bytes). No profiling or tracing.
cudaError_t launch_experts_decode_scratch(Layer& L, const void* x, void* y, float* y_f32, const float* part,
                                          float* logits, int32_t* ids, float* wts, float* h, cudaStream_t s) {
    const int ns = L.d.top_k + L.d.n_shared;
    cudaError_t e = launch_gateup(L, x, part, h, 1, ids, wts, logits, nullptr, 0, ns, L.pdl, nullptr, s);
    if (e != cudaSuccess) return e;
    return launch_down(L, part, h, 1, y, y_f32, ids, wts, L.pdl, nullptr, s);
}

// Streamed layers: the selection (ids, wts of one token) is already on the
// device and the routed experts' records are resident. `jj0..jj1` are the
// row-order slots of gate/up to run (0 = the shared expert when there is one);
// `down` adds the down + combine kernel. Plain launches (no programmatic
// overlap): the caller orders them against the cache's copies with events.
cudaError_t launch_experts_decode_sel(Layer& L, const void* x, void* y, float* y_f32, const int32_t* ids,
                                      const float* wts, int jj0, int jj1, bool down, cudaStream_t s, bool pdl) {
    cudaError_t e = cudaSuccess;
    if (jj1 > jj0) {
        prof_begin(L, K_GATEUP_DECODE, s);
        e = launch_gateup(L, x, nullptr, L.h, L.h_copies, nullptr, nullptr, nullptr, ids, jj0, jj1, pdl && L.pdl,
                          nullptr, s);
        prof_end(L, s);
        if (e != cudaSuccess) return e;
    }
    if (down) {
        prof_begin(L, K_DOWN_DECODE, s);
        e = launch_down(L, nullptr, L.h, L.h_copies, y, y_f32, ids, wts, pdl && L.pdl, nullptr, s);
        prof_end(L, s);
    }
    return e;
}

}  // namespace moe
