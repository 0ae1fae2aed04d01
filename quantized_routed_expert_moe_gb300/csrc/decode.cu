// Three-kernel decode, expert part: gate/up dequant-GEMV with SwiGLU, then
// down dequant-GEMV with the weighted combine.
//
// The kernels are chained with programmatic dependent launch (PDL):
//   router   -- the token's logits and, in its last block, the top-k selection
//               and routing weights (router.cu), then a ready flag;
//   gate/up  -- starts while the router runs: stages the activations and
//               computes the shared expert's rows, which do not depend on the
//               routing, then counts the CTA as done with them; waits
//               (bounded) for the ready flag rather than for the router grid
//               to retire, then computes the routed experts' rows. Row pairs
//               are spread over every warp of the grid, one or two pairs per
//               warp at a time; each SwiGLU output is written (fp32) into
//               every replica of the output block with plain stores, so no
//               warp ever waits on another;
//   down     -- starts as gate/up CTAs retire: once every gate/up CTA has
//               counted its shared rows, quantises the shared expert's SwiGLU
//               outputs into shared memory and computes their output rows;
//               then waits for gate/up, quantises the routed experts' outputs
//               and computes their rows and the weighted combine.
// Each warp issues all of a row's weight loads (128-bit, streaming) before it
// computes. The 4-bit codes are multiplied with 16-bit fixed-point activations
// by integer dp4a (common.cuh).
//
// Scaling: the token's activations are staged as x * 2^a, with a chosen so that
// max |x| * 2^a lies in [1, 2). The dot products then come out times 2^a, the
// SwiGLU outputs times 2^2a, and the combine multiplies by 2^-2a: exact powers
// of two, so tokens of any magnitude keep fp32's relative precision
// throughout (no overflow of large activations, no flush of tiny ones).
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
// Down CTAs: a warp keeps one work item in flight at a time, so the bytes in
// flight per SM grow with its warps. 4-bit items of one slot per warp (J = 1)
// fit two 384-thread CTAs per SM (80 registers); the others need more
// registers and keep 256.
template <int BITS, int J>
constexpr int down_threads() { return BITS == 4 && J == 1 ? 384 : 256; }
constexpr int kGuBlock = 6;           // half-groups per lane whose loads are in flight together (gate/up)
constexpr int kDownRows = 4;          // output rows per down work item (share the staged activations)
constexpr int kDownMaxRows = 96;      // output rows one CTA owns in the down kernel
constexpr uint64_t kWaitNs = 200000000ull;   // bounded device waits: 0.2 s
constexpr int kHCopies = kDecodeHCopies;   // replicas of the staged SwiGLU outputs: the down CTAs' reads spread over L2

__device__ __forceinline__ void load_run(const void* x, int x_bf16, int r, float (&v)[8]) {
    if (x_bf16) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + r);
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w4[i] << 16);
            v[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(x) + 2 * r;
        const float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// max |x_i| over K activations, every thread of the block gets it (NaN ignored)
__device__ float block_absmax(const void* x, int x_bf16, int K, float* s_red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float m = 0.f;
    for (int r = threadIdx.x; r < K / 8; r += blockDim.x) {
        float v[8];
        load_run(x, x_bf16, r, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, s_red[w]);
    __syncthreads();
    return r;
}

// Stage K activations times xs (a power of two) into 16-bit fixed-point runs
// xq[4][K/32] with per-half-group inverse scale and sum. Block-wide,
// warp-uniform trip counts.
__device__ void stage_vector_q16(const void* x, int x_bf16, int K, float xs, uint4* xq, float* inv, float* X) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrun = K / 8, KG = K / 32;
    for (int rb = warp * 32; rb < ((nrun + 31) / 32) * 32; rb += blockDim.x) {
        const int r = rb + lane;
        const bool valid = r < nrun;
        float v[8];
        if (valid) {
            load_run(x, x_bf16, r, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= xs;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        stage_q16_run(v, valid, r, KG, xq, inv, X);
    }
}

// The token exponent a (max|x| 2^a in [1, 2)) and the staged runs of x 2^a, in
// one pass over x: warp w takes blocks of 32 runs w, w + warps, ... (as
// stage_vector_q16 does), keeps them in registers across the block-wide
// maximum and quantises them from there. Requires at most kMaxB blocks per
// warp.
template <int kMaxB>
__device__ int stage_token_q16(const void* x, int x_bf16, int K, float* s_red, uint4* xq, float* inv, float* X) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (int)(blockDim.x >> 5);
    const int nrun = K / 8, KG = K / 32, nblk = (nrun + 31) / 32;
    float v[kMaxB][8];
    float m = 0.f;
#pragma unroll
    for (int t = 0; t < kMaxB; ++t) {
        const int r = (warp + t * nw) * 32 + lane;
        if (r < nrun) {
            load_run(x, x_bf16, r, v[t]);
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[t][i]));
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[t][i] = 0.f;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float mx = 0.f;
    for (int w = 0; w < nw; ++w) mx = fmaxf(mx, s_red[w]);
    const int ta = token_exp(mx);
    const float xs = exp2i(ta);
#pragma unroll
    for (int t = 0; t < kMaxB; ++t) {
        const int b = warp + t * nw;
        if (b < nblk) {   // warp-uniform
            const int r = b * 32 + lane;
#pragma unroll
            for (int i = 0; i < 8; ++i) v[t][i] *= xs;
            stage_q16_run(v[t], r < nrun, r, KG, xq, inv, X);
        }
    }
    return ta;
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------
//
// h[j][i] = silu(gate_i . x) * (up_i . x) for row-order slot j: the shared
// expert first (when there is one), then the routed slots in selection order.
// The kernel writes h * 2^2a in fp32, [slot][I].

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

// Dot products of NQ row pairs (gate row at g[q], up row at g[q] + rbH) with
// the staged activations; every lane gets the warp sums gv[q], uv[q]. A lane
// issues all loads of its half-groups (4-bit: kGuBlock / NQ at a time; 2-bit:
// whole groups, kGuBlock / 2 at a time) of every row before it computes.
template <int BITS, int NQ>
__device__ __forceinline__ void pair_dots(const uint8_t* const (&g)[NQ], const bool (&live)[NQ], int H, size_t rbH,
                                          const uint4* xq, const float* Iv, const float* Xx, uint64_t pol,
                                          float (&gv)[NQ], float (&uv)[NQ]) {
    const int lane = threadIdx.x & 31, HG = H / 32;
    float acc_g[NQ], acc_u[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc_g[q] = acc_u[q] = 0.f;
    if constexpr (BITS == 2) {
        constexpr int B2 = kGuBlock / 2;
        const int GH = HG / 2, M2 = (GH + 31) / 32;
        for (int m0 = 0; m0 < M2; m0 += B2) {
            uint4 cg[NQ][B2], cu[NQ][B2];
            uint32_t mg[NQ][B2], mu[NQ][B2];
#pragma unroll
            for (int q = 0; q < NQ; ++q)
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
            for (int q = 0; q < NQ; ++q)
#pragma unroll
                for (int mm = 0; mm < B2; ++mm) {
                    const int G = lane + 32 * (m0 + mm);
                    if (live[q] && m0 + mm < M2 && G < GH)
                        group2_dot_gu(cg[q][mm], cu[q][mm], mg[q][mm], mu[q][mm], xq, HG, G, Iv, Xx, acc_g[q],
                                      acc_u[q]);
                }
        }
    } else {
        constexpr int BQ = kGuBlock / NQ;
        const int M = (HG + 31) / 32;
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
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        gv[q] = warp_sum(acc_g[q]);
        uv[q] = warp_sum(acc_u[q]);
    }
}

// Row pairs p0, p0 + step, ... (< pend) of one phase, NQ at a time; ptr(p)
// gives the gate row of pair p; done(p, g, u, live) is called by every lane
// with the (scaled) dot products of pair p.
template <int BITS, int NQ, typename PtrF, typename DoneF>
__device__ __forceinline__ void gu_phase(int p0, int step, int pend, PtrF ptr, DoneF done, int H, size_t rbH,
                                         const uint4* xq, const float* Iv, const float* Xx, uint64_t pol) {
    for (int p = p0; p < pend; p += NQ * step) {
        const uint8_t* g[NQ];
        bool live[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int pq = p + q * step;
            live[q] = pq < pend;
            g[q] = ptr(live[q] ? pq : p);
        }
        float gv[NQ], uv[NQ];
        pair_dots<BITS, NQ>(g, live, H, rbH, xq, Iv, Xx, pol, gv, uv);
#pragma unroll
        for (int q = 0; q < NQ; ++q) done(p + q * step, gv[q], uv[q], live[q]);
    }
}

// Wait until *ctr >= target (acquire), for at most limit_ns of GPU time.
__device__ __forceinline__ bool wait_count(const unsigned* ctr, unsigned target, uint64_t limit_ns) {
    const uint64_t t0 = bw::gtimer();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((i & 15) == 15 && bw::gtimer() - t0 > limit_ns) return false;
        __nanosleep(64);
    }
    return false;
}

// Poll the 64-bit word *p until its high half is `tag`, for at most limit_ns
// of GPU time; *out gets the last value read. False when the limit passed.
__device__ __forceinline__ bool poll_tagged(const unsigned long long* p, unsigned tag, uint64_t limit_ns,
                                            unsigned long long* out) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    const uint64_t t0 = bw::gtimer();
    for (uint32_t i = 0; (unsigned)(v >> 32) != tag; ++i) {
        if ((i & 15) == 15 && bw::gtimer() - t0 > limit_ns) {
            *out = v;
            return false;
        }
        __nanosleep(32);
        asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    }
    *out = v;
    return true;
}

__device__ __forceinline__ void st_tagged(unsigned long long* p, unsigned tag, uint32_t lo) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(((unsigned long long)tag << 32) | lo) : "memory");
}

// Words of shared memory the per-CTA selection uses: keys [E], then sigmoid
// scores [E] (the layout the router's selecting block uses).
__host__ __device__ inline int select_words(int E) { return 2 * E; }

// This token's selection, computed by the whole CTA from the router's tagged
// partial logits part_tag[splits][E]: each word is polled until it carries the
// token's tag (for at most limit_ns; then the router grid's completion is
// waited for instead and the error bit set), the splits are summed in order
// (the same arithmetic as the router's selecting block, so the selection is the
// same), and the top k are selected with their weights into ids_out / w_out
// (shared memory). Ends with the block synchronised.
__device__ void select_from_tagged(const unsigned long long* part_tag, unsigned tag, int splits, int E, int k,
                                   const float* bias, RouteMode mode, float* sm, int32_t* ids_out, float* w_out,
                                   unsigned* err) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        unsigned long long v[kMaxRouterSplits];
#pragma unroll
        for (int s = 0; s < kMaxRouterSplits; ++s)
            if (s < splits)
                asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v[s]) : "l"(part_tag + (size_t)s * E + e)
                             : "memory");
        const uint64_t t0 = bw::gtimer();
        bool late = false;
        for (uint32_t it = 0;; ++it) {
            bool all = true;
#pragma unroll
            for (int s = 0; s < kMaxRouterSplits; ++s)
                if (s < splits && (unsigned)(v[s] >> 32) != tag) {
                    all = false;
                    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v[s]) : "l"(part_tag + (size_t)s * E + e)
                                 : "memory");
                }
            if (all) break;
            if (late || ((it & 15) == 15 && bw::gtimer() - t0 > kWaitNs)) {
                if (late) break;   // read after the router's completion: take what is there
                late = true;
                atomicOr(err, 1u << 28);
                pdl_wait();        // the router grid is complete: its partials are all written
            }
            __nanosleep(32);
        }
        float l = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxRouterSplits; ++s)
            if (s < splits) l += __uint_as_float((uint32_t)v[s]);
        sm[e] = route_key(l, bias ? bias[e] : 0.f, mode, sm + E + e);
    }
    __syncthreads();
    block_topk(sm, E, k, ids_out, w_out, mode.sigmoid ? sm + E : nullptr, mode.scale);
}

struct GuArgs {
    const uint8_t* const* rec_tab;   // [E + 1] expert records (index E: the shared expert)
    int k, E, n_shared;
    const void* x;
    int x_bf16;
    int H, I;
    size_t rbH;                      // bytes of one gate/up row record
    const int32_t* ids;              // the token's selection [k] (the router's, or a streamed layer's)
    const unsigned* ids_ready;       // nullable: set by the router's selecting block once ids are written
    const unsigned long long* part_tag;   // nullable: tagged router partials; every CTA selects from them
    const unsigned* seq;             // with part_tag: the layer's decode count (the token's tag)
    int splits;                      // with part_tag: router K-splits
    const float* bias;               // with part_tag: router bias [E] or null
    RouteMode mode;
    int32_t* sel_ids;                // with part_tag: CTA 0 publishes the selection here (down reads it)
    float* sel_wts;
    unsigned long long* sel_tag;     // with part_tag: CTA 0 also publishes ids [k], weights [k] and the
                                     // token exponent as tagged words (the down kernel polls them)
    float* h;                        // copies x [ns][I] SwiGLU outputs times 2^2a, row-order slots
    int copies;                      // replicas of the output block (<= 32): the down CTAs' reads spread over L2
    int* scale_out;                  // the token exponent a (CTA 0 writes it)
    unsigned* shared_done;           // nullable: gate/up CTAs done with the shared expert's rows
    int jj0, jj1;                    // row-order slots this launch computes
    const uint8_t* pf;               // next layer's router weights to warm into L2 (nullable)
    size_t pf_bytes;
    unsigned* err;
    unsigned long long* tr;
    int stall_shared;                // test hook: do not count the CTAs done with the shared expert's rows
};

template <int BITS, int NQ>
__global__ void __launch_bounds__(kThreads, 2) k_gateup(const GuArgs a) {
    extern __shared__ uint4 smq[];
    __shared__ int32_t s_ids[MOE_MAX_TOP_K];
    __shared__ float s_wsel[MOE_MAX_TOP_K];
    __shared__ float s_red[kWarps];
    __shared__ int s_skip, s_ok;
    const int H = a.H, I = a.I, HG = H / 32, ns = a.k + a.n_shared;
    uint4* xq = smq;                                                   // [4][HG]
    float* Iv = reinterpret_cast<float*>(smq + 4 * HG);                // [HG] 2^-f
    float* Xx = Iv + HG;                                               // [HG]
    float* s_sel = Xx + HG;                                            // [select_words(E)] (part_tag only)
    // [E + 1] the record table (part_tag only: a resident layer's, fixed)
    const uint8_t** s_rtab = reinterpret_cast<const uint8_t**>(s_sel + select_words(a.E));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ktrace(a.tr, blockIdx.x, 0);
    // the token's tag, read before any wait (the previous token's down kernel,
    // which advanced the count, completed before the router started)
    const unsigned tag = a.part_tag ? decode_tag(__ldcg(a.seq)) : 0u;
    // a resident layer's record table into shared memory while the router
    // runs: the routed rows' addresses then need no load after the selection
    if (a.part_tag)
        for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_rtab[i] = a.rec_tab[i];
    const uint8_t* const* tab = a.part_tag ? s_rtab : a.rec_tab;
    if (a.pf && threadIdx.x == 0) {
        // the next layer's router weights into L2 (moe_layer_set_next): this
        // CTA's share, in 16-byte multiples, no more than 64 KB a request
        const size_t per = (a.pf_bytes / gridDim.x + 15) / 16 * 16;
        const size_t b0 = per * blockIdx.x, b1 = min(a.pf_bytes, b0 + per);
        for (size_t o = b0; o < b1; o += 65536) prefetch_l2(a.pf + o, (uint32_t)min((size_t)65536, b1 - o));
    }
    // this warp's shared-expert row pairs into L2 while x is staged (HBM is
    // idle then: the router reads its weights from L2), so that their loads
    // after the staging hit L2
    if (a.n_shared && a.jj0 == 0 && lane == 0) {
        const uint8_t* rec = a.rec_tab[a.E];
        for (int p = blockIdx.x * kWarps + warp; p < I; p += gridDim.x * kWarps)
            prefetch_l2(rec + (size_t)2 * p * a.rbH, (uint32_t)(2 * a.rbH));
    }
    // the token's scale and staged activations (the router waited for the
    // producer of x before this kernel could start, so x is final)
    int ta;
    if ((H / 8 + 31) / 32 <= 4 * kWarps) {   // H <= 8192: one pass over x
        ta = stage_token_q16<4>(a.x, a.x_bf16, H, s_red, xq, Iv, Xx);
    } else {
        ta = token_exp(block_absmax(a.x, a.x_bf16, H, s_red));
        stage_vector_q16(a.x, a.x_bf16, H, exp2i(ta), xq, Iv, Xx);
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.scale_out) *a.scale_out = ta;   // for the down kernel
    const float inv_a = exp2i(-ta);
    const uint64_t pol = policy_evict_first();
    const bool has_shared = a.n_shared && a.jj0 == 0;
    const int jr0 = has_shared ? 1 : a.jj0;   // first routed row-order slot
    const size_t blk = (size_t)ns * I;   // floats of one replica
    // pair (slot jj, row i) done: every lane holds the same warp sums, and lane
    // c < copies writes h * 2^2a = (g 2^a)(u 2^a) sigmoid(g) into replica c
    auto done = [&](int jj, int i, float gs, float us, bool live) {
        if (live && lane < a.copies) {
            const float sg = 1.0f / (1.0f + expf(-(gs * inv_a)));
            a.h[lane * blk + (size_t)jj * I + i] = gs * us * sg;
        }
    };
    // the shared expert's rows need no routing: they overlap the router
    if (has_shared) {
        const uint8_t* rec = tab[a.E];   // fixed for the layer's lifetime
        gu_phase<BITS, NQ>(
            blockIdx.x * kWarps + warp, gridDim.x * kWarps, I, [&](int p) { return rec + (size_t)2 * p * a.rbH; },
            [&](int p, float gs, float us, bool live) { done(0, p, gs, us, live); }, H, a.rbH, xq, Iv, Xx, pol);
    }
    ktrace(a.tr, blockIdx.x, 1);
    // this CTA's shared rows are written: count it for the down kernel's early
    // start (every writer fences its stores before the barrier)
    if (has_shared && a.shared_done) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0 && !a.stall_shared) atomicAdd(a.shared_done, 1u);
    }
    if (a.part_tag) {
        // the selection, computed here from the router's tagged partials as
        // soon as they are written (no wait for the router grid to retire)
        select_from_tagged(a.part_tag, tag, a.splits, a.E, a.k, a.bias, a.mode, s_sel, s_ids, s_wsel, a.err);
        if (blockIdx.x == 0 && threadIdx.x < a.k) {   // for the down kernel and moe_layer_selection
            a.sel_ids[threadIdx.x] = s_ids[threadIdx.x];
            a.sel_wts[threadIdx.x] = s_wsel[threadIdx.x];
            st_tagged(a.sel_tag + threadIdx.x, tag, (uint32_t)s_ids[threadIdx.x]);
            st_tagged(a.sel_tag + a.k + threadIdx.x, tag, __float_as_uint(s_wsel[threadIdx.x]));
            if (threadIdx.x == 0) st_tagged(a.sel_tag + 2 * a.k, tag, (uint32_t)ta);
        }
    } else {
        // the router's selecting block raises the ready flag as soon as the
        // ids are written; a wait that runs out falls back to the ordinary
        // dependency wait
        if (threadIdx.x == 0) {
            int ok = 0;
            if (a.ids_ready) {
                ok = wait_count(a.ids_ready, 1u, kWaitNs) ? 1 : 0;
                if (!ok) atomicOr(a.err, 1u << 28);
            }
            s_ok = ok;
        }
        __syncthreads();
        if (!s_ok) pdl_wait();   // the router (or, streamed, the staging of the records) is complete
        if (threadIdx.x < a.k) s_ids[threadIdx.x] = __ldcg(a.ids + threadIdx.x);
        __syncthreads();
    }
    pdl_trigger();   // the down kernel may launch: it starts with the shared expert's rows
    ktrace(a.tr, blockIdx.x, 2);
    if (a.jj1 > jr0) {
        // streamed layers: a launch made before the host has staged this
        // token's experts finds a missing expert's record null and does
        // nothing (the host launches again once every expert is resident); a
        // resident layer's records are never null
        if (!a.part_tag) {
            if (threadIdx.x == 0) {
                int bad = 0;
                for (int jj = jr0; jj < a.jj1; ++jj)
                    bad |= a.rec_tab[row_slot_expert(jj, a.k, a.E, a.n_shared, s_ids)] == nullptr;
                s_skip = bad;
            }
            __syncthreads();
        }
        if (a.part_tag || !s_skip)
            gu_phase<BITS, NQ>(
                blockIdx.x * kWarps + warp, gridDim.x * kWarps, (a.jj1 - jr0) * I,
                [&](int p) {
                    const int jj = jr0 + p / I, i = p - (p / I) * I;
                    return tab[row_slot_expert(jj, a.k, a.E, a.n_shared, s_ids)] + (size_t)2 * i * a.rbH;
                },
                [&](int p, float gs, float us, bool live) {
                    const int jj = jr0 + p / I;
                    done(jj, p - (jj - jr0) * I, gs, us, live);
                },
                H, a.rbH, xq, Iv, Xx, pol);
    }
    pdl_wait();   // this grid's completion then implies the router's (returns at once by now)
    ktrace(a.tr, blockIdx.x, 3);
}

// ---------------------------------------------------------------------------
// down + combine
// ---------------------------------------------------------------------------
//
// CTA c owns output rows [c*H/G, (c+1)*H/G). The staged SwiGLU outputs (16-bit
// fixed point per half-group, written by gate/up) are loaded once per CTA.
// Work items are (4 rows, slot); a warp computes the 4 rows' dot products with
// that slot's outputs, keeping the results per (slot, row); the rows are then
// combined in a fixed order: shared expert first (weight 1), then the routed
// slots in selection order, and scaled back by 2^-2a.

// Quantise slots [s0, s1) of the SwiGLU outputs src[ns][I] (fp32, written by
// the gate/up kernel, read through L2) into the staged form the dot products
// read: slot s at hq + 4 IG s, Iv + IG s, Xh + IG s. Block-wide: each warp takes
// blocks of 32 runs (8 half-groups) of a slot and issues the loads of
// kStageBatch blocks before it quantises them.
template <int kStageBatch>
__device__ __forceinline__ void stage_slots_q16(const float* src, int s0, int s1, int I, uint4* hq, float* Iv,
                                                float* Xh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (int)(blockDim.x >> 5);
    const int nrun = I / 8, IG = I / 32, nrb = (nrun + 31) / 32;
    const int ntask = (s1 - s0) * nrb;
    for (int t0 = warp; t0 < ntask; t0 += kStageBatch * nw) {
        float v[kStageBatch][8];
        int slot[kStageBatch], run[kStageBatch];
        bool valid[kStageBatch];
#pragma unroll
        for (int b = 0; b < kStageBatch; ++b) {
            const int t = t0 + b * nw;
            const int q = t / nrb;
            slot[b] = s0 + q;
            run[b] = (t - q * nrb) * 32 + lane;
            valid[b] = t < ntask && run[b] < nrun;
            if (valid[b]) {
                const float4* p = reinterpret_cast<const float4*>(src + (size_t)slot[b] * I) + 2 * run[b];
                const float4 x0 = __ldcg(p), x1 = __ldcg(p + 1);
                v[b][0] = x0.x; v[b][1] = x0.y; v[b][2] = x0.z; v[b][3] = x0.w;
                v[b][4] = x1.x; v[b][5] = x1.y; v[b][6] = x1.z; v[b][7] = x1.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[b][i] = 0.f;
            }
        }
#pragma unroll
        for (int b = 0; b < kStageBatch; ++b)
            if (t0 + b * nw < ntask)   // warp-uniform
                stage_q16_run(v[b], valid[b], run[b], IG, hq + (size_t)slot[b] * 4 * IG, Iv + slot[b] * IG,
                              Xh + slot[b] * IG);
    }
}

// Work items (quad of rows, slot) for slots [s0, s1) of this CTA's rows
// [own0, own1): per-(slot, row) results into ypart[slot][row - own0].
template <int BITS, int J>
__device__ __forceinline__ void down_items(int s0, int s1, int own0, int own1, int I, size_t rbI,
                                           const uint8_t* const* s_rows, const uint4* hq, const float* Iv,
                                           const float* Xh, float* ypart) {
    constexpr int kDW = down_threads<BITS, J>() / 32;   // the kernel's warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int IG = I / 32, nsl = s1 - s0;
    const int nquad = (own1 - own0 + kDownRows - 1) / kDownRows;
    const int nit = nquad * nsl;
    if constexpr (BITS == 2) {
        // a lane takes whole groups of 64 codes (16 bytes each); a warp works
        // on J items at a time, so that it keeps as many bytes in flight as
        // with 4-bit codes
        const int GI = IG / 2;
        for (int it0 = warp; it0 < nit; it0 += J * kDW) {
            const uint8_t* rr[J][kDownRows];
            int s2[J], n0s[J], nrs[J];
            bool live[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int it = it0 + j * kDW;
                live[j] = it < nit;
                const int itv = live[j] ? it : it0;
                const int q = itv / nsl;
                s2[j] = s0 + (itv - q * nsl);
                n0s[j] = own0 + q * kDownRows;
                nrs[j] = min(kDownRows, own1 - n0s[j]);
#pragma unroll
                for (int r = 0; r < kDownRows; ++r) rr[j][r] = s_rows[s2[j]] + (size_t)(n0s[j] + min(r, nrs[j] - 1)) * rbI;
            }
            float acc[J][kDownRows];
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
                for (int r = 0; r < kDownRows; ++r) acc[j][r] = 0.f;
            for (int G = lane; G < GI; G += 32) {
                uint4 c[J][kDownRows];
                uint32_t mt[J][kDownRows];
#pragma unroll
                for (int j = 0; j < J; ++j)
#pragma unroll
                    for (int r = 0; r < kDownRows; ++r)
                        if (live[j]) {
                            c[j][r] = ldg_stream(rr[j][r] + 16 * G);
                            mt[j][r] = ldg_u32(rr[j][r] + I / 4 + 4 * G);
                        }
#pragma unroll
                for (int j = 0; j < J; ++j)
                    if (live[j]) {
                        const uint4* xs = hq + (size_t)s2[j] * 4 * IG;
#pragma unroll
                        for (int r = 0; r < kDownRows; ++r)
                            acc[j][r] = group2_dot(c[j][r], mt[j][r], xs, IG, G, Iv + s2[j] * IG, Xh + s2[j] * IG,
                                                   acc[j][r]);
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
    } else {
        // 4-bit codes. A warp works on J items at a time, and each lane issues
        // the loads of MB half-groups of every row of them before it computes.
        // Short rows (one half-group per lane) take two items at a time
        // (J = 2), so that as many bytes are in flight per warp as with long
        // rows.
        constexpr int MB = 2 / J;
        const int M = (IG + 31) / 32;
        for (int it0 = warp; it0 < nit; it0 += J * kDW) {
            const uint8_t* rr[J][kDownRows];
            int s2[J], n0s[J], nrs[J];
            bool live[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int it = it0 + j * kDW;
                live[j] = it < nit;
                const int itv = live[j] ? it : it0;
                const int q = itv / nsl;
                s2[j] = s0 + (itv - q * nsl);
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
                                for (int r = 0; r < kDownRows; ++r) word_dp4a(u4w(c[j][mm][r], wi), xv, ah[r], al[r]);
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

struct DownArgs {
    const uint8_t* const* rec_tab;
    int k, E, n_shared, H, I;
    size_t rbI, gu_block;            // bytes of one down row record; offset of the down block in a record
    const float* h;                  // copies x [ns][I] SwiGLU outputs (gate/up wrote them)
    int copies;
    unsigned gu_ctas;                // gate/up CTAs that count their shared rows
    void* y;
    int y_bf16;
    float* y32;
    const int32_t* sel_ids;          // the selection (the router's, or the streamed layer's)
    const float* sel_wts;
    const int* scale_in;             // the token exponent a
    unsigned* shared_done;           // with n_shared: early start on the shared rows (nullable; set only
                                     // under the bounded-wait test hook)
    unsigned* ids_ready;             // the router's ready flag (nullable); cleared with the counters
    unsigned* down_done;             // the last CTA clears the counters
    unsigned* seq;                   // nullable: the layer's decode count, advanced by the last CTA
    const unsigned long long* sel_tag;   // nullable (with seq): the selection and token exponent as
                                     // tagged words, read before the wait for gate/up
    unsigned* err;
    unsigned long long* tr;
};

template <int BITS, int J>
__device__ __forceinline__ void down_body(const DownArgs& a) {
    extern __shared__ uint4 smh[];
    ktrace(a.tr, blockIdx.x, 0);
    const int I = a.I, IG = I / 32, ns = a.k + a.n_shared;
    uint4* hq = smh;                                                     // [ns][4][IG]
    float* Iv = reinterpret_cast<float*>(hq + (size_t)ns * 4 * IG);     // [ns][IG]
    float* Xh = Iv + ns * IG;                                            // [ns][IG]
    float* ypart = Xh + ns * IG;                                         // [ns][kDownMaxRows]
    __shared__ const uint8_t* s_rows[MOE_MAX_TOP_K + 1];
    __shared__ float s_w[MOE_MAX_TOP_K + 1];
    __shared__ int s_skip, s_early, s_scale, s_have;
    // whole quads of rows per CTA (a partial quad costs a full work item)
    const int nquads_all = (a.H + kDownRows - 1) / kDownRows;
    const int own0 = kDownRows * (int)((long long)nquads_all * blockIdx.x / gridDim.x);
    const int own1 = min(a.H, kDownRows * (int)((long long)nquads_all * (blockIdx.x + 1) / gridDim.x));
    const bool counted = a.n_shared && a.shared_done;
    const float* src = a.h + (size_t)(blockIdx.x % a.copies) * ns * I;   // this CTA's replica
    if (threadIdx.x == 0) {
        // the shared expert's outputs are all written once every gate/up CTA
        // has counted itself: its rows run before the wait for gate/up
        int ok = 0;
        if (counted) {
            ok = wait_count(a.shared_done, a.gu_ctas, kWaitNs) ? 1 : 0;
            if (!ok) atomicOr(a.err, 1u << 27);
        }
        s_early = ok;
        s_skip = 0;
        s_have = a.sel_tag ? 1 : 0;
        if (a.n_shared) {   // slot 0: the shared expert (its record is fixed), weight 1
            s_rows[0] = a.rec_tab[a.E] + a.gu_block;
            s_w[0] = 1.0f;
        }
    }
    __syncthreads();
    if (a.sel_tag) {
        // the selection and the token exponent, published by gate/up CTA 0 long
        // before this kernel starts, resolved before the wait for gate/up (a
        // resident layer's record table does not change between launches)
        const unsigned tag = decode_tag(__ldcg(a.seq));
        const int nw = 2 * a.k + 1;
        if (threadIdx.x < nw) {
            unsigned long long v;
            if (!poll_tagged(a.sel_tag + threadIdx.x, tag, kWaitNs, &v)) {
                atomicOr(a.err, 1u << 25);
                s_have = 0;   // read after the wait instead
            }
            const uint32_t lo = (uint32_t)v;
            const int t = threadIdx.x;
            if (t < a.k) {
                int e = (int)lo;
                if ((unsigned)e >= (unsigned)a.E) e = 0;   // a valid selection never needs the clamp
                s_rows[a.n_shared + t] = a.rec_tab[e] + a.gu_block;
            } else if (t < 2 * a.k) {
                s_w[a.n_shared + t - a.k] = __uint_as_float(lo);
            } else {
                s_scale = (int)lo;
            }
        }
        __syncthreads();
    }
    // Every thread of this CTA has read the decode count and the counters: the
    // CTA counts itself now, and the one counted last clears them at its end
    // (every CTA has read them by then). The count's return is needed only
    // there, so its round trip overlaps the work; the next token's kernels see
    // the cleared words once this grid has completed.
    unsigned order = 0;
    if (a.down_done && threadIdx.x == 0) order = atomicAdd(a.down_done, 1u);
    const int early = s_early;
    if (early) {
        stage_slots_q16<BITS == 4 ? 4 : 2>(src, 0, 1, I, hq, Iv, Xh);
        __syncthreads();
        down_items<BITS, J>(0, 1, own0, own1, I, a.rbI, s_rows, hq, Iv, Xh, ypart);
    }
    pdl_wait();     // gate/up complete: the staged SwiGLU outputs are final
    pdl_trigger();  // the next token's router may start prefetching its weights
    ktrace(a.tr, blockIdx.x, 1);
    const bool have = s_have;
    __syncthreads();   // every thread has read s_have
    if (!have && threadIdx.x >= a.n_shared && threadIdx.x < ns) {   // the routed slots
        const int s = threadIdx.x, j = s - a.n_shared;
        int e = a.sel_ids[j];
        if ((unsigned)e >= (unsigned)a.E) e = 0;   // a valid selection never needs the clamp
        const uint8_t* rec = a.rec_tab[e];
        if (!rec) s_skip = 1;   // streamed layer, expert not resident yet: see below
        s_rows[s] = rec + a.gu_block;
        s_w[s] = a.sel_wts[j];
    }
    if (!have && threadIdx.x == 0) s_scale = a.scale_in ? *a.scale_in : 0;
    stage_slots_q16<BITS == 4 ? 4 : 2>(src, early, ns, I, hq, Iv, Xh);
    __syncthreads();
    ktrace(a.tr, blockIdx.x, 2);
    // a launch made before the host staged this token's experts (streamed
    // layers) does nothing; the host launches again when every expert is resident
    if (!s_skip) {
        down_items<BITS, J>(early, ns, own0, own1, I, a.rbI, s_rows, hq, Iv, Xh, ypart);
        __syncthreads();
        const float inv_a = exp2i(-s_scale);
        for (int n = own0 + threadIdx.x; n < own1; n += blockDim.x) {
            float acc = 0.f;
            for (int s = 0; s < ns; ++s) acc = fmaf(s_w[s], ypart[s * kDownMaxRows + (n - own0)], acc);
            acc = acc * inv_a * inv_a;   // two exact steps (one rounding if the result is subnormal)
            if (a.y32) a.y32[n] = acc;
            if (a.y) {
                if (a.y_bf16) static_cast<__nv_bfloat16*>(a.y)[n] = __float2bfloat16_rn(acc);
                else static_cast<float*>(a.y)[n] = acc;
            }
        }
    }
    if (a.down_done && threadIdx.x == 0 && order == gridDim.x - 1) {
        if (a.shared_done) *a.shared_done = 0u;
        if (a.ids_ready) *a.ids_ready = 0u;
        if (a.seq) *a.seq += 1u;   // the next token's tag
        *a.down_done = 0u;
    }
    ktrace(a.tr, blockIdx.x, 3);
}

template <int BITS, int J = 1>
__global__ void __launch_bounds__(down_threads<BITS, J>()) k_down(const DownArgs a) {
    down_body<BITS, J>(a);
}
template <>
__global__ void __launch_bounds__(down_threads<4, 1>(), 2) k_down<4, 1>(const DownArgs a) {
    down_body<4, 1>(a);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

// staged activations, then the per-CTA selection's scratch
static size_t gu_smem_for(const Layer& L) {
    const int H = L.d.hidden;
    return (size_t)H * 2 + (size_t)(H / 32) * 8 + (size_t)select_words(L.d.n_experts) * 4 +
           (size_t)(L.d.n_experts + 1) * 8;
}
static size_t down_smem(int I, int ns) {
    return (size_t)ns * I * 2 + (size_t)ns * (I / 32) * 8 + (size_t)ns * kDownMaxRows * 4;
}
static int down_grid(const Layer& L) { return L.num_sms * L.occ_down; }
// gate/up CTAs: every resident CTA, but not more than there are row pairs per warp
static int gu_grid(const Layer& L) {
    const int pairs = (L.d.top_k + L.d.n_shared) * L.d.inter;
    return std::max(1, std::min(L.num_sms * L.occ_gu, (pairs + kWarps - 1) / kWarps));
}

using GuKernel = decltype(&k_gateup<4, 1>);
using DownKernel = decltype(&k_down<4, 1>);
// 4-bit rows of at most kGuBlock / 2 half-groups per lane (H <= 3072): two
// row pairs per warp at a time; down rows of one half-group per lane
// (I <= 1024): two items per warp at a time; 2-bit codes: two of each
static GuKernel gu_kernel(const Layer& L) {
    if (L.wbits == 2) return k_gateup<2, 2>;
    return (L.d.hidden / 32 + 31) / 32 <= kGuBlock / 2 ? k_gateup<4, 2> : k_gateup<4, 1>;
}
static DownKernel down_kernel(const Layer& L) {
    if (L.wbits == 2) return k_down<2, 2>;
    return (L.d.inter / 32 + 31) / 32 == 1 ? k_down<4, 2> : k_down<4, 1>;
}
static int down_block(const Layer& L) {
    if (L.wbits == 2) return down_threads<2, 2>();
    return (L.d.inter / 32 + 31) / 32 == 1 ? down_threads<4, 2>() : down_threads<4, 1>();
}


cudaError_t decode_kernel_setup(Layer& L) {
    const int H = L.d.hidden, I = L.d.inter, ns = L.d.top_k + L.d.n_shared;
    cudaError_t e = router_kernel_setup(L);
    if (e != cudaSuccess) return e;
    L.gu_smem = gu_smem_for(L);
    const void* gu = (const void*)gu_kernel(L);
    const void* dn = (const void*)down_kernel(L);
    e = cudaFuncSetAttribute(gu, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.gu_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)down_smem(I, ns));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_gu, gu, kThreads, L.gu_smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ_down, dn, down_block(L), down_smem(I, ns));
    if (e != cudaSuccess) return e;
    if (L.occ_gu < 1 || L.occ_down < 1) return cudaErrorInvalidConfiguration;
    // rows owned by one down CTA must fit its partial-sum buffer
    while (kDownRows * (((H + kDownRows - 1) / kDownRows + down_grid(L) - 1) / down_grid(L)) > kDownMaxRows) {
        if (L.occ_down >= 64) return cudaErrorInvalidConfiguration;
        ++L.occ_down;   // more (smaller) CTAs per SM are launched in waves
    }
    return cudaSuccess;
}

static cudaError_t launch_gateup(Layer& L, const void* x, const DecodeScratch& b, int jj0, int jj1, bool pdl,
                                 unsigned long long* tr, cudaStream_t s) {
    const auto& d = L.d;
    GuArgs a{};
    a.rec_tab = (const uint8_t* const*)L.rec_table;
    a.k = d.top_k;
    a.E = d.n_experts;
    a.n_shared = d.n_shared;
    a.x = x;
    a.x_bf16 = d.act_dtype == MOE_BF16 ? 1 : 0;
    a.H = d.hidden;
    a.I = d.inter;
    a.rbH = row_bytes(d.hidden, L.wbits);
    a.ids = b.ids;
    a.ids_ready = b.ids_ready;
    a.part_tag = b.part_tag;
    a.seq = b.seq;
    a.splits = L.router_splits;
    a.bias = (const float*)L.router_bias;
    a.mode = L.route_mode();
    a.sel_ids = b.ids;
    a.sel_wts = b.wts;
    a.sel_tag = b.sel_tag;
    a.h = b.h;
    a.copies = b.copies;
    a.scale_out = b.scale;
    // The count of CTAs done with the shared expert's rows (a fence and a
    // barrier in every CTA before its selection) feeds the down kernel's early
    // start on the shared expert; down CTAs start only as gate/up CTAs retire,
    // so that start gains nothing and the fence costs the selection a loaded
    // round trip. Only the bounded-wait test hook turns it on.
    a.shared_done = L.test_stall_shared ? b.shared_done : nullptr;
    a.jj0 = jj0;
    a.jj1 = jj1;
    a.pf = (const uint8_t*)L.next_router;
    a.pf_bytes = L.next_router_bytes;
    a.err = error_word(L);
    a.tr = tr;
    a.stall_shared = L.test_stall_shared;
    return launch_pdl(gu_kernel(L), dim3(gu_grid(L)), dim3(kThreads), L.gu_smem, s, pdl, a);
}

static cudaError_t launch_down(Layer& L, const DecodeScratch& b, void* y, float* y_f32, bool pdl,
                               unsigned long long* tr, cudaStream_t s) {
    const auto& d = L.d;
    const int ns = d.top_k + d.n_shared;
    DownArgs a{};
    a.rec_tab = (const uint8_t* const*)L.rec_table;
    a.k = d.top_k;
    a.E = d.n_experts;
    a.n_shared = d.n_shared;
    a.H = d.hidden;
    a.I = d.inter;
    a.rbI = row_bytes(d.inter, L.wbits);
    a.gu_block = gu_block_bytes(d.hidden, d.inter, L.wbits);
    a.h = b.h;
    a.copies = b.copies;
    a.gu_ctas = (unsigned)gu_grid(L);
    a.y = y;
    a.y_bf16 = d.act_dtype == MOE_BF16 ? 1 : 0;
    a.y32 = y_f32;
    a.sel_ids = b.ids;
    a.sel_wts = b.wts;
    a.scale_in = b.scale;
    a.shared_done = L.test_stall_shared ? b.shared_done : nullptr;   // see launch_gateup
    a.ids_ready = b.ids_ready;
    a.seq = b.seq;
    a.sel_tag = b.seq ? b.sel_tag : nullptr;
    a.down_done = (b.shared_done || b.ids_ready || b.seq) ? b.down_done : nullptr;
    a.err = error_word(L);
    a.tr = tr;
    return launch_pdl(down_kernel(L), dim3(down_grid(L)), dim3(down_block(L)), down_smem(d.inter, ns), s, pdl, a);
}

// gate/up over row-order slots jj0..jj1-1 and (with `down`) down + combine,
// over the scratch `b`; the selection b.ids / b.wts is published by the
// router (or given, streamed layers).
cudaError_t launch_experts_decode(Layer& L, const void* x, void* y, float* y_f32, const DecodeScratch& b, int jj0,
                                  int jj1, bool down, bool pdl, bool trace, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (jj1 > jj0) {
        prof_begin(L, K_GATEUP_DECODE, s);
        e = launch_gateup(L, x, b, jj0, jj1, pdl && L.pdl, trace ? L.split_trace(1) : nullptr, s);
        prof_end(L, s);
        if (e != cudaSuccess) return e;
    }
    if (down) {
        prof_begin(L, K_DOWN_DECODE, s);
        e = launch_down(L, b, y, y_f32, pdl && L.pdl, trace ? L.split_trace(2) : nullptr, s);
        prof_end(L, s);
    }
    return e;
}

DecodeScratch layer_decode_scratch(Layer& L, bool fast) {
    DecodeScratch b;
    b.part = L.logits_part;
    b.logits = L.logits;
    b.ids = L.ids;
    b.wts = L.wts;
    b.scale = reinterpret_cast<int*>(L.counters + CNT_TOKEN_SCALE);
    b.router_cnt = L.counters + CNT_ROUTER;
    b.h = L.h;
    b.copies = kHCopies;
    if (fast) {
        b.part_tag = L.part_tag;
        b.seq = L.counters + CNT_DECODE_SEQ;
        b.sel_tag = L.sel_tag;
        b.shared_done = L.counters + CNT_SHARED_DONE;
        b.down_done = L.counters + CNT_DOWN_DONE;
    }
    return b;
}

// Streamed layers: the selection (L.ids, L.wts) is already on the device and
// the routed experts' records are resident. `jj0..jj1` are the row-order
// slots of gate/up to run (0 = the shared expert when there is one); `down`
// adds the down + combine kernel. The caller orders them against the cache's
// copies (events, or programmatic launch after the kernels that staged them).
cudaError_t launch_experts_decode_sel(Layer& L, const void* x, void* y, float* y_f32, int jj0, int jj1, bool down,
                                      cudaStream_t s, bool pdl) {
    return launch_experts_decode(L, x, y, y_f32, layer_decode_scratch(L, false), jj0, jj1, down, pdl, false, s);
}

}  // namespace moe
