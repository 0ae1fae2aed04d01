// Prefill chunk path: the T tokens' (token, slot) pairs are grouped by expert,
// gathered as fp16, run through a grouped GEMM on the tcgen05 tensor cores
// (gate/up with the SwiGLU in the epilogue, then down) with the 4-bit weights
// dequantised into shared memory, and combined per token in a fixed order.
//
// Grouping follows the "Union" step of the Colibri analysis report (section 2):
// each distinct expert's weights are read once per chunk however many tokens
// selected it. The TurboFieldfare article ("token generation") chunks prefill
// at 128 tokens.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <string>
#include <vector>

#include "common.cuh"
#include "moe_internal.h"
#include "sm100.cuh"

namespace moe {
namespace {

using namespace bw;

// The dequantiser turns one 32-bit word of codes (8 elements) into four fp16
// pairs in the order (0,4) (1,5) (2,6) (3,7): masking the nibbles at bits 0
// and 16, then 4 and 20, and so on. The activation operands (x gathered here,
// h written by the gate/up epilogue) are stored in the same order within every
// block of 8 along K (element j at place ((j & 3) << 1) | (j >> 2)), so the
// products pair up as in the plain dot product.

// ---------------------------------------------------------------------------
// permutation (histogram, exclusive scan, stable scatter) -- one CTA
// ---------------------------------------------------------------------------

constexpr int kPermThreads = 1024;

__global__ void __launch_bounds__(kPermThreads) k_pf_permute(const int32_t* __restrict__ ids, int T, int k, int E,
                                                             int n_shared, int32_t* __restrict__ gexp,
                                                             int32_t* __restrict__ goff, int32_t* __restrict__ gcnt,
                                                             int32_t* __restrict__ n_groups,
                                                             int32_t* __restrict__ perm_token,
                                                             int32_t* __restrict__ pos) {
    __shared__ int s_cnt[1024];
    __shared__ int s_start[1024];
    __shared__ int s_gidx[1024];
    __shared__ uint32_t s_bits[1024][MOE_MAX_CHUNK / 32];   // [expert][token bit]: token selected the expert
    __shared__ int s_wa[32], s_wb[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = T * k;   // <= 1024
    s_cnt[tid] = 0;
#pragma unroll
    for (int q = 0; q < MOE_MAX_CHUNK / 32; ++q) s_bits[tid][q] = 0u;
    __syncthreads();
    int my_e = 0;
    if (tid < P) {
        my_e = ids[tid];
        if ((unsigned)my_e >= (unsigned)E) my_e = 0;   // a valid selection never needs this
        const int t = tid / k;
        atomicAdd(&s_cnt[my_e], 1);
        atomicOr(&s_bits[my_e][t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    // exclusive scans over experts (thread e): row starts, and group index of
    // each expert that has rows (groups in ascending expert id)
    const int c = tid < E ? s_cnt[tid] : 0, nz = c > 0;
    int a = c, b = nz;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ua = __shfl_up_sync(0xffffffffu, a, o), ub = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) { a += ua; b += ub; }
    }
    if (lane == 31) { s_wa[warp] = a; s_wb[warp] = b; }
    __syncthreads();
    if (warp == 0) {
        int wa = s_wa[lane], wb = s_wb[lane];
        const int ta = wa, tb = wb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ua = __shfl_up_sync(0xffffffffu, wa, o), ub = __shfl_up_sync(0xffffffffu, wb, o);
            if (lane >= o) { wa += ua; wb += ub; }
        }
        s_wa[lane] = wa - ta;   // exclusive prefix of warp totals
        s_wb[lane] = wb - tb;
        if (lane == 31) s_gidx[1023] = wb;   // number of routed groups (read below, after the sync)
    }
    __syncthreads();
    const int n_routed = s_gidx[1023];
    __syncthreads();
    if (tid < E) {
        s_start[tid] = a - c + s_wa[warp];
        s_gidx[tid] = b - nz + s_wb[warp];
    }
    __syncthreads();
    if (tid < P) {
        // stable: a token selects an expert at most once, so the rank among
        // earlier pairs with the same expert is the number of earlier tokens
        // that selected it (bits below t in the expert's token mask)
        const int e = my_e;
        const int t = tid / k, j = tid - t * k;
        int r = 0;
#pragma unroll
        for (int q = 0; q < MOE_MAX_CHUNK / 32; ++q) {
            const uint32_t m = s_bits[e][q];
            r += (q < (t >> 5)) ? __popc(m) : (q == (t >> 5)) ? __popc(m & ((1u << (t & 31)) - 1u)) : 0;
        }
        const int row = s_start[e] + r;
        perm_token[row] = t;
        pos[t * (k + 1) + j] = row;
    }
    if (tid < E && c > 0) {
        const int g = s_gidx[tid];
        gexp[g] = tid;
        goff[g] = s_start[tid];
        gcnt[g] = c;
    }
    if (n_shared) {
        for (int t = tid; t < T; t += blockDim.x) {
            perm_token[P + t] = t;
            pos[t * (k + 1) + k] = P + t;
        }
        if (tid == 0) {
            gexp[n_routed] = E;
            goff[n_routed] = P;
            gcnt[n_routed] = T;
        }
    }
    if (tid == 0) *n_groups = n_routed + (n_shared ? 1 : 0);
}

// ---------------------------------------------------------------------------
// gather: xp[row] = fp16(x[perm_token[row]]), blocks of 8 in operand order
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) k_pf_gather(const void* __restrict__ x, int x_bf16,
                                                   const int32_t* __restrict__ perm_token, int rows, int H,
                                                   const int32_t* __restrict__ xexp, uint4* __restrict__ xp,
                                                   int32_t* __restrict__ rexp, unsigned* __restrict__ hmax) {
    const int nb = H / 8;
    const long total = (long)rows * nb;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int row = (int)(idx / nb), blk = (int)(idx - (long)row * nb);
        const int t = __ldg(perm_token + row);
        const int a = __ldg(xexp + t);   // the token's exponent: x * 2^a in binary16 without overflow
        if (blk == 0) {
            rexp[row] = a;
            hmax[row] = 0u;   // the gate/up epilogue accumulates the row's max |h| here
        }
        const float sc = exp2i(a);
        float v[8];
        if (x_bf16) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + (size_t)t * H) + blk);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[2 * q] = __uint_as_float(w[q] << 16);
                v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)t * H) + 2 * blk;
            const float4 p = __ldg(src), q = __ldg(src + 1);
            v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
            v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // position 2q holds element q, 2q + 1 holds element q + 4
            const __half2 h = __floats2half2_rn(v[q] * sc, v[q + 4] * sc);
            o[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
        xp[idx] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------------------------------
// grouped GEMM on tcgen05
// ---------------------------------------------------------------------------
//
// Work items are (group g, 128-row weight tile mt). One persistent CTA per SM
// walks the items; per item it computes D[128 weight rows][N tokens] over K in
// chunks of 64 (one quantisation group), 4 chunks (one raw block) at a time:
//   * one TMA thread copies the packed codes of a block (128 rows x 128 B, with
//     the 128-byte swizzle so that the dequantisers' reads are conflict-free)
//     and their (scale, bias) pairs (128 rows x 16 B) into a raw ring, as far
//     ahead as the ring allows; another copies the group's token rows of the
//     fp16 activations for the block's chunks (N x 128 B each, 128-byte
//     swizzle) into a shared-memory operand slot once the MMA thread has
//     released it (one thread for both kept the raw ring from running ahead);
//   * 16 dequantiser warps turn the codes into fp16 w = code * scale + bias
//     (one fp16 fma: correctly rounded) and store them straight into tensor
//     memory (tcgen05.st): warp w owns tensor-memory lanes 32 (w % 4) .. + 31
//     (one weight row each) and a quarter of each chunk's 64 columns of K. The
//     weight operand never touches shared memory: stores from the SM's threads
//     into shared memory slow the tensor core's operand reads, copies by the
//     TMA unit and stores into tensor memory do not;
//   * one thread issues tcgen05.mma (A from tensor memory, B from shared
//     memory; M = 128, N = round16(tokens), K = 16), 16 per block, into a
//     tensor-memory accumulator (two, alternating by item);
//   * 4 epilogue warps read the accumulator (warp w owns lanes 32w..32w+31) and
//     write either h = silu(gate) * up in fp16 (gate/up: the weight tile holds
//     64 interleaved gate/up row pairs) or the fp32 expert outputs (down).
// Operand slots change hands a block at a time (one barrier wait and one commit
// per 16 MMAs): the MMA thread shares its scheduler with four dequantiser warps
// that keep it busy, and per-chunk hand-offs left the tensor core idle.
//
// Tensor memory (512 columns): accumulators at columns 0 and 128; weight
// operand stages of 32 columns (128 x 64 fp16) from column 256, two slots of
// four.

constexpr int kStages = 8, kRawStages = 4, kChunksPerRaw = 4;
constexpr int kBatchSlots = kStages / kChunksPerRaw;   // operand stages are handed over a raw block at a time
constexpr int kEpiWarps = 4, kDqWarps = 16;
constexpr int kTmaWarp = kEpiWarps + kDqWarps, kTokWarp = kTmaWarp + 1, kMmaWarp = kTokWarp + 1;
constexpr int kGemmThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kB16 = 128 * 128;
constexpr uint32_t kRawCodes = 128 * 128, kRawMeta = 128 * 16, kRaw = kRawCodes + kRawMeta;
// 2-bit codes: a raw block is 128 rows x 64 bytes (64-byte swizzle), then the same meta
constexpr uint32_t kRawCodes2 = 128 * 64, kRaw2Tx = kRawCodes2 + kRawMeta;
constexpr uint32_t kTmemCols = 512, kTmemA = 256, kACols = 32;
constexpr size_t kBarBytes = 8 * (2 * kStages + 2 * kRawStages + 4) + 16;
constexpr size_t kZfBytes = 2 * 128 * 8;   // down epilogue: the tile's row factors, two tiles
constexpr size_t kGemmSmem = 1024 + (size_t)kStages * kB16 + (size_t)kRawStages * kRaw + kBarBytes + kZfBytes;
static_assert(kRaw % 1024 == 0 && kB16 % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kTmemA + kStages * kACols <= kTmemCols, "weight stages exceed tensor memory");

struct GemmArgs {
    const int32_t* gexp;
    const int32_t* goff;
    const int32_t* gcnt;
    const int32_t* n_groups;
    int K;          // reduction length (H for gate/up, I for down)
    int n_mt;       // 128-row weight tiles per expert
    int rows_out;   // weight rows that exist (2I or H)
    void* out;      // gate/up: fp32 h * 2^(2a) [rows][I]; down: fp32 [rows][H]
    int ld_out;
    const int32_t* rexp;   // gate/up: each permuted row's activation exponent a
    unsigned* hmax;        // gate/up: each row's max |h * 2^(2a)| (float bits)
    const float2* zfac;    // down: each row's (2^-e, 2^-a); its operand is h * 2^(e + 2a) in binary16
    unsigned* err;
    unsigned long long* tr;   // [gridDim][4]: wait cycles of copy / dequant / MMA, total cycles; or null
};

// mbarrier wait that, when tracing, adds the SM clock cycles spent waiting to `acc`
struct TimedWait {
    unsigned long long* tr;
    unsigned long long acc;
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity, volatile int* abort, unsigned* err,
                                               unsigned code) {
        if (!tr) return mbar_wait(bar, parity, abort, err, code);
        const long long t0 = clock64();
        const bool ok = mbar_wait(bar, parity, abort, err, code);
        acc += (unsigned long long)(clock64() - t0);
        return ok;
    }
    __device__ __forceinline__ void store(int slot, unsigned long long v) {
        if (tr) tr[blockIdx.x * 4 + slot] = v;
    }
};

// error bits (moe_layer_check): bit 16 + role
enum { ERR_TMA = 1u << 16, ERR_DQ = 1u << 17, ERR_MMA = 1u << 18, ERR_EPI = 1u << 19, ERR_DRAIN = 1u << 20 };

// fp16 pair from two nibbles placed at bits 0..3 and 16..19 of t: code * s + b.
// The nibble becomes the low mantissa bits of 1024.0 (unit in the last place 1),
// so subtracting 1024 leaves the code exactly.
__device__ __forceinline__ uint32_t dq_pair(uint32_t t, uint32_t s2, uint32_t b2) {
    uint32_t r;
    asm("{.reg .b32 c; lop3.b32 c, %1, 0x000F000F, 0x64006400, 0xEA;"   // (t & mask) | 1024.0
        " sub.f16x2 c, c, %4; fma.rn.f16x2 %0, c, %2, %3;}"
        : "=r"(r)
        : "r"(t), "r"(s2), "r"(b2), "r"(0x64006400u));
    return r;
}
// The same for nibbles at bits 4..7 and 20..23, without a shift: there they are
// mantissa bits 4..7, which in 64.0 (unit in the last place 1/16) weigh 1 each.
__device__ __forceinline__ uint32_t dq_pair_hi(uint32_t t, uint32_t s2, uint32_t b2) {
    uint32_t r;
    asm("{.reg .b32 c; lop3.b32 c, %1, 0x00F000F0, 0x54005400, 0xEA;"   // (t & mask) | 64.0
        " sub.f16x2 c, c, %4; fma.rn.f16x2 %0, c, %2, %3;}"
        : "=r"(r)
        : "r"(t), "r"(s2), "r"(b2), "r"(0x54005400u));
    return r;
}

// fp16 pair from two 2-bit codes at bits F..F+1 and 16+F..17+F of t: code * s
// + b. The code lands in mantissa bits F..F+1 of a power of two whose unit in
// the last place is 2^-F (1024.0, 256.0, 64.0, 16.0 for F = 0, 2, 4, 6), where
// it weighs 1, so subtracting the power of two leaves the code exactly.
template <int F>
__device__ __forceinline__ uint32_t dq2_pair(uint32_t t, uint32_t s2, uint32_t b2) {
    constexpr uint32_t mask = 0x00030003u << F;
    constexpr uint32_t base = F == 0 ? 0x64006400u : F == 2 ? 0x5C005C00u : F == 4 ? 0x54005400u : 0x4C004C00u;
    uint32_t r;
    asm("{.reg .b32 c; lop3.b32 c, %1, %4, %5, 0xEA;"   // (t & mask) | base
        " sub.f16x2 c, c, %6; fma.rn.f16x2 %0, c, %2, %3;}"
        : "=r"(r)
        : "r"(t), "r"(s2), "r"(b2), "n"(mask), "n"(base), "r"(base));
    return r;
}

template <int MODE, int BITS>
__global__ void __launch_bounds__(kGemmThreads, 1) k_pf_gemm(const __grid_constant__ CUtensorMap tm_codes,
                                                             const __grid_constant__ CUtensorMap tm_meta,
                                                             const __grid_constant__ CUtensorMap tm_b16,
                                                             const __grid_constant__ CUtensorMap tm_b32,
                                                             const __grid_constant__ CUtensorMap tm_b64,
                                                             const __grid_constant__ CUtensorMap tm_b128,
                                                             const GemmArgs a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint8_t* bst = smem;                          // token operand stages
    uint8_t* raw = smem + kStages * kB16;         // raw code / meta ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw + kRawStages * kRaw);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 2 * kRawStages + 4);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    float2* s_zf = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);   // [2][128]
    const uint32_t b_full = saddr(bars), b_empty = b_full + 8 * kStages;
    const uint32_t b_rfull = b_empty + 8 * kStages, b_rempty = b_rfull + 8 * kRawStages;
    const uint32_t b_afull = b_rempty + 8 * kRawStages, b_aempty = b_afull + 16;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kBatchSlots; ++s) {
            mbar_init(b_full + 8 * s, kDqWarps + 1);   // dequantisers' stores + the token copies
            mbar_init(b_empty + 8 * s, 1);
        }
        for (int r = 0; r < kRawStages; ++r) {
            mbar_init(b_rfull + 8 * r, 1);
            mbar_init(b_rempty + 8 * r, kDqWarps);
        }
        for (int c = 0; c < 2; ++c) {
            mbar_init(b_afull + 8 * c, 1);
            mbar_init(b_aempty + 8 * c, kEpiWarps);
        }
        *s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) tmem_alloc(saddr(s_tmem), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long t_start = clock64();
    const int n_items = *a.n_groups * a.n_mt;
    const int nk = a.K / 64;
    TimedWait tw{a.tr, 0ull};

    if (warp == kTmaWarp) {
        // raw codes and (scale, bias) pairs, as far ahead as the raw ring allows.
        // The whole warp walks the loop (waits included) and one elected lane
        // issues each copy, so the warp stays converged.
        if (elect_one()) {
            tma_prefetch_desc(&tm_codes);
            tma_prefetch_desc(&tm_meta);
        }
        __syncwarp();
        const uint64_t pol_w = l2_evict_first();
        uint32_t rit = 0;   // copies issued
        bool go = true;
        for (int w = blockIdx.x; go && w < n_items; w += gridDim.x) {
            const int g = w / a.n_mt, mt = w - g * a.n_mt;
            const int e = a.gexp[g];
            for (int kb = 0; kb * kChunksPerRaw < nk; ++kb, ++rit) {
                const uint32_t rs = rit % kRawStages;
                const bool ok = tw(b_rempty + 8 * rs, ((rit / kRawStages) & 1) ^ 1, s_abort, a.err, ERR_TMA);
                // after an abort nothing more is issued: a stage is only ever
                // refilled once its consumers have released it, so each stage
                // has at most one copy in flight and the drain below sees them all
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { go = false; break; }
                if (elect_one()) {
                    mbar_arrive_tx(b_rfull + 8 * rs, BITS == 4 ? kRaw : kRaw2Tx);
                    const uint32_t rd = saddr(raw + rs * kRaw);
                    // a block: 4 chunks of 64 codes per row (128 or 64 bytes), then their meta
                    tma_load_3d(rd, &tm_codes, kb * (BITS == 4 ? 128 : 64), mt * 128, e, b_rfull + 8 * rs, pol_w);
                    tma_load_3d(rd + kRawCodes, &tm_meta, a.K * BITS / 8 + kb * 16, mt * 128, e, b_rfull + 8 * rs,
                                pol_w);
                }
                __syncwarp();
            }
        }
        // every copy issued lands before the CTA exits, also after an abort
        // (on the normal path the consumers have already waited for all of them)
        const uint32_t n_tail = rit < (uint32_t)kRawStages ? rit : (uint32_t)kRawStages;
        for (uint32_t q = rit - n_tail; q < rit; ++q) {
            int dummy = 0;
            mbar_wait(b_rfull + 8 * (q % kRawStages), (q / kRawStages) & 1, &dummy, a.err, ERR_DRAIN, 50000000ull);
        }
        if (lane == 0) tw.store(0, tw.acc);
    } else if (warp == kTokWarp) {
        // the group's token tiles of a block, into the operand slot the MMA thread has released
        if (elect_one()) {
            tma_prefetch_desc(&tm_b16);
            tma_prefetch_desc(&tm_b32);
            tma_prefetch_desc(&tm_b64);
            tma_prefetch_desc(&tm_b128);
        }
        __syncwarp();
        const uint64_t pol_b = l2_evict_last();
        uint32_t bt = 0;   // operand blocks issued
        bool go = true;
        for (int w = blockIdx.x; go && w < n_items; w += gridDim.x) {
            const int g = w / a.n_mt;
            const int off = a.goff[g], m = a.gcnt[g];
            // one copy per chunk: the smallest box of 16, 32, 64 or 128 token rows that holds the group
            const CUtensorMap* tmb = m <= 16 ? &tm_b16 : m <= 32 ? &tm_b32 : m <= 64 ? &tm_b64 : &tm_b128;
            const uint32_t b_bytes = (m <= 16 ? 16u : m <= 32 ? 32u : m <= 64 ? 64u : 128u) * 128u;
            for (int kb = 0; kb * kChunksPerRaw < nk; ++kb, ++bt) {
                const uint32_t bs = bt % kBatchSlots;
                const int kc0 = kb * kChunksPerRaw, nc = min(nk - kc0, kChunksPerRaw);
                const bool ok = tw(b_empty + 8 * bs, ((bt / kBatchSlots) & 1) ^ 1, s_abort, a.err, ERR_TMA);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { go = false; break; }   // as the raw copies
                if (elect_one()) {
                    mbar_arrive_tx(b_full + 8 * bs, (uint32_t)nc * b_bytes);
                    for (int c = 0; c < nc; ++c)
                        tma_load_2d(saddr(bst + (bs * kChunksPerRaw + c) * kB16), tmb, (kc0 + c) * 64, off,
                                    b_full + 8 * bs, pol_b);
                }
                __syncwarp();
            }
        }
        // every copy issued lands before the CTA exits: the operand barrier's
        // phase of an issued block completes once its copy has landed (the
        // dequantisers arrive for every block, after an abort too)
        const uint32_t n_tail = bt < (uint32_t)kBatchSlots ? bt : (uint32_t)kBatchSlots;
        for (uint32_t q = bt - n_tail; q < bt; ++q) {
            int dummy = 0;
            mbar_wait(b_full + 8 * (q % kBatchSlots), (q / kBatchSlots) & 1, &dummy, a.err, ERR_DRAIN, 50000000ull);
        }
    } else if (warp >= kEpiWarps && warp < kEpiWarps + kDqWarps) {
        // lane quarter q (tensor-memory lanes 32q..32q+31 = weight rows) and
        // part pt: 4-bit codes, 16 elements of every chunk's K (columns 8 pt ..
        // 8 pt + 7 of each chunk); 2-bit codes, the whole of chunk pt
        const int dw = warp - kEpiWarps, q = dw & 3, pt = dw >> 2;
        const int r = 32 * q + lane;
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kTmemA + 8 * pt;   // 4-bit: K part pt
        const uint32_t ta2 = tmem + ((uint32_t)(32 * q) << 16) + kTmemA;            // 2-bit: whole chunks
        uint32_t rit = 0;
        for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
            for (int kb = 0; kb * kChunksPerRaw < nk; ++kb, ++rit) {
                // one raw block (up to 4 chunks) at a time: all of its codes are
                // read and converted before any is stored, for instruction-level
                // parallelism across the chunks
                const uint32_t rs = rit % kRawStages;
                tw(b_rfull + 8 * rs, (rit / kRawStages) & 1, s_abort, a.err, ERR_DQ);
                const uint8_t* rw = raw + rs * kRaw;
                const uint4 mq = *reinterpret_cast<const uint4*>(rw + kRawCodes + r * 16);
                const int kc0 = kb * kChunksPerRaw, nc = min(nk - kc0, kChunksPerRaw);
                // 4-bit: o[c] = this warp's 8 columns (K part pt) of chunk c;
                // 2-bit: o[w] = columns 8w .. 8w + 7 of chunk pt (the warp's chunk)
                uint32_t o[kChunksPerRaw][8];
                if constexpr (BITS == 4) {
                    uint2 cw[kChunksPerRaw];
#pragma unroll
                    for (int c = 0; c < kChunksPerRaw; ++c) {
                        // bytes 8 pt .. 8 pt + 7 of chunk c (16-byte unit 2c + pt / 2),
                        // at their 128-byte-swizzled place
                        const int u = (c << 1) | (pt >> 1);
                        cw[c] = *reinterpret_cast<const uint2*>(rw + r * 128 + ((u ^ (r & 7)) << 4) + 8 * (pt & 1));
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_rempty + 8 * rs);
#pragma unroll
                    for (int c = 0; c < kChunksPerRaw; ++c) {
                        const uint32_t mw = u4w(mq, c);
                        const uint32_t s2 = __byte_perm(mw, 0, 0x1010), b2 = __byte_perm(mw, 0, 0x3232);
                        const uint32_t vw[2] = {cw[c].x, cw[c].y};
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t v = vw[j], v8 = v >> 8;
                            o[c][4 * j + 0] = dq_pair(v, s2, b2);
                            o[c][4 * j + 1] = dq_pair_hi(v, s2, b2);
                            o[c][4 * j + 2] = dq_pair(v8, s2, b2);
                            o[c][4 * j + 3] = dq_pair_hi(v8, s2, b2);
                        }
                    }
                } else {
                    // the 16 bytes of chunk pt (64 codes), at their 64-byte-swizzled
                    // place: 16-byte unit pt of row r is unit pt ^ ((r / 2) % 4)
                    const uint4 cw = *reinterpret_cast<const uint4*>(rw + r * 64 + ((pt ^ ((r >> 1) & 3)) << 4));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_rempty + 8 * rs);
                    const uint32_t mw = u4w(mq, pt);
                    const uint32_t s2 = __byte_perm(mw, 0, 0x1010), b2 = __byte_perm(mw, 0, 0x3232);
                    // word w holds codes 16w .. 16w + 15: byte i carries codes 2i, 2i + 1,
                    // 8 + 2i, 9 + 2i at bits 0, 2, 4, 6 (the 2-bit kernel layout), so the
                    // pairs (j, j + 4) of each block of 8 come out of one mask each
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t v = u4w(cw, w), v8 = v >> 8;
                        o[w][0] = dq2_pair<0>(v, s2, b2);    // codes 0, 4
                        o[w][1] = dq2_pair<2>(v, s2, b2);    // 1, 5
                        o[w][2] = dq2_pair<0>(v8, s2, b2);   // 2, 6
                        o[w][3] = dq2_pair<2>(v8, s2, b2);   // 3, 7
                        o[w][4] = dq2_pair<4>(v, s2, b2);    // 8, 12
                        o[w][5] = dq2_pair<6>(v, s2, b2);    // 9, 13
                        o[w][6] = dq2_pair<4>(v8, s2, b2);   // 10, 14
                        o[w][7] = dq2_pair<6>(v8, s2, b2);   // 11, 15
                    }
                }
                const uint32_t bs = rit % kBatchSlots;
                tw(b_empty + 8 * bs, ((rit / kBatchSlots) & 1) ^ 1, s_abort, a.err, ERR_DQ);
                tc_fence_after();
                if constexpr (BITS == 4) {
#pragma unroll
                    for (int c = 0; c < kChunksPerRaw; ++c)
                        if (c < nc) tmem_st8(ta + (bs * kChunksPerRaw + c) * kACols, o[c]);
                } else if (pt < nc) {   // warp-uniform
#pragma unroll
                    for (int w = 0; w < 4; ++w) tmem_st8(ta2 + (bs * kChunksPerRaw + pt) * kACols + 8 * w, o[w]);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_full + 8 * bs);
            }
        }
        if (dw == 0 && lane == 0) tw.store(1, tw.acc);
    } else if (warp == kMmaWarp) {
        // converged warp; one elected lane issues the MMAs and commits
        uint32_t bt = 0, tile = 0;
        for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++tile) {
            const int g = w / a.n_mt;
            const int m = a.gcnt[g];
            const int N = ((m + 15) >> 4) << 4;
            const uint32_t idesc = idesc_f16_f32(128, N);
            const uint32_t acc = tile & 1;
            tw(b_aempty + 8 * acc, ((tile >> 1) & 1) ^ 1, s_abort, a.err, ERR_MMA);
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * 128;
            for (int kb = 0; kb * kChunksPerRaw < nk; ++kb, ++bt) {
                // one wait and one commit per block of up to 4 chunks (16 MMAs)
                const uint32_t bs = bt % kBatchSlots;
                const int kc0 = kb * kChunksPerRaw, nc = min(nk - kc0, kChunksPerRaw);
                tw(b_full + 8 * bs, (bt / kBatchSlots) & 1, s_abort, a.err, ERR_MMA);
                tc_fence_after();
                if (elect_one()) {
                    for (int c = 0; c < nc; ++c) {
                        const uint32_t A = tmem + kTmemA + (bs * kChunksPerRaw + c) * kACols;
                        const uint32_t B = saddr(bst + (bs * kChunksPerRaw + c) * kB16);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16_ta(d_tmem, A + kk * 8, desc_sw128(B + kk * 32), idesc, ((kc0 + c) | kk) != 0);
                    }
                    mma_commit(b_empty + 8 * bs);
                }
                __syncwarp();
            }
            if (elect_one()) mma_commit(b_afull + 8 * acc);
            __syncwarp();
        }
        // every MMA completes before the tensor memory is released
        if (tile > 0) {
            int dummy = 0;
            mbar_wait(b_afull + 8 * ((tile - 1) & 1), ((tile - 1) >> 1) & 1, &dummy, a.err, ERR_DRAIN, 50000000ull);
        }
        if (lane == 0) tw.store(2, tw.acc);
    } else {   // epilogue warps 0..3: tensor-memory lanes 32*warp .. 32*warp + 31
        const int row = warp * 32 + lane;
        uint32_t tile = 0;
        for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++tile) {
            const int g = w / a.n_mt, mt = w - g * a.n_mt;
            const int off = a.goff[g], m = a.gcnt[g];
            const int N = ((m + 15) >> 4) << 4;
            const uint32_t acc = tile & 1;
            // down: each thread fetches one of the tile's row factors while the
            // accumulator is still being computed; the four epilogue warps then
            // share them through shared memory (double-buffered by tile)
            float2 fz = make_float2(0.f, 0.f);
            if (MODE == 1 && row < m) fz = __ldg(a.zfac + off + row);
            tw(b_afull + 8 * acc, (tile >> 1) & 1, s_abort, a.err, ERR_EPI);
            tc_fence_after();
            if (MODE == 1) {
                s_zf[acc * 128 + row] = fz;
                asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
            }
            const uint32_t tb = tmem + ((uint32_t)(warp * 32) << 16) + acc * 128;
            for (int c0 = 0; c0 < N; c0 += 16) {
                float v[16];
                tmem_ld16(tb + c0, v);
                if (MODE == 0) {
                    // lanes 2p and 2p + 1 hold gate and up of pair i for these 16
                    // tokens; the even lane finishes the even tokens and the odd
                    // lane the odd ones, after one exchange per token pair. The
                    // products come out times 2^a (the token's scale), so
                    // g * u * sigmoid(g 2^-a) is h * 2^(2a); the row's max |h|
                    // goes to hmax for the conversion to binary16.
                    const int i = mt * 64 + (row >> 1);
                    const bool odd = row & 1;
                    float* hp = static_cast<float*>(a.out) + i;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float got = __shfl_xor_sync(0xffffffffu, odd ? v[2 * q] : v[2 * q + 1], 1);
                        const float g = odd ? got : v[2 * q], u = odd ? v[2 * q + 1] : got;
                        const int col = c0 + 2 * q + (odd ? 1 : 0);
                        uint32_t mb = 0u;
                        if (col < m) {
                            const int prow = off + col;
                            const float gt = g * exp2i(-__ldg(a.rexp + prow));
                            // the fast exponential and division are far inside the
                            // binary16 rounding the value gets next
                            const float h = g * u * __fdividef(1.0f, 1.0f + __expf(-gt));
                            hp[(size_t)prow * a.ld_out] = h;
                            mb = __float_as_uint(h) & 0x7fffffffu;
                        }
                        // max over the warp's 16 pairs, even and odd tokens apart
                        const uint32_t me = __reduce_max_sync(0xffffffffu, odd ? 0u : mb);
                        const uint32_t mo = __reduce_max_sync(0xffffffffu, odd ? mb : 0u);
                        if (lane < 2 && col < m) atomicMax(a.hmax + off + col, lane ? mo : me);
                    }
                } else {
                    // the operand was h * 2^(e + 2a): scale back by 2^-e, 2^-a
                    // and 2^-a, exact powers of two (one rounding only if the
                    // result is subnormal)
                    const int n = mt * 128 + row;
                    float* yp = static_cast<float*>(a.out);
                    if (n < a.rows_out) {
                        float2 f[16];   // the same for every lane
#pragma unroll
                        for (int j = 0; j < 16; ++j) f[j] = s_zf[acc * 128 + c0 + j];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < m)
                                yp[(size_t)(off + c0 + j) * a.ld_out + n] = v[j] * f[j].x * f[j].y * f[j].y;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_aempty + 8 * acc);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) tw.store(3, (unsigned long long)(clock64() - t_start));
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// SwiGLU outputs to the down GEMM's binary16 operand
// ---------------------------------------------------------------------------
//
// Row r of the listed groups: hp[r] = fp16(h32[r] * 2^e_r) in the
// dequantiser's order within each block of 8, e_r from the row's max |h32|
// (fp16_fit_exp), so that hp[r] = h * 2^(e_r + 2 a_r); zfac[r] = (2^-e_r,
// 2^-a_r), by which the down GEMM's epilogue scales the row back. Grid
// (groups of the list, blocks per group); a CTA past the list's group count
// does nothing.
// all_rows > 0: every row of [0, all_rows) (a whole chunk), the grid strided
// over (row, block of 8) pairs; the group list is not read.
__global__ void __launch_bounds__(256) k_pf_hconv(const float* __restrict__ h32, const unsigned* __restrict__ hmax,
                                                  const int32_t* __restrict__ rexp, const int32_t* __restrict__ goff,
                                                  const int32_t* __restrict__ gcnt, const int32_t* __restrict__ n_groups,
                                                  int all_rows, int I, uint4* __restrict__ hp,
                                                  float2* __restrict__ zfac) {
    const int nb = I / 8;
    int off = 0, cnt = all_rows;
    long idx0 = (long)blockIdx.x * blockDim.x + threadIdx.x, stride = (long)gridDim.x * blockDim.x;
    if (all_rows == 0) {
        const int g = blockIdx.x;
        if (g >= *n_groups) return;
        off = goff[g];
        cnt = gcnt[g];
        idx0 = (long)blockIdx.y * blockDim.x + threadIdx.x;
        stride = (long)gridDim.y * blockDim.x;
    }
    for (long idx = idx0; idx < (long)cnt * nb; idx += stride) {
        const int r = off + (int)(idx / nb), b = (int)(idx - (idx / nb) * nb);
        const int e = fp16_fit_exp(__uint_as_float(__ldcg(hmax + r)));
        const float sc = exp2i(e);
        const float4* src = reinterpret_cast<const float4*>(h32 + (size_t)r * I + 8 * b);
        const float4 p = __ldcg(src), q = __ldcg(src + 1);
        const float v[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // position 2j holds element j, 2j + 1 holds element j + 4
            const __half2 h = __floats2half2_rn(v[j] * sc, v[j + 4] * sc);
            o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        hp[(size_t)r * nb + b] = make_uint4(o[0], o[1], o[2], o[3]);
        if (b == 0) zfac[r] = make_float2(exp2i(-e), exp2i(-rexp[r]));   // |e|, |a| <= 126: normal floats
    }
}

// ---------------------------------------------------------------------------
// combine: y[t] = y_shared[t] + sum_j w[t][j] * y_{S_j}[t], fixed order
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) k_pf_combine(const float* __restrict__ yp, const int32_t* __restrict__ pos,
                                                    const float* __restrict__ wts, int k, int n_shared, int H,
                                                    void* __restrict__ y, int y_bf16, float* __restrict__ y32) {
    const int t = blockIdx.x;
    const int n = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (n >= H) return;
    const int32_t* pt = pos + (size_t)t * (k + 1);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (n_shared) acc = __ldcg(reinterpret_cast<const float4*>(yp + (size_t)pt[k] * H + n));
    // every slot's outputs in flight at once, then summed in slot order
    float4 v[MOE_MAX_TOP_K];
    float w[MOE_MAX_TOP_K];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOP_K; ++j)
        if (j < k) {
            w[j] = wts[(size_t)t * k + j];
            v[j] = __ldcg(reinterpret_cast<const float4*>(yp + (size_t)pt[j] * H + n));
        }
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOP_K; ++j)
        if (j < k) {
            acc.x = fmaf(w[j], v[j].x, acc.x);
            acc.y = fmaf(w[j], v[j].y, acc.y);
            acc.z = fmaf(w[j], v[j].z, acc.z);
            acc.w = fmaf(w[j], v[j].w, acc.w);
        }
    const size_t o = (size_t)t * H + n;
    if (y32) *reinterpret_cast<float4*>(y32 + o) = acc;
    if (y) {
        if (y_bf16) {
            __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y) + o;
            yb[0] = __float2bfloat16_rn(acc.x);
            yb[1] = __float2bfloat16_rn(acc.y);
            yb[2] = __float2bfloat16_rn(acc.z);
            yb[3] = __float2bfloat16_rn(acc.w);
        } else {
            *reinterpret_cast<float4*>(static_cast<float*>(y) + o) = acc;
        }
    }
}

// ---------------------------------------------------------------------------
// host: tensor maps and launches
// ---------------------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// rows of packed weights (bytes), one plane per expert record
bool map_weight_rows(CUtensorMap* tm, const uint8_t* base, size_t row_b, int rows, int recs, size_t rec_b,
                     uint32_t box_x, CUtensorMapSwizzle swz) {
    const cuuint64_t dims[3] = {row_b, (cuuint64_t)rows, (cuuint64_t)recs};
    const cuuint64_t strides[2] = {row_b, rec_b};
    const cuuint32_t box[3] = {box_x, 128, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return encoder()(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 activations [rows][K], `box_rows` x 64-column boxes with the 128-byte swizzle
bool map_act(CUtensorMap* tm, void* base, int K, int rows, uint32_t box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return encoder()(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The four weight maps of a set of records (gate/up codes, gate/up meta, down
// codes, down meta): rows of the record layout, one plane per record. A raw
// block of codes is 4 chunks of 64 codes per row: 128 bytes with the 128-byte
// swizzle (4-bit) or 64 bytes with the 64-byte swizzle (2-bit).
static bool map_weights(const Layer& L, CUtensorMap* tm, const uint8_t* recs_base, int recs) {
    const int H = L.d.hidden, I = L.d.inter, b = L.wbits;
    const uint8_t* gu = recs_base;
    const uint8_t* dn = recs_base + gu_block_bytes(H, I, b);
    const auto SW = b == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const auto NS = CU_TENSOR_MAP_SWIZZLE_NONE;
    const uint32_t bx = b == 4 ? 128 : 64;
    return map_weight_rows(&tm[0], gu, row_bytes(H, b), 2 * I, recs, L.rec_bytes, bx, SW) &&
           map_weight_rows(&tm[1], gu, row_bytes(H, b), 2 * I, recs, L.rec_bytes, 16, NS) &&
           map_weight_rows(&tm[2], dn, row_bytes(I, b), H, recs, L.rec_bytes, bx, SW) &&
           map_weight_rows(&tm[3], dn, row_bytes(I, b), H, recs, L.rec_bytes, 16, NS);
}

cudaError_t prefill_kernel_setup(Layer& L) {
    const auto& d = L.d;
    if (!L.pf.xp) return cudaSuccess;
    const auto g0 = L.wbits == 4 ? k_pf_gemm<0, 4> : k_pf_gemm<0, 2>;
    const auto g1 = L.wbits == 4 ? k_pf_gemm<1, 4> : k_pf_gemm<1, 2>;
    cudaError_t e = cudaFuncSetAttribute(g0, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(g1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e != cudaSuccess) return e;
    if (!encoder()) return cudaErrorSymbolNotFound;
    const int H = d.hidden, I = d.inter;
    // device records: every expert and the shared one (resident layers), or
    // the shared one alone (streamed layers: routed experts live in the cache slots)
    const int recs = d.cache_slots > 0 ? d.n_shared : d.n_experts + d.n_shared;
    bool ok = recs == 0 || map_weights(L, &L.pf.tm[0], L.experts, recs);
    for (int j = 0; j < 4 && ok; ++j)   // token boxes of 16, 32, 64 and 128 rows
        ok = map_act(&L.pf.tm[4 + j], L.pf.xp, H, L.pf.max_rows, 16u << j) &&
             map_act(&L.pf.tm[8 + j], L.pf.hp, I, L.pf.max_rows, 16u << j);
    if (!ok) return cudaErrorInvalidValue;
    L.pf.ready = d.cache_slots == 0;   // streamed layers: once the slot maps exist
    return cudaSuccess;
}

moe_status prefill_cache_maps(Layer& L) {
    auto& pf = L.pf;
    if (!pf.xp) return MOE_OK;
    const uint8_t* slots = cache_slots_base(L);
    const int n = cache_slot_count(L);   // LFU slots, then pinned experts
    if (!map_weights(L, &pf.tm[12], slots, n)) return fail(MOE_E_CUDA, "tensor maps over the cache slots");
    return MOE_OK;
}

moe_status prefill_cache_setup(Layer& L) {
    const auto& d = L.d;
    auto& pf = L.pf;
    if (!pf.xp) return MOE_OK;
    const int E = d.n_experts;
    const moe_status sm = prefill_cache_maps(L);
    if (sm != MOE_OK) return sm;
    MOE_CUDA_TRY(cudaHostAlloc(&pf.groups_host, (size_t)(1 + 3 * (E + 1)) * 4, cudaHostAllocDefault));
    MOE_CUDA_TRY(cudaHostAlloc(&pf.waves_host, (size_t)4 * (E + 2) * 4, cudaHostAllocDefault));
    MOE_CUDA_TRY(cudaMalloc(&pf.waves_dev, (size_t)4 * (E + 2) * 4));
    L.device_bytes += (size_t)4 * (E + 2) * 4;
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&pf.groups_ready, cudaEventDisableTiming));
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&pf.waves_free, cudaEventDisableTiming));
    MOE_CUDA_TRY(cudaEventRecord(pf.waves_free, 0));
    pf.ready = true;
    return MOE_OK;
}

namespace {

// permute the chunk's (token, slot) pairs by expert and gather the activations
cudaError_t launch_permute_gather(Layer& L, const void* x, int T, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden, k = d.top_k, E = d.n_experts, ns = d.n_shared;
    const int rows = T * k + T * ns;
    auto& pf = L.pf;
    prof_begin(L, K_PF_PERMUTE, s);
    k_pf_permute<<<1, kPermThreads, 0, s>>>(L.ids, T, k, E, ns, pf.group_expert, pf.group_off, pf.group_cnt,
                                            pf.n_groups, pf.perm_token, pf.pos);
    prof_end(L, s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prof_begin(L, K_PF_GATHER, s);
    const long blocks = ((long)rows * (H / 8) + 255) / 256;
    k_pf_gather<<<(int)std::min<long>(blocks, (long)L.num_sms * 8), 256, 0, s>>>(
        x, d.act_dtype == MOE_BF16 ? 1 : 0, pf.perm_token, rows, H, pf.xexp, static_cast<uint4*>(pf.xp), pf.rexp,
        pf.hmax);
    prof_end(L, s);
    return cudaGetLastError();
}

// gate/up + SwiGLU and down GEMMs over a list of groups; `wmap` selects the
// weight maps (0: device records, 12: cache slots); group g's expert field is
// the record (or slot) index the maps address
// all_rows > 0: the groups cover rows [0, all_rows) (a whole chunk); 0: a
// wave's subset of the groups
cudaError_t launch_gemm_pair(Layer& L, int wmap, const int32_t* gexp, const int32_t* goff, const int32_t* gcnt,
                             const int32_t* n_groups, int all_rows, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden, I = d.inter;
    auto& pf = L.pf;
    GemmArgs gu{gexp, goff, gcnt, n_groups, H, I / 64, 2 * I, pf.h32, I, pf.rexp, pf.hmax, nullptr, pf.err,
                L.split_trace(3)};
    prof_begin(L, K_PF_GEMM_GU, s);
    (L.wbits == 4 ? k_pf_gemm<0, 4> : k_pf_gemm<0, 2>)<<<L.num_sms, kGemmThreads, kGemmSmem, s>>>(
        pf.tm[wmap + 0], pf.tm[wmap + 1], pf.tm[4], pf.tm[5], pf.tm[6], pf.tm[7], gu);
    prof_end(L, s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prof_begin(L, K_PF_HCONV, s);
    if (all_rows > 0) {
        const long items = (long)all_rows * (I / 8);
        k_pf_hconv<<<(int)std::min<long>((items + 255) / 256, (long)L.num_sms * 4), 256, 0, s>>>(
            pf.h32, pf.hmax, pf.rexp, goff, gcnt, n_groups, all_rows, I, static_cast<uint4*>(pf.hp), pf.zfac);
    } else {
        k_pf_hconv<<<dim3(d.n_experts + 1, 8), 256, 0, s>>>(pf.h32, pf.hmax, pf.rexp, goff, gcnt, n_groups, 0, I,
                                                             static_cast<uint4*>(pf.hp), pf.zfac);
    }
    prof_end(L, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    GemmArgs dn{gexp, goff, gcnt, n_groups, I, (H + 127) / 128, H, pf.yp, H, nullptr, nullptr, pf.zfac, pf.err,
                L.split_trace(4)};
    prof_begin(L, K_PF_GEMM_DOWN, s);
    (L.wbits == 4 ? k_pf_gemm<1, 4> : k_pf_gemm<1, 2>)<<<L.num_sms, kGemmThreads, kGemmSmem, s>>>(
        pf.tm[wmap + 2], pf.tm[wmap + 3], pf.tm[8], pf.tm[9], pf.tm[10], pf.tm[11], dn);
    prof_end(L, s);
    return cudaGetLastError();
}

cudaError_t launch_combine(Layer& L, int T, void* y, float* y_f32, cudaStream_t s) {
    const auto& d = L.d;
    const int H = d.hidden;
    prof_begin(L, K_PF_COMBINE, s);
    k_pf_combine<<<dim3(T, (H / 4 + 255) / 256), 256, 0, s>>>(L.pf.yp, L.pf.pos, L.wts, d.top_k, d.n_shared, H, y,
                                                              d.act_dtype == MOE_BF16 ? 1 : 0, y_f32);
    prof_end(L, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(Layer& L, const void* x, int T, void* y, float* y_f32, cudaStream_t s) {
    if (!L.pf.ready) return cudaErrorNotSupported;
    auto& pf = L.pf;
    cudaError_t e = launch_permute_gather(L, x, T, s);
    if (e != cudaSuccess) return e;
    e = launch_gemm_pair(L, 0, pf.group_expert, pf.group_off, pf.group_cnt, pf.n_groups,
                         T * (L.d.top_k + L.d.n_shared), s);
    if (e != cudaSuccess) return e;
    return launch_combine(L, T, y, y_f32, s);
}

// Batch union through the cache (Colibri report section 2, "Union": each
// distinct expert of a batch is loaded once and applied to every row that
// routes to it; Colibri README, "What's implemented": batch-union MoE in
// prefill). The chunk's distinct routed experts pass through the layer's
// cache slots in waves: first the experts already resident (no copies), then
// the rest, at most cache_slots at a time. Each wave is one moe_cache_stage
// (the LFU counts one use per expert per wave), then the grouped GEMMs run on
// that wave's groups with the weight maps over the slots. The shared expert's
// group runs first, from its device record, while the first copies are in
// flight. Every group's rows are computed exactly as on a resident layer, so
// the chunk's output is the same bit for bit.
moe_status launch_prefill_streamed(Layer& L, const void* x, int T, void* y, float* y_f32, cudaStream_t s) {
    auto& pf = L.pf;
    if (!pf.ready) return fail(MOE_E_UNSUPPORTED, "prefill scratch missing (max_tokens == 1)");
    const auto& d = L.d;
    const int E = d.n_experts, ns = d.n_shared, S = d.cache_slots;
    MOE_CUDA_TRY(launch_permute_gather(L, x, T, s));
    // the groups, read back (count, then expert / offset / size arrays)
    int32_t* gh = pf.groups_host;
    MOE_CUDA_TRY(cudaMemcpyAsync(gh, pf.n_groups, 4, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(gh + 1, pf.group_expert, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(gh + 1 + (E + 1), pf.group_off, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(gh + 1 + 2 * (E + 1), pf.group_cnt, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaEventRecord(pf.groups_ready, s));
    moe_status st = host_wait_event(L, pf.groups_ready, "prefill groups");
    if (st != MOE_OK) return st;
    // the previous chunk's wave-list uploads have run before the pinned lists are rewritten
    st = host_wait_event(L, pf.waves_free, "wave list buffer reuse");
    if (st != MOE_OK) return st;
    const int ng = gh[0];
    const int32_t* gexp = gh + 1;
    const int32_t* goff = gh + 1 + (E + 1);
    const int32_t* gcnt = gh + 1 + 2 * (E + 1);
    const int nr = ng - ns;   // routed groups (ascending expert id); the shared group is last
    if (nr < 0 || nr > E) return fail(MOE_E_STATE, "prefill group count out of range");
    int32_t* wh = pf.waves_host;
    int32_t* wd = pf.waves_dev;
    int o = 0;   // next free int in the wave lists
    // one wave list: [n, index x n, off x n, cnt x n], uploaded on `s`, then the GEMMs
    auto run_wave = [&](int wmap, const int* gsel, int n, const int32_t* index) -> moe_status {
        int32_t* w = wh + o;
        w[0] = n;
        for (int i = 0; i < n; ++i) {
            w[1 + i] = index[i];
            w[1 + n + i] = goff[gsel[i]];
            w[1 + 2 * n + i] = gcnt[gsel[i]];
        }
        const int len = 1 + 3 * n;
        MOE_CUDA_TRY(cudaMemcpyAsync(wd + o, w, (size_t)len * 4, cudaMemcpyHostToDevice, s));
        MOE_CUDA_TRY(launch_gemm_pair(L, wmap, wd + o + 1, wd + o + 1 + n, wd + o + 1 + 2 * n, wd + o, 0, s));
        o += len;
        ++pf.waves;
        return MOE_OK;
    };
    if (ns) {
        const int gs = ng - 1;
        const int32_t rec0 = 0;   // the shared expert is the layer's only device record
        st = run_wave(0, &gs, 1, &rec0);
        if (st != MOE_OK) return st;
    }
    // waves: the resident experts first, then the others in ascending id
    std::vector<int> order;
    order.reserve(nr);
    for (int g = 0; g < nr; ++g)
        if (cache_slot_of(L, gexp[g]) >= 0) order.push_back(g);
    const int n_res = (int)order.size();
    for (int g = 0; g < nr; ++g)
        if (cache_slot_of(L, gexp[g]) < 0) order.push_back(g);
    std::vector<int32_t> ids, slot;
    for (int w0 = 0; w0 < nr;) {
        // the resident experts form the first wave (at most S in the LFU slots, plus
        // the pinned ones)
        const int w1 = (w0 == 0 && n_res > 0) ? n_res : std::min(nr, w0 + S);
        const int n = w1 - w0;
        ids.resize(n);
        slot.resize(n);
        for (int i = 0; i < n; ++i) ids[i] = gexp[order[w0 + i]];
        st = cache_stage(L, ids.data(), n, s, nullptr, nullptr);
        if (st != MOE_OK) break;
        for (int i = 0; i < n; ++i) {
            slot[i] = cache_slot_of(L, ids[i]);
            if (slot[i] < 0) st = fail(MOE_E_STATE, "expert " + std::to_string(ids[i]) + " is not resident");
        }
        if (st != MOE_OK) break;
        st = run_wave(12, order.data() + w0, n, slot.data());
        if (st != MOE_OK) break;
        w0 = w1;
    }
    MOE_CUDA_TRY(cudaEventRecord(pf.waves_free, s));
    if (st != MOE_OK) return st;
    MOE_CUDA_TRY(launch_combine(L, T, y, y_f32, s));
    return MOE_OK;
}

}  // namespace moe
