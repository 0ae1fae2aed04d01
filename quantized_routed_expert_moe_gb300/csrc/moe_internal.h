// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda.h>

#include "moe.h"
#include "route_mode.h"

namespace moe {

// ---- errors -----------------------------------------------------------------

void set_error(const std::string& msg);
moe_status fail(moe_status s, const std::string& msg);
moe_status cuda_fail(cudaError_t e, const char* what);

#define MOE_CUDA_TRY(expr)                                            \
    do {                                                              \
        cudaError_t _e = (expr);                                      \
        if (_e != cudaSuccess) return ::moe::cuda_fail(_e, #expr);    \
    } while (0)

// Makes `dev` current for the guard's lifetime; restores the previous device.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err != cudaSuccess) return;
        if (prev != dev) err = cudaSetDevice(dev);
        ok = (err == cudaSuccess);
    }
    ~DeviceGuard() {
        if (ok && prev >= 0) {
            int cur = -1;
            if (cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
        }
    }
};

// ---- kernel layout of the weights ---------------------------------------------
//
// A quantised row of K inputs is stored as one "row record":
//   [ codes: 4-bit experts: K/2 bytes, canonical nibble order (element k in
//     byte k/2, low nibble for even k). 2-bit experts: K/4 bytes; per group
//     of 64, 4 words of 16 codes; word w holds elements 16w + j, j < 16, with
//     byte i, bits 2f: f = 0: j = 2i, f = 1: j = 2i + 1, f = 2: j = 8 + 2i,
//     f = 3: j = 9 + 2i (so that (word >> 2f) & 0x03030303 is the even or
//     odd half of one run of 8, one code per byte) ]
//   [ meta: K/64 pairs (scale, bias) as two binary16 values, scale first;
//     zero-padded to a multiple of 16 bytes ]
// so one row is a single contiguous, 16-byte aligned run of bytes.
//
// An expert record is
//   GU block: for i in 0..I-1: gate row i, then up row i   (2*I rows of K = H)
//   D block:  for n in 0..H-1: down row n                  (H rows of K = I)
//
// The 8-bit router is stored as codes [E][H] followed by meta [E][H/64]
// (scale, bias) binary16 pairs.

inline size_t row_meta_bytes(int K) { return ((size_t)(K / 64) * 4 + 15) / 16 * 16; }
inline size_t row_bytes(int K, int bits = 4) { return (size_t)K * bits / 8 + row_meta_bytes(K); }
inline size_t gu_block_bytes(int H, int I, int bits = 4) { return 2 * (size_t)I * row_bytes(H, bits); }
inline size_t record_bytes(int H, int I, int bits = 4) {
    return gu_block_bytes(H, I, bits) + (size_t)H * row_bytes(I, bits);
}

void pack_expert(int H, int I, int bits, const moe_expert& e, uint8_t* dst);

// ---- layer ------------------------------------------------------------------

struct PrefillScratch {
    // permutation of the (token, slot) pairs by expert: groups of rows, one
    // group per distinct routed expert (ascending id), then the shared group
    int32_t* group_expert = nullptr;  // [E + 1] record index of each group
    int32_t* group_off = nullptr;     // [E + 1] first permuted row
    int32_t* group_cnt = nullptr;     // [E + 1] rows (tokens) in the group
    int32_t* n_groups = nullptr;      // [1]
    int32_t* perm_token = nullptr;    // [rows] token of each permuted row
    int32_t* pos = nullptr;           // [T][k + 1] permuted row of (t, slot j); slot k = shared
    unsigned* err = nullptr;          // [1] error bits of the grouped GEMM (bounded waits)
    void* xp = nullptr;               // [rows][H] fp16 x * 2^a (8-element blocks permuted)
    void* hp = nullptr;               // [rows][I] fp16 SwiGLU outputs * 2^z (same block permutation)
    float* yp = nullptr;              // [rows][H] fp32 expert outputs (unweighted)
    float* h32 = nullptr;             // [rows][I] fp32 SwiGLU outputs * 2^(2a) (gate/up epilogue)
    int32_t* xexp = nullptr;          // [T] token activation exponents a
    int32_t* rexp = nullptr;          // [rows] a of each permuted row's token
    unsigned* hmax = nullptr;         // [rows] max |h32| of each row (float bits)
    float2* zfac = nullptr;           // [rows] (2^-e, 2^-a) of each row: hp = h * 2^(e + 2a)
    int max_rows = 0;
    // TMA descriptors: gate/up codes, gate/up meta, down codes, down meta, then
    // xp and hp with boxes of 16, 32, 64 and 128 token rows; on streamed layers
    // 12..15 are the four weight maps over the cache slots
    CUtensorMap tm[16];
    bool ready = false;
    // streamed layers: the chunk's groups read back to the host, and the group
    // lists of the staging waves ([n, expert or slot x n, off x n, cnt x n] per
    // wave, waves back to back), in pinned host memory and on the device
    int32_t* groups_host = nullptr;   // pinned [1 + 3 (E + 1)]
    int32_t* waves_host = nullptr;    // pinned [4 (E + 2)]
    int32_t* waves_dev = nullptr;     // device [4 (E + 2)]
    cudaEvent_t groups_ready = nullptr, waves_free = nullptr;
    uint64_t waves = 0;               // staging waves run by streamed prefill chunks
};

struct CacheState;  // streamed mode (cache.cu)

// Device-managed cache (MOE_OPT_CACHE_DEVICE): the LFU state of a streamed
// layer in device memory, kept per slot (an expert's count and last use are
// dropped on eviction, so only residents carry any), updated by the router's
// selecting block, and the fills it decides, which k_cache_fill copies from
// host-mapped records. All pointers are device pointers.
struct DevCacheArgs {
    int32_t* slot_expert = nullptr;     // [slots] expert held, -1 when free
    uint32_t* slot_count = nullptr;     // [slots] uses since admission
    uint32_t* slot_last = nullptr;      // [slots] clock of the last use
    uint32_t* clock = nullptr;          // [1] tokens seen
    int32_t* fills = nullptr;           // [1 + 2 MOE_MAX_TOP_K]: n, then (expert, slot) pairs
    unsigned long long* stats = nullptr;   // [4] tokens, hits, misses, bytes
    const uint8_t** rec_table = nullptr;   // the layer's record table [E + 1]
    const uint8_t* const* src = nullptr;   // [E] device views of the host records
    const uint8_t* pinned = nullptr;    // [E] 1: pinned (resident outside the slots, never in the LFU)
    unsigned long long* usage = nullptr;   // [E] selections since the state came to the device
    uint8_t* slots_base = nullptr;      // [slots][rb]
    unsigned long long rb = 0;          // record bytes
    int slots = 0;
    unsigned* err = nullptr;            // error word (bit 26: no victim found)
};
struct Profiler;    // per-kernel event timing (profile.cu)

// Kernel kinds for per-kernel timing.
enum KernelKind {
    K_ROUTER_DECODE = 0,
    K_ROUTER_TOKENS,
    K_TOPK_TOKENS,
    K_GATEUP_DECODE,
    K_DOWN_DECODE,
    K_PF_PERMUTE,
    K_PF_GATHER,
    K_PF_GEMM_GU,
    K_PF_HCONV,
    K_PF_GEMM_DOWN,
    K_PF_COMBINE,
    K_CACHE_FILL,
    K_NUM_KINDS
};

struct Layer {
    moe_layer_desc d{};
    int device = 0;
    size_t rec_bytes = 0;

    // router
    void* router = nullptr;         // fp32 [E][H], or 8-bit codes + meta
    size_t router_nbytes = 0;
    // moe_layer_set_next: the router weights of the layer that runs next,
    // warmed into L2 by this layer's gate/up kernel (nullable)
    const void* next_router = nullptr;
    size_t next_router_bytes = 0;
    float* router_bias = nullptr;   // fp32 [E] or null
    int router_scoring = MOE_SCORE_SOFTMAX;   // moe_layer_set_router_scoring
    float routed_scaling = 1.0f;
    RouteMode route_mode() const { return RouteMode{router_scoring == MOE_SCORE_SIGMOID ? 1 : 0, routed_scaling}; }

    // experts (resident mode): (E + n_shared) records; the shared expert is index E
    uint8_t* experts = nullptr;
    const uint8_t** rec_table = nullptr;  // device [E + 1] record pointer per expert

    // decode scratch
    float* logits_part = nullptr;   // [max(router_splits, router_splits_tok)][max_tokens][E]
    float* logits = nullptr;        // [max_tokens][E]
    unsigned long long* part_tag = nullptr;   // [router_splits][E] tagged partial logits (fast decode)
    unsigned long long* sel_tag = nullptr;    // [2k + 1] the fast decode's selection, tagged
    int32_t* ids = nullptr;         // [max_tokens][k]
    float* wts = nullptr;           // [max_tokens][k]
    float* h = nullptr;             // SwiGLU outputs, kDecodeHCopies x [k + 1][I] fp32 (times 2^2a, the token scale)
    unsigned* counters = nullptr;   // [64] counters and words of the decode kernels (CNT_*)
    int router_splits = 1;       // split-K of the one-token router
    int router_splits_tok = 1;   // split-K of the multi-token router (<= 16)

    PrefillScratch pf;
    CacheState* cache = nullptr;
    Profiler* prof = nullptr;

    // host I/O staging for moe_decode_tokens_host
    void* io_x = nullptr;
    void* io_y = nullptr;
    int io_cap = 0;

    size_t device_bytes = 0;
    int num_sms = 0;
    int occ_gu = 0, occ_down = 0;  // resident CTAs per SM of the decode expert kernels
    size_t gu_smem = 0;            // gate/up dynamic shared memory (upper bound)

    // three-kernel decode: programmatic dependent launch between the kernels
    bool pdl = true;

    // host waits (streamed layers): deadline, and a test hook that holds the
    // copy stream for this long before each stage's fills
    int host_timeout_ms = 30000;
    int test_stall_copies_ms = 0;

    int wbits = 4;   // expert code width: 4 (MOE_W_Q4G64) or 2 (MOE_W_Q2G64)
    int test_stall_shared = 0;   // MOE_OPT_TEST_STALL_SHARED
    unsigned long long* trace_split = nullptr;  // device [MOE_TRACE_KERNELS][MOE_TRACE_MAX_CTAS][4]
    bool trace_on = false;
    unsigned long long* split_trace(int kernel) const {
        return (trace_on && trace_split) ? trace_split + (size_t)kernel * MOE_TRACE_MAX_CTAS * 4 : nullptr;
    }
};

// Words of Layer::counters. The counters are zero between launches.
enum {
    CNT_ROUTER = 0,        // router blocks done (the last one selects), moe_route / streamed layers
    CNT_SHARED_DONE = 1,   // decode gate/up CTAs whose shared-expert rows are written
    CNT_DOWN_DONE = 2,     // decode down CTAs done (the last one clears the decode counters)
    CNT_IDS_READY = 3,     // the router's selecting block has published the selection (decode)
    CNT_DECODE_SEQ = 4,    // fast decodes of the layer so far (the tag of the next one's router partials)
    CNT_TOKEN_SCALE = 8,   // the token exponent a of the last decode (int)
    CNT_ERR = 20           // error bits of bounded device waits (moe_layer_check)
};
inline unsigned* error_word(Layer& L) { return L.counters + CNT_ERR; }

// ---- launchers (decode.cu / prefill.cu) -----------------------------------------

// ids_pub / seq_pub (host-mapped, nullable): with select, the ids are also
// written there and then seq, for a host that polls instead of copying
// dc (nullable): the selecting block also runs the device-managed cache's LFU step
// Scratch one decode token works on: the router's outputs (partials, keys,
// selection, and the ready flag the decode's gate/up waits for), the SwiGLU
// outputs (`copies` replicas of [k + 1][I] fp32), and the fast decode's tagged
// words and counters (null: the router's last block selects, and the down
// kernel waits for gate/up before anything).
struct DecodeScratch {
    float* part = nullptr;
    float* logits = nullptr;
    int32_t* ids = nullptr;
    float* wts = nullptr;
    int* scale = nullptr;
    unsigned* router_cnt = nullptr;
    unsigned* ids_ready = nullptr;
    float* h = nullptr;
    int copies = 1;
    // fast decode: the router's partials as tagged 64-bit words [splits][E]
    // (tag in the high half), from which every gate/up CTA selects; seq
    // counts the layer's decodes (the down kernel's last CTA advances it)
    unsigned long long* part_tag = nullptr;
    unsigned* seq = nullptr;
    unsigned long long* sel_tag = nullptr;   // [2k + 1]: ids, weights, token exponent (tagged)
    unsigned* shared_done = nullptr;   // gate/up CTAs done with the shared rows (the test hook's early start)
    unsigned* down_done = nullptr;     // down CTAs counted (the last clears the counters)
};
// the layer's own scratch; `fast`: with the tagged words, the decode count and
// the counters
DecodeScratch layer_decode_scratch(Layer& L, bool fast);

// out (nullable): where the partials, keys and selection go (default: the
// layer's scratch, no ready flag)
cudaError_t launch_route_decode(Layer& L, const void* x, cudaStream_t s, int select, int32_t* ids_pub = nullptr,
                                unsigned* seq_pub = nullptr, unsigned seq = 0, const DevCacheArgs* dc = nullptr,
                                const DecodeScratch* out = nullptr);
// xexp (nullable): each token's activation exponent for a prefill chunk
cudaError_t launch_route_tokens(Layer& L, const void* x, int T, cudaStream_t s, int32_t* xexp = nullptr);
// pdl: both launches may start early (the preceding kernel in `s` must be ours)
cudaError_t launch_experts_decode_sel(Layer& L, const void* x, void* y, float* y_f32, int jj0, int jj1, bool down,
                                      cudaStream_t s, bool pdl = false);
// K-splits of the prefill router GEMM: at most this many partial logit sets
// are summed (in a fixed order) per token.
constexpr int kMaxTokSplits = 32;
constexpr int kMaxRouterSplits = 16;   // K-splits of the one-token router (moe_abi.cu)
constexpr int kDecodeHCopies = 8;   // replicas of the decode SwiGLU outputs (decode.cu), <= 32
// gate/up over row-order slots jj0..jj1-1 and (down) the down kernel, over scratch b
cudaError_t launch_experts_decode(Layer& L, const void* x, void* y, float* y_f32, const DecodeScratch& b, int jj0,
                                  int jj1, bool down, bool pdl, bool trace, cudaStream_t s);
cudaError_t launch_prefill(Layer& L, const void* x, int T, void* y, float* y_f32, cudaStream_t s);
cudaError_t decode_kernel_setup(Layer& L);
cudaError_t router_kernel_setup(Layer& L);
cudaError_t prefill_kernel_setup(Layer& L);

// Launch with programmatic dependent launch allowed (the kernel may start
// before the preceding kernel in the stream completes and must call
// griddepcontrol.wait before touching that kernel's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Event marks around a launch; no-ops unless profiling was started.
void prof_begin(Layer& L, int kind, cudaStream_t s);
void prof_end(Layer& L, cudaStream_t s);
void prof_destroy(Layer& L);


// ---- streamed cache (cache.cu) ---------------------------------------------------

moe_status cache_create(Layer& L, const void* const* records, moe_expert_source src, void* user);
void cache_destroy(Layer& L);
moe_status cache_stage(Layer& L, const int32_t* ids, int n, cudaStream_t s, int* hits, int* misses);
moe_status cache_decode(Layer& L, const void* x, void* y, float* y_f32, cudaStream_t s);
// MOE_OPT_CACHE_DEVICE: hand the LFU state to the device (on) or back to the host (off)
moe_status cache_set_device(Layer& L, bool on);
bool cache_is_device(const Layer& L);
// tensor maps of the streamed prefill over the slots (LFU slots, then pinned experts)
moe_status prefill_cache_maps(Layer& L);
int cache_slot_of(const Layer& L, int expert);   // slot holding `expert`, -1 when not resident
const uint8_t* cache_slots_base(const Layer& L); // device [cache_slot_count][rec_bytes]
int cache_slot_count(const Layer& L);            // LFU slots + pinned experts
// host wait for `ev` with the layer's deadline (MOE_OPT_HOST_TIMEOUT_MS)
moe_status host_wait_event(const Layer& L, cudaEvent_t ev, const char* what);
// prefill chunk on a streamed layer (router already launched): waves through the cache
moe_status launch_prefill_streamed(Layer& L, const void* x, int T, void* y, float* y_f32, cudaStream_t s);
// streamed layers: tensor maps over the cache slots and the pinned buffers (after cache_create)
moe_status prefill_cache_setup(Layer& L);

}  // namespace moe

struct moe_layer {
    moe::Layer L;
};
