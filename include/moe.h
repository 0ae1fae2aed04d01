/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed Mixture-of-Experts FFN step.
 *
 * One layer object holds a routed-MoE FFN: a router, n_experts routed experts
 * and an optional always-resident shared expert, every expert a gated (SwiGLU)
 * FFN over affine group-64 4-bit weights. The calls below compute, per token x:
 *
 *   l      = W_r x (+ bias)                      router logits
 *   S      = first top_k experts by (-l_e, e)     exact top-k, ties to lower index
 *   w_j    = softmax over the selected logits     renormalised routing weights
 *   f_e(x) = W_down,e (silu(W_gate,e x) * W_up,e x)
 *   y      = f_shared(x) + sum_j w_j f_{S_j}(x)
 *
 * Passages that define these operations:
 *   - router, LFU cache, shared expert and combine: TurboFieldfare article
 *     (GeekNews), section "token generation";
 *   - weight format (affine 4-bit group 64; 8-bit router): same article,
 *     section "execution architecture";
 *   - exact top-8: Inferno README, "Current Scope"; Colibri report, section 3;
 *   - gate/up/down experts stored side by side: Inferno README, "Model";
 *   - prefill chunk (up to 128 tokens) and batch-union MoE: TurboFieldfare
 *     "token generation"; Colibri report, section 2 ("Union"); Colibri README,
 *     "What's implemented".
 *
 * Conventions for every call:
 *   - Every call returns a moe_status and never aborts or exits. On failure
 *     moe_last_error() returns a thread-local detail string.
 *   - "device" pointers are CUDA global-memory pointers on the layer's device;
 *     "host" pointers are ordinary (pageable or pinned) host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Work is enqueued on it; calls return without waiting unless
 *     stated otherwise.
 *   - A layer serves one call at a time; calls on one layer must not overlap
 *     from several host threads, and work enqueued on different streams for
 *     the same layer must not overlap on the GPU (they share scratch).
 *   - Nothing falls back to the CPU: without a usable CUDA device every
 *     compute call fails with MOE_E_CUDA.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1u
#define MOE_MAX_TOP_K 8
#define MOE_MAX_CHUNK 128
#define MOE_GROUP 64

typedef enum {
    MOE_OK = 0,
    MOE_E_INVALID = 1,     /* bad argument or descriptor */
    MOE_E_UNSUPPORTED = 2, /* valid but not built (format, shape) */
    MOE_E_NOMEM = 3,       /* device or pinned host memory exhausted (checked up front) */
    MOE_E_CUDA = 4,        /* a CUDA runtime error; detail in moe_last_error() */
    MOE_E_TIMEOUT = 5,     /* a host wait passed its deadline */
    MOE_E_STATE = 6,       /* layer state forbids the call (e.g. an expert slot is not valid) */
    MOE_E_SOURCE = 7       /* the expert source callback failed or returned a short read */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum { MOE_W_F32 = 0, MOE_W_Q8G64 = 1, MOE_W_Q4G64 = 2, MOE_W_Q2G64 = 3 } moe_wfmt;

/* Affine group-64 matrix [N][K] in canonical storage (host memory):
 *   codes: 4-bit: uint8 [N][K/2], element k in byte k/2, low nibble for even k;
 *          2-bit: uint8 [N][K/4], element k in byte k/4 at bits 2*(k%4) (low bits first);
 *          8-bit: uint8 [N][K];
 *   scale, bias: IEEE binary16 bit patterns [N][K/64];
 *   element (n, k) = code(n, k) * scale[n][k/64] + bias[n][k/64]. */
typedef struct {
    const uint8_t* codes;
    const uint16_t* scale;
    const uint16_t* bias;
} moe_qmat;

/* One expert: gate [I][H], up [I][H], down [H][I], all in the layer's
 * expert_fmt (4-bit or 2-bit group-64). */
typedef struct {
    moe_qmat gate, up, down;
} moe_expert;

/* Router weights [E][H]: `w` (fp32, row-major) when router_fmt == MOE_W_F32,
 * `q` (8-bit group-64) when router_fmt == MOE_W_Q8G64. */
typedef struct {
    const float* w;
    moe_qmat q;
} moe_router;

typedef struct {
    uint32_t abi_version;  /* MOE_ABI_VERSION */
    int32_t hidden;        /* H, multiple of 64 */
    int32_t inter;         /* I, multiple of 64 */
    int32_t n_experts;     /* E, top_k <= E <= 1024 */
    int32_t top_k;         /* 1..MOE_MAX_TOP_K */
    int32_t n_shared;      /* 0 or 1 */
    int32_t router_fmt;    /* MOE_W_F32 or MOE_W_Q8G64 */
    int32_t expert_fmt;    /* MOE_W_Q4G64 or MOE_W_Q2G64 */
    int32_t group;         /* 64 */
    int32_t act_dtype;     /* MOE_F32 or MOE_BF16: dtype of x and y */
    int32_t max_tokens;    /* largest T for moe_route / moe_prefill_chunk, 1..MOE_MAX_CHUNK */
    int32_t cache_slots;   /* 0: all experts device-resident; > 0: streamed, that many slots (>= top_k) */
} moe_layer_desc;

typedef struct moe_layer moe_layer;

/* Expert source for streamed layers: copy expert `expert`'s packed record
 * (moe_expert_record_bytes bytes) into `dst`, host memory owned by the layer.
 * Return 0 on success and nonzero on failure (short read, I/O error). */
typedef int (*moe_expert_source)(void* user, int32_t expert, void* dst, size_t bytes);

typedef struct {
    uint64_t tokens;       /* tokens staged */
    uint64_t hits;         /* expert lookups served from a resident slot */
    uint64_t misses;       /* expert lookups that needed a host-to-device fill */
    uint64_t bytes_h2d;    /* bytes copied host -> device for fills */
    uint64_t stage_ns;     /* host time spent in moe_cache_stage */
} moe_cache_stats_t;

/* ---- layer lifetime ------------------------------------------------------ */

/* Create a layer on CUDA device `device`.
 *   router:       host, required. Copied and repacked; the caller may free it after.
 *   router_bias:  host fp32 [E] or NULL. With softmax scoring (the default)
 *                 it is added to the logits before selection and before the
 *                 softmax; with sigmoid scoring (moe_layer_set_router_scoring)
 *                 it is added to the sigmoid scores for the selection only.
 *   shared:       host, required iff n_shared == 1.
 *   experts:      host array of E experts, required when cache_slots == 0
 *                 (copied, repacked into the kernel layout in device memory).
 *                 Ignored when cache_slots > 0.
 *   records:      streamed mode only (cache_slots > 0): host array of E
 *                 pointers to packed expert records (moe_pack_expert_record),
 *                 borrowed -- they must stay valid until the layer is
 *                 destroyed; page-locked memory gives the fastest fills. May be
 *                 NULL when `source` is given.
 *   source/user:  streamed mode only: fills a layer-owned pinned staging
 *                 buffer on demand when `records` is NULL.
 * Capacity is checked against free device memory before anything is
 * allocated (MOE_E_NOMEM). An invalid device fails with MOE_E_CUDA. */
moe_status moe_layer_create(const moe_layer_desc* desc, const moe_router* router,
                            const float* router_bias, const moe_expert* shared,
                            const moe_expert* experts, const void* const* records,
                            moe_expert_source source, void* source_user,
                            int32_t device, moe_layer** out);

/* Release every device and host resource of the layer (NULL is ignored).
 * Synchronises with the layer's own streams first. */
void moe_layer_destroy(moe_layer* layer);

/* Bytes of one packed expert record for this descriptor (0 if invalid). */
size_t moe_expert_record_bytes(const moe_layer_desc* desc);

/* Pack one expert from canonical storage into the library's record layout
 * (host to host). `dst` must hold moe_expert_record_bytes(desc) bytes. */
moe_status moe_pack_expert_record(const moe_layer_desc* desc, const moe_expert* expert, void* dst);

/* Device bytes the layer holds (weights + slots + scratch). */
size_t moe_layer_device_bytes(const moe_layer* layer);

/* The layer that runs after `layer` (same device; NULL clears it). While
 * `layer` decodes, its gate/up kernel prefetches `next`'s router weights into
 * L2, so that the next layer's router reads them from L2 rather than HBM. A
 * hint only: results do not depend on it. `next` must stay alive while it is
 * set. Errors: MOE_E_INVALID for a NULL layer or a layer on another device. */
moe_status moe_layer_set_next(moe_layer* layer, const moe_layer* next);

/* ---- router scoring ---------------------------------------------------------- */

/* How router logits become a selection and routing weights. */
enum {
    /* softmax top-k (the default): key_e = l_e + bias_e; the k largest keys
     * (ties to the lower index) are selected and weighted by the softmax of
     * their keys, renormalised over the selection. */
    MOE_SCORE_SOFTMAX = 0,
    /* sigmoid top-k, the DeepSeek-V3-style router of the Colibri README
     * ("What's implemented": sigmoid router, noaux_tc,
     * routed_scaling_factor): s_e = 1 / (1 + exp(-l_e)); key_e = s_e + bias_e,
     * the bias steering the selection only; the k largest keys (ties to the
     * lower index, all experts in one group) are selected and weighted by
     * w_j = routed_scaling * s_j / sum over the selection of s. */
    MOE_SCORE_SIGMOID = 1
};

/* Set the layer's router scoring (default MOE_SCORE_SOFTMAX, scaling 1).
 * routed_scaling must be finite and positive; it multiplies the sigmoid
 * weights and is ignored for softmax. The layer's router_bias (moe_layer_create)
 * is the bias_e above. Applies to every later moe_route, moe_decode,
 * moe_decode_static_scratch and moe_prefill_chunk call; set it before the
 * first of them (the call does not wait for work in flight). Errors:
 * MOE_E_INVALID for a NULL layer, an unknown scoring or a bad routed_scaling. */
moe_status moe_layer_set_router_scoring(moe_layer* layer, int32_t scoring, float routed_scaling);

/* ---- compute --------------------------------------------------------------- */

/* Router only, for T tokens (1 <= T <= max_tokens).
 *   x:   device [T][H] of act_dtype.
 *   ids: device int32 [T][top_k], selection order (descending key, ties to lower index).
 *   w:   device fp32 [T][top_k], the routing weights of the layer's scoring
 *        (moe_layer_set_router_scoring): softmax over the selected keys, or the
 *        scaled, renormalised sigmoid scores.
 * Router GEMV/GEMM with fp32 accumulation; selection and weights in fp32. */
moe_status moe_route(moe_layer* layer, const void* x, int32_t T, int32_t* ids, float* w, void* stream);

/* The expert selection of the last moe_route, moe_decode or moe_prefill_chunk
 * on this layer -- the one that call itself computed and combined with -- for
 * tokens 0..T-1 (T = 1 after moe_decode): ids device int32 [T][top_k] in
 * selection order, w device fp32 [T][top_k], both caller-owned. The copies are
 * enqueued on `stream` (order it after that call, e.g. the same stream).
 * Every call selects once per token (moe_decode in its router kernel's last
 * block, which the gate/up and down kernels then read; moe_prefill_chunk in
 * one block per token); moe_decode_static_scratch keeps its selection in the
 * static region and does not update this one. TurboFieldfare article, "token generation" (top-8 selection);
 * Inferno README, "Current Scope" (exact top-8). Errors: MOE_E_INVALID. */
moe_status moe_layer_selection(moe_layer* layer, int32_t T, int32_t* ids, float* w, void* stream);

/* One decode token.
 *   x:     device [H] of act_dtype.
 *   y:     device [H] of act_dtype (bf16 rounded to nearest even), may be NULL;
 *   y_f32: device fp32 [H] or NULL (at least one of y, y_f32 non-NULL).
 * Resident layers: no host synchronisation. Streamed layers: the host waits
 * (with a deadline) for the router's expert IDs, stages the misses on the
 * layer's copy stream while the shared expert runs, then runs the routed
 * experts (MOE_E_TIMEOUT / MOE_E_SOURCE / MOE_E_STATE on failure). */
moe_status moe_decode(moe_layer* layer, const void* x, void* y, float* y_f32, void* stream);

/* Largest scratch moe_decode_static_scratch can use on one device, in bytes. */
#define MOE_STATIC_SCRATCH_BYTES (256u * 1024u)

/* One decode token like moe_decode, with its scratch in a fixed region of the
 * library's own device image instead of the layer's scratch. The pages have no
 * counterpart to this call: it serves callers that must not allocate device
 * memory while they serve tokens. cudaMalloc and cudaFree can synchronise the
 * whole device and so stall work queued on every other stream; an engine that
 * has already divided HBM between weights, caches and activations has nothing
 * left to hand out; and a caching allocator asked for a new block at that
 * point may have to grow or trim its pool. This call makes no allocation of
 * any kind, by CUDA, by a library or by the binding above it.
 *
 * Arguments, layouts, result and errors are those of moe_decode, with these
 * differences:
 *   - The same three kernels run; the router's last block selects and gate/up
 *     waits for the router grid rather than polling tagged partials, and the
 *     down kernel reads the selection after its wait for gate/up. Streamed
 *     layers (cache_slots > 0) get MOE_E_UNSUPPORTED.
 *   - The scratch holds the router's partial logits [splits][E], the logits
 *     [E], ids [k], weights [k] and the SwiGLU outputs [k + 1][I] (each
 *     rounded up to 256 bytes). A layer that needs more than
 *     MOE_STATIC_SCRATCH_BYTES gets MOE_E_INVALID, with the sizes in
 *     moe_last_error(), before anything is launched.
 *   - The first call on a device does a one-time set-up with that device
 *     current: it looks up the region's device address, which may load the
 *     library's kernels onto the device. Make that first call before any
 *     stream capture begins on the device.
 *   - Nothing in the region has to start at zero: each call writes every word
 *     it later reads, so no clear is issued.
 *   - There is one region per device, shared by every layer and stream: two
 *     calls whose work overlaps on the device (other streams, other threads,
 *     other layers) overwrite each other's scratch. Order them, for example on
 *     one stream. */
moe_status moe_decode_static_scratch(moe_layer* layer, const void* x, void* y, float* y_f32, void* stream);

/* A prefill chunk of T tokens (1 <= T <= max_tokens), resident layers.
 *   x: device [T][H]; y: device [T][H] or NULL; y_f32: device fp32 [T][H] or NULL.
 * Row t equals moe_decode of token t up to rounding: the tokens are grouped by
 * expert (each distinct expert's weights read once per chunk), run through a
 * grouped GEMM on the tensor cores with fp16 operands (weights dequantised to
 * fp16 in shared memory, activations and SwiGLU outputs rounded to fp16) and
 * fp32 accumulation, and combined per token in a fixed order. fp16 rather than
 * bf16: its 11-bit significand keeps the chunk within the layer tolerance,
 * which bf16 operands do not. Activations and SwiGLU outputs must lie within
 * the fp16 range (|v| < 65504).
 * Streamed layers (cache_slots > 0) run the chunk as a batch union through the
 * cache (Colibri report section 2, "Union"): the chunk's distinct routed
 * experts are staged in waves, first those already resident, then the others
 * at most cache_slots at a time, and each wave's groups are computed from the
 * slots. Each wave is one moe_cache_stage (the host waits for the chunk's
 * routing, with the layer's deadline), so a failing source returns
 * MOE_E_SOURCE and a deadline MOE_E_TIMEOUT. The output equals that of the
 * same layer held resident, bit for bit. */
moe_status moe_prefill_chunk(moe_layer* layer, const void* x, int32_t T, void* y, float* y_f32,
                             void* stream);

/* T decode tokens from HOST buffers, one after another through moe_decode.
 *   x_host: [T][H] act_dtype; y_host: [T][H] act_dtype.
 * Copies the inputs to the device, runs the T decode steps and copies the
 * outputs back, all on `stream`, then waits for the stream. */
moe_status moe_decode_tokens_host(moe_layer* layer, const void* x_host, int32_t T, void* y_host,
                                  void* stream);

/* ---- streamed expert cache ------------------------------------------------- */

/* Make the given experts resident (streamed layers). ids: host int32 [n]
 * (n <= cache_slots, no repeats). Hits refresh the LFU counts; misses evict
 * the least-frequently-used resident not in `ids` and are copied host ->
 * device on the layer's copy stream; `stream` waits for those copies.
 * n_hits / n_misses may be NULL. */
moe_status moe_cache_stage(moe_layer* layer, const int32_t* ids, int32_t n, void* stream,
                           int32_t* n_hits, int32_t* n_misses);

/* Router lookahead (Colibri analysis report, caching and prefetch: the state
 * entering layer L, passed through the routing function of layer L + 1,
 * predicts that layer's experts one layer ahead, and the predicted weights are
 * loaded while layer L computes). Call it on the NEXT layer (streamed) with
 * the CURRENT layer's input x (device, [H] act_dtype), before running the
 * current layer. Once the work already queued on `stream` is done, the next
 * layer's router runs on x on the layer's copy stream. The host waits for the
 * predicted ids (the layer's deadline applies), then copies the predicted
 * experts that are not resident into slots on the copy stream. `stream` does
 * not wait for these copies; the layer's next moe_decode / moe_prefill_chunk
 * does.
 * Policy: a predicted expert is admitted with a use count of 0 (a later use
 * counts as a hit); residents keep their counts and recency; victims are
 * chosen as in moe_cache_stage, outside the prediction.
 * n_resident / n_fills (may be NULL): predicted experts already resident, and
 * copies issued. Errors: MOE_E_UNSUPPORTED on a resident layer, MOE_E_SOURCE
 * if the source fails (that expert is left out), MOE_E_TIMEOUT. */
moe_status moe_cache_prefetch(moe_layer* layer, const void* x, void* stream, int32_t* n_resident,
                              int32_t* n_fills);

/* Lookahead counters since creation: out4 = {calls, predicted experts already
 * resident, fills, bytes copied for fills}. Prefetch fills are not counted in
 * moe_cache_stats. */
moe_status moe_cache_prefetch_stats(const moe_layer* layer, uint64_t* out4);

/* Counters since creation. */
moe_status moe_cache_stats(const moe_layer* layer, moe_cache_stats_t* out);

/* Slot residency (streamed layers): slot_expert host int32 [cache_slots],
 * -1 for an empty slot. */
moe_status moe_cache_residency(const moe_layer* layer, int32_t* slot_expert);

/* The learning cache (Colibri README, "Self-learning cache": the engine records
 * which experts the usage routes to and pins the hottest in spare memory).
 *
 * moe_cache_usage: counts (host uint64 [n_experts]) of how often each expert was
 * selected on this streamed layer since creation: every decode token's ids and
 * every expert of every streamed-prefill wave; lookahead predictions do not
 * count. In device-managed mode it synchronises the device first.
 *
 * moe_cache_pin: replaces the set of pinned experts by experts[0..n) (host
 * int32, distinct, 0 <= id < n_experts; n = 0 unpins all). Pinned experts are
 * copied once into device memory beside the cache slots (n records more) and
 * stay resident: their lookups are hits that leave the LFU state alone. An
 * expert pinned while it held a slot frees the slot; an unpinned expert is not
 * resident until a token stages it. Not a token (the LFU clock stays). Copies
 * come from the borrowed records or the source callback. Synchronises the
 * device (slots move); MOE_E_INVALID for bad ids, MOE_E_STATE on a resident
 * layer, MOE_E_SOURCE / MOE_E_CUDA if a copy fails (the previous state is
 * kept). Choosing the set (e.g. the hottest by moe_cache_usage, ties to the
 * lower id) is the caller's. */
moe_status moe_cache_usage(const moe_layer* layer, uint64_t* counts);
moe_status moe_cache_pin(moe_layer* layer, const int32_t* experts, int32_t n);

/* The hottest experts by a usage count: out (host int32 [n]) receives the n
 * experts with the largest counts[e] (host uint64 [n_experts]), the lower id
 * first among equal counts. Host only, no device. MOE_E_INVALID for NULL
 * pointers or n outside 0..n_experts. */
moe_status moe_hottest(const uint64_t* counts, int32_t n_experts, int32_t n, int32_t* out);

/* The learning cache's step in one call: moe_cache_usage, then moe_cache_pin
 * of the n hottest experts by those counts (moe_hottest's order). The same
 * errors and synchronisation as the two calls. */
moe_status moe_cache_pin_hottest(moe_layer* layer, int32_t n);

/* The cache policy alone, on the host (no device, no layer): runs n_tokens
 * tokens of k distinct expert ids each (ids: host int32 [n_tokens][k], values
 * in 0..n_experts-1) through an empty `slots`-slot cache exactly as a streamed
 * layer's moe_cache_stage does, and writes per (token, slot j): hit[t][j] = 1
 * if the expert was resident before the token, and slot[t][j] = the slot that
 * holds it afterwards. Policy (TurboFieldfare article, "token generation",
 * with the readings the pages leave open): counts start at 1 on admission and
 * grow by one per use, the victim is the least-used resident the token does
 * not need (ties: least recently used, then lower id), a miss takes the lowest
 * free slot while there is one, hits are counted before misses. */
moe_status moe_lfu_trace(int32_t slots, int32_t n_experts, int32_t k, int32_t n_tokens, const int32_t* ids,
                         int32_t* slot, uint8_t* hit);

/* The same host-only run with the learning cache: experts pinned[0..n_pinned)
 * (distinct, in range) are pinned before the first token, as moe_cache_pin
 * does. A pinned expert is a hit that leaves the LFU state alone; its slot[t][j]
 * is slots + its index in `pinned` (where moe_cache_pin places it). usage
 * (nullable, uint64 [n_experts]) receives each expert's selection count, as
 * moe_cache_usage reports it. Colibri README, "Self-learning cache". */
moe_status moe_lfu_trace_pinned(int32_t slots, int32_t n_experts, int32_t k, int32_t n_tokens, const int32_t* ids,
                                const int32_t* pinned, int32_t n_pinned, int32_t* slot, uint8_t* hit,
                                uint64_t* usage);

/* ---- options and health ----------------------------------------------------------- */

/* moe_decode on a resident layer runs three kernels chained with programmatic
 * dependent launch: the router (partial logits over K-splits, each written
 * with the token's tag in one 64-bit word); gate/up + SwiGLU (computes the
 * shared expert's rows while the router runs, then every CTA polls the tagged
 * partials, selects the top k itself and computes its share of the routed
 * experts' rows; CTA 0 publishes the selection as tagged words); down +
 * combine (reads the published selection before its wait, then waits for
 * gate/up and computes the shared and routed experts' rows and the fixed-order
 * combine). Device-side polls are bounded (0.2 s) and fall back to the
 * ordinary dependency wait, recording MOE_E_TIMEOUT for moe_layer_check. */
enum {
    /* Test hook for failure detection: while nonzero, the decode kernels also
     * run an early start on the shared expert (gate/up counts its CTAs done
     * with the shared expert's rows; down computes them once all are counted),
     * and gate/up never counts, so the down kernel's bounded wait on the count
     * runs out (0.2 s), records MOE_E_TIMEOUT for moe_layer_check and computes
     * the shared expert after its ordinary wait instead (the output is
     * unchanged). */
    MOE_OPT_TEST_STALL_SHARED = 2,
    /* Phase tracing of the decode kernels and the prefill GEMMs: while
     * nonzero, every CTA records timestamps; read them with
     * moe_trace_read_split. Costs a few stores per CTA. */
    MOE_OPT_TRACE = 3,
    /* Deadline of every host-side wait of a streamed layer (expert ids coming
     * back, staging and table buffers free for reuse), in milliseconds
     * (default 30000); a wait that passes it returns MOE_E_TIMEOUT. */
    MOE_OPT_HOST_TIMEOUT_MS = 4,
    /* Test hook for failure detection on streamed layers: while nonzero, each
     * stage first holds the layer's copy stream for this many milliseconds (a
     * host callback that sleeps), so that a short MOE_OPT_HOST_TIMEOUT_MS runs
     * out on the host. No device work is involved. */
    MOE_OPT_TEST_STALL_COPIES_MS = 5,
    /* Device-managed cache of a streamed layer (0: off, the default; 1: on).
     * While on, moe_decode makes no host round trip: the router's selecting
     * block runs the LFU step (the same policy as host staging, on the same
     * state), a copy kernel moves the missing records from host memory into
     * their slots, reading them through their device mapping, and the expert
     * kernels follow; a decode can be captured in a CUDA graph. Needs borrowed
     * records (records != NULL at create) in page-locked host memory, 16-byte
     * aligned (else MOE_E_UNSUPPORTED / MOE_E_INVALID). Switching on waits for
     * the layer's host copies; switching off synchronises the device and
     * hands the state back to the host. While on, moe_cache_stage and
     * moe_cache_prefetch return MOE_E_STATE; a streamed moe_prefill_chunk
     * hands the state to the host for the chunk's staging waves and back after
     * it (synchronising the device twice);
     * moe_cache_stats and moe_cache_residency synchronise the device and
     * report the device state (stage_ns does not grow). A token whose ids
     * found no victim slot (impossible while top_k <= cache_slots) sets a bit
     * that moe_layer_check reports. TurboFieldfare article ("token
     * generation"): the 16-slot LFU cache and its misses loaded per token. */
    MOE_OPT_CACHE_DEVICE = 6
};

/* Traces of the last three-kernel decode and of the last prefill chunk's two
 * grouped GEMMs (while MOE_OPT_TRACE is on): out receives
 * MOE_TRACE_KERNELS * MOE_TRACE_MAX_CTAS * 4 uint64 values ordered kernel,
 * CTA, slot; 0 where a CTA or slot did not run. Waits for the device.
 *   kernels 0..2 (decode router, gate/up, down): global-timer stamps (ns) at
 *     start, dependency satisfied, main work done, end;
 *   kernels 3..4 (prefill gate/up GEMM, down GEMM): SM clock cycles spent
 *     waiting by the copy thread, by one dequantiser thread and by the MMA
 *     thread, then the CTA's total cycles.
 * cap must be at least MOE_TRACE_KERNELS * MOE_TRACE_MAX_CTAS * 4. */
#define MOE_TRACE_MAX_CTAS 1024
#define MOE_TRACE_KERNELS 5
moe_status moe_trace_read_split(moe_layer* layer, uint64_t* out, int32_t cap);

moe_status moe_layer_set_option(moe_layer* layer, int32_t option, int64_t value);

/* Wait for the layer's device work, then report device-side failures since
 * the last check: MOE_E_TIMEOUT if a bounded wait inside a kernel gave up
 * (bits, if non-NULL, receives the raw error bits), MOE_OK otherwise. The
 * error state is cleared. */
moe_status moe_layer_check(moe_layer* layer, uint32_t* bits);

/* ---- per-kernel timing ---------------------------------------------------------- */

/* Device time of one kernel kind, accumulated between moe_profile_start and
 * moe_profile_stop. `name` points to a static string of the library. */
typedef struct {
    const char* name;
    uint64_t launches;
    double total_ms;
} moe_kernel_time;

/* Start recording a CUDA event pair around every kernel the layer launches
 * (on the stream the kernel runs on), for at most `max_launches` launches;
 * later launches are not recorded. Costs one event record per kernel edge. */
moe_status moe_profile_start(moe_layer* layer, int32_t max_launches);

/* Stop recording, wait for the recorded events, and return per-kernel-kind
 * totals in `out` (host array of `cap` entries); *n_kinds receives the number
 * of kinds with at least one launch. */
moe_status moe_profile_stop(moe_layer* layer, moe_kernel_time* out, int32_t cap, int32_t* n_kinds);

/* ---- errors ----------------------------------------------------------------- */

const char* moe_status_str(moe_status s);
/* Detail of the last failure on the calling thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
