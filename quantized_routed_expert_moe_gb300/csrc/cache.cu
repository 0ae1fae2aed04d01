// Streamed expert cache: per-layer device slots holding the records of the
// experts used recently, managed least-frequently-used and filled from host
// memory by cudaMemcpyAsync on the layer's own copy stream.
//
// TurboFieldfare article ("token generation"): the router's expert IDs are
// matched against a per-layer 16-slot LFU cache and the misses are loaded,
// overlapped with the always-resident shared expert's compute. Inferno README
// ("Memory Strategy") keeps hot experts resident and streams the rest.
//
// Policy (the pages leave the details open; this is the reading the oracle's
// LFU simulation follows):
//   * an expert's count starts at 1 when it is admitted and grows by 1 on every
//     use while resident; the count is dropped on eviction;
//   * the victim is the resident expert with the smallest count that the
//     current token does not need; ties go to the least recently used, then to
//     the lower expert id;
//   * a token's IDs are processed in selection order, hits before misses, and
//     a miss takes the lowest free slot while there is one.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstring>
#include <thread>
#include <vector>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// LFU policy (host)
// ---------------------------------------------------------------------------

struct Fill {
    int expert, slot, victim;
};

class Lfu {
public:
    Lfu(int slots, int E)
        : slots_(slots), slot_of_(E, -1), expert_in_(slots, -1), count_(E, 0), last_(E, 0), pinned_(E, 0), usage_(E, 0) {}

    // One token's IDs (distinct, at most `slots`): updates the counts and
    // returns the fills (expert, slot, evicted expert or -1) in admission order.
    void access(const int32_t* ids, int n, int* hits, std::vector<Fill>& fills) {
        ++clock_;
        fills.clear();
        int h = 0;
        for (int i = 0; i < n; ++i) {
            const int e = ids[i];
            ++usage_[e];
            if (pinned_[e]) {   // served outside the slots; the LFU state stays
                ++h;
            } else if (slot_of_[e] >= 0) {
                ++h;
                ++count_[e];
                last_[e] = clock_;
            }
        }
        for (int i = 0; i < n; ++i) {
            const int e = ids[i];
            if (slot_of_[e] >= 0 || pinned_[e]) continue;
            int slot = -1, victim = -1;
            for (int s = 0; s < slots_; ++s)
                if (expert_in_[s] < 0) { slot = s; break; }
            if (slot < 0) {
                for (int s = 0; s < slots_; ++s) {
                    const int r = expert_in_[s];
                    bool needed = false;
                    for (int j = 0; j < n; ++j) needed |= (ids[j] == r);
                    if (needed) continue;
                    if (victim < 0 || count_[r] < count_[victim] ||
                        (count_[r] == count_[victim] &&
                         (last_[r] < last_[victim] || (last_[r] == last_[victim] && r < victim))))
                        victim = r;
                }
                slot = slot_of_[victim];
                drop(victim);
            }
            slot_of_[e] = slot;
            expert_in_[slot] = e;
            count_[e] = 1;
            last_[e] = clock_;
            fills.push_back({e, slot, victim});
        }
        *hits = h;
    }

    // A prediction (router lookahead): admits each predicted expert that is
    // not resident, with count 0 (it has not been used yet), and leaves the
    // residents' counts and recency alone. Victims as in access: the least
    // used resident outside the prediction, ties to the least recently used,
    // then the lower id.
    void prefetch(const int32_t* ids, int n, int* resident, std::vector<Fill>& fills) {
        ++clock_;
        fills.clear();
        int r0 = 0;
        for (int i = 0; i < n; ++i) r0 += slot_of_[ids[i]] >= 0 || pinned_[ids[i]];
        for (int i = 0; i < n; ++i) {
            const int e = ids[i];
            if (slot_of_[e] >= 0 || pinned_[e]) continue;
            int slot = -1, victim = -1;
            for (int s = 0; s < slots_; ++s)
                if (expert_in_[s] < 0) { slot = s; break; }
            if (slot < 0) {
                for (int s = 0; s < slots_; ++s) {
                    const int r = expert_in_[s];
                    bool predicted = false;
                    for (int j = 0; j < n; ++j) predicted |= (ids[j] == r);
                    if (predicted) continue;
                    if (victim < 0 || count_[r] < count_[victim] ||
                        (count_[r] == count_[victim] &&
                         (last_[r] < last_[victim] || (last_[r] == last_[victim] && r < victim))))
                        victim = r;
                }
                if (victim < 0) break;   // every slot holds a predicted expert
                slot = slot_of_[victim];
                drop(victim);
            }
            slot_of_[e] = slot;
            expert_in_[slot] = e;
            count_[e] = 0;
            last_[e] = clock_;
            fills.push_back({e, slot, victim});
        }
        *resident = r0;
    }

    // Forget a resident expert (eviction, or a fill that failed).
    void drop(int e) {
        if (slot_of_[e] < 0) return;
        expert_in_[slot_of_[e]] = -1;
        slot_of_[e] = -1;
        count_[e] = 0;
        last_[e] = 0;
    }

    // The learning cache (Colibri README, "Self-learning cache"): a new set
    // of pinned experts, resident outside the slots. An expert pinned while it
    // holds a slot leaves the slot; an unpinned one is not resident until a
    // token stages it. Not a token: the clock stays.
    void pin(const int32_t* ids, int n) {
        std::fill(pinned_.begin(), pinned_.end(), 0);
        for (int i = 0; i < n; ++i) {
            drop(ids[i]);
            pinned_[ids[i]] = 1;
        }
    }
    bool pinned(int e) const { return pinned_[e] != 0; }
    // selections of each expert so far (tokens and prefill waves; not predictions)
    uint64_t usage(int e) const { return usage_[e]; }
    void add_usage(int e, uint64_t v) { usage_[e] += v; }

    int slot_of(int e) const { return slot_of_[e]; }
    int expert_in(int s) const { return expert_in_[s]; }
    uint64_t count(int e) const { return count_[e]; }
    uint64_t last(int e) const { return last_[e]; }
    uint64_t clock() const { return clock_; }

    // Replace the state by a per-slot one (the device-managed cache's).
    void load(const int32_t* expert_in, const uint32_t* count, const uint32_t* last, uint64_t clock) {
        std::fill(slot_of_.begin(), slot_of_.end(), -1);
        std::fill(count_.begin(), count_.end(), 0);
        std::fill(last_.begin(), last_.end(), 0);
        for (int s = 0; s < slots_; ++s) {
            expert_in_[s] = expert_in[s];
            if (expert_in[s] < 0) continue;
            slot_of_[expert_in[s]] = s;
            count_[expert_in[s]] = count[s];
            last_[expert_in[s]] = last[s];
        }
        clock_ = clock;
    }

private:
    int slots_;
    uint64_t clock_ = 0;
    std::vector<int> slot_of_, expert_in_;
    std::vector<uint64_t> count_, last_;
    std::vector<char> pinned_;
    std::vector<uint64_t> usage_;
};

// ---------------------------------------------------------------------------
// cache state
// ---------------------------------------------------------------------------

struct CacheState {
    int slots = 0;
    uint8_t* dev_slots = nullptr;             // [slots][rec_bytes]
    Lfu lfu{1, 1};
    const void* const* records = nullptr;     // borrowed host records, or null
    std::vector<const void*> records_copy;    // the caller's pointer array, copied
    moe_expert_source src = nullptr;
    void* user = nullptr;
    uint8_t* staging[2] = {nullptr, nullptr}; // pinned, for the source path
    cudaEvent_t staging_ev[2] = {nullptr, nullptr};
    int staging_idx = 0;
    const uint8_t** tab_pinned[2] = {nullptr, nullptr};   // record table upload buffers
    cudaEvent_t tab_ev[2] = {nullptr, nullptr};
    int tab_idx = 0;
    std::vector<const uint8_t*> table;        // host copy of the device record table [E + 1]
    int32_t* ids_host = nullptr;              // pinned [top_k]
    cudaEvent_t ids_ready = nullptr, stream_mark = nullptr, copies_done = nullptr;
    cudaStream_t copy = nullptr;
    moe_cache_stats_t stats{};
    std::vector<Fill> fills;
    uint64_t pf_calls = 0, pf_resident = 0, pf_fills = 0, pf_bytes = 0;   // router lookahead
    bool copies_pending = false;   // copies (lookahead fills) the caller's stream has not waited for
    // the router's selection published into host-mapped memory: ids, then a
    // sequence number the host polls (speculative decode)
    int32_t* pub_ids = nullptr;    // host view [top_k]
    unsigned* pub_seq = nullptr;   // host view [1]
    int32_t* pub_ids_dev = nullptr;
    unsigned* pub_seq_dev = nullptr;
    unsigned seq = 0;
    // device-managed mode (MOE_OPT_CACHE_DEVICE): the LFU state lives in
    // dev_state, the host copies above are stale until the mode is left
    bool device = false;
    void* dev_state = nullptr;
    DevCacheArgs dca;
    // pinned experts: pinned[i] lives at dev_slots + (slots + i) * rec_bytes
    std::vector<int32_t> pinned;
    std::vector<int32_t> pin_index;   // [E] index into pinned, or -1
};

namespace {

using clk = std::chrono::steady_clock;

// Host wait for `ev` with the layer's deadline (MOE_OPT_HOST_TIMEOUT_MS).
moe_status wait_event(const Layer& L, cudaEvent_t ev, const char* what) {
    const auto t0 = clk::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return MOE_OK;
        if (e != cudaErrorNotReady) return cuda_fail(e, what);
        const auto waited = clk::now() - t0;
        if (waited > std::chrono::milliseconds(L.host_timeout_ms))
            return fail(MOE_E_TIMEOUT, std::string(what) + ": host wait passed its deadline");
        // a decode token's round trip is tens of microseconds: spin first,
        // then give the core back
        if (waited > std::chrono::milliseconds(2)) std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

// Host wait until the router has published sequence number `want` into
// host-mapped memory (deadline as for events); then the ids are visible.
moe_status wait_published(const Layer& L, const volatile unsigned* seq, unsigned want) {
    const auto t0 = clk::now();
    for (;;) {
        if (*seq == want) {
            std::atomic_thread_fence(std::memory_order_acquire);
            return MOE_OK;
        }
        const auto waited = clk::now() - t0;
        if (waited > std::chrono::milliseconds(L.host_timeout_ms))
            return fail(MOE_E_TIMEOUT, "expert ids: host wait passed its deadline");
        if (waited > std::chrono::milliseconds(2)) {
            // a failed launch never publishes: report it instead of waiting out the deadline
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e, "expert ids");
            std::this_thread::sleep_for(std::chrono::microseconds(50));
        }
    }
}

void CUDART_CB sleep_host(void* ms) {
    std::this_thread::sleep_for(std::chrono::milliseconds((intptr_t)ms));
}

}  // namespace

moe_status cache_create(Layer& L, const void* const* records, moe_expert_source src, void* user) {
    const auto& d = L.d;
    CacheState* C = new (std::nothrow) CacheState();
    if (!C) return fail(MOE_E_NOMEM, "host allocation failed");
    L.cache = C;
    C->slots = d.cache_slots;
    C->lfu = Lfu(d.cache_slots, d.n_experts);
    C->pin_index.assign(d.n_experts, -1);
    if (records) {
        C->records_copy.assign(records, records + d.n_experts);
        for (int e = 0; e < d.n_experts; ++e)
            if (!C->records_copy[e]) return fail(MOE_E_INVALID, "records[" + std::to_string(e) + "] is NULL");
        C->records = C->records_copy.data();
    }
    C->src = src;
    C->user = user;
    const size_t rb = L.rec_bytes;
    MOE_CUDA_TRY(cudaMalloc(&C->dev_slots, (size_t)C->slots * rb));
    L.device_bytes += (size_t)C->slots * rb;
    MOE_CUDA_TRY(cudaStreamCreateWithFlags(&C->copy, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&C->tab_ev[i], cudaEventDisableTiming));
        MOE_CUDA_TRY(cudaHostAlloc(&C->tab_pinned[i], (size_t)(d.n_experts + 1) * sizeof(void*), cudaHostAllocDefault));
        if (!records) {
            MOE_CUDA_TRY(cudaHostAlloc(&C->staging[i], rb, cudaHostAllocDefault));
            MOE_CUDA_TRY(cudaEventCreateWithFlags(&C->staging_ev[i], cudaEventDisableTiming));
        }
    }
    MOE_CUDA_TRY(cudaHostAlloc(&C->ids_host, (size_t)d.top_k * 4, cudaHostAllocDefault));
    MOE_CUDA_TRY(cudaHostAlloc(&C->pub_ids, (size_t)d.top_k * 4, cudaHostAllocMapped));
    MOE_CUDA_TRY(cudaHostAlloc(&C->pub_seq, 64, cudaHostAllocMapped));
    *C->pub_seq = 0;
    MOE_CUDA_TRY(cudaHostGetDevicePointer((void**)&C->pub_ids_dev, C->pub_ids, 0));
    MOE_CUDA_TRY(cudaHostGetDevicePointer((void**)&C->pub_seq_dev, C->pub_seq, 0));
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&C->ids_ready, cudaEventDisableTiming));
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&C->stream_mark, cudaEventDisableTiming));
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&C->copies_done, cudaEventDisableTiming));
    // the record table as create left it: no routed expert resident, the
    // shared expert (index E) in device memory
    C->table.assign(d.n_experts + 1, nullptr);
    MOE_CUDA_TRY(cudaMemcpy(C->table.data(), L.rec_table, C->table.size() * sizeof(void*), cudaMemcpyDeviceToHost));
    for (int e = 0; e < d.n_experts; ++e) C->table[e] = nullptr;
    return MOE_OK;
}

void cache_destroy(Layer& L) {
    CacheState* C = L.cache;
    if (!C) return;
    if (C->copy) cudaStreamSynchronize(C->copy);
    for (int i = 0; i < 2; ++i) {
        if (C->staging[i]) cudaFreeHost(C->staging[i]);
        if (C->staging_ev[i]) cudaEventDestroy(C->staging_ev[i]);
        if (C->tab_pinned[i]) cudaFreeHost(C->tab_pinned[i]);
        if (C->tab_ev[i]) cudaEventDestroy(C->tab_ev[i]);
    }
    if (C->ids_host) cudaFreeHost(C->ids_host);
    if (C->pub_ids) cudaFreeHost(C->pub_ids);
    if (C->pub_seq) cudaFreeHost(C->pub_seq);
    if (C->ids_ready) cudaEventDestroy(C->ids_ready);
    if (C->stream_mark) cudaEventDestroy(C->stream_mark);
    if (C->copies_done) cudaEventDestroy(C->copies_done);
    if (C->copy) cudaStreamDestroy(C->copy);
    if (C->dev_slots) cudaFree(C->dev_slots);
    if (C->dev_state) cudaFree(C->dev_state);
    delete C;
    L.cache = nullptr;
}

moe_status fill_slots(Layer& L, int& filled, bool prefetch);

moe_status cache_stage(Layer& L, const int32_t* ids, int n, cudaStream_t s, int* hits, int* misses) {
    CacheState& C = *L.cache;
    const auto& d = L.d;
    if (C.device) return fail(MOE_E_STATE, "the cache is device-managed (MOE_OPT_CACHE_DEVICE): host staging is off");
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= d.n_experts) return fail(MOE_E_INVALID, "expert id out of range");
        for (int j = 0; j < i; ++j)
            if (ids[j] == ids[i]) return fail(MOE_E_INVALID, "repeated expert id");
    }
    const auto t0 = clk::now();
    // the record-table upload buffer used now must be free before anything
    // changes, so that a timeout leaves the cache as it was
    {
        const moe_status sw = wait_event(L, C.tab_ev[C.tab_idx], "record table buffer reuse");
        if (sw != MOE_OK) return sw;
    }
    int h = 0;
    C.lfu.access(ids, n, &h, C.fills);
    if (C.fills.empty() && !C.copies_pending) {
        // every expert resident and no copy in flight: the slots and the
        // record table already hold what the kernels read
        C.stats.tokens += 1;
        C.stats.hits += (uint64_t)h;
        C.stats.stage_ns += (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(clk::now() - t0).count();
        if (hits) *hits = h;
        if (misses) *misses = 0;
        return MOE_OK;
    }
    // work already queued on `s` may still read the slots that are about to be refilled
    MOE_CUDA_TRY(cudaEventRecord(C.stream_mark, s));
    MOE_CUDA_TRY(cudaStreamWaitEvent(C.copy, C.stream_mark, 0));
    if (L.test_stall_copies_ms > 0)
        MOE_CUDA_TRY(cudaLaunchHostFunc(C.copy, sleep_host, (void*)(intptr_t)L.test_stall_copies_ms));
    int filled = 0;
    moe_status st = fill_slots(L, filled, false);
    // publish the record table (double-buffered pinned upload)
    {
        const int b = C.tab_idx;   // free: waited for above
        std::memcpy(C.tab_pinned[b], C.table.data(), C.table.size() * sizeof(void*));
        MOE_CUDA_TRY(cudaMemcpyAsync(L.rec_table, C.tab_pinned[b], C.table.size() * sizeof(void*),
                                     cudaMemcpyHostToDevice, C.copy));
        MOE_CUDA_TRY(cudaEventRecord(C.tab_ev[b], C.copy));
        C.tab_idx ^= 1;
    }
    MOE_CUDA_TRY(cudaEventRecord(C.copies_done, C.copy));
    MOE_CUDA_TRY(cudaStreamWaitEvent(s, C.copies_done, 0));
    C.copies_pending = false;
    C.stats.tokens += 1;
    C.stats.hits += (uint64_t)h;
    C.stats.misses += (uint64_t)C.fills.size();
    C.stats.stage_ns += (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(clk::now() - t0).count();
    if (hits) *hits = h;
    if (misses) *misses = (int)C.fills.size();
    return st;
}

// The copies of C.fills on the copy stream (the slots' previous readers are
// already ordered before them); a failing fill leaves its expert, and the
// ones after it, out of the cache.
moe_status fill_slots(Layer& L, int& filled, bool prefetch) {
    CacheState& C = *L.cache;
    const size_t rb = L.rec_bytes;
    moe_status st = MOE_OK;
    for (const Fill& f : C.fills) {
        uint8_t* dst = C.dev_slots + (size_t)f.slot * rb;
        if (f.victim >= 0) C.table[f.victim] = nullptr;
        C.table[f.expert] = nullptr;
        if (st != MOE_OK) {   // an earlier fill of this token failed: admit nothing more
            C.lfu.drop(f.expert);
            continue;
        }
        const void* src = nullptr;
        if (C.records) {
            src = C.records[f.expert];
        } else {
            const int b = C.staging_idx;
            st = wait_event(L, C.staging_ev[b], "staging buffer reuse");
            if (st == MOE_OK && C.src(C.user, f.expert, C.staging[b], rb) != 0)
                st = fail(MOE_E_SOURCE, "expert source failed for expert " + std::to_string(f.expert));
            if (st != MOE_OK) {
                C.lfu.drop(f.expert);
                continue;
            }
            src = C.staging[b];
            C.staging_idx ^= 1;
        }
        const cudaError_t ce = cudaMemcpyAsync(dst, src, rb, cudaMemcpyHostToDevice, C.copy);
        if (ce != cudaSuccess) {
            st = cuda_fail(ce, "expert fill copy");
            C.lfu.drop(f.expert);
            continue;
        }
        if (!C.records) MOE_CUDA_TRY(cudaEventRecord(C.staging_ev[C.staging_idx ^ 1], C.copy));
        C.table[f.expert] = dst;
        (prefetch ? C.pf_bytes : C.stats.bytes_h2d) += rb;
        ++filled;
    }
    return st;
}

// Router lookahead (Colibri analysis report, caching and prefetch: the state
// entering layer L, passed through the router of layer L + 1, predicts that
// layer's experts one layer ahead, and the predicted weights are loaded while
// layer L computes). On this (next) layer: its router runs on `x` on the copy
// stream once the work queued on `s` so far is done, the predicted ids come
// back to the host, and the predicted experts that are not resident are
// copied into slots on the copy stream. `s` does not wait for those copies;
// the layer's next stage (its next decode or prefill chunk) does.
moe_status cache_prefetch(Layer& L, const void* x, cudaStream_t s, int* resident, int* fills) {
    CacheState& C = *L.cache;
    const int k = L.d.top_k;
    if (C.device) return fail(MOE_E_STATE, "the cache is device-managed (MOE_OPT_CACHE_DEVICE): host staging is off");
    {
        const moe_status sw = wait_event(L, C.tab_ev[C.tab_idx], "record table buffer reuse");
        if (sw != MOE_OK) return sw;
    }
    MOE_CUDA_TRY(cudaEventRecord(C.stream_mark, s));
    MOE_CUDA_TRY(cudaStreamWaitEvent(C.copy, C.stream_mark, 0));
    cudaError_t e = launch_route_decode(L, x, C.copy, 1);
    if (e != cudaSuccess) return cuda_fail(e, "lookahead router launch");
    MOE_CUDA_TRY(cudaMemcpyAsync(C.ids_host, L.ids, (size_t)k * 4, cudaMemcpyDeviceToHost, C.copy));
    MOE_CUDA_TRY(cudaEventRecord(C.ids_ready, C.copy));
    moe_status st = wait_event(L, C.ids_ready, "predicted expert ids");
    if (st != MOE_OK) return st;
    int r = 0, filled = 0;
    C.lfu.prefetch(C.ids_host, k, &r, C.fills);
    st = fill_slots(L, filled, true);
    if (!C.fills.empty()) {
        const int b = C.tab_idx;
        std::memcpy(C.tab_pinned[b], C.table.data(), C.table.size() * sizeof(void*));
        MOE_CUDA_TRY(cudaMemcpyAsync(L.rec_table, C.tab_pinned[b], C.table.size() * sizeof(void*),
                                     cudaMemcpyHostToDevice, C.copy));
        MOE_CUDA_TRY(cudaEventRecord(C.tab_ev[b], C.copy));
        C.tab_idx ^= 1;
        C.copies_pending = true;
    }
    C.pf_calls += 1;
    C.pf_resident += (uint64_t)r;
    C.pf_fills += (uint64_t)filled;
    if (resident) *resident = r;
    if (fills) *fills = (int)C.fills.size();
    return st;
}

int cache_slot_of(const Layer& L, int expert) {
    const CacheState& C = *L.cache;
    const int p = C.pin_index[expert];
    return p >= 0 ? C.slots + p : C.lfu.slot_of(expert);
}

const uint8_t* cache_slots_base(const Layer& L) { return L.cache->dev_slots; }

int cache_slot_count(const Layer& L) { return L.cache->slots + (int)L.cache->pinned.size(); }

moe_status host_wait_event(const Layer& L, cudaEvent_t ev, const char* what) { return wait_event(L, ev, what); }

// ---------------------------------------------------------------------------
// device-managed mode
// ---------------------------------------------------------------------------

constexpr int kFillThreads = 256;

// Copy the records the router's LFU step admitted (fills: n, then (expert,
// slot) pairs) from host memory, read through its device mapping, into their
// slots: each thread moves 16-byte units, 8 in flight. Nothing to do on an
// all-hit token.
__global__ void __launch_bounds__(kFillThreads) k_cache_fill(const int32_t* fills, const uint8_t* const* src,
                                                             uint8_t* slots, unsigned long long rb) {
    pdl_wait();      // the router's LFU step is complete
    pdl_trigger();
    const int n = fills[0];
    const size_t units = rb / 16, stride = (size_t)gridDim.x * blockDim.x;
    for (int f = 0; f < n; ++f) {
        const uint4* from = reinterpret_cast<const uint4*>(src[fills[1 + 2 * f]]);
        uint4* to = reinterpret_cast<uint4*>(slots + (size_t)fills[2 + 2 * f] * rb);
        for (size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < units; i0 += 8 * stride) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const size_t i = i0 + u * stride;
                if (i < units) v[u] = from[i];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const size_t i = i0 + u * stride;
                if (i < units) to[i] = v[u];
            }
        }
    }
}

bool cache_is_device(const Layer& L) { return L.cache && L.cache->device; }

// On: the host LFU state goes to the device (after any host copies in flight
// have landed), and every decode runs its LFU step and fills on the device.
// Off: the device state comes back (after the device is idle) and host staging
// resumes from it. Needs borrowed records in page-locked host memory, 16-byte
// aligned: a source callback cannot run on the device.
moe_status cache_set_device(Layer& L, bool on) {
    CacheState& C = *L.cache;
    const int E = L.d.n_experts, S = C.slots;
    if (on == C.device) return MOE_OK;
    if (on) {
        if (!C.records)
            return fail(MOE_E_UNSUPPORTED, "a device-managed cache needs borrowed host records, not a source callback");
        if (L.rec_bytes % 16) return fail(MOE_E_UNSUPPORTED, "record size is not a multiple of 16 bytes");
        std::vector<const uint8_t*> src(E);
        for (int e = 0; e < E; ++e) {
            void* p = nullptr;
            if (cudaHostGetDevicePointer(&p, const_cast<void*>(C.records[e]), 0) != cudaSuccess) {
                cudaGetLastError();
                return fail(MOE_E_UNSUPPORTED, "record " + std::to_string(e) +
                                                   " is not in page-locked host memory the device can read");
            }
            if (reinterpret_cast<uintptr_t>(p) % 16)
                return fail(MOE_E_INVALID, "record " + std::to_string(e) + " is not 16-byte aligned");
            src[e] = static_cast<const uint8_t*>(p);
        }
        if (!C.dev_state) {
            // slot_expert, slot_count, slot_last [S] | clock | fills [1 + 2 MOE_MAX_TOP_K] | stats [4] (8-aligned)
            // | src [E] | usage [E] | pinned flags [E]
            const size_t words = 3 * (size_t)S + 1 + 1 + 2 * MOE_MAX_TOP_K;
            const size_t stats_off = (words * 4 + 7) / 8 * 8, src_off = stats_off + 4 * 8;
            const size_t usage_off = src_off + (size_t)E * sizeof(void*), pin_off = usage_off + (size_t)E * 8;
            MOE_CUDA_TRY(cudaMalloc(&C.dev_state, pin_off + (size_t)E));
            uint8_t* b = static_cast<uint8_t*>(C.dev_state);
            C.dca.slot_expert = reinterpret_cast<int32_t*>(b);
            C.dca.slot_count = reinterpret_cast<uint32_t*>(b) + S;
            C.dca.slot_last = reinterpret_cast<uint32_t*>(b) + 2 * S;
            C.dca.clock = reinterpret_cast<uint32_t*>(b) + 3 * S;
            C.dca.fills = reinterpret_cast<int32_t*>(b) + 3 * S + 1;
            C.dca.stats = reinterpret_cast<unsigned long long*>(b + stats_off);
            C.dca.src = reinterpret_cast<const uint8_t* const*>(b + src_off);
            C.dca.usage = reinterpret_cast<unsigned long long*>(b + usage_off);
            C.dca.pinned = b + pin_off;
            C.dca.rec_table = (const uint8_t**)L.rec_table;
            C.dca.rb = L.rec_bytes;
            C.dca.slots = S;
            C.dca.err = error_word(L);
        }
        // host copies (lookahead fills, table uploads) land first
        MOE_CUDA_TRY(cudaStreamSynchronize(C.copy));
        C.copies_pending = false;
        std::vector<int32_t> se(S);
        std::vector<uint32_t> cnt(S), last(S);
        for (int s = 0; s < S; ++s) {
            se[s] = C.lfu.expert_in(s);
            cnt[s] = se[s] < 0 ? 0u : (uint32_t)C.lfu.count(se[s]);
            last[s] = se[s] < 0 ? 0u : (uint32_t)C.lfu.last(se[s]);
        }
        const uint32_t clk = (uint32_t)C.lfu.clock();
        const int32_t zero_fills = 0;
        const unsigned long long zero_stats[4] = {0, 0, 0, 0};
        MOE_CUDA_TRY(cudaMemcpy(C.dca.slot_expert, se.data(), S * 4, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemcpy(C.dca.slot_count, cnt.data(), S * 4, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemcpy(C.dca.slot_last, last.data(), S * 4, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemcpy(C.dca.clock, &clk, 4, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemcpy(C.dca.fills, &zero_fills, 4, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemcpy(C.dca.stats, zero_stats, sizeof zero_stats, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemcpy((void*)C.dca.src, src.data(), (size_t)E * sizeof(void*), cudaMemcpyHostToDevice));
        std::vector<uint8_t> pin(E);
        for (int e = 0; e < E; ++e) pin[e] = C.lfu.pinned(e) ? 1 : 0;
        MOE_CUDA_TRY(cudaMemcpy((void*)C.dca.pinned, pin.data(), (size_t)E, cudaMemcpyHostToDevice));
        MOE_CUDA_TRY(cudaMemset(C.dca.usage, 0, (size_t)E * 8));
        C.dca.slots_base = C.dev_slots;   // the slots may have moved (pinning)
        C.device = true;
        return MOE_OK;
    }
    // off: every decode already queued has run
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    std::vector<int32_t> se(S);
    std::vector<uint32_t> cnt(S), last(S);
    uint32_t clk = 0;
    unsigned long long st[4];
    MOE_CUDA_TRY(cudaMemcpy(se.data(), C.dca.slot_expert, S * 4, cudaMemcpyDeviceToHost));
    MOE_CUDA_TRY(cudaMemcpy(cnt.data(), C.dca.slot_count, S * 4, cudaMemcpyDeviceToHost));
    MOE_CUDA_TRY(cudaMemcpy(last.data(), C.dca.slot_last, S * 4, cudaMemcpyDeviceToHost));
    MOE_CUDA_TRY(cudaMemcpy(&clk, C.dca.clock, 4, cudaMemcpyDeviceToHost));
    MOE_CUDA_TRY(cudaMemcpy(st, C.dca.stats, sizeof st, cudaMemcpyDeviceToHost));
    std::vector<unsigned long long> use(E);
    MOE_CUDA_TRY(cudaMemcpy(use.data(), C.dca.usage, (size_t)E * 8, cudaMemcpyDeviceToHost));
    C.lfu.load(se.data(), cnt.data(), last.data(), clk);
    for (int e = 0; e < E; ++e) C.lfu.add_usage(e, use[e]);
    C.stats.tokens += st[0];
    C.stats.hits += st[1];
    C.stats.misses += st[2];
    C.stats.bytes_h2d += st[3];
    // the host mirror of the record table (the device's already matches):
    // LFU residents and pinned experts
    for (int e = 0; e < E; ++e) {
        const int sl = cache_slot_of(L, e);
        C.table[e] = sl < 0 ? nullptr : C.dev_slots + (size_t)sl * L.rec_bytes;
    }
    C.device = false;
    return MOE_OK;
}

// The learning cache (Colibri README, "Self-learning cache": the engine records
// which experts the usage routes to and pins the hottest in spare memory).
// A new pinned set: the records are copied into a slot array that now holds
// the LFU slots followed by the pinned experts, the record table points at
// them, and the LFU forgets them (an expert pinned while it held a slot frees
// the slot). Synchronises the device; a failed copy leaves everything as it was.
moe_status cache_pin(Layer& L, const int32_t* ids, int n) {
    CacheState& C = *L.cache;
    const int E = L.d.n_experts, S = C.slots;
    const size_t rb = L.rec_bytes;
    if (n < 0 || n > E) return fail(MOE_E_INVALID, "n out of range 0..n_experts");
    if (n > 0 && !ids) return fail(MOE_E_INVALID, "NULL ids");
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return fail(MOE_E_INVALID, "expert id out of range");
        for (int j = 0; j < i; ++j)
            if (ids[j] == ids[i]) return fail(MOE_E_INVALID, "repeated expert id");
    }
    const bool was_device = C.device;
    if (was_device) {
        const moe_status st = cache_set_device(L, false);
        if (st != MOE_OK) return st;
    }
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    MOE_CUDA_TRY(cudaStreamSynchronize(C.copy));
    C.copies_pending = false;
    uint8_t* nb = nullptr;
    MOE_CUDA_TRY(cudaMalloc(&nb, (size_t)(S + n) * rb));
    moe_status st = MOE_OK;
    cudaError_t ce = cudaMemcpy(nb, C.dev_slots, (size_t)S * rb, cudaMemcpyDeviceToDevice);
    if (ce != cudaSuccess) st = cuda_fail(ce, "slot move");
    for (int i = 0; i < n && st == MOE_OK; ++i) {
        const void* src = nullptr;
        if (C.records) {
            src = C.records[ids[i]];
        } else if (C.src(C.user, ids[i], C.staging[0], rb) != 0) {
            st = fail(MOE_E_SOURCE, "expert source failed for expert " + std::to_string(ids[i]));
            break;
        } else {
            src = C.staging[0];
        }
        ce = cudaMemcpy(nb + (size_t)(S + i) * rb, src, rb, cudaMemcpyHostToDevice);
        if (ce != cudaSuccess) st = cuda_fail(ce, "pinned expert copy");
    }
    if (st != MOE_OK) {
        cudaFree(nb);
        if (was_device) cache_set_device(L, true);
        return st;
    }
    C.lfu.pin(ids, n);
    cudaFree(C.dev_slots);
    L.device_bytes = L.device_bytes - (size_t)(S + C.pinned.size()) * rb + (size_t)(S + n) * rb;
    C.dev_slots = nb;
    C.pinned.assign(ids, ids + n);
    std::fill(C.pin_index.begin(), C.pin_index.end(), -1);
    for (int i = 0; i < n; ++i) C.pin_index[ids[i]] = i;
    // the record table: LFU residents, then pinned experts (the shared expert's entry stays)
    for (int e = 0; e < E; ++e) {
        const int sl = cache_slot_of(L, e);
        C.table[e] = sl < 0 ? nullptr : nb + (size_t)sl * rb;
    }
    MOE_CUDA_TRY(cudaMemcpy(L.rec_table, C.table.data(), C.table.size() * sizeof(void*), cudaMemcpyHostToDevice));
    st = prefill_cache_maps(L);
    if (st != MOE_OK) return st;
    if (was_device) return cache_set_device(L, true);
    return MOE_OK;
}

moe_status cache_decode(Layer& L, const void* x, void* y, float* y_f32, cudaStream_t s) {
    CacheState& C = *L.cache;
    const auto& d = L.d;
    const int k = d.top_k;
    const int jj0 = d.n_shared ? 1 : 0;
    if (C.device) {
        // no host step: the router's selecting block runs the LFU step, the
        // fill kernel copies the misses, the experts read the updated table
        cudaError_t e = launch_route_decode(L, x, s, 1, nullptr, nullptr, 0, &C.dca);
        if (e != cudaSuccess) return cuda_fail(e, "router launch");
        prof_begin(L, K_CACHE_FILL, s);
        e = launch_pdl(k_cache_fill, dim3(2 * L.num_sms), dim3(kFillThreads), 0, s, L.pdl,
                       (const int32_t*)C.dca.fills, C.dca.src, C.dca.slots_base, (unsigned long long)L.rec_bytes);
        prof_end(L, s);
        if (e != cudaSuccess) return cuda_fail(e, "cache fill launch");
        e = launch_experts_decode_sel(L, x, y, y_f32, 0, jj0 + k, true, s, true);
        if (e != cudaSuccess) return cuda_fail(e, "expert launch");
        return MOE_OK;
    }
    // Speculative launch: every expert (shared and routed) runs right after
    // the router, from the record table as it stands. If the token needs an
    // expert that is not resident, its record is null there and the kernels do
    // nothing; the host then stages and launches again. With every expert
    // resident (the common case) the host's wait for the ids overlaps the
    // experts' compute. The router publishes the ids straight into
    // host-mapped memory, so no copy sits between it and the experts. Not
    // while a lookahead's copies are in flight (their slots are not ready
    // yet): then the shared expert's gate/up alone runs while the host stages.
    const bool spec = !C.copies_pending && L.test_stall_copies_ms == 0;
    const unsigned want = ++C.seq;
    cudaError_t e = spec ? launch_route_decode(L, x, s, 1, C.pub_ids_dev, C.pub_seq_dev, want)
                         : launch_route_decode(L, x, s, 1);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");
    moe_status st = MOE_OK;
    if (spec) {
        e = launch_experts_decode_sel(L, x, y, y_f32, 0, jj0 + k, true, s);
        if (e != cudaSuccess) return cuda_fail(e, "expert launch");
        st = wait_published(L, C.pub_seq, want);
        if (st != MOE_OK) return st;
        for (int j = 0; j < k; ++j) C.ids_host[j] = ((volatile int32_t*)C.pub_ids)[j];
    } else {
        if (d.n_shared) {
            e = launch_experts_decode_sel(L, x, y, y_f32, 0, 1, false, s);
            if (e != cudaSuccess) return cuda_fail(e, "shared expert launch");
        }
        MOE_CUDA_TRY(cudaMemcpyAsync(C.ids_host, L.ids, (size_t)k * 4, cudaMemcpyDeviceToHost, s));
        MOE_CUDA_TRY(cudaEventRecord(C.ids_ready, s));
        st = wait_event(L, C.ids_ready, "expert ids");
        if (st != MOE_OK) return st;
    }
    int h = 0, m = 0;
    st = cache_stage(L, C.ids_host, k, s, &h, &m);
    if (st != MOE_OK) return st;
    for (int j = 0; j < k; ++j)
        if (cache_slot_of(L, C.ids_host[j]) < 0)
            return fail(MOE_E_STATE, "expert " + std::to_string(C.ids_host[j]) + " is not resident");
    if (spec && m == 0) return MOE_OK;   // the speculative launch had every expert
    // after a speculative launch that met a miss every slot runs again;
    // otherwise the shared expert's gate/up has run already
    e = launch_experts_decode_sel(L, x, y, y_f32, spec ? 0 : jj0, jj0 + k, true, s);
    if (e != cudaSuccess) return cuda_fail(e, "routed expert launch");
    return MOE_OK;
}

}  // namespace moe

extern "C" {

moe_status moe_cache_prefetch(moe_layer* layer, const void* x, void* stream, int32_t* n_resident,
                              int32_t* n_fills) {
    if (!layer || !x) return moe::fail(MOE_E_INVALID, "NULL argument");
    moe::Layer& L = layer->L;
    if (!L.cache) return moe::fail(MOE_E_UNSUPPORTED, "router lookahead needs a streamed layer (cache_slots > 0)");
    moe::DeviceGuard g(L.device);
    if (!g.ok) return moe::cuda_fail(g.err, "cudaSetDevice");
    int r = 0, f = 0;
    const moe_status st = moe::cache_prefetch(L, x, static_cast<cudaStream_t>(stream), &r, &f);
    if (n_resident) *n_resident = r;
    if (n_fills) *n_fills = f;
    return st;
}

moe_status moe_cache_prefetch_stats(const moe_layer* layer, uint64_t* out4) {
    if (!layer || !out4) return moe::fail(MOE_E_INVALID, "NULL argument");
    const moe::Layer& L = layer->L;
    if (!L.cache) return moe::fail(MOE_E_UNSUPPORTED, "not a streamed layer");
    const moe::CacheState& C = *L.cache;
    out4[0] = C.pf_calls;
    out4[1] = C.pf_resident;
    out4[2] = C.pf_fills;
    out4[3] = C.pf_bytes;
    return MOE_OK;
}

moe_status moe_cache_stats(const moe_layer* layer, moe_cache_stats_t* out) {
    if (!layer || !out) return moe::fail(MOE_E_INVALID, "NULL argument");
    if (!layer->L.cache) return moe::fail(MOE_E_STATE, "layer is not streamed");
    const moe::CacheState& C = *layer->L.cache;
    *out = C.stats;
    if (C.device) {   // plus the device's counts so far (every decode queued included)
        moe::DeviceGuard g(layer->L.device);
        if (!g.ok) return moe::cuda_fail(g.err, "cudaSetDevice");
        MOE_CUDA_TRY(cudaDeviceSynchronize());
        unsigned long long st[4];
        MOE_CUDA_TRY(cudaMemcpy(st, C.dca.stats, sizeof st, cudaMemcpyDeviceToHost));
        out->tokens += st[0];
        out->hits += st[1];
        out->misses += st[2];
        out->bytes_h2d += st[3];
    }
    return MOE_OK;
}

moe_status moe_cache_pin(moe_layer* layer, const int32_t* experts, int32_t n) {
    if (!layer) return moe::fail(MOE_E_INVALID, "NULL layer");
    moe::Layer& L = layer->L;
    if (!L.cache) return moe::fail(MOE_E_STATE, "layer is not streamed (cache_slots == 0)");
    moe::DeviceGuard g(L.device);
    if (!g.ok) return moe::cuda_fail(g.err, "cudaSetDevice");
    return moe::cache_pin(L, experts, n);
}

moe_status moe_hottest(const uint64_t* counts, int32_t n_experts, int32_t n, int32_t* out) {
    if (!counts || (!out && n > 0)) return moe::fail(MOE_E_INVALID, "NULL argument");
    if (n_experts < 0 || n < 0 || n > n_experts) return moe::fail(MOE_E_INVALID, "n must be in 0..n_experts");
    std::vector<int32_t> order(n_experts);
    for (int32_t e = 0; e < n_experts; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return counts[a] > counts[b]; });
    for (int32_t i = 0; i < n; ++i) out[i] = order[i];
    return MOE_OK;
}

moe_status moe_cache_pin_hottest(moe_layer* layer, int32_t n) {
    if (!layer) return moe::fail(MOE_E_INVALID, "NULL layer");
    if (!layer->L.cache) return moe::fail(MOE_E_STATE, "layer is not streamed (cache_slots == 0)");
    const int32_t E = layer->L.d.n_experts;
    if (n < 0 || n > E) return moe::fail(MOE_E_INVALID, "n must be in 0..n_experts");
    std::vector<uint64_t> use(E);
    moe_status st = moe_cache_usage(layer, use.data());
    if (st != MOE_OK) return st;
    std::vector<int32_t> hot(n);
    st = moe_hottest(use.data(), E, n, hot.data());
    if (st != MOE_OK) return st;
    return moe_cache_pin(layer, n ? hot.data() : nullptr, n);
}

moe_status moe_cache_usage(const moe_layer* layer, uint64_t* counts) {
    if (!layer || !counts) return moe::fail(MOE_E_INVALID, "NULL argument");
    const moe::Layer& L = layer->L;
    if (!L.cache) return moe::fail(MOE_E_STATE, "layer is not streamed (cache_slots == 0)");
    const moe::CacheState& C = *L.cache;
    const int E = L.d.n_experts;
    for (int e = 0; e < E; ++e) counts[e] = C.lfu.usage(e);
    if (C.device) {   // plus the device's counts so far (every decode queued included)
        moe::DeviceGuard g(L.device);
        if (!g.ok) return moe::cuda_fail(g.err, "cudaSetDevice");
        MOE_CUDA_TRY(cudaDeviceSynchronize());
        std::vector<unsigned long long> use(E);
        MOE_CUDA_TRY(cudaMemcpy(use.data(), C.dca.usage, (size_t)E * 8, cudaMemcpyDeviceToHost));
        for (int e = 0; e < E; ++e) counts[e] += use[e];
    }
    return MOE_OK;
}

moe_status moe_cache_residency(const moe_layer* layer, int32_t* slot_expert) {
    if (!layer || !slot_expert) return moe::fail(MOE_E_INVALID, "NULL argument");
    if (!layer->L.cache) return moe::fail(MOE_E_STATE, "layer is not streamed");
    const moe::CacheState& C = *layer->L.cache;
    if (C.device) {
        moe::DeviceGuard g(layer->L.device);
        if (!g.ok) return moe::cuda_fail(g.err, "cudaSetDevice");
        MOE_CUDA_TRY(cudaDeviceSynchronize());
        MOE_CUDA_TRY(cudaMemcpy(slot_expert, C.dca.slot_expert, (size_t)C.slots * 4, cudaMemcpyDeviceToHost));
        return MOE_OK;
    }
    for (int s = 0; s < C.slots; ++s) slot_expert[s] = C.lfu.expert_in(s);
    return MOE_OK;
}

moe_status moe_lfu_trace(int32_t slots, int32_t n_experts, int32_t k, int32_t n_tokens, const int32_t* ids,
                         int32_t* slot, uint8_t* hit) {
    if (!ids || !slot || !hit) return moe::fail(MOE_E_INVALID, "NULL argument");
    if (slots < 1 || n_experts < 1 || k < 1 || k > slots || n_tokens < 0)
        return moe::fail(MOE_E_INVALID, "need 1 <= k <= slots, n_experts >= 1, n_tokens >= 0");
    moe::Lfu lfu(slots, n_experts);
    std::vector<moe::Fill> fills;
    for (int t = 0; t < n_tokens; ++t) {
        const int32_t* row = ids + (size_t)t * k;
        for (int i = 0; i < k; ++i) {
            if (row[i] < 0 || row[i] >= n_experts) return moe::fail(MOE_E_INVALID, "expert id out of range");
            for (int j = 0; j < i; ++j)
                if (row[j] == row[i]) return moe::fail(MOE_E_INVALID, "repeated expert id");
        }
        for (int i = 0; i < k; ++i) hit[(size_t)t * k + i] = lfu.slot_of(row[i]) >= 0 ? 1 : 0;
        int h = 0;
        lfu.access(row, k, &h, fills);
        for (int i = 0; i < k; ++i) slot[(size_t)t * k + i] = lfu.slot_of(row[i]);
    }
    return MOE_OK;
}

moe_status moe_lfu_trace_pinned(int32_t slots, int32_t n_experts, int32_t k, int32_t n_tokens, const int32_t* ids,
                                const int32_t* pinned, int32_t n_pinned, int32_t* slot, uint8_t* hit,
                                uint64_t* usage) {
    if (!ids || !slot || !hit || (n_pinned > 0 && !pinned)) return moe::fail(MOE_E_INVALID, "NULL argument");
    if (slots < 1 || n_experts < 1 || k < 1 || k > slots || n_tokens < 0)
        return moe::fail(MOE_E_INVALID, "need 1 <= k <= slots, n_experts >= 1, n_tokens >= 0");
    if (n_pinned < 0 || n_pinned > n_experts) return moe::fail(MOE_E_INVALID, "n_pinned out of range 0..n_experts");
    std::vector<int32_t> pin_index(n_experts, -1);
    for (int i = 0; i < n_pinned; ++i) {
        if (pinned[i] < 0 || pinned[i] >= n_experts) return moe::fail(MOE_E_INVALID, "pinned id out of range");
        if (pin_index[pinned[i]] >= 0) return moe::fail(MOE_E_INVALID, "repeated pinned id");
        pin_index[pinned[i]] = i;
    }
    moe::Lfu lfu(slots, n_experts);
    lfu.pin(pinned, n_pinned);
    std::vector<moe::Fill> fills;
    for (int t = 0; t < n_tokens; ++t) {
        const int32_t* row = ids + (size_t)t * k;
        for (int i = 0; i < k; ++i) {
            if (row[i] < 0 || row[i] >= n_experts) return moe::fail(MOE_E_INVALID, "expert id out of range");
            for (int j = 0; j < i; ++j)
                if (row[j] == row[i]) return moe::fail(MOE_E_INVALID, "repeated expert id");
        }
        for (int i = 0; i < k; ++i)
            hit[(size_t)t * k + i] = (lfu.pinned(row[i]) || lfu.slot_of(row[i]) >= 0) ? 1 : 0;
        int h = 0;
        lfu.access(row, k, &h, fills);
        for (int i = 0; i < k; ++i) {
            const int p = pin_index[row[i]];
            slot[(size_t)t * k + i] = p >= 0 ? slots + p : lfu.slot_of(row[i]);
        }
    }
    if (usage)
        for (int e = 0; e < n_experts; ++e) usage[e] = lfu.usage(e);
    return MOE_OK;
}

}  // extern "C"
