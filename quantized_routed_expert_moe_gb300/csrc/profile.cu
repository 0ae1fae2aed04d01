// Per-kernel device timing: a pool of CUDA event pairs recorded around each
// launch on the launch's own stream, summed per kernel kind on stop.
#include <vector>

#include "moe_internal.h"

namespace moe {

static const char* kKindNames[K_NUM_KINDS] = {
    "router_decode", "router_tokens", "topk_tokens", "gateup_decode", "down_decode",
    "prefill_permute", "prefill_gather", "prefill_gemm_gateup", "prefill_hconv", "prefill_gemm_down", "prefill_combine",
    "cache_fill"};

struct Profiler {
    bool on = false;
    std::vector<cudaEvent_t> a, b;
    std::vector<int> kind;
    int used = 0;
    int open_kind = -1;
};

void prof_begin(Layer& L, int kind, cudaStream_t s) {
    Profiler* p = L.prof;
    if (!p || !p->on || p->used >= (int)p->a.size()) return;
    if (cudaEventRecord(p->a[p->used], s) == cudaSuccess) p->open_kind = kind;
}

void prof_end(Layer& L, cudaStream_t s) {
    Profiler* p = L.prof;
    if (!p || !p->on || p->open_kind < 0) return;
    if (cudaEventRecord(p->b[p->used], s) == cudaSuccess) {
        p->kind[p->used] = p->open_kind;
        ++p->used;
    }
    p->open_kind = -1;
}

void prof_destroy(Layer& L) {
    if (!L.prof) return;
    for (auto e : L.prof->a) cudaEventDestroy(e);
    for (auto e : L.prof->b) cudaEventDestroy(e);
    delete L.prof;
    L.prof = nullptr;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_profile_start(moe_layer* layer, int32_t max_launches) {
    if (!layer || max_launches < 1) return fail(MOE_E_INVALID, "bad argument");
    Layer& L = layer->L;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(L.device);
    if (!L.prof) L.prof = new Profiler();
    Profiler& p = *L.prof;
    while ((int)p.a.size() < max_launches) {
        cudaEvent_t ea, eb;
        cudaError_t e = cudaEventCreate(&ea);
        if (e == cudaSuccess) e = cudaEventCreate(&eb);
        if (e != cudaSuccess) {
            if (prev >= 0) cudaSetDevice(prev);
            return cuda_fail(e, "cudaEventCreate");
        }
        p.a.push_back(ea);
        p.b.push_back(eb);
        p.kind.push_back(-1);
    }
    p.used = 0;
    p.open_kind = -1;
    p.on = true;
    if (prev >= 0) cudaSetDevice(prev);
    return MOE_OK;
}

moe_status moe_profile_stop(moe_layer* layer, moe_kernel_time* out, int32_t cap, int32_t* n_kinds) {
    if (!layer) return fail(MOE_E_INVALID, "bad argument");
    Layer& L = layer->L;
    if (!L.prof) return fail(MOE_E_STATE, "profiling was not started");
    Profiler& p = *L.prof;
    p.on = false;
    uint64_t cnt[K_NUM_KINDS] = {};
    double ms[K_NUM_KINDS] = {};
    for (int i = 0; i < p.used; ++i) {
        cudaError_t e = cudaEventSynchronize(p.b[i]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        float t = 0.f;
        e = cudaEventElapsedTime(&t, p.a[i], p.b[i]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        cnt[p.kind[i]] += 1;
        ms[p.kind[i]] += t;
    }
    int n = 0;
    for (int k = 0; k < K_NUM_KINDS; ++k) {
        if (!cnt[k]) continue;
        if (out && n < cap) out[n] = moe_kernel_time{kKindNames[k], cnt[k], ms[k]};
        ++n;
    }
    if (n_kinds) *n_kinds = n;
    p.used = 0;
    return MOE_OK;
}

}  // extern "C"
