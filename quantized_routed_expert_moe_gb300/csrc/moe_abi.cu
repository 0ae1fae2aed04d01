// C ABI entry points: layer lifetime, argument checks, scratch, dispatch.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "moe_internal.h"

namespace moe {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

moe_status fail(moe_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return MOE_E_CUDA;
}

static moe_status check_desc(const moe_layer_desc* d) {
    if (!d) return fail(MOE_E_INVALID, "desc is NULL");
    if (d->abi_version != MOE_ABI_VERSION) return fail(MOE_E_INVALID, "abi_version mismatch");
    if (d->hidden <= 0 || d->hidden % 64) return fail(MOE_E_INVALID, "hidden must be a positive multiple of 64");
    if (d->inter <= 0 || d->inter % 64) return fail(MOE_E_INVALID, "inter must be a positive multiple of 64");
    if (d->hidden > 16384 || d->inter > 16384)
        return fail(MOE_E_UNSUPPORTED, "hidden and inter are limited to 16384");
    if (d->top_k < 1 || d->top_k > MOE_MAX_TOP_K) return fail(MOE_E_INVALID, "top_k must be in 1..8");
    if (d->n_experts < d->top_k || d->n_experts > 1024)
        return fail(MOE_E_INVALID, "n_experts must be in top_k..1024");
    if (d->n_shared != 0 && d->n_shared != 1) return fail(MOE_E_INVALID, "n_shared must be 0 or 1");
    if (d->router_fmt != MOE_W_F32 && d->router_fmt != MOE_W_Q8G64)
        return fail(MOE_E_UNSUPPORTED, "router_fmt must be MOE_W_F32 or MOE_W_Q8G64");
    if (d->expert_fmt != MOE_W_Q4G64 && d->expert_fmt != MOE_W_Q2G64)
        return fail(MOE_E_UNSUPPORTED, "expert_fmt must be MOE_W_Q4G64 or MOE_W_Q2G64");
    if (d->group != MOE_GROUP) return fail(MOE_E_UNSUPPORTED, "group must be 64");
    if (d->act_dtype != MOE_F32 && d->act_dtype != MOE_BF16) return fail(MOE_E_INVALID, "act_dtype");
    if (d->max_tokens < 1 || d->max_tokens > MOE_MAX_CHUNK)
        return fail(MOE_E_INVALID, "max_tokens must be in 1..128");
    if (d->cache_slots < 0) return fail(MOE_E_INVALID, "cache_slots must be >= 0");
    if (d->cache_slots > 0 && d->cache_slots < d->top_k)
        return fail(MOE_E_INVALID, "cache_slots must be >= top_k");
    if (d->cache_slots > d->n_experts) return fail(MOE_E_INVALID, "cache_slots must be <= n_experts");
    return MOE_OK;
}

static size_t act_size(const moe_layer_desc& d) { return d.act_dtype == MOE_BF16 ? 2 : 4; }

static size_t router_bytes(const moe_layer_desc& d) {
    const size_t E = d.n_experts, H = d.hidden;
    if (d.router_fmt == MOE_W_F32) return E * H * 4;
    return E * H + E * (H / 64) * 4;
}

// K-splits of the one-token router: the most (at most kMaxRouterSplits, each
// a whole number of 64-wide groups) that keep its grid of ceil(E/8) x splits
// CTAs within two per SM, so that small layers still spread over the GPU
static int pick_router_splits(int H, int E, int num_sms) {
    const int cta_cols = (E + 7) / 8;
    for (int s = kMaxRouterSplits; s > 1; --s)
        if ((H / 64) % s == 0 && cta_cols * s <= 2 * std::max(num_sms, 1)) return s;
    return 1;
}

struct Alloc {
    size_t total = 0;
    size_t add(size_t b) {
        size_t off = total;
        total += (b + 255) / 256 * 256;
        return off;
    }
};

static void free_layer(Layer& L) {
    if (L.cache) cache_destroy(L);
    prof_destroy(L);
    auto f = [](void* p) { if (p) cudaFree(p); };
    f(L.router);
    f(L.router_bias);
    f(L.experts);
    f(L.rec_table);
    f(L.logits_part);  // scratch block base (see create)
    f(L.io_x);
    f(L.io_y);
    f(L.pf.xp);        // prefill block base
    f(L.pf.waves_dev);
    if (L.pf.groups_host) cudaFreeHost(L.pf.groups_host);
    if (L.pf.waves_host) cudaFreeHost(L.pf.waves_host);
    if (L.pf.groups_ready) cudaEventDestroy(L.pf.groups_ready);
    if (L.pf.waves_free) cudaEventDestroy(L.pf.waves_free);
    f(L.trace_split);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_E_INVALID: return "MOE_E_INVALID";
        case MOE_E_UNSUPPORTED: return "MOE_E_UNSUPPORTED";
        case MOE_E_NOMEM: return "MOE_E_NOMEM";
        case MOE_E_CUDA: return "MOE_E_CUDA";
        case MOE_E_TIMEOUT: return "MOE_E_TIMEOUT";
        case MOE_E_STATE: return "MOE_E_STATE";
        case MOE_E_SOURCE: return "MOE_E_SOURCE";
    }
    return "MOE_E_?";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

size_t moe_expert_record_bytes(const moe_layer_desc* desc) {
    if (check_desc(desc) != MOE_OK) return 0;
    return record_bytes(desc->hidden, desc->inter, desc->expert_fmt == MOE_W_Q2G64 ? 2 : 4);
}

moe_status moe_pack_expert_record(const moe_layer_desc* desc, const moe_expert* expert, void* dst) {
    moe_status st = check_desc(desc);
    if (st != MOE_OK) return st;
    if (!expert || !dst) return fail(MOE_E_INVALID, "expert and dst must be non-NULL");
    const moe_qmat* m[3] = {&expert->gate, &expert->up, &expert->down};
    for (auto q : m)
        if (!q->codes || !q->scale || !q->bias) return fail(MOE_E_INVALID, "expert matrix pointer is NULL");
    pack_expert(desc->hidden, desc->inter, desc->expert_fmt == MOE_W_Q2G64 ? 2 : 4, *expert,
                static_cast<uint8_t*>(dst));
    return MOE_OK;
}

size_t moe_layer_device_bytes(const moe_layer* layer) { return layer ? layer->L.device_bytes : 0; }

moe_status moe_layer_create(const moe_layer_desc* desc, const moe_router* router,
                            const float* router_bias, const moe_expert* shared,
                            const moe_expert* experts, const void* const* records,
                            moe_expert_source source, void* source_user, int32_t device,
                            moe_layer** out) {
    if (!out) return fail(MOE_E_INVALID, "out is NULL");
    *out = nullptr;
    moe_status st = check_desc(desc);
    if (st != MOE_OK) return st;
    const moe_layer_desc& d = *desc;
    if (!router) return fail(MOE_E_INVALID, "router is NULL");
    if (d.router_fmt == MOE_W_F32 && !router->w) return fail(MOE_E_INVALID, "router->w is NULL");
    if (d.router_fmt == MOE_W_Q8G64 && (!router->q.codes || !router->q.scale || !router->q.bias))
        return fail(MOE_E_INVALID, "router->q has a NULL pointer");
    if (d.n_shared && !shared) return fail(MOE_E_INVALID, "shared expert is NULL but n_shared == 1");
    if (d.cache_slots == 0 && !experts) return fail(MOE_E_INVALID, "experts is NULL in resident mode");
    if (d.cache_slots > 0 && !records && !source)
        return fail(MOE_E_INVALID, "streamed mode needs records or a source");

    int ndev = 0;
    cudaError_t ce = cudaGetDeviceCount(&ndev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDeviceCount");
    if (device < 0 || device >= ndev) return fail(MOE_E_CUDA, "invalid CUDA device index");
    DeviceGuard g(device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");

    moe_layer* layer = new (std::nothrow) moe_layer();
    if (!layer) return fail(MOE_E_NOMEM, "host allocation failed");
    Layer& L = layer->L;
    L.d = d;
    L.device = device;
    L.wbits = d.expert_fmt == MOE_W_Q2G64 ? 2 : 4;
    L.rec_bytes = record_bytes(d.hidden, d.inter, L.wbits);
    cudaDeviceGetAttribute(&L.num_sms, cudaDevAttrMultiProcessorCount, device);
    L.router_splits = pick_router_splits(d.hidden, d.n_experts, L.num_sms);
    // prefill router GEMM: enough K-splits for two CTAs per SM at 128 tokens
    // (each split a whole number of 64-wide groups)
    L.router_splits_tok = ((d.hidden / 64) % kMaxTokSplits == 0) ? kMaxTokSplits
                          : ((d.hidden / 64) % 16 == 0) ? 16 : L.router_splits;

    const int E = d.n_experts, H = d.hidden, I = d.inter, k = d.top_k, T = d.max_tokens;
    const size_t n_rec = (d.cache_slots == 0) ? (size_t)E + d.n_shared : (size_t)d.n_shared;

    // scratch block layout
    Alloc sc;
    size_t o_part = sc.add((size_t)std::max(L.router_splits, L.router_splits_tok) * E * 4 * std::max(1, T));
    size_t o_logits = sc.add((size_t)T * E * 4);
    size_t o_ptag = sc.add((size_t)L.router_splits * E * 8);
    size_t o_stag = sc.add((size_t)(2 * k + 1) * 8);
    size_t o_ids = sc.add((size_t)T * k * 4);
    size_t o_w = sc.add((size_t)T * k * 4);
    size_t o_h = sc.add((size_t)kDecodeHCopies * (k + 1) * I * 4);
    size_t o_cnt = sc.add(64 * 4);
    // prefill block layout
    const int rows = T * k + T * d.n_shared;
    Alloc pf;
    size_t o_xp = pf.add((size_t)rows * H * 2);
    size_t o_hp = pf.add((size_t)rows * I * 2);
    size_t o_yp = pf.add((size_t)rows * H * 4);
    size_t o_h32 = pf.add((size_t)rows * I * 4);
    size_t o_xexp = pf.add((size_t)T * 4);
    size_t o_rexp = pf.add((size_t)rows * 4);
    size_t o_hmax = pf.add((size_t)rows * 4);
    size_t o_zexp = pf.add((size_t)rows * 8);
    size_t o_gexp = pf.add((size_t)(E + 1) * 4);
    size_t o_goff = pf.add((size_t)(E + 1) * 4);
    size_t o_gcnt = pf.add((size_t)(E + 1) * 4);
    size_t o_ptok = pf.add((size_t)rows * 4);
    size_t o_pos = pf.add((size_t)T * (k + 1) * 4);
    size_t o_ng = pf.add(16);

    size_t need = router_bytes(d) + (size_t)E * 4 + n_rec * L.rec_bytes + (size_t)(E + 1) * 8 +
                  (size_t)d.cache_slots * L.rec_bytes +
                  sc.total + (T > 1 ? pf.total : 0);
    size_t free_b = 0, total_b = 0;
    ce = cudaMemGetInfo(&free_b, &total_b);
    if (ce != cudaSuccess) { delete layer; return cuda_fail(ce, "cudaMemGetInfo"); }
    const size_t headroom = (size_t)256 << 20;
    if (need + headroom > free_b) {
        delete layer;
        char buf[160];
        std::snprintf(buf, sizeof buf, "layer needs %zu bytes of device memory, %zu free", need, free_b);
        return fail(MOE_E_NOMEM, buf);
    }

#define TRY_ALLOC(ptr, bytes)                                             \
    do {                                                                  \
        cudaError_t _e = cudaMalloc((void**)&(ptr), (bytes));             \
        if (_e != cudaSuccess) {                                          \
            free_layer(L); delete layer;                                  \
            return _e == cudaErrorMemoryAllocation ? fail(MOE_E_NOMEM, "cudaMalloc failed") \
                                                   : cuda_fail(_e, "cudaMalloc"); \
        }                                                                 \
    } while (0)
#define TRY_CUDA(expr)                                                    \
    do {                                                                  \
        cudaError_t _e = (expr);                                          \
        if (_e != cudaSuccess) { free_layer(L); delete layer; return cuda_fail(_e, #expr); } \
    } while (0)

    // router
    TRY_ALLOC(L.router, router_bytes(d));
    L.router_nbytes = router_bytes(d);
    if (d.router_fmt == MOE_W_F32) {
        TRY_CUDA(cudaMemcpy(L.router, router->w, (size_t)E * H * 4, cudaMemcpyHostToDevice));
    } else {
        std::vector<uint8_t> tmp(router_bytes(d));
        std::memcpy(tmp.data(), router->q.codes, (size_t)E * H);
        uint8_t* meta = tmp.data() + (size_t)E * H;
        const size_t G = (size_t)E * (H / 64);
        for (size_t gi = 0; gi < G; ++gi) {
            std::memcpy(meta + 4 * gi, router->q.scale + gi, 2);
            std::memcpy(meta + 4 * gi + 2, router->q.bias + gi, 2);
        }
        TRY_CUDA(cudaMemcpy(L.router, tmp.data(), tmp.size(), cudaMemcpyHostToDevice));
    }
    if (router_bias) {
        TRY_ALLOC(L.router_bias, (size_t)E * 4);
        TRY_CUDA(cudaMemcpy(L.router_bias, router_bias, (size_t)E * 4, cudaMemcpyHostToDevice));
    }

    // experts: pack on the host into pinned staging, copy in chunks
    TRY_ALLOC(L.experts, n_rec * L.rec_bytes);
    {
        const size_t rb = L.rec_bytes;
        uint8_t* stage[2] = {nullptr, nullptr};
        cudaEvent_t ev[2] = {nullptr, nullptr};
        cudaStream_t cs = nullptr;
        cudaError_t e2 = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
        for (int b = 0; b < 2 && e2 == cudaSuccess; ++b) {
            e2 = cudaMallocHost((void**)&stage[b], rb);
            if (e2 == cudaSuccess) e2 = cudaEventCreateWithFlags(&ev[b], cudaEventDisableTiming);
        }
        for (size_t r = 0; r < n_rec && e2 == cudaSuccess; ++r) {
            const int b = (int)(r & 1);
            if (r >= 2) e2 = cudaEventSynchronize(ev[b]);
            if (e2 != cudaSuccess) break;
            const moe_expert* src = (d.cache_slots == 0 && r < (size_t)E) ? &experts[r] : shared;
            pack_expert(H, I, L.wbits, *src, stage[b]);
            e2 = cudaMemcpyAsync(L.experts + r * rb, stage[b], rb, cudaMemcpyHostToDevice, cs);
            if (e2 == cudaSuccess) e2 = cudaEventRecord(ev[b], cs);
        }
        if (cs) {
            cudaError_t e3 = cudaStreamSynchronize(cs);
            if (e2 == cudaSuccess) e2 = e3;
            cudaStreamDestroy(cs);
        }
        for (int b = 0; b < 2; ++b) {
            if (stage[b]) cudaFreeHost(stage[b]);
            if (ev[b]) cudaEventDestroy(ev[b]);
        }
        if (e2 != cudaSuccess) { free_layer(L); delete layer; return cuda_fail(e2, "expert upload"); }
    }

    // record table: routed experts then the shared expert at index E
    TRY_ALLOC(L.rec_table, (size_t)(E + 1) * sizeof(void*));
    {
        std::vector<const uint8_t*> tab(E + 1, nullptr);
        if (d.cache_slots == 0)
            for (int e = 0; e < E; ++e) tab[e] = L.experts + (size_t)e * L.rec_bytes;
        if (d.n_shared) tab[E] = L.experts + (n_rec - 1) * L.rec_bytes;
        TRY_CUDA(cudaMemcpy(L.rec_table, tab.data(), tab.size() * sizeof(void*), cudaMemcpyHostToDevice));
    }

    // scratch
    {
        uint8_t* base = nullptr;
        TRY_ALLOC(base, sc.total);
        TRY_CUDA(cudaMemset(base, 0, sc.total));
        L.logits_part = reinterpret_cast<float*>(base + o_part);
        L.logits = reinterpret_cast<float*>(base + o_logits);
        L.part_tag = reinterpret_cast<unsigned long long*>(base + o_ptag);
        L.sel_tag = reinterpret_cast<unsigned long long*>(base + o_stag);
        L.ids = reinterpret_cast<int32_t*>(base + o_ids);
        L.wts = reinterpret_cast<float*>(base + o_w);
        L.h = reinterpret_cast<float*>(base + o_h);
        L.counters = reinterpret_cast<unsigned*>(base + o_cnt);
    }
    if (T > 1) {
        uint8_t* base = nullptr;
        TRY_ALLOC(base, pf.total);
        TRY_CUDA(cudaMemset(base, 0, pf.total));
        L.pf.xp = base + o_xp;
        L.pf.hp = base + o_hp;
        L.pf.yp = reinterpret_cast<float*>(base + o_yp);
        L.pf.h32 = reinterpret_cast<float*>(base + o_h32);
        L.pf.xexp = reinterpret_cast<int32_t*>(base + o_xexp);
        L.pf.rexp = reinterpret_cast<int32_t*>(base + o_rexp);
        L.pf.hmax = reinterpret_cast<unsigned*>(base + o_hmax);
        L.pf.zfac = reinterpret_cast<float2*>(base + o_zexp);
        L.pf.group_expert = reinterpret_cast<int32_t*>(base + o_gexp);
        L.pf.group_off = reinterpret_cast<int32_t*>(base + o_goff);
        L.pf.group_cnt = reinterpret_cast<int32_t*>(base + o_gcnt);
        L.pf.perm_token = reinterpret_cast<int32_t*>(base + o_ptok);
        L.pf.pos = reinterpret_cast<int32_t*>(base + o_pos);
        L.pf.n_groups = reinterpret_cast<int32_t*>(base + o_ng);
        L.pf.err = reinterpret_cast<unsigned*>(base + o_ng + 4);
        L.pf.max_rows = rows;
    }
    L.device_bytes = need;

    TRY_CUDA(decode_kernel_setup(L));
    if (T > 1) TRY_CUDA(prefill_kernel_setup(L));

    if (d.cache_slots > 0) {
        st = cache_create(L, records, source, source_user);
        if (st == MOE_OK && T > 1) st = prefill_cache_setup(L);
        if (st != MOE_OK) { std::string m = g_last_error; free_layer(L); delete layer; return fail(st, m); }
    }
#undef TRY_ALLOC
#undef TRY_CUDA
    *out = layer;
    return MOE_OK;
}

void moe_layer_destroy(moe_layer* layer) {
    if (!layer) return;
    DeviceGuard g(layer->L.device);
    cudaDeviceSynchronize();
    free_layer(layer->L);
    delete layer;
}

moe_status moe_route(moe_layer* layer, const void* x, int32_t T, int32_t* ids, float* w, void* stream) {
    if (!layer || !x || !ids || !w) return fail(MOE_E_INVALID, "NULL argument");
    Layer& L = layer->L;
    if (T < 1 || T > L.d.max_tokens) return fail(MOE_E_INVALID, "T out of range 1..max_tokens");
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = (T == 1) ? launch_route_decode(L, x, s, 1) : launch_route_tokens(L, x, T, s);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    const size_t nb = (size_t)T * L.d.top_k * 4;
    MOE_CUDA_TRY(cudaMemcpyAsync(ids, L.ids, nb, cudaMemcpyDeviceToDevice, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(w, L.wts, nb, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

moe_status moe_decode(moe_layer* layer, const void* x, void* y, float* y_f32, void* stream) {
    if (!layer || !x) return fail(MOE_E_INVALID, "NULL argument");
    if (!y && !y_f32) return fail(MOE_E_INVALID, "y and y_f32 are both NULL");
    Layer& L = layer->L;
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L.d.cache_slots > 0) return cache_decode(L, x, y, y_f32, s);
    // the router writes tagged partial logits, every gate/up CTA selects from
    // them; the down kernel starts early on the shared expert
    const DecodeScratch b = layer_decode_scratch(L, true);
    cudaError_t e = launch_route_decode(L, x, s, 1, nullptr, nullptr, 0, nullptr, &b);
    if (e == cudaSuccess) e = launch_experts_decode(L, x, y, y_f32, b, 0, L.d.top_k + L.d.n_shared, true, true, true, s);
    if (e != cudaSuccess) {
        // the token did not run to its end, so the decode count did not
        // advance: clear the tagged partials so that the next token cannot
        // take this one's for its own
        cudaMemsetAsync(L.part_tag, 0, (size_t)L.router_splits * L.d.n_experts * 8, s);
        cudaMemsetAsync(L.sel_tag, 0, (size_t)(2 * L.d.top_k + 1) * 8, s);
        return cuda_fail(e, "decode launch");
    }
    return MOE_OK;
}

moe_status moe_prefill_chunk(moe_layer* layer, const void* x, int32_t T, void* y, float* y_f32,
                             void* stream) {
    if (!layer || !x) return fail(MOE_E_INVALID, "NULL argument");
    if (!y && !y_f32) return fail(MOE_E_INVALID, "y and y_f32 are both NULL");
    Layer& L = layer->L;
    if (T < 1 || T > L.d.max_tokens) return fail(MOE_E_INVALID, "T out of range 1..max_tokens");
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 1) return moe_decode(layer, x, y, y_f32, stream);
    cudaError_t e = launch_route_tokens(L, x, T, s, L.pf.xexp);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");
    if (L.d.cache_slots > 0) {
        if (!cache_is_device(L)) return launch_prefill_streamed(L, x, T, y, y_f32, s);
        // device-managed cache: a chunk's waves are staged by the host, so the
        // LFU state comes to the host for the chunk and goes back after it (two
        // synchronisations, against a chunk of milliseconds); one LFU run throughout
        moe_status st = cache_set_device(L, false);
        if (st != MOE_OK) return st;
        st = launch_prefill_streamed(L, x, T, y, y_f32, s);
        const moe_status back = cache_set_device(L, true);
        return st != MOE_OK ? st : back;
    }
    e = launch_prefill(L, x, T, y, y_f32, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return MOE_OK;
}

moe_status moe_decode_tokens_host(moe_layer* layer, const void* x_host, int32_t T, void* y_host,
                                  void* stream) {
    if (!layer || !x_host || !y_host) return fail(MOE_E_INVALID, "NULL argument");
    if (T < 1) return fail(MOE_E_INVALID, "T must be >= 1");
    Layer& L = layer->L;
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t row = (size_t)L.d.hidden * act_size(L.d);
    if (T > L.io_cap) {
        MOE_CUDA_TRY(cudaStreamSynchronize(s));
        if (L.io_x) cudaFree(L.io_x);
        if (L.io_y) cudaFree(L.io_y);
        L.io_x = L.io_y = nullptr;
        L.io_cap = 0;
        MOE_CUDA_TRY(cudaMalloc(&L.io_x, row * T));
        MOE_CUDA_TRY(cudaMalloc(&L.io_y, row * T));
        L.io_cap = T;
    }
    MOE_CUDA_TRY(cudaMemcpyAsync(L.io_x, x_host, row * T, cudaMemcpyHostToDevice, s));
    for (int t = 0; t < T; ++t) {
        const uint8_t* xt = static_cast<const uint8_t*>(L.io_x) + row * t;
        uint8_t* yt = static_cast<uint8_t*>(L.io_y) + row * t;
        moe_status st = moe_decode(layer, xt, yt, nullptr, stream);
        if (st != MOE_OK) return st;
    }
    MOE_CUDA_TRY(cudaMemcpyAsync(y_host, L.io_y, row * T, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    return MOE_OK;
}

moe_status moe_layer_set_next(moe_layer* layer, const moe_layer* next) {
    if (!layer) return fail(MOE_E_INVALID, "NULL layer");
    Layer& L = layer->L;
    if (!next) {
        L.next_router = nullptr;
        L.next_router_bytes = 0;
        return MOE_OK;
    }
    if (next->L.device != L.device) return fail(MOE_E_INVALID, "next layer is on another device");
    L.next_router = next->L.router;
    L.next_router_bytes = next->L.router_nbytes / 16 * 16;   // the prefetch moves multiples of 16 bytes
    return MOE_OK;
}

moe_status moe_layer_set_router_scoring(moe_layer* layer, int32_t scoring, float routed_scaling) {
    if (!layer) return fail(MOE_E_INVALID, "NULL layer");
    Layer& L = layer->L;
    if (scoring != MOE_SCORE_SOFTMAX && scoring != MOE_SCORE_SIGMOID) return fail(MOE_E_INVALID, "unknown router scoring");
    if (!(routed_scaling > 0.0f) || !std::isfinite(routed_scaling))
        return fail(MOE_E_INVALID, "routed_scaling must be finite and positive");
    L.router_scoring = scoring;
    L.routed_scaling = routed_scaling;
    return MOE_OK;
}

moe_status moe_layer_set_option(moe_layer* layer, int32_t option, int64_t value) {
    if (!layer) return fail(MOE_E_INVALID, "NULL layer");
    Layer& L = layer->L;
    switch (option) {
        case MOE_OPT_TEST_STALL_SHARED:
            L.test_stall_shared = value ? 1 : 0;
            return MOE_OK;
        case MOE_OPT_TRACE:
            if (value && !L.trace_split) {
                DeviceGuard g(L.device);
                if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
                const size_t ns = (size_t)MOE_TRACE_KERNELS * MOE_TRACE_MAX_CTAS * 4 * 8;
                MOE_CUDA_TRY(cudaMalloc(&L.trace_split, ns));
                MOE_CUDA_TRY(cudaMemset(L.trace_split, 0, ns));
            }
            L.trace_on = value != 0;
            return MOE_OK;
        case MOE_OPT_HOST_TIMEOUT_MS:
            if (value < 0 || value > 3600000) return fail(MOE_E_INVALID, "host timeout out of range 0..3600000 ms");
            L.host_timeout_ms = (int)value;
            return MOE_OK;
        case MOE_OPT_TEST_STALL_COPIES_MS:
            if (value < 0 || value > 10000) return fail(MOE_E_INVALID, "copy stall out of range 0..10000 ms");
            L.test_stall_copies_ms = (int)value;
            return MOE_OK;
        case MOE_OPT_CACHE_DEVICE: {
            if (value != 0 && value != 1) return fail(MOE_E_INVALID, "MOE_OPT_CACHE_DEVICE takes 0 or 1");
            if (!L.cache) return fail(MOE_E_STATE, "layer is not streamed (cache_slots == 0)");
            DeviceGuard g(L.device);
            if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
            return cache_set_device(L, value != 0);
        }
    }
    return fail(MOE_E_INVALID, "unknown option");
}

moe_status moe_layer_selection(moe_layer* layer, int32_t T, int32_t* ids, float* w, void* stream) {
    if (!layer || !ids || !w) return fail(MOE_E_INVALID, "NULL argument");
    Layer& L = layer->L;
    if (T < 1 || T > L.d.max_tokens) return fail(MOE_E_INVALID, "T out of range 1..max_tokens");
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nb = (size_t)T * L.d.top_k * 4;
    MOE_CUDA_TRY(cudaMemcpyAsync(ids, L.ids, nb, cudaMemcpyDeviceToDevice, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(w, L.wts, nb, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

moe_status moe_trace_read_split(moe_layer* layer, uint64_t* out, int32_t cap) {
    if (!layer || !out) return fail(MOE_E_INVALID, "NULL argument");
    Layer& L = layer->L;
    if (!L.trace_split) return fail(MOE_E_STATE, "tracing was never enabled (MOE_OPT_TRACE)");
    const int n = MOE_TRACE_KERNELS * MOE_TRACE_MAX_CTAS * 4;
    if (cap < n) return fail(MOE_E_INVALID, "cap smaller than MOE_TRACE_KERNELS * MOE_TRACE_MAX_CTAS * 4");
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    MOE_CUDA_TRY(cudaMemcpy(out, L.trace_split, (size_t)n * 8, cudaMemcpyDeviceToHost));
    return MOE_OK;
}

moe_status moe_layer_check(moe_layer* layer, uint32_t* bits) {
    if (!layer) return fail(MOE_E_INVALID, "NULL layer");
    Layer& L = layer->L;
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    uint32_t v = 0, vp = 0;
    unsigned* w = error_word(L);
    MOE_CUDA_TRY(cudaMemcpy(&v, w, 4, cudaMemcpyDeviceToHost));
    if (L.pf.err) MOE_CUDA_TRY(cudaMemcpy(&vp, L.pf.err, 4, cudaMemcpyDeviceToHost));
    v |= vp;   // the prefill GEMM reports in bits 16 and up
    if (bits) *bits = v;
    if (v) {
        MOE_CUDA_TRY(cudaMemset(w, 0, 4));
        if (L.pf.err) MOE_CUDA_TRY(cudaMemset(L.pf.err, 0, 4));
        return fail(MOE_E_TIMEOUT, "a bounded device-side wait gave up (error bits " + std::to_string(v) + ")");
    }
    return MOE_OK;
}

moe_status moe_cache_stage(moe_layer* layer, const int32_t* ids, int32_t n, void* stream,
                           int32_t* n_hits, int32_t* n_misses) {
    if (!layer || !ids) return fail(MOE_E_INVALID, "NULL argument");
    Layer& L = layer->L;
    if (L.d.cache_slots == 0) return fail(MOE_E_STATE, "layer is not streamed (cache_slots == 0)");
    if (n < 0 || n > L.d.cache_slots) return fail(MOE_E_INVALID, "n out of range 0..cache_slots");
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    int h = 0, m = 0;
    moe_status st = cache_stage(L, ids, n, static_cast<cudaStream_t>(stream), &h, &m);
    if (n_hits) *n_hits = h;
    if (n_misses) *n_misses = m;
    return st;
}

}  // extern "C"
