// moe_decode_static_scratch: the split decode path over scratch that lives in
// a fixed region of this library's device image, so the call allocates
// nothing. It exists for callers that may not allocate device memory while
// serving: cudaMalloc/cudaFree can synchronise the device and stall every
// other stream, an engine that has already divided HBM among weights and
// caches has no room to give, and a caching allocator asked for a block then
// may have to grow its pool. The weights and the layer itself are set up once,
// at creation; this file adds no allocation of any kind on the call path.
#include <mutex>

#include <cuda.h>

#include "moe_internal.h"

namespace moe {
namespace {

// One region per device (a __device__ variable is instantiated on every
// device the module is loaded on).
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// per device: the region's address and the context it was looked up in (a
// device reset gives the device a new primary context, where the region has
// another address, so the lookup is redone when the context changes)
void* g_base[kMaxDevices] = {};
CUcontext g_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

inline size_t up256(size_t n) { return (n + 255) / 256 * 256; }

constexpr int kParts = 7;

// Byte offsets of the pieces within the region; the last entry is the total.
void layout(const Layer& L, size_t off[kParts]) {
    const auto& d = L.d;
    const size_t E = d.n_experts, k = d.top_k, I = d.inter;
    off[0] = 0;                                                  // partial logits [splits][E]
    off[1] = off[0] + up256((size_t)L.router_splits * E * 4);    // keys [E]
    off[2] = off[1] + up256(E * 4);                              // ids [k]
    off[3] = off[2] + up256(k * 4);                              // weights [k]
    off[4] = off[3] + up256(k * 4);                              // the token's scale exponent
    off[5] = off[4] + up256(4);                                  // SwiGLU outputs [k + 1][I] fp32 (one replica)
    off[6] = off[5] + up256((k + 1) * I * 4);
}

DecodeScratch carve(Layer& L, unsigned char* base) {
    size_t off[kParts];
    layout(L, off);
    DecodeScratch s;
    s.part = reinterpret_cast<float*>(base + off[0]);
    s.logits = reinterpret_cast<float*>(base + off[1]);
    s.ids = reinterpret_cast<int32_t*>(base + off[2]);
    s.wts = reinterpret_cast<float*>(base + off[3]);
    s.scale = reinterpret_cast<int*>(base + off[4]);
    s.router_cnt = L.counters + CNT_ROUTER;   // the layer's own (zero between launches)
    s.h = reinterpret_cast<float*>(base + off[5]);
    s.copies = 1;
    return s;   // no ready flag and no early start: nothing else in the region must start at zero
}

// Device address of this device's region, looked up once per device (per
// context of that device) with that device current. The caller holds a
// DeviceGuard for `dev`.
moe_status region_for(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_E_UNSUPPORTED, "device ordinal above the static-scratch table");
    // binds the device's primary context to this thread (a thread that never
    // used the runtime has none current yet)
    const cudaError_t se = cudaSetDevice(dev);
    if (se != cudaSuccess) return cuda_fail(se, "cudaSetDevice");
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return fail(MOE_E_CUDA, "cuCtxGetCurrent is not available from the driver");
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return fail(MOE_E_CUDA, "no current CUDA context for the device");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_base[dev] || g_ctx[dev] != ctx) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        if (!p) return fail(MOE_E_CUDA, "cudaGetSymbolAddress(static scratch) returned NULL");
        g_base[dev] = p;
        g_ctx[dev] = ctx;
    }
    *out = static_cast<unsigned char*>(g_base[dev]);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_decode_static_scratch(moe_layer* layer, const void* x, void* y, float* y_f32,
                                                void* stream) {
    if (!layer || !x) return fail(MOE_E_INVALID, "NULL argument");
    if (!y && !y_f32) return fail(MOE_E_INVALID, "y and y_f32 are both NULL");
    Layer& L = layer->L;
    if (L.d.cache_slots > 0) return fail(MOE_E_UNSUPPORTED, "static-scratch decode of a streamed layer");
    // size check first: an oversized layer is rejected before any CUDA call
    size_t off[kParts];
    layout(L, off);
    const size_t need = off[kParts - 1];
    if (need > MOE_STATIC_SCRATCH_BYTES)
        return fail(MOE_E_INVALID, "layer needs " + std::to_string(need) +
                                       " bytes of decode scratch; the static region holds " +
                                       std::to_string((size_t)MOE_STATIC_SCRATCH_BYTES));
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    unsigned char* base = nullptr;
    const moe_status st = region_for(L.device, &base);
    if (st != MOE_OK) return st;
    const DecodeScratch sc = carve(L, base);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_route_decode(L, x, s, 1, nullptr, nullptr, 0, nullptr, &sc);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");
    e = launch_experts_decode(L, x, y, y_f32, sc, 0, L.d.top_k + L.d.n_shared, true, true, false, s);
    if (e != cudaSuccess) return cuda_fail(e, "expert launch");
    return MOE_OK;
}
