// moe_decode_static_scratch: the split decode path over scratch that lives in
// a fixed region of this library's device image, so the call allocates
// nothing. It exists for callers that may not allocate device memory while
// serving: cudaMalloc/cudaFree can synchronise the device and stall every
// other stream, an engine that has already divided HBM among weights and
// caches has no room to give, and a caching allocator asked for a block then
// may have to grow its pool. The weights and the layer itself are set up once,
// at creation; this file adds no allocation of any kind on the call path.
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

// One region per device (a __device__ variable is instantiated on every
// device the module is loaded on).
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_base[kMaxDevices] = {};

inline size_t up256(size_t n) { return (n + 255) / 256 * 256; }

struct StaticScratch {
    float* part;
    float* logits;
    int32_t* ids;
    float* wts;
    float* h;
    size_t bytes;
};

// Byte offsets of the pieces within the region; the last entry is the total.
void layout(const Layer& L, size_t off[6]) {
    const auto& d = L.d;
    const size_t E = d.n_experts, k = d.top_k;
    off[0] = 0;                                                  // partial logits [splits][E]
    off[1] = off[0] + up256((size_t)L.router_splits * E * 4);    // logits [E]
    off[2] = off[1] + up256(E * 4);                              // ids [k]
    off[3] = off[2] + up256(k * 4);                              // weights [k]
    off[4] = off[3] + up256(k * 4);                              // SwiGLU outputs [k + 1][I]
    off[5] = off[4] + up256((k + 1) * (size_t)d.inter * 4);
}

StaticScratch carve(const Layer& L, unsigned char* base) {
    size_t off[6];
    layout(L, off);
    StaticScratch s{};
    s.part = reinterpret_cast<float*>(base + off[0]);
    s.logits = reinterpret_cast<float*>(base + off[1]);
    s.ids = reinterpret_cast<int32_t*>(base + off[2]);
    s.wts = reinterpret_cast<float*>(base + off[3]);
    s.h = reinterpret_cast<float*>(base + off[4]);
    s.bytes = off[5];
    return s;
}

// Device address of this device's region, looked up once per device with
// that device current. The caller holds a DeviceGuard for `dev`.
moe_status region_for(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_E_UNSUPPORTED, "device ordinal above the static-scratch table");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_base[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        if (!p) return fail(MOE_E_CUDA, "cudaGetSymbolAddress(static scratch) returned NULL");
        g_base[dev] = p;
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
    size_t off[6];
    layout(L, off);
    const size_t need = off[5];
    if (need > MOE_STATIC_SCRATCH_BYTES)
        return fail(MOE_E_INVALID, "layer needs " + std::to_string(need) +
                                       " bytes of decode scratch; the static region holds " +
                                       std::to_string((size_t)MOE_STATIC_SCRATCH_BYTES));
    DeviceGuard g(L.device);
    if (!g.ok) return cuda_fail(g.err, "cudaSetDevice");
    unsigned char* base = nullptr;
    const moe_status st = region_for(L.device, &base);
    if (st != MOE_OK) return st;
    const StaticScratch sc = carve(L, base);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_route_decode_partials(L, x, sc.part, s);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");
    e = launch_experts_decode_scratch(L, x, y, y_f32, sc.part, sc.logits, sc.ids, sc.wts, sc.h, s);
    if (e != cudaSuccess) return cuda_fail(e, "expert launch");
    return MOE_OK;
}
