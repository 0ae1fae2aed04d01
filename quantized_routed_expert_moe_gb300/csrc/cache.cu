// Streamed expert cache (per-layer LFU slots filled from host records).
#include "moe_internal.h"

namespace moe {

struct CacheState {};

moe_status cache_create(Layer&, const void* const*, moe_expert_source, void*) {
    return fail(MOE_E_UNSUPPORTED, "streamed mode is not built yet");
}
void cache_destroy(Layer& L) { delete L.cache; L.cache = nullptr; }
moe_status cache_stage(Layer&, const int32_t*, int, cudaStream_t, int*, int*) {
    return fail(MOE_E_UNSUPPORTED, "streamed mode is not built yet");
}
moe_status cache_decode(Layer&, const void*, void*, float*, cudaStream_t) {
    return fail(MOE_E_UNSUPPORTED, "streamed mode is not built yet");
}

}  // namespace moe

extern "C" {
moe_status moe_cache_stats(const moe_layer* layer, moe_cache_stats_t* out) {
    if (!layer || !out) return moe::fail(MOE_E_INVALID, "NULL argument");
    *out = moe_cache_stats_t{};
    return MOE_OK;
}
moe_status moe_cache_residency(const moe_layer* layer, int32_t*) {
    if (!layer) return moe::fail(MOE_E_INVALID, "NULL argument");
    return moe::fail(MOE_E_STATE, "layer is not streamed");
}
}
