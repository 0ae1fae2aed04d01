// Router scoring of a layer as the kernels see it (host and device).
#pragma once

namespace moe {

// sigmoid: 1 for MOE_SCORE_SIGMOID, 0 for MOE_SCORE_SOFTMAX; scale: the routed
// scaling factor that multiplies the sigmoid weights.
struct RouteMode {
    int sigmoid;
    float scale;
};

}  // namespace moe
