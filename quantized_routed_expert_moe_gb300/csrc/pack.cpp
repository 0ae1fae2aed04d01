// Host-side packing of canonical quantised experts into the kernel layout
// (row records, gate/up rows interleaved; see moe_internal.h).
#include <cstring>

#include "moe_internal.h"

namespace moe {

static void pack_row(const uint8_t* codes, const uint16_t* scale, const uint16_t* bias, int K,
                     uint8_t* dst) {
    std::memcpy(dst, codes, (size_t)K / 2);
    uint8_t* meta = dst + K / 2;
    const int G = K / 64;
    for (int g = 0; g < G; ++g) {
        std::memcpy(meta + 4 * g, scale + g, 2);
        std::memcpy(meta + 4 * g + 2, bias + g, 2);
    }
    std::memset(meta + 4 * G, 0, row_meta_bytes(K) - 4 * (size_t)G);
}

void pack_expert(int H, int I, const moe_expert& e, uint8_t* dst) {
    const size_t rbH = row_bytes(H), rbI = row_bytes(I);
    const int GH = H / 64, GI = I / 64;
    for (int i = 0; i < I; ++i) {
        pack_row(e.gate.codes + (size_t)i * (H / 2), e.gate.scale + (size_t)i * GH,
                 e.gate.bias + (size_t)i * GH, H, dst + (size_t)(2 * i) * rbH);
        pack_row(e.up.codes + (size_t)i * (H / 2), e.up.scale + (size_t)i * GH,
                 e.up.bias + (size_t)i * GH, H, dst + (size_t)(2 * i + 1) * rbH);
    }
    uint8_t* d = dst + gu_block_bytes(H, I);
    for (int n = 0; n < H; ++n)
        pack_row(e.down.codes + (size_t)n * (I / 2), e.down.scale + (size_t)n * GI,
                 e.down.bias + (size_t)n * GI, I, d + (size_t)n * rbI);
}

}  // namespace moe
