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

// 2-bit row: canonical codes (element k in byte k/4, bits 2 (k % 4)) into the
// kernel's per-run arrangement (moe_internal.h), then the meta as for 4 bits.
static void pack_row2(const uint8_t* codes, const uint16_t* scale, const uint16_t* bias, int K,
                      uint8_t* dst) {
    auto code = [&](int k) { return (codes[k >> 2] >> (2 * (k & 3))) & 3; };
    for (int w = 0; w < K / 16; ++w)
        for (int i = 0; i < 4; ++i) {
            const int k0 = 16 * w;
            dst[4 * w + i] = (uint8_t)(code(k0 + 2 * i) | code(k0 + 2 * i + 1) << 2 | code(k0 + 8 + 2 * i) << 4 |
                                       code(k0 + 9 + 2 * i) << 6);
        }
    uint8_t* meta = dst + K / 4;
    const int G = K / 64;
    for (int g = 0; g < G; ++g) {
        std::memcpy(meta + 4 * g, scale + g, 2);
        std::memcpy(meta + 4 * g + 2, bias + g, 2);
    }
    std::memset(meta + 4 * G, 0, row_meta_bytes(K) - 4 * (size_t)G);
}

void pack_expert(int H, int I, int bits, const moe_expert& e, uint8_t* dst) {
    const size_t rbH = row_bytes(H, bits), rbI = row_bytes(I, bits);
    auto row = [&](const moe_qmat& q, size_t r, int K, uint8_t* out) {
        const int G = K / 64;
        const uint8_t* c = q.codes + r * ((size_t)K * bits / 8);
        if (bits == 2) pack_row2(c, q.scale + r * G, q.bias + r * G, K, out);
        else pack_row(c, q.scale + r * G, q.bias + r * G, K, out);
    };
    for (int i = 0; i < I; ++i) {
        row(e.gate, i, H, dst + (size_t)(2 * i) * rbH);
        row(e.up, i, H, dst + (size_t)(2 * i + 1) * rbH);
    }
    uint8_t* d = dst + gu_block_bytes(H, I, bits);
    for (int n = 0; n < H; ++n) row(e.down, n, I, d + (size_t)n * rbI);
}

}  // namespace moe
