// Prints, for every E8M0 scale byte and every E2M1 code, the bf16 pattern the
// tensor-core kernels' MXFP4 conversion produces (host build of the same code).
#include <cstdio>

#include "mxfp4.cuh"

int main()
{
    for (unsigned s = 0; s < 256; ++s) {
        const moe::Fp4Table t = moe::mxfp4_table(s);
        // codes 0..7 in one word and 8..15 in another, plus a mixed word
        const uint32_t words[3] = {0x76543210u, 0xfedcba98u, 0x1f2e3d4cu};
        for (uint32_t w : words) {
            uint32_t o[4];
            moe::mxfp4_to_bf16x8(w, t, o);
            for (int i = 0; i < 8; ++i) {
                const unsigned code = (w >> (4 * i)) & 0xfu;
                const unsigned bits = (o[i / 2] >> (16 * (i & 1))) & 0xffffu;
                printf("%u %u %u\n", s, code, bits);
            }
        }
    }
    return 0;
}
