// Prints the bf16 patterns the tensor-core kernels' low-bit conversions
// produce (host build of the same code, the bf16 pair FMAs emulated with one
// rounding each): "M s code bits" for every MXFP4 scale byte and code,
// "Q d code bits" for sampled binary16 Q4 scales.
#include <cstdio>

#include "lowbit.cuh"

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
                printf("M %u %u %u\n", s, code, bits);
            }
        }
    }
    for (unsigned h = 0; h < 65536; h += 251) {
        const unsigned hs[2] = {h, h ^ 0x8000u};
        for (unsigned d16 : hs) {
            if (((d16 >> 10) & 31u) == 31u) continue;  // scales are finite
            uint32_t hi2, lo2;
            moe::q4_split_scale(d16, hi2, lo2);
            const uint32_t words[2] = {0x76543210u, 0xfedcba98u};
            for (uint32_t w : words) {
                uint32_t o[4];
                moe::q4_to_bf16x8(w, hi2, lo2, o);
                for (int i = 0; i < 8; ++i) {
                    const unsigned code = (w >> (4 * moe::q4_nibble_of(i))) & 0xfu;
                    const unsigned bits = (o[i / 2] >> (16 * (i & 1))) & 0xffffu;
                    printf("Q %u %u %u\n", d16, code, bits);
                }
            }
        }
    }
    return 0;
}
