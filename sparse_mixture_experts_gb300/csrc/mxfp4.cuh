// mxfp4.cuh -- MXFP4 (E2M1 codes, one E8M0 scale per 32 elements) to bf16,
// exactly, for the tensor-core kernels' weight operands.
//
// Format ("Phase 19: MoE -- gpt-oss-20b", the MXFP4 packing note under the
// measured tensor layout, and section 3 on MXFP4 dequantisation): an element is
// e2m1(code) * 2^(e8m0 - 127); the low nibble of a byte is the even element.
// E2M1 (sign, 2 exponent bits, 1 mantissa bit) has the magnitudes 0, 0.5, 1,
// 1.5, 2, 3, 4, 6.  Every magnitude times a power of two has at most two
// significant bits, so it is a bf16 number whenever it is an fp32 number: for
// every scale byte 0..254 (2^-127 is the fp32 subnormal 0x00400000; products
// beyond the fp32 range are infinite, as in IEEE arithmetic), and byte 255
// (NaN) gives NaN.
//
// Conversion: per scale byte, a 16-byte table of the eight magnitudes' bf16
// patterns (high bytes, then low bytes) computed with fp32 arithmetic; per
// eight codes (one 32-bit word), four byte-permutes look up the high and low
// bytes of the magnitudes, two more place the sign bits into the high bytes,
// and four interleave the bytes into bf16 pairs (even element in the low
// half).  The same code compiles for the host (with the byte permute written
// out), which is how it is tested against the format's definition.
#pragma once

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define MXFP4_HD __host__ __device__ __forceinline__
#else
#define MXFP4_HD inline
#endif

namespace moe {

// the eight byte tables of one scale: magnitude m's bf16 pattern is
// (hi[m] << 8) | lo[m]; hi[0..3] in ah, hi[4..7] in bh, likewise lo
struct Fp4Table {
    uint32_t ah, bh, al, bl;
};

MXFP4_HD float mxfp4_bits_float(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

MXFP4_HD uint32_t mxfp4_float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

// byte permute: result byte i = byte (c >> 4i) & 7 of the pair {a (bytes 0-3), b (bytes 4-7)}
MXFP4_HD uint32_t mxfp4_prmt(uint32_t a, uint32_t b, uint32_t c)
{
#if defined(__CUDA_ARCH__)
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
#else
    const uint64_t ab = ((uint64_t)b << 32) | a;
    uint32_t d = 0;
    for (int i = 0; i < 4; ++i) {
        const uint32_t sel = (c >> (4 * i)) & 0xfu;
        uint32_t byte = (uint32_t)(ab >> (8 * (sel & 7u))) & 0xffu;
        if (sel & 8u) byte = (byte & 0x80u) ? 0xffu : 0u;  // sign-replicate mode (unused here)
        d |= byte << (8 * i);
    }
    return d;
#endif
}

// the table of scale byte s (0..255)
MXFP4_HD Fp4Table mxfp4_table(uint32_t s)
{
    // 2^(s - 127): the fp32 exponent field is s itself, except s = 0
    // (2^-127, a subnormal) and s = 255 (NaN in E8M0)
    const float scale = mxfp4_bits_float(s == 0 ? 0x00400000u : s == 255 ? 0x7fc00000u : (s << 23));
    const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint32_t hi[8], lo[8];
    for (int m = 0; m < 8; ++m) {
        const uint32_t v = mxfp4_float_bits(mag[m] * scale) >> 16;  // exact: at most two significant bits
        hi[m] = v >> 8;
        lo[m] = v & 0xffu;
    }
    Fp4Table t;
    t.ah = hi[0] | hi[1] << 8 | hi[2] << 16 | hi[3] << 24;
    t.bh = hi[4] | hi[5] << 8 | hi[6] << 16 | hi[7] << 24;
    t.al = lo[0] | lo[1] << 8 | lo[2] << 16 | lo[3] << 24;
    t.bl = lo[4] | lo[5] << 8 | lo[6] << 16 | lo[7] << 24;
    return t;
}

// eight codes (nibble i = element i) -> four bf16 pairs: o[j] holds elements
// 2j (low half) and 2j + 1
MXFP4_HD void mxfp4_to_bf16x8(uint32_t w, const Fp4Table &t, uint32_t (&o)[4])
{
    const uint32_t idx = w & 0x77777777u;           // magnitudes
    uint32_t hi0 = mxfp4_prmt(t.ah, t.bh, idx);       // high bytes of elements 0..3
    uint32_t lo0 = mxfp4_prmt(t.al, t.bl, idx);
    uint32_t hi1 = mxfp4_prmt(t.ah, t.bh, idx >> 16); // elements 4..7
    uint32_t lo1 = mxfp4_prmt(t.al, t.bl, idx >> 16);
    // sign of element i (bit 4i + 3) to bit 7 of high byte i
    const uint32_t ev = (w << 4) & 0x80808080u;      // elements 0, 2, 4, 6 at bit 7 of bytes 0..3
    const uint32_t od = w & 0x80808080u;             // elements 1, 3, 5, 7
    hi0 |= mxfp4_prmt(ev, od, 0x5140u);
    hi1 |= mxfp4_prmt(ev, od, 0x7362u);
    o[0] = mxfp4_prmt(lo0, hi0, 0x5140u);
    o[1] = mxfp4_prmt(lo0, hi0, 0x7362u);
    o[2] = mxfp4_prmt(lo1, hi1, 0x5140u);
    o[3] = mxfp4_prmt(lo1, hi1, 0x7362u);
}

}  // namespace moe
