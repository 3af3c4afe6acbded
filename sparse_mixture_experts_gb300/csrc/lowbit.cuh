// lowbit.cuh -- the low-bit expert formats, widened exactly (MXFP4) or
// rounded once (Q4) to bf16 for the tensor-core kernels' weight operands, and
// the packed block both kernels stream: per (128 weight rows, 64-wide K block)
// the codes as [2 halves][128 rows][16 B] (half h = K elements 32h .. 32h+31,
// byte b of a row's 16 = elements 2b (low nibble) and 2b + 1 (high nibble)),
// then the scales as [2 halves][128 rows] (one E8M0 byte, or one binary16).
//
// MXFP4 ("Phase 19: MoE -- gpt-oss-20b", the MXFP4 packing note under the
// measured tensor layout, and section 3 on MXFP4 dequantisation): an element
// is e2m1(code) * 2^(e8m0 - 127); the low nibble of a byte is the even element.
// E2M1 (sign, 2 exponent bits, 1 mantissa bit) has the magnitudes 0, 0.5, 1,
// 1.5, 2, 3, 4, 6.  Every magnitude times a power of two has at most two
// significant bits, so it is a bf16 number whenever it is an fp32 number: for
// every scale byte 0..254 (2^-127 is the fp32 subnormal 0x00400000; products
// beyond the fp32 range are infinite, as in IEEE arithmetic), and byte 255
// (NaN) gives NaN.  Conversion: per scale byte, a 16-byte table of the eight
// magnitudes' bf16 patterns (high bytes, then low bytes) computed with fp32
// arithmetic; per eight codes (one 32-bit word), four byte-permutes look up
// the high and low bytes of the magnitudes, two more place the sign bits into
// the high bytes, and four interleave the bytes into bf16 pairs (even element
// in the low half).
//
// Q4 ("Engine" (cherenkov), section "Prefill": Q4 GEMMs with half weights and
// float accumulation; records as the ggml-Q4_0 rows named under "Qwen3.5-MoE
// Model Implementation", KV Cache): 32 elements share a binary16 scale d, an
// element is (code - 8) * d.  code - 8 is exact in fp32 (the code is placed in
// the mantissa of 2^23 and 2^23 + 8 subtracted), and so is its product with d
// (4 bits times 11); the product is rounded once to bf16, nearest even -- the
// 16-bit ("half") weight of the pages, in the layer's activation type.
//
// The same code compiles for the host (the byte permute and the rounding
// written out), which is how it is tested against the formats' definitions.
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

// ---- Q4 ----

// binary16 bit pattern -> float (exact)
MXFP4_HD float q4_half_to_float(uint32_t h)
{
    const uint32_t sign = (h & 0x8000u) << 16, e = (h >> 10) & 31u, m = h & 1023u;
    if (e == 0) {
        // zero or subnormal: m * 2^-24, exact in fp32
        const float v = (float)m * mxfp4_bits_float(0x33800000u);  // 2^-24
        return sign ? -v : v;
    }
    if (e == 31) return mxfp4_bits_float(sign | 0x7f800000u | (m << 13));
    return mxfp4_bits_float(sign | ((e + 112u) << 23) | (m << 13));
}

// float -> bf16 bits, round to nearest even (NaN stays NaN)
MXFP4_HD uint32_t q4_bf16_rne(float f)
{
#if defined(__CUDA_ARCH__)
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
#else
    const uint32_t u = mxfp4_float_bits(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) return (u >> 16) | 0x40u;
    return (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
#endif
}

MXFP4_HD float q4_bf16_float(uint32_t b) { return mxfp4_bits_float(b << 16); }

// binary16 bit pattern -> float (exact): the hardware conversion on the device
MXFP4_HD float q4_scale_float(uint32_t h)
{
#if defined(__CUDA_ARCH__)
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((unsigned short)h));
    return f;
#else
    return q4_half_to_float(h);
#endif
}

// A Q4 scale d (binary16 bits) split into two bf16 values, d = hi + lo
// exactly: hi = d truncated to bf16 (toward zero: the high half of d's fp32
// pattern), lo = d - hi, computed exactly in fp32; d has at most 11
// significant bits and hi keeps the first 8, so lo has at most three and d's
// sign and is a bf16 value too (the high half of its fp32 pattern).  A zero
// lo carries d's sign as well, so that code 8 times d gives the zero of d's
// sign; lo = 0 (with d's sign) for an infinite or NaN d.  Returned as bf16
// pairs (the value in both halves).
MXFP4_HD void q4_split_scale(uint32_t h16, uint32_t &hi2, uint32_t &lo2)
{
    const float d = q4_scale_float(h16);
    const uint32_t db = mxfp4_float_bits(d);
    const uint32_t hi = db >> 16;
    const float r = d - mxfp4_bits_float(db & 0xffff0000u);  // exact
    uint32_t lo = ((mxfp4_float_bits(r) >> 16) & 0x7fffu) | (h16 & 0x8000u);
    if (((h16 >> 10) & 31u) == 31u) lo = h16 & 0x8000u;
    hi2 = hi | (hi << 16);
    lo2 = lo | (lo << 16);
}

// d = a * b + c on bf16 pairs with one rounding (to nearest even) per half
MXFP4_HD uint32_t q4_fma_bf16x2(uint32_t a, uint32_t b, uint32_t c)
{
#if defined(__CUDA_ARCH__)
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
#else
    // the operands of the conversion below keep a * b + c exact in fp32:
    // products of at most 12 significant bits, sums spanning at most 22
    uint32_t d = 0;
    for (int k = 0; k < 2; ++k) {
        const float x = q4_bf16_float((a >> (16 * k)) & 0xffffu), y = q4_bf16_float((b >> (16 * k)) & 0xffffu),
                    z = q4_bf16_float((c >> (16 * k)) & 0xffffu);
        d |= q4_bf16_rne(x * y + z) << (16 * k);
    }
    return d;
#endif
}

// Eight codes of a packed Q4 word with the split scale of their record ->
// four bf16 pairs: o[j] holds elements 2j (low half) and 2j + 1.  The packed
// word keeps element 2j in nibble j and element 2j + 1 in nibble j + 4, so
// one mask takes both codes of a pair into the low bits of a bf16 pair:
//   p = 128 + code (bf16: exponent 7, the code in the low mantissa bits),
//   v = p - 136 = code - 8 (exact), t = v * lo (exact: at most 7 bits),
//   o = v * hi + t, rounded once: the bf16 rounding of (code - 8) * d.
MXFP4_HD void q4_to_bf16x8(uint32_t w, uint32_t hi2, uint32_t lo2, uint32_t (&o)[4])
{
#if defined(__CUDACC__)
#pragma unroll
#endif
    for (int j = 0; j < 4; ++j) {
        const uint32_t p = ((w >> (4 * j)) & 0x000f000fu) | 0x43004300u;
        const uint32_t v = q4_fma_bf16x2(p, 0x3f803f80u, 0xc308c308u);  // p * 1 - 136
        const uint32_t t = q4_fma_bf16x2(v, lo2, 0x80008000u);           // v * lo - 0
        o[j] = q4_fma_bf16x2(v, hi2, t);
    }
}

// nibble position, in its packed word, of element i (0..7) of the word
MXFP4_HD int q4_nibble_of(int i) { return (i & 1) ? 4 + (i >> 1) : (i >> 1); }

// bytes of one packed block: codes, then the scales
constexpr int LOWBIT_CODE_BYTES = 128 * 32;
constexpr int LOWBIT_BLK_MXFP4 = LOWBIT_CODE_BYTES + 128 * 2;      // an E8M0 byte per row and half
constexpr int LOWBIT_BLK_Q4 = LOWBIT_CODE_BYTES + 128 * 2 * 2;     // a binary16 per row and half

#if defined(__CUDACC__)
// Row r of a packed low-bit block as loaded from shared memory: its eight
// code words (K elements 0..31, then 32..63) and its two scales (an E8M0
// byte, or a binary16, per half).
struct LowbitRow {
    uint32_t w[8];
    uint32_t s0, s1;
};

// The loads of row r of a block (both halves first, so that their latencies
// overlap).  The caller may release the block once this returns.
template <int QF>
__device__ __forceinline__ void lowbit_load_row(const uint8_t *blk, int r, LowbitRow &row)
{
    const uint4 c0 = *reinterpret_cast<const uint4 *>(blk + r * 16);
    const uint4 c1 = *reinterpret_cast<const uint4 *>(blk + (128 + r) * 16);
    row.w[0] = c0.x; row.w[1] = c0.y; row.w[2] = c0.z; row.w[3] = c0.w;
    row.w[4] = c1.x; row.w[5] = c1.y; row.w[6] = c1.z; row.w[7] = c1.w;
    if constexpr (QF == 1) {
        row.s0 = blk[LOWBIT_CODE_BYTES + r];
        row.s1 = blk[LOWBIT_CODE_BYTES + 128 + r];
    } else {
        const uint16_t *sc = reinterpret_cast<const uint16_t *>(blk + LOWBIT_CODE_BYTES);
        row.s0 = sc[r];
        row.s1 = sc[128 + r];
    }
}

// A loaded row widened to bf16: v[c] holds elements 2c (low half) and 2c + 1,
// c = 0..31, i.e. the 64 K elements of the block in order.  MXFP4: exact, by
// the scale byte's table (tabs, in shared memory); Q4: (code - 8) * d rounded
// once to bf16.
template <int QF>
__device__ __forceinline__ void lowbit_widen_row(const LowbitRow &row, const Fp4Table *tabs, uint32_t (&v)[32])
{
    if constexpr (QF == 1) {
        const Fp4Table t0 = tabs[row.s0];
        const Fp4Table t1 = tabs[row.s1];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t o[4];
            mxfp4_to_bf16x8(row.w[q], q < 4 ? t0 : t1, o);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[q * 4 + i] = o[i];
        }
    } else {
        uint32_t hi0, lo0, hi1, lo1;
        q4_split_scale(row.s0, hi0, lo0);
        q4_split_scale(row.s1, hi1, lo1);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t o[4];
            q4_to_bf16x8(row.w[q], q < 4 ? hi0 : hi1, q < 4 ? lo0 : lo1, o);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[q * 4 + i] = o[i];
        }
    }
}

// Half h (K elements 32h .. 32h+31) of row r of a packed block: its four code
// words and its scale.
struct LowbitHalf {
    uint32_t w[4];
    uint32_t s;
};

template <int QF>
__device__ __forceinline__ void lowbit_load_half(const uint8_t *blk, int r, int h, LowbitHalf &x)
{
    const uint4 c = *reinterpret_cast<const uint4 *>(blk + (h * 128 + r) * 16);
    x.w[0] = c.x; x.w[1] = c.y; x.w[2] = c.z; x.w[3] = c.w;
    if constexpr (QF == 1) x.s = blk[LOWBIT_CODE_BYTES + h * 128 + r];
    else x.s = reinterpret_cast<const uint16_t *>(blk + LOWBIT_CODE_BYTES)[h * 128 + r];
}

// A loaded half widened to bf16: v[c] holds its elements 2c (low half) and 2c + 1
template <int QF>
__device__ __forceinline__ void lowbit_widen_half(const LowbitHalf &x, const Fp4Table *tabs, uint32_t (&v)[16])
{
    if constexpr (QF == 1) {
        const Fp4Table t = tabs[x.s];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t o[4];
            mxfp4_to_bf16x8(x.w[q], t, o);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[q * 4 + i] = o[i];
        }
    } else {
        uint32_t hi, lo;
        q4_split_scale(x.s, hi, lo);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t o[4];
            q4_to_bf16x8(x.w[q], hi, lo, o);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[q * 4 + i] = o[i];
        }
    }
}

// Row r of a packed low-bit block (QF 1: MXFP4, 2: Q4) widened to bf16 (the
// two row steps above).
template <int QF>
__device__ __forceinline__ void lowbit_dequant_row(const uint8_t *blk, int r, const Fp4Table *tabs, uint32_t (&v)[32])
{
    LowbitRow row;
    lowbit_load_row<QF>(blk, r, row);
    lowbit_widen_row<QF>(row, tabs, v);
}
#endif

}  // namespace moe
