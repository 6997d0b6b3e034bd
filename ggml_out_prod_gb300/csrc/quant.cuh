// quant.cuh -- src0 element types: block sizes and one-element decoders.
//
// The element types of src0 that OUT_PROD takes ("Metal
// kernel_mul_mat_id_back", first bullet: the op is instantiated for f32, f16,
// bf16, q4_0, q4_1, q5_0, q5_1, q8_0 and q2_K .. q6_K, out_prod's set; the
// dense timings of "metal: OUT_PROD multiplies in float staging", answer (2),
// use a q4_K weight).  The block layouts are ggml's published formats; the
// type ids are ggml's.  Every decoder returns the element's value rounded once
// to fp32: the integer parts are exact, products of a binary16 scale and a
// small integer are exact, and a scale-times-code minus an offset is one fused
// multiply-add.
#pragma once

#include <cstdint>

#include "oop_internal.cuh"

namespace oop {

// Elements per block (1 for the plain types) and bytes per block.
template <int TYPE>
struct QFormat;
template <> struct QFormat<OOP_TYPE_F32>  { static constexpr int QK = 1, BYTES = 4; };
template <> struct QFormat<OOP_TYPE_F16>  { static constexpr int QK = 1, BYTES = 2; };
template <> struct QFormat<OOP_TYPE_BF16> { static constexpr int QK = 1, BYTES = 2; };
template <> struct QFormat<OOP_TYPE_Q4_0> { static constexpr int QK = 32, BYTES = 18; };
template <> struct QFormat<OOP_TYPE_Q4_1> { static constexpr int QK = 32, BYTES = 20; };
template <> struct QFormat<OOP_TYPE_Q5_0> { static constexpr int QK = 32, BYTES = 22; };
template <> struct QFormat<OOP_TYPE_Q5_1> { static constexpr int QK = 32, BYTES = 24; };
template <> struct QFormat<OOP_TYPE_Q8_0> { static constexpr int QK = 32, BYTES = 34; };
template <> struct QFormat<OOP_TYPE_Q2_K> { static constexpr int QK = 256, BYTES = 84; };
template <> struct QFormat<OOP_TYPE_Q3_K> { static constexpr int QK = 256, BYTES = 110; };
template <> struct QFormat<OOP_TYPE_Q4_K> { static constexpr int QK = 256, BYTES = 144; };
template <> struct QFormat<OOP_TYPE_Q5_K> { static constexpr int QK = 256, BYTES = 176; };
template <> struct QFormat<OOP_TYPE_Q6_K> { static constexpr int QK = 256, BYTES = 210; };

// Whether a value of the type, split into TF32 hi + lo, leaves a remainder
// that needs rounding: types whose values have at most 22 significant bits
// (a binary16 scale times a code of up to 8 bits, with no offset) split
// exactly; f32 and the types with an offset (or a 6-bit scale times a 6-bit
// code) can carry all 24.
template <int TYPE>
constexpr bool split_needs_rounding() {
    return TYPE == OOP_TYPE_F32 || TYPE == OOP_TYPE_Q4_1 || TYPE == OOP_TYPE_Q5_1 ||
           TYPE == OOP_TYPE_Q2_K || TYPE == OOP_TYPE_Q4_K || TYPE == OOP_TYPE_Q5_K ||
           TYPE == OOP_TYPE_Q6_K;
}

// Values that are TF32 values already (11 significant bits or fewer, in
// fp32's exponent range): their lo term is zero.
template <int TYPE>
constexpr bool is_tf32_exact() {
    return TYPE == OOP_TYPE_BF16 || TYPE == OOP_TYPE_F16;
}

template <int TYPE>
constexpr bool is_plain_type() {
    return QFormat<TYPE>::QK == 1;
}

namespace qdec {

__device__ __forceinline__ uint32_t u8(const uint8_t *p) { return p[0]; }
// Little-endian 16- and 32-bit fields at 2-byte aligned addresses.
__device__ __forceinline__ uint32_t u16(const uint8_t *p) {
    return *reinterpret_cast<const uint16_t *>(p);
}
__device__ __forceinline__ uint32_t u32(const uint8_t *p) {
    return u16(p) | (u16(p + 2) << 16);
}
__device__ __forceinline__ float f16(const uint8_t *p) {
    return half_bits_to_float(static_cast<uint16_t>(u16(p)));
}

// The 6-bit scale and offset of sub-block j (0..7) from the 12 packed bytes
// of q4_K / q5_K: j < 4 in the low six bits of bytes j and j+4; j >= 4 in
// the nibbles of byte j+4 with their top two bits in the top bits of bytes
// j-4 and j.
__device__ __forceinline__ void scale_min_k4(const uint8_t *sc, int j, uint32_t &s, uint32_t &m) {
    if (j < 4) {
        s = sc[j] & 63u;
        m = sc[j + 4] & 63u;
    } else {
        s = (sc[j + 4] & 0xFu) | ((sc[j - 4] >> 6) << 4);
        m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
}

// The 6-bit scale s (0..15) of q3_K from its 12 packed bytes: the low four
// bits in a nibble of bytes 0..7 (low nibbles for s < 8, high for s >= 8), the
// top two in bits 2*(s/4) of byte 8 + s%4.
__device__ __forceinline__ int scale_q3k(const uint8_t *sc, int s) {
    const uint32_t lo = s < 8 ? (sc[s] & 0xFu) : (sc[s - 8] >> 4);
    const uint32_t hi = (sc[8 + (s & 3)] >> (2 * (s >> 2))) & 3u;
    return static_cast<int>(lo | (hi << 4)) - 32;
}

}  // namespace qdec

// Element j of the block at `blk` (j < QK; for the plain types blk points at
// the element itself and j is 0).
template <int TYPE>
__device__ __forceinline__ float decode(const uint8_t *blk, int j) {
    using namespace qdec;
    if constexpr (TYPE == OOP_TYPE_F32) {
        return *reinterpret_cast<const float *>(blk);
    } else if constexpr (TYPE == OOP_TYPE_F16) {
        return f16(blk);
    } else if constexpr (TYPE == OOP_TYPE_BF16) {
        return bf16_bits_to_float(static_cast<uint16_t>(u16(blk)));
    } else if constexpr (TYPE == OOP_TYPE_Q8_0) {
        return f16(blk) * static_cast<float>(static_cast<int8_t>(blk[2 + j]));
    } else if constexpr (TYPE == OOP_TYPE_Q4_0 || TYPE == OOP_TYPE_Q4_1) {
        // 16 bytes of codes after the header: byte i holds element i (low
        // nibble) and element i + 16 (high nibble)
        constexpr int H = TYPE == OOP_TYPE_Q4_0 ? 2 : 4;
        const uint32_t byte = blk[H + (j & 15)];
        const int v = static_cast<int>(j < 16 ? (byte & 0xFu) : (byte >> 4));
        if constexpr (TYPE == OOP_TYPE_Q4_0) return f16(blk) * static_cast<float>(v - 8);
        else return fmaf(f16(blk), static_cast<float>(v), f16(blk + 2));
    } else if constexpr (TYPE == OOP_TYPE_Q5_0 || TYPE == OOP_TYPE_Q5_1) {
        // header, then 32 fifth bits (bit i of the little-endian word is
        // element i's), then the 16 bytes of low nibbles as in q4_0
        constexpr int QH = TYPE == OOP_TYPE_Q5_0 ? 2 : 4;
        const uint32_t byte = blk[QH + 4 + (j & 15)];
        const uint32_t lo = j < 16 ? (byte & 0xFu) : (byte >> 4);
        const uint32_t hb = (u32(blk + QH) >> j) & 1u;
        const int v = static_cast<int>(lo | (hb << 4));
        if constexpr (TYPE == OOP_TYPE_Q5_0) return f16(blk) * static_cast<float>(v - 16);
        else return fmaf(f16(blk), static_cast<float>(v), f16(blk + 2));
    } else if constexpr (TYPE == OOP_TYPE_Q4_K || TYPE == OOP_TYPE_Q5_K) {
        // d, dmin, 12 bytes of packed 6-bit scales and offsets of the eight
        // 32-element sub-blocks, [q5_K: 32 bytes of fifth bits, bit sb of
        // byte l for element l of sub-block sb,] then 128 bytes of nibbles:
        // bytes 32*p .. 32*p+31 hold sub-block 2p (low) and 2p+1 (high)
        constexpr int QS = TYPE == OOP_TYPE_Q4_K ? 16 : 48;
        const int sb = j >> 5, l = j & 31;
        uint32_t sc, mn;
        scale_min_k4(blk + 4, sb, sc, mn);
        uint32_t q = (blk[QS + 32 * (sb >> 1) + l] >> (4 * (sb & 1))) & 0xFu;
        if constexpr (TYPE == OOP_TYPE_Q5_K) q |= ((blk[16 + l] >> sb) & 1u) << 4;
        return fmaf(f16(blk) * static_cast<float>(sc), static_cast<float>(q),
                    -(f16(blk + 2) * static_cast<float>(mn)));
    } else if constexpr (TYPE == OOP_TYPE_Q6_K) {
        // 128 bytes of low nibbles, 64 of two-bit high parts, 16 int8 scales,
        // then d.  Half h (128 elements) takes low-nibble bytes 64h..,
        // high-part bytes 32h.. and scales 8h..; its element 32g + l (g < 4)
        // has the low nibble of byte 64h + l + 32(g&1) (high nibble for g >= 2),
        // bits 2g..2g+1 of high-part byte 32h + l and scale 8h + l/16 + 2g.
        const int h = j >> 7, g = (j >> 5) & 3, l = j & 31;
        const uint32_t byte = blk[64 * h + l + 32 * (g & 1)];
        const uint32_t lo = g >= 2 ? (byte >> 4) : (byte & 0xFu);
        const uint32_t hi = (blk[128 + 32 * h + l] >> (2 * g)) & 3u;
        const int q = static_cast<int>(lo | (hi << 4)) - 32;
        const int sc = static_cast<int8_t>(blk[192 + 8 * h + (l >> 4) + 2 * g]);
        return f16(blk + 208) * static_cast<float>(sc) * static_cast<float>(q);
    } else if constexpr (TYPE == OOP_TYPE_Q2_K) {
        // 16 scale bytes (low nibble scale, high nibble offset), 64 bytes of
        // 2-bit codes, d, dmin.  Element 128h + 32g + l: bits 2g..2g+1 of code
        // byte 32h + l, scale byte 8h + 2g + l/16.
        const int h = j >> 7, g = (j >> 5) & 3, l = j & 31;
        const uint32_t q = (blk[16 + 32 * h + l] >> (2 * g)) & 3u;
        const uint32_t s = blk[8 * h + 2 * g + (l >> 4)];
        return fmaf(f16(blk + 80) * static_cast<float>(s & 0xFu), static_cast<float>(q),
                    -(f16(blk + 82) * static_cast<float>(s >> 4)));
    } else if constexpr (TYPE == OOP_TYPE_Q3_K) {
        // 32 bytes of third bits, 64 bytes of 2-bit codes, 12 bytes of packed
        // 6-bit scales, d.  Element 128h + 32g + l: bits 2g..2g+1 of code byte
        // 32h + l, third bit 4h + g of byte l (clear: the code is less 4),
        // scale 8h + 2g + l/16 (stored plus 32).
        const int h = j >> 7, g = (j >> 5) & 3, l = j & 31;
        const int q2 = static_cast<int>((blk[32 + 32 * h + l] >> (2 * g)) & 3u);
        const int q = q2 - (((blk[l] >> (4 * h + g)) & 1u) ? 0 : 4);
        const int sc = scale_q3k(blk + 96, 8 * h + 2 * g + (l >> 4));
        return f16(blk + 108) * static_cast<float>(sc) * static_cast<float>(q);
    }
}

// Element m of a row of M elements of `TYPE` starting at `row`.
template <int TYPE>
__device__ __forceinline__ float decode_row(const uint8_t *row, int64_t m) {
    using F = QFormat<TYPE>;
    return decode<TYPE>(row + (m / F::QK) * F::BYTES, static_cast<int>(m % F::QK));
}

}  // namespace oop
