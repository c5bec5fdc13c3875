// kq_common.cuh -- shared device helpers and launch descriptors of libkq.
//
// Block layouts follow "Chapter 6 - The kquant family on the reference
// lane": Q4_K (Figure 6.2: d, dmin, 12-byte scale field, 128 B nibbles),
// Q5_K (Figure 6.4: the same plus a 32-byte high-bit plane before the
// nibbles), Q6_K (Figure 6.5: ql 128 B, qh 64 B, 16 int8 scales, f16 d last).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace kq {

constexpr int kFmtQ4K = 12;
constexpr int kFmtQ5K = 13;
constexpr int kFmtQ6K = 14;
constexpr int kMaxSet = 16;
constexpr int kMaxNtok = 8;

// One member of a launch: a matrix, its input planes and its output.
struct MatDesc {
    const uint8_t *W;   // rows * nb super-blocks, row-major
    const float *x;     // [ntok][nb * 256]
    float *y;           // [ntok][rows]
    int64_t rows;
    int32_t nb;         // super-blocks per row (cols / 256)
    int32_t fmt;        // kFmtQ4K / kFmtQ5K / kFmtQ6K
    int32_t cta_begin;  // first CTA of the grid that works on this member
    int32_t rpc;        // rows per CTA for this member
};

struct SetParams {
    MatDesc m[kMaxSet];
    int32_t n;
};

// ------------------------------------------------------------ conversions
// IEEE binary16 bits -> f32 (CUDA's conversion intrinsic).
__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}

// Integer 0 <= v < 2^23 -> f32, exactly: OR v into the mantissa of 2^23 and
// subtract 2^23 (both operands within a factor of two: the difference is
// exact).  Avoids the slow integer-to-float conversion unit.
__device__ __forceinline__ float u2f(uint32_t v) {
    return __int_as_float(0x4B000000u | v) - 8388608.0f;
}

// The signed byte held in the low 8 bits of v -> f32, exactly (bias by 128
// into 0..255, convert as above, remove the bias).
__device__ __forceinline__ float s8_to_f32(uint32_t v) {
    return __int_as_float(0x4B000000u | ((v ^ 0x80u) & 0xFFu)) -
           8388736.0f;  // 2^23 + 128
}

// ------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ldg_v4(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ uint32_t ldg_u32(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ float4 ldg_f4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// Input accessors for kq_blocks.cuh: x.ld(t, e) = inputs e..e+3 of token t.
struct XGlobal {  // read-only global loads (L1-cached)
    const float *p;
    int64_t plane;  // floats between token planes
    __device__ __forceinline__ float4 ld(int t, int e) const {
        return ldg_f4(p + t * plane + e);
    }
};
struct XShared {  // shared-memory copy of x
    uint32_t a;     // shared address of this block's first input, token 0
    uint32_t plane; // bytes between token planes
    __device__ __forceinline__ float4 ld(int t, int e) const {
        float4 v;
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                     : "r"(a + t * plane + 4 * e));
        return v;
    }
};

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ------------------------------------------------------------ scale field
// The 12-byte Q4_K/Q5_K scale field as three little-endian words s0,s1,s2
// (bytes 4..7, 8..11, 12..15 of the block).  Figure 6.3's rule, applied to
// four bytes at a time: the low words hold sc/m of sub-blocks 0..3 in their
// low six bits; sub-blocks 4..7 join the nibbles of s2 with the spare top
// two bits of s0 (scales) and s1 (mins).
struct ScaleWords {
    uint32_t sc_lo, m_lo, sc_hi, m_hi;  // byte j -> sub-block j (lo) / j+4
};

__device__ __forceinline__ ScaleWords unpack_scale_words(uint32_t s0,
                                                         uint32_t s1,
                                                         uint32_t s2) {
    ScaleWords w;
    w.sc_lo = s0 & 0x3F3F3F3Fu;
    w.m_lo = s1 & 0x3F3F3F3Fu;
    w.sc_hi = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
    w.m_hi = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
    return w;
}

// 6-bit scale and min of sub-block s (compile-time s after unrolling).
__device__ __forceinline__ void scale_min(const ScaleWords &w, int s,
                                          uint32_t &sc, uint32_t &m) {
    const uint32_t scw = s < 4 ? w.sc_lo : w.sc_hi;
    const uint32_t mw = s < 4 ? w.m_lo : w.m_hi;
    const int sh = 8 * (s & 3);
    sc = (scw >> sh) & 0xFFu;
    m = (mw >> sh) & 0xFFu;
}

}  // namespace kq
