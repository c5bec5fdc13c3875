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
    const uint8_t *rec; // input records [ntok][nb] (kq_xrec.cuh), global memory;
                        // tensor-core launches: the records of kq_xtc.cuh
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
    int32_t ntok;  // token columns of the launch (tensor-core launches are
                   // compiled for a multiple of 8)
};

// ------------------------------------------------------------ conversions
// IEEE binary16 bits -> f32 (CUDA's conversion intrinsic).
__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}

// Word k (0..3) of a 16-byte chunk.
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
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

}  // namespace kq
