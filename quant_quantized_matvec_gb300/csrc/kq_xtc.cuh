// kq_xtc.cuh -- the input vectors in the form the tensor-core block sums
// (kq_tc.cuh) use: calls of kTcMinNtok or more token columns, all formats.
//
// The tensor cores take the codes as the A operand (16 rows x 16 inputs)
// and up to eight token columns at a time as the B operand (16 inputs x 8
// tokens), in f16 with f32 accumulation.  Each token's 256-input column is
// scaled by one power of two and written as two f16 terms:
//
//   E     the smallest integer with max_{j in column} |x_j| < 2^E, clamped
//         to [-100, 128];  u = 2^(E - 14)
//   x'_j  = x_j / u  (exact; |x'_j| < 2^14)
//   hi_j  = f16(x'_j),  lo_j = f16(x'_j - hi_j)   (round to nearest even)
//
// so x_j ~ (hi_j + lo_j) * u with |x'_j - hi_j - lo_j| <= max(2^-22 |x'_j|,
// 2^-25) (the second term where lo_j is an f16 subnormal), i.e. an input
// error of at most max(2^-22 |x_j|, 2^(E - 39)).  The MMA chain
// D = A*B_hi + A*B_lo adds both terms; every product code * f16 is exact
// and only the tensor core's f32 sums round.  A non-finite input makes u of
// its column NaN, so that every output that reads the column is NaN.
//
// Records, in global memory, for `noct` octets of tokens (octet o holds
// tokens 8o..8o+7; tokens past ntok are zero) and nb columns, one column
// after another (tc_col_bytes(noct) each, so that the columns of a stage
// are one contiguous copy):
//
//   fragments  [o][k][lane] x 16 bytes, k = 0..15 the k-step (inputs
//              16k..16k+15 of the column); lane L = 4g + t holds, for token
//              8o + g, the f16 pairs (hi[16k+4t], hi[16k+4t+2]),
//              (hi[16k+4t+1], hi[16k+4t+3]), then the same two pairs of lo
//              -- the m16n8k16 B layout with the k index permuted (k-slot
//              2t <-> input 4t, 2t+1 <-> 4t+2, 2t+8 <-> 4t+1, 2t+9 <->
//              4t+3; the A side uses the same order), hi and lo side by
//              side so that one 16-byte load fetches both
//   aux        [token 0..8 noct - 1] x kTcAuxFloats: S32[0..7], the f32 sums
//              of hi + lo over the 32-input sub-blocks in a fixed order (the
//              Q4_K / Q5_K min term); then u.  Tokens past ntok are not
//              written and never read.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace kq {

constexpr int kTcMinNtok = 4;   // calls with at least this many token columns
constexpr int kTcMaxOct = 2;    // octets of tokens per launch (16 tokens)
constexpr int kTcFragOctBytes = 16 * 32 * 16;  // one octet of one column
constexpr int kTcAuxFloats = 16;                // per token of one column
constexpr int kTcAuxS32 = 0;
constexpr int kTcAuxU = 8;

__host__ __device__ constexpr int tc_col_bytes(int noct) {
    return noct * (kTcFragOctBytes + 8 * kTcAuxFloats * 4);
}
__host__ __device__ constexpr int64_t tc_record_bytes(int ntok, int nb) {
    return (int64_t)nb * tc_col_bytes((ntok + 7) / 8);
}
// Byte offset of (k-step, lane) inside one octet of one column.
__host__ __device__ __forceinline__ int tc_frag_offset(int k, int lane) {
    return (k * 32 + lane) * 16;
}

__device__ __forceinline__ uint32_t half2_bits(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

// The records of one octet o and one column j, k-steps 4q..4q+3, built by
// warp q (0..3) of a block of four: each warp loads only its quarter of the
// column (64 inputs of each of 8 tokens), the column's maximum per token is
// taken over the four quarters' maxima in shared memory (smax, [4][8]
// words).  x is [ntok][nb * 256]; `frag` points at this (octet, column)'s
// fragments and `aux` at the column's aux of token 0.  Every thread of the
// block calls this (it holds one block barrier).
constexpr int kTcPrepSplit = 4;

__device__ __forceinline__ void build_tc_record(const float *x, int ntok, int nb, int o, int j,
                                                int q, uint8_t *frag, float *aux, int lane,
                                                uint32_t *smax) {
    const int g = lane >> 2, t = lane & 3;
    const int tok = 8 * o + g;
    const bool live = tok < ntok;
    const float *xc = x + (int64_t)tok * nb * 256 + (int64_t)j * 256 + 4 * t;
    float4 v[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        v[kk] = live ? __ldg(reinterpret_cast<const float4 *>(xc + 16 * (4 * q + kk)))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t m = 0;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        m = max(m, __float_as_uint(v[kk].x) & 0x7FFFFFFFu);
        m = max(m, __float_as_uint(v[kk].y) & 0x7FFFFFFFu);
        m = max(m, __float_as_uint(v[kk].z) & 0x7FFFFFFFu);
        m = max(m, __float_as_uint(v[kk].w) & 0x7FFFFFFFu);
    }
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    if (t == 0) smax[q * 8 + g] = m;
    __syncthreads();
#pragma unroll
    for (int qq = 0; qq < kTcPrepSplit; ++qq) m = max(m, smax[qq * 8 + g]);
    const bool finite = m < 0x7F800000u;
    // m < 2^E for E = (biased exponent of m) - 126; zero and subnormal
    // maxima take the exponent of the smallest normal
    int E = (int)(m >> 23);
    E = (E < 1 ? 1 : E) - 126;
    E = E < -100 ? -100 : (E > 128 ? 128 : E);
    const float s = __uint_as_float((uint32_t)(127 + 14 - E) << 23);
    const float u = finite ? __uint_as_float((uint32_t)(127 + E - 14) << 23)
                           : __uint_as_float(0x7FC00000u);
    float s16[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int k = 4 * q + kk;
        const float4 vk = v[kk];
        const float xs[4] = {vk.x * s, vk.y * s, vk.z * s, vk.w * s};
        __half hi[4], lo[4];
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hi[i] = __float2half_rn(xs[i]);
            const float h = __half2float(hi[i]);
            lo[i] = __float2half_rn(xs[i] - h);  // xs - h is exact in f32
            part += h + __half2float(lo[i]);     // h + lo is exact in f32
        }
        *reinterpret_cast<uint4 *>(frag + tc_frag_offset(k, lane)) =
            make_uint4(half2_bits(hi[0], hi[2]), half2_bits(hi[1], hi[3]),
                       half2_bits(lo[0], lo[2]), half2_bits(lo[1], lo[3]));
        // the k-step's sum over the four lanes of this token (same value in all four)
        part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
        part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
        s16[kk] = part;
    }
    if (live && t == 0) {
        float *a = aux + tok * kTcAuxFloats;
        *reinterpret_cast<float2 *>(a + kTcAuxS32 + 2 * q) =
            make_float2(s16[0] + s16[1], s16[2] + s16[3]);
        if (q == 0) a[kTcAuxU] = u;
    }
}

}  // namespace kq
