// kq_xrec.cuh -- the input vector in the form the block dot products use.
//
// Every product code_j * x_j of a super-block is summed exactly, in
// integers, with the four-way byte dot product (dp4a).  For that each
// group of 32 consecutive inputs (one Q4_K / Q5_K sub-block, two Q6_K
// sub-blocks) is written in fixed point with its own power-of-two step:
//
//   E    the smallest integer with max_{j in group} |x_j| < 2^E, clamped to
//        [-100, 128] (so that both 2^(23-E) and 2^(E-23) are normal floats)
//   X_j  = rint(x_j * 2^(23-E)), limited to 2^23 - 1, so |X_j| <= 2^23
//   x_j ~ X_j * u  with  u = 2^(E-23);  |x_j - X_j * u| <= u/2 <= 2^-24 * 2^E
//
// X_j is split into three bytes, X = b2 * 2^16 + b1 * 2^8 + b0, with b0 and
// b1 unsigned and b2 signed.  A sub-block's sum_j code_j * X_j is then three
// exact integer sums sum_j code_j * b_l, and only their combination,
// (S2 * 256 + S1) * 256 + S0, is rounded (once, in the conversion to f32).
// The whole error of a block's dot product is the input rounding above,
// at most 2^-24 * 2^E per input -- below 2^-23 * max|x| of its group.
//
// A non-finite input makes u of its group NaN, so that every output that
// reads it is NaN.
//
// One record per (token, super-block column), in shared or global memory:
//
//   bytes   0..255   b0 of inputs 0..255 (input e at byte e)
//         256..511   b1
//         512..767   b2
//         768..799   u of the eight groups (f32)
//   Q4_K / Q5_K (kRecQ45 = 832 bytes):
//         800..831   X_s = (sum_{j in s} X_j) * u_s, s = 0..7 (f32): the
//                    sub-block input sums of the min term, from the same
//                    rounded inputs
//   Q6_K (kRecQ6 = 1056 bytes):
//         800..1055  for the 16 sub-blocks of 16: int32 x4
//                    (-32 * sum b0, -32 * sum b1, -32 * sum b2, 0), the
//                    starting values of the limb sums, which make them sums
//                    of (code - 32) * b_l
//
// The record depends on the inputs and the format family only, and is
// built by the same code wherever it is built, so every kernel that reads
// it sees the same bytes.
#pragma once

#include <stdint.h>

namespace kq {

constexpr int kRecQ45 = 832;
constexpr int kRecQ6 = 1056;
constexpr int kRecU = 768;
constexpr int kRecSums = 800;

__host__ __device__ constexpr int rec_bytes(bool q6) { return q6 ? kRecQ6 : kRecQ45; }

// Records for one 128-input half of a super-block column, built by one warp:
// lane i converts inputs 128h + 4i .. 128h + 4i + 3 (v) of one token.  `rec`
// points at the column's record for that token.
__device__ __forceinline__ void build_record_half(float4 v, uint8_t *rec, int h, bool q6,
                                                  int lane) {
    const int e = 128 * h + 4 * lane;
    const uint32_t a0 = __float_as_uint(v.x) & 0x7FFFFFFFu, a1 = __float_as_uint(v.y) & 0x7FFFFFFFu;
    const uint32_t a2 = __float_as_uint(v.z) & 0x7FFFFFFFu, a3 = __float_as_uint(v.w) & 0x7FFFFFFFu;
    uint32_t m = max(max(a0, a1), max(a2, a3));
    // maximum over the eight lanes of the group (inputs 32 * (e / 32) ..)
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    const bool finite = m < 0x7F800000u;
    // m < 2^E for E = (biased exponent of m) - 126; subnormal and zero
    // maxima take the exponent of the smallest normal
    int E = (int)(m >> 23);
    E = (E < 1 ? 1 : E) - 126;
    E = E < -100 ? -100 : (E > 128 ? 128 : E);
    const float s = __uint_as_float((uint32_t)(127 + 23 - E) << 23);
    const float u = finite ? __uint_as_float((uint32_t)(127 + E - 23) << 23) : __uint_as_float(0x7FC00000u);
    int X[4];
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = __float2int_rn(vv[i] * s);
        X[i] = finite ? min(q, 8388607) : 0;
    }
    // byte planes: bytes l of X[0..3] -> one word per plane
    const uint32_t w01 = __byte_perm((uint32_t)X[0], (uint32_t)X[1], 0x5140);
    const uint32_t w23 = __byte_perm((uint32_t)X[2], (uint32_t)X[3], 0x5140);
    const uint32_t p0 = __byte_perm(w01, w23, 0x5410);
    const uint32_t p1 = __byte_perm(w01, w23, 0x7632);
    const uint32_t p2 = __byte_perm(__byte_perm((uint32_t)X[0], (uint32_t)X[1], 0x0062),
                                    __byte_perm((uint32_t)X[2], (uint32_t)X[3], 0x0062), 0x5410);
    *reinterpret_cast<uint32_t *>(rec + e) = p0;
    *reinterpret_cast<uint32_t *>(rec + 256 + e) = p1;
    *reinterpret_cast<uint32_t *>(rec + 512 + e) = p2;
    if ((lane & 7) == 0) *reinterpret_cast<float *>(rec + kRecU + 4 * (e >> 5)) = u;
    if (!q6) {
        int sx = (X[0] + X[1]) + (X[2] + X[3]);
        sx += __shfl_xor_sync(0xFFFFFFFFu, sx, 1);
        sx += __shfl_xor_sync(0xFFFFFFFFu, sx, 2);
        sx += __shfl_xor_sync(0xFFFFFFFFu, sx, 4);
        if ((lane & 7) == 0)
            *reinterpret_cast<float *>(rec + kRecSums + 4 * (e >> 5)) = __int2float_rn(sx) * u;
    } else {
        // limb sums over the sub-block of 16 (four lanes)
        int s0 = 0, s1 = 0, s2 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s0 += X[i] & 0xFF;
            s1 += (X[i] >> 8) & 0xFF;
            s2 += X[i] >> 16;
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, o);
            s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, o);
            s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
        }
        if ((lane & 3) == 0)
            *reinterpret_cast<int4 *>(rec + kRecSums + 16 * (e >> 4)) = make_int4(-32 * s0, -32 * s1, -32 * s2, 0);
    }
}

// The four inputs lane `lane` converts for half i (= 2 * j + h) of token t.
__device__ __forceinline__ float4 record_inputs(const float *x, int64_t cols, int t, int i,
                                                int lane) {
    const float *q = x + t * cols + (int64_t)(i >> 1) * 256 + 128 * (i & 1) + 4 * lane;
    float4 v;
    // volatile: issued in program order after the caller's signal
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(q));
    return v;
}

// All records of one input plane set: ntok tokens x nb columns, records
// token-major ([t][j]) at `recs`.  Work is dealt in warp-sized halves over
// `nwarps` warps (`w` is this warp's index), kRecBatch halves a warp at a
// time: all loads of a batch are issued before any conversion.  `issued()`
// is called once, as the first batch's loads go out (they are issued right
// after it), so that the caller can start other memory traffic with them.
constexpr int kRecBatch = 5;

template <bool Q6, class F>
__device__ __forceinline__ void build_records(const float *x, int64_t cols, int ntok, int nb,
                                              uint8_t *recs, int w, int nwarps, int lane,
                                              F issued) {
    constexpr bool q6 = Q6;
    const int rb = rec_bytes(q6);
    const int n = nb * 2;  // halves per token
    bool first = true;
#pragma unroll 1
    for (int t = 0; t < ntok; ++t) {
        uint8_t *rt = recs + (int64_t)t * nb * rb;
#pragma unroll 1
        for (int base = w; base < n || first; base += kRecBatch * nwarps) {
            if (first) {
                issued();
                first = false;
            }
            float4 v[kRecBatch];
#pragma unroll
            for (int k = 0; k < kRecBatch; ++k) {
                const int i = base + k * nwarps;
                if (i < n) v[k] = record_inputs(x, cols, t, i, lane);
            }
#pragma unroll
            for (int k = 0; k < kRecBatch; ++k) {
                const int i = base + k * nwarps;
                if (i < n) build_record_half(v[k], rt + (i >> 1) * rb, i & 1, q6, lane);
            }
        }
    }
}

}  // namespace kq
