// kq_rows.cu -- rows of a K-quant matrix gathered by index and dequantized
// to f32: the embedding lookup ("Chapter 6 - The kquant family on the
// reference lane", section 6.7: muser_embedding_q4k resolves the token's
// row, row_bytes = (hidden / 256) * 144, and dequantizes it element by
// element with section 6.3's formula), here for Q4_K, Q5_K and Q6_K.
//
// One warp per (output row, super-block).  Every value is formed exactly
// and rounded once:
//   Q4_K / Q5_K   fma(d*sc, q, -(dmin*m))   (d*sc, dmin*m and the product
//                 d*sc*q are exact in f32, so only the sum rounds)
//   Q6_K          (d*sc) * (q - 32)        (exact: at most 23 significant
//                 bits)
// so the result is the correctly rounded weight, the same bits any exact
// evaluation order gives.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kq_common.cuh"
#include "kq_launch.cuh"

namespace kq {

constexpr int kRowsThreads = 256;  // 8 warps, one super-block each

// Scale and min of sub-block s from the three scale-field words (Figure 6.3).
__device__ __forceinline__ void scale_min_of(const ScaleWords &w, int s, uint32_t &sc,
                                             uint32_t &m) {
    const uint32_t scw = s < 4 ? w.sc_lo : w.sc_hi;
    const uint32_t mw = s < 4 ? w.m_lo : w.m_hi;
    sc = (scw >> (8 * (s & 3))) & 0xFFu;
    m = (mw >> (8 * (s & 3))) & 0xFFu;
}

__global__ void __launch_bounds__(kRowsThreads)
    kq_rows_kernel(int fmt, const uint8_t *__restrict__ W, int64_t rows, int nb,
                   const int32_t *__restrict__ ids, int64_t n, float *__restrict__ out) {
    const int64_t gw = ((int64_t)blockIdx.x * kRowsThreads + threadIdx.x) >> 5;
    if (gw >= n * nb) return;
    const int lane = threadIdx.x & 31;
    const int64_t i = gw / nb;
    const int b = (int)(gw - i * nb);
    const int64_t cols = (int64_t)nb * 256;
    float *o = out + i * cols + (int64_t)b * 256;
    const int32_t id = __ldg(ids + i);
    if (id < 0 || (int64_t)id >= rows) {
        // an index outside the matrix yields a row of NaN
        const float nan = __int_as_float(0x7FC00000);
#pragma unroll
        for (int k = 0; k < 8; ++k) o[lane + 32 * k] = nan;
        return;
    }
    if (fmt == kFmtQ4K || fmt == kFmtQ5K) {
        const bool q5 = fmt == kFmtQ5K;
        const int bb = q5 ? 176 : 144;
        const uint8_t *blk = W + ((int64_t)id * nb + b) * bb;
        const uint4 h = __ldg(reinterpret_cast<const uint4 *>(blk));
        const float d = h2f(h.x), dmin = h2f(h.x >> 16);
        const ScaleWords sw = unpack_scale_words(h.y, h.z, h.w);
        // lane: group g (64 weights), qs bytes 4p..4p+3 of the group
        const int g = lane >> 3, p = lane & 7;
        const uint8_t *qs = blk + (q5 ? 48 : 16);
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(qs + 32 * g + 4 * p));
        const uint32_t hb = q5 ? __ldg(reinterpret_cast<const uint32_t *>(blk + 16 + 4 * p)) : 0u;
        uint32_t sc0, m0, sc1, m1;
        scale_min_of(sw, 2 * g, sc0, m0);
        scale_min_of(sw, 2 * g + 1, sc1, m1);
        const float ds0 = d * (float)sc0, dm0 = dmin * (float)m0;
        const float ds1 = d * (float)sc1, dm1 = dmin * (float)m1;
        float lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t ql = (w >> (8 * k)) & 0xFu, qh = (w >> (8 * k + 4)) & 0xFu;
            if (q5) {
                ql |= ((hb >> (8 * k + 2 * g)) & 1u) << 4;
                qh |= ((hb >> (8 * k + 2 * g + 1)) & 1u) << 4;
            }
            lo[k] = fmaf(ds0, (float)ql, -dm0);
            hi[k] = fmaf(ds1, (float)qh, -dm1);
        }
        *reinterpret_cast<float4 *>(o + 64 * g + 4 * p) = make_float4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<float4 *>(o + 64 * g + 32 + 4 * p) = make_float4(hi[0], hi[1], hi[2], hi[3]);
    } else {
        // Q6_K (Figure 6.5): ql 0..127, qh 128..191, int8 scales 192..207,
        // f16 d 208..209; 2-byte aligned, so bytes are read one by one.
        const uint8_t *blk = W + ((int64_t)id * nb + b) * 210;
        const float d = h2f((uint32_t)__ldg(blk + 208) | ((uint32_t)__ldg(blk + 209) << 8));
        // lane: half hh, positions l = 2p, 2p + 1 of the half's 32
        const int hh = lane >> 4, p = lane & 15;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int l = 2 * p + u;
            const uint32_t a = __ldg(blk + 64 * hh + l);
            const uint32_t c = __ldg(blk + 64 * hh + 32 + l);
            const uint32_t q = __ldg(blk + 128 + 32 * hh + l);
            const int code[4] = {(int)((a & 0xFu) | ((q & 3u) << 4)),
                                 (int)((c & 0xFu) | (((q >> 2) & 3u) << 4)),
                                 (int)((a >> 4) | (((q >> 4) & 3u) << 4)),
                                 (int)((c >> 4) | (((q >> 6) & 3u) << 4))};
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const int e = 128 * hh + 32 * qd + l;
                const int8_t sc = (int8_t)__ldg(blk + 192 + e / 16);
                o[e] = (d * (float)sc) * (float)(code[qd] - 32);
            }
        }
    }
}

}  // namespace kq

namespace kqlaunch {

cudaError_t rows(int fmt, const uint8_t *W, int64_t rows, int nb, const int32_t *ids, int64_t n,
                 float *out, cudaStream_t s) {
    const int64_t warps = n * nb;
    const int64_t blocks = (warps * 32 + kq::kRowsThreads - 1) / kq::kRowsThreads;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    kq::kq_rows_kernel<<<(unsigned)blocks, kq::kRowsThreads, 0, s>>>(fmt, W, rows, nb, ids, n, out);
    return cudaGetLastError();
}

}  // namespace kqlaunch
