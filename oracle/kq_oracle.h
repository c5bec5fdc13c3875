/*
 * kq_oracle.h -- plain, slow, CPU-only reference for the K-quant matvec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) may include, link or call this code; only the tests,
 * the package's smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (sources are the pages' titles and sections):
 *   - "Chapter 13 - The QKV + gate matvec family", section 13.1:
 *       y_i = sum_{j=0..cols-1} W[i,j] * x[j], one dot product per row.
 *   - "Chapter 6 - The kquant family on the reference lane":
 *       Figure 6.1 (block bytes / elements), section 6.2 and Figure 6.2/6.3
 *       (Q4_K super-block, 6-bit scale/min packing, nibble interleave),
 *       section 6.4 with Figures 6.4 and 6.5 (Q5_K and Q6_K layouts).
 *
 * Precision: each block is dequantized to f32 exactly as section 6.2's
 * dequantizer does (f32 effective scale and min, one f32 subtraction), and
 * every dot product is accumulated in f64, in element order j = 0..cols-1.
 * Alongside y the oracle returns S_i = sum_j |W[i,j] * x[j]| (f64), the
 * magnitude the parity tolerance is scaled by.
 *
 * Readings where the pages leave a step open (see the .c file for each):
 *   R1  Q5_K high-bit order: bit 2g / 2g+1 of qh[l] for the low / high
 *       nibble of qs[32g+l].          -- element order parity unpinned
 *   R2  Q6_K code order inside each 128-element half.
 *                                     -- element order parity unpinned
 *   R3  f16 fields decoded as IEEE binary16, subnormals included.
 */
#ifndef KQ_ORACLE_H
#define KQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GgmlType codes of the three formats (Chapter 6, section 6.1). */
enum { KQO_Q4_K = 12, KQO_Q5_K = 13, KQO_Q6_K = 14 };

/* Bytes per 256-element super-block (Figure 6.1); -1 for an unknown code. */
int kqo_block_bytes(int fmt);

/* IEEE binary16 bits -> value (R3). */
float kqo_f16_to_f32(uint16_t h);

/* 6-bit scale and min of sub-block j (0..7) from the 12-byte field
 * (Q4_K and Q5_K; section 6.2, Figure 6.3). */
void kqo_scale_min_k4(const uint8_t scales[12], int j, int *sc, int *m);

/* One super-block -> 256 f32 weights.  Returns 0, or -1 for unknown fmt. */
int kqo_dequant_block(int fmt, const uint8_t *block, float out[256]);

/* One row of a row-major matrix (cols/256 consecutive super-blocks) -> f32.
 * Returns 0, or -1 on a bad fmt / cols. */
int kqo_dequant_row(int fmt, const uint8_t *W, int64_t cols, int64_t row,
                    float *out);

/* Dense f32 matvec with f64 accumulation: y[t*rows+i] = sum_j W[i*cols+j] *
 * x[t*cols+j] (Figure 13.1's arithmetic).  S as above. */
void kqo_matvec_f32(const float *W, int64_t rows, int64_t cols,
                    const float *x, int ntok, double *y, double *S);

/* The K-quant matvec for a chosen list of rows (all rows: pass row_idx NULL
 * and n = rows).  x is [ntok][cols] f32; y and S are [ntok][n] f64, column
 * k of y belonging to row row_idx[k].  Returns 0, or -1 on bad arguments. */
int kqo_matvec_rows(int fmt, const uint8_t *W, int64_t rows, int64_t cols,
                    const float *x, int ntok, const int64_t *row_idx,
                    int64_t n, double *y, double *S);

#ifdef __cplusplus
}
#endif

#endif /* KQ_ORACLE_H */
