/*
 * mlq_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * block-quantized decode matrix-vector product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline (and its "--impl reference" arm) may use it.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * Build: C11, -O2 -ffp-contract=off, no -ffast-math, so that every float
 * operation below is one IEEE-754 binary32 operation rounded to nearest and
 * no multiply/add pair is fused.
 *
 * Source of every definition: the page "Legacy-ISA ML Inference Runtime --
 * Design Spec":
 *   Sec. 4 (Quantization Formats): QK = 32 symmetric blocks; Q8_0 quants are
 *     int8 clamped to [-127, 127] with one float32 scale per block; Q4_0 is
 *     16 bytes per block, low nibble = element 0..15, high nibble = element
 *     16..31, value = nibble - 8; q and d are separate arrays per tensor;
 *     d = max|x| / 127, d = 0 gives an all-zero block; per block the integer
 *     dot sumi = sum(qw * qx) is an int32 and the output accumulates
 *     sum += (float)sumi * dw * dx in float32.
 *   Sec. 5 (Kernel Interface): matvec processes rows [r0, r1); quantize_q8
 *     rounds with q = trunc(x*id + copysign(0.5, x)), id = 127/amax; Q4
 *     kernels unpack nibbles (and 0x0F, shift 4, subtract 8) into int8 and
 *     then reuse the Q8 path.
 * Readings where the page is silent (each is listed in the design doc):
 *   - the rounding formula of Sec. 5 is normative over "round(x/d)" of Sec. 4;
 *     d is stored as amax/127, not as 1/id;
 *   - a NaN produced by 0 * inf (amax so small that 127/amax overflows) is
 *     stored as 0; +-inf clamps to +-127;
 *   - block order inside q and d is row-major: block b of row r is at
 *     q byte offset (r*nb + b)*bytes_per_block and scale index r*nb + b;
 *   - y is indexed by absolute row (y[r]); rows outside [r0, r1) are not
 *     written;
 *   - the small-M product treats each of the M activation rows as an
 *     independent M = 1 product with its own per-block scales; row m of the
 *     output starts at Y + m*ldy.
 *
 * Parity pins (tests/test_oracle_pins.py): hand-computed blocks, the d = 0
 * rule, the clamp, the Sec. 7 dequantisation bound, the int32 bound
 * 32*127*127 < 2^31, the all-ones-scale special case (a plain integer
 * matvec), and fp64 brute force over dequantised elements on tiny inputs.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_QK 32

enum { ORACLE_Q8_0 = 0, ORACLE_Q4_0 = 1 };

/* ---- Sec. 4 / Sec. 5: Q8_0 quantisation of one block of 32 floats ---- */
static void quantize_block(int8_t *q, float *d, const float *x)
{
    float amax = 0.0f;
    for (int j = 0; j < ORACLE_QK; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float dd = amax / 127.0f;                        /* d = max|x| / 127      */
    float id = (amax != 0.0f) ? 127.0f / amax : 0.0f; /* id = 127 / amax      */
    for (int j = 0; j < ORACLE_QK; ++j) {
        float v = x[j] * id;                         /* one rounded multiply  */
        v = v + copysignf(0.5f, x[j]);               /* one rounded add       */
        v = truncf(v);
        int8_t qq;
        if (v >= 127.0f)       qq = 127;             /* clamp to [-127, 127]  */
        else if (v <= -127.0f) qq = -127;
        else if (v != v)       qq = 0;               /* NaN (0 * inf) -> 0    */
        else                   qq = (int8_t)v;
        q[j] = qq;
    }
    *d = dd;
}

/* Quantise m rows of k floats (row-major) into q[m*k] and d[m*(k/32)].
 * Returns 0, or -1 when k is not a multiple of 32 or m < 0. */
int mlqo_quantize_q8(int8_t *q, float *d, const float *x, int m, int k)
{
    if (k % ORACLE_QK != 0 || k < 0 || m < 0) return -1;
    int nb = k / ORACLE_QK;
    for (int row = 0; row < m; ++row)
        for (int b = 0; b < nb; ++b)
            quantize_block(q + (size_t)row * k + (size_t)b * ORACLE_QK,
                           d + (size_t)row * nb + b,
                           x + (size_t)row * k + (size_t)b * ORACLE_QK);
    return 0;
}

/* ---- Sec. 4: Q4_0 nibble map, unpacked to int8 as Sec. 5 describes ---- */
static void unpack_q4_block(int8_t *w, const uint8_t *bytes16)
{
    for (int j = 0; j < 16; ++j) {
        w[j]      = (int8_t)((int)(bytes16[j] & 0x0F) - 8); /* element j      */
        w[j + 16] = (int8_t)((int)(bytes16[j] >> 4) - 8);   /* element j + 16 */
    }
}

/* ---- Sec. 4: integer dot of one block, int32 ---- */
static int32_t block_dot(const int8_t *w, const int8_t *x)
{
    int32_t s = 0;
    for (int j = 0; j < ORACLE_QK; ++j) s += (int32_t)w[j] * (int32_t)x[j];
    return s;
}

/* Weight block (r, b) as 32 int8 values. */
static void weight_block(int8_t *w, int type, const uint8_t *wq, int nb, int r, int b)
{
    if (type == ORACLE_Q4_0) {
        unpack_q4_block(w, wq + ((size_t)r * nb + b) * 16);
    } else {
        memcpy(w, wq + ((size_t)r * nb + b) * ORACLE_QK, ORACLE_QK);
    }
}

/* Per-block int32 sums for rows [r0, r1): sumi[(r - r0)*nb + b]. */
int mlqo_block_sumi(int32_t *sumi, int type, const uint8_t *wq, int rows, int cols,
                    const int8_t *xq, int r0, int r1)
{
    if (cols % ORACLE_QK != 0 || r0 < 0 || r1 < r0 || r1 > rows) return -1;
    if (type != ORACLE_Q4_0 && type != ORACLE_Q8_0) return -1;
    int nb = cols / ORACLE_QK;
    int8_t w[ORACLE_QK];
    for (int r = r0; r < r1; ++r)
        for (int b = 0; b < nb; ++b) {
            weight_block(w, type, wq, nb, r, b);
            sumi[(size_t)(r - r0) * nb + b] = block_dot(w, xq + (size_t)b * ORACLE_QK);
        }
    return 0;
}

/* ---- Sec. 4 / Sec. 5: y[r] = sum_b ((float)sumi * dw) * dx, r in [r0, r1) ----
 * Blocks are taken in increasing b, float32 throughout, nothing fused. */
int mlqo_matvec(float *y, int type, const uint8_t *wq, const float *wd, int rows, int cols,
                const int8_t *xq, const float *xd, int r0, int r1)
{
    if (cols % ORACLE_QK != 0 || r0 < 0 || r1 < r0 || r1 > rows) return -1;
    if (type != ORACLE_Q4_0 && type != ORACLE_Q8_0) return -1;
    int nb = cols / ORACLE_QK;
    int8_t w[ORACLE_QK];
    for (int r = r0; r < r1; ++r) {
        float sum = 0.0f;
        for (int b = 0; b < nb; ++b) {
            weight_block(w, type, wq, nb, r, b);
            int32_t sumi = block_dot(w, xq + (size_t)b * ORACLE_QK);
            float t = (float)sumi * wd[(size_t)r * nb + b];
            t = t * xd[b];
            sum = sum + t;
        }
        y[r] = sum;
    }
    return 0;
}

/* Small-M product: M independent activation rows, each an M = 1 product.
 * Xq is M x cols int8, Xd is M x nb float; Y[m*ldy + r] for r in [r0, r1). */
int mlqo_gemm_small_m(float *Y, int ldy, int type, const uint8_t *wq, const float *wd,
                      int rows, int cols, const int8_t *Xq, const float *Xd, int M,
                      int r0, int r1)
{
    if (cols % ORACLE_QK != 0 || M < 0 || ldy < r1) return -1;
    int nb = cols / ORACLE_QK;
    for (int m = 0; m < M; ++m) {
        int rc = mlqo_matvec(Y + (size_t)m * ldy, type, wq, wd, rows, cols,
                             Xq + (size_t)m * cols, Xd + (size_t)m * nb, r0, r1);
        if (rc != 0) return rc;
    }
    return 0;
}
