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
 * Readings taken where the page is silent:
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
#include <stdlib.h>
#include <string.h>

#define ORACLE_QK 32

enum { ORACLE_Q8_0 = 0, ORACLE_Q4_0 = 1 };

/* ---- Sec. 4 / Sec. 5: Q8_0 quantisation of `len` floats with one scale ---- */
static void quantize_span(int8_t *q, float *d, const float *x, int len)
{
    float amax = 0.0f;
    for (int j = 0; j < len; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float dd = amax / 127.0f;                        /* d = max|x| / 127      */
    float id = (amax != 0.0f) ? 127.0f / amax : 0.0f; /* id = 127 / amax      */
    for (int j = 0; j < len; ++j) {
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

/* One block of 32 floats (Sec. 4: QK = 32). */
static void quantize_block(int8_t *q, float *d, const float *x)
{
    quantize_span(q, d, x, ORACLE_QK);
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


/* ========================================================================
 * The floating-point steps of a decode layer around the products.
 *
 * Source: the page "Legacy-ISA ML Inference Runtime -- Design Spec",
 * Sec. 5 (Kernel Interface: ml_k_rmsnorm, ml_k_softmax, ml_k_rope,
 * ml_k_silu_mul, ml_k_add, ml_k_dot_f32, ml_k_axpy_f32, and the notes on
 * RoPE: interleaved pairs (2i, 2i+1), freq_i = theta^(-2i/head_dim),
 * cos/sin tables of [max_seq][head_dim/2] precomputed at load) and Sec. 6
 * (Forward pass per token: attention per head as dot_f32 / sqrt(hd),
 * softmax, sum of axpy over positions; GQA: the KV head of query head h is
 * h / (n_heads / n_kv_heads)).  The page fixes float32 interfaces but not
 * the internal precision of these steps, so they are computed here in
 * double and rounded to float once per output (readings taken where the
 * page is silent):
 *   - rmsnorm: o_j = w_j * x_j / sqrt(sum_i x_i^2 / n + eps)
 *   - softmax: x_j = exp(x_j - max) / sum_i exp(x_i - max)
 *   - silu_mul: g_j = g_j / (1 + exp(-g_j)) * u_j
 *   - rope: (a, b) -> (a cos - b sin, a sin + b cos) on every pair of every
 *     q head and k head, with the float tables given
 *   - attention over positions t = 0..n_pos-1 of a float32 KV cache whose
 *     row t holds the n_kv_heads heads of K (or V) one after another.
 * ====================================================================== */

int mlqo_rmsnorm(float *o, const float *x, const float *w, int n, float eps)
{
    if (n <= 0) return -1;
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
    const double inv = 1.0 / sqrt(ss / (double)n + (double)eps);
    for (int j = 0; j < n; ++j) o[j] = (float)((double)w[j] * ((double)x[j] * inv));
    return 0;
}

int mlqo_softmax(float *x, int n)
{
    if (n <= 0) return -1;
    double mx = x[0];
    for (int i = 1; i < n; ++i) if (x[i] > mx) mx = x[i];
    double sum = 0.0;
    for (int i = 0; i < n; ++i) sum += exp((double)x[i] - mx);
    for (int j = 0; j < n; ++j) x[j] = (float)(exp((double)x[j] - mx) / sum);
    return 0;
}

int mlqo_silu_mul(float *g, const float *u, int n)
{
    if (n < 0) return -1;
    for (int j = 0; j < n; ++j) {
        const double a = g[j];
        g[j] = (float)(a / (1.0 + exp(-a)) * (double)u[j]);
    }
    return 0;
}

int mlqo_add(float *y, const float *x, int n)
{
    if (n < 0) return -1;
    for (int j = 0; j < n; ++j) y[j] = (float)((double)y[j] + (double)x[j]);
    return 0;
}

/* Row `pos` of the cos/sin tables: angle_i = pos * theta^(-2i/head_dim). */
int mlqo_rope_tables(float *cos_t, float *sin_t, int max_seq, int head_dim, float theta)
{
    if (head_dim <= 0 || head_dim % 2 != 0 || max_seq <= 0) return -1;
    const int half = head_dim / 2;
    for (int pos = 0; pos < max_seq; ++pos)
        for (int i = 0; i < half; ++i) {
            const double freq = pow((double)theta, -2.0 * i / (double)head_dim);
            const double ang = (double)pos * freq;
            cos_t[(size_t)pos * half + i] = (float)cos(ang);
            sin_t[(size_t)pos * half + i] = (float)sin(ang);
        }
    return 0;
}

static void rope_head(float *v, const float *c, const float *s, int head_dim)
{
    for (int i = 0; i < head_dim / 2; ++i) {
        const double a = v[2 * i], b = v[2 * i + 1];
        v[2 * i] = (float)(a * c[i] - b * s[i]);
        v[2 * i + 1] = (float)(a * s[i] + b * c[i]);
    }
}

/* q: n_heads x head_dim, k: n_kv_heads x head_dim, both rotated in place;
 * cos_t, sin_t: the table rows of the position (head_dim/2 each). */
int mlqo_rope(float *q, float *k, const float *cos_t, const float *sin_t, int head_dim,
              int n_heads, int n_kv_heads)
{
    if (head_dim <= 0 || head_dim % 2 != 0 || n_heads < 0 || n_kv_heads < 0) return -1;
    for (int h = 0; h < n_heads; ++h) rope_head(q + (size_t)h * head_dim, cos_t, sin_t, head_dim);
    for (int h = 0; h < n_kv_heads; ++h) rope_head(k + (size_t)h * head_dim, cos_t, sin_t, head_dim);
    return 0;
}

/* o: n_heads x head_dim.  For query head h with KV head g = h / (n_heads /
 * n_kv_heads): s_t = dot(q_h, K[t][g]) / sqrt(head_dim) for t < n_pos,
 * softmax over t, o_h = sum_t p_t V[t][g] accumulated in t order. */
int mlqo_attention(float *o, const float *q, const float *kc, const float *vc, int n_pos,
                   int head_dim, int n_heads, int n_kv_heads)
{
    if (n_pos <= 0 || head_dim <= 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads != 0)
        return -1;
    const int kv_dim = n_kv_heads * head_dim, group = n_heads / n_kv_heads;
    double *p = (double *)malloc((size_t)n_pos * sizeof(double));
    if (p == NULL) return -2;
    for (int h = 0; h < n_heads; ++h) {
        const int g = h / group;
        const float *qh = q + (size_t)h * head_dim;
        /* scores: dot_f32(q_h, K_t) / sqrt(hd) */
        for (int t = 0; t < n_pos; ++t) {
            const float *kt = kc + (size_t)t * kv_dim + (size_t)g * head_dim;
            double dot = 0.0;
            for (int i = 0; i < head_dim; ++i) dot += (double)qh[i] * (double)kt[i];
            p[t] = dot / sqrt((double)head_dim);
        }
        /* softmax over the positions */
        double mx = p[0], sum = 0.0;
        for (int t = 1; t < n_pos; ++t) if (p[t] > mx) mx = p[t];
        for (int t = 0; t < n_pos; ++t) { p[t] = exp(p[t] - mx); sum += p[t]; }
        for (int t = 0; t < n_pos; ++t) p[t] /= sum;
        /* o_h = sum over t of axpy(p_t, V_t) */
        double *acc = (double *)calloc((size_t)head_dim, sizeof(double));
        if (acc == NULL) { free(p); return -2; }
        for (int t = 0; t < n_pos; ++t) {
            const float *vt = vc + (size_t)t * kv_dim + (size_t)g * head_dim;
            for (int i = 0; i < head_dim; ++i) acc[i] += p[t] * (double)vt[i];
        }
        for (int i = 0; i < head_dim; ++i) o[(size_t)h * head_dim + i] = (float)acc[i];
        free(acc);
    }
    free(p);
    return 0;
}

/* ========================================================================
 * Q4_K-style super-blocks with the sub-block scale folded in the integer
 * domain.
 *
 * Source: the page "SKaiNET-native-kernels", section "Proving an
 * optimization is safe before writing it": 4-bit weight nibbles w in
 * [0, 15], 32 elements per sub-block, a 6-bit sub-block scale s <= 63,
 * 8 sub-blocks per block, activations quantised to int8 (|a| <= 127); the
 * sum over the 8 sub-blocks of s_b * sum_i a_i w_i fits int32 with ~70x
 * headroom (8*63*32*127*15 = 3.07e7), so it is formed in integers and
 * converted to float once per block; the format keeps per-32 asymmetric
 * minima.  Readings taken where the page is silent:
 *   - a block ("super-block") is 256 elements = 8 sub-blocks of 32; per
 *     super-block a float32 scale d and a float32 scale of the minima dmin;
 *     per sub-block a 6-bit scale s_b and a 6-bit minimum m_b, one per byte;
 *     element value = d*s_b*n - dmin*m_b;
 *   - layout, rows row-major: q = the nibbles, 16 bytes per sub-block in
 *     the Q4_0 order (byte j: element j in the low nibble, element j+16 in
 *     the high nibble); s = 16 bytes per super-block, the 8 sub-block
 *     scales then the 8 sub-block minima; d and dmin = one float32 each per
 *     super-block;
 *   - activations quantised per 256 elements with the Q8_0 rounding rule
 *     (one float32 scale per 256), plus the int32 sum of each 32-element
 *     sub-block of the quants;
 *   - per super-block ISUM = sum_b s_b * sum_i a_i n_i and MSUM = sum_b m_b *
 *     sum_i a_i, both int32, and y += ((float)ISUM * d - (float)MSUM * dmin)
 *     * dx in float32, super-blocks in increasing order, nothing fused.
 * ====================================================================== */
#define ORACLE_QKK 256
#define ORACLE_SUBS (ORACLE_QKK / ORACLE_QK)

int mlqo_quantize_q8k(int8_t *q, float *d, int32_t *bsums, const float *x, int m, int k)
{
    if (k <= 0 || k % ORACLE_QKK != 0 || m < 0) return -1;
    const int nsb = k / ORACLE_QKK;
    for (int r = 0; r < m; ++r)
        for (int B = 0; B < nsb; ++B) {
            const size_t e0 = (size_t)r * k + (size_t)B * ORACLE_QKK;
            quantize_span(q + e0, d + (size_t)r * nsb + B, x + e0, ORACLE_QKK);
            for (int b = 0; b < ORACLE_SUBS; ++b) {
                int32_t t = 0;
                for (int i = 0; i < ORACLE_QK; ++i) t += q[e0 + (size_t)b * ORACLE_QK + i];
                bsums[((size_t)r * nsb + B) * ORACLE_SUBS + b] = t;
            }
        }
    return 0;
}

/* ISUM and MSUM of row r, super-block B (the integer-domain fold). */
static void q4k_block_sums(int32_t *isum, int32_t *msum, const uint8_t *wq, const uint8_t *ws,
                           int nsb, int r, int B, const int8_t *xq, const int32_t *xbs)
{
    const uint8_t *sm = ws + ((size_t)r * nsb + B) * 16;   /* scales, then minima */
    int32_t is = 0, ms = 0;
    for (int b = 0; b < ORACLE_SUBS; ++b) {
        const size_t sb = (size_t)B * ORACLE_SUBS + b;             /* sub-block of the row */
        const uint8_t *bytes = wq + ((size_t)r * nsb * ORACLE_SUBS + sb) * 16;
        const int8_t *a = xq + sb * ORACLE_QK;
        int32_t dot = 0;
        for (int j = 0; j < 16; ++j) {
            dot += (int32_t)(bytes[j] & 0x0F) * a[j];
            dot += (int32_t)(bytes[j] >> 4) * a[j + 16];
        }
        is += (int32_t)sm[b] * dot;
        ms += (int32_t)sm[8 + b] * xbs[sb];
    }
    *isum = is;
    *msum = ms;
}

int mlqo_block_sums_q4k(int32_t *isum, int32_t *msum, const uint8_t *wq, const uint8_t *ws,
                        int rows, int cols, const int8_t *xq, const int32_t *xbs, int r0, int r1)
{
    if (cols <= 0 || cols % ORACLE_QKK != 0 || r0 < 0 || r1 > rows || r0 > r1) return -1;
    const int nsb = cols / ORACLE_QKK;
    for (int r = r0; r < r1; ++r)
        for (int B = 0; B < nsb; ++B)
            q4k_block_sums(isum + (size_t)(r - r0) * nsb + B, msum + (size_t)(r - r0) * nsb + B,
                           wq, ws, nsb, r, B, xq, xbs);
    return 0;
}

int mlqo_matvec_q4k(float *y, const uint8_t *wq, const uint8_t *ws, const float *wd,
                    const float *wdmin, int rows, int cols, const int8_t *xq, const float *xd,
                    const int32_t *xbs, int r0, int r1)
{
    if (cols <= 0 || cols % ORACLE_QKK != 0 || r0 < 0 || r1 > rows || r0 > r1) return -1;
    const int nsb = cols / ORACLE_QKK;
    for (int r = r0; r < r1; ++r) {
        float yr = 0.0f;
        for (int B = 0; B < nsb; ++B) {
            int32_t is, ms;
            q4k_block_sums(&is, &ms, wq, ws, nsb, r, B, xq, xbs);
            const float t = (float)is * wd[(size_t)r * nsb + B];
            const float u = (float)ms * wdmin[(size_t)r * nsb + B];
            const float v = (t - u) * xd[B];
            yr = yr + v;
        }
        y[r] = yr;
    }
    return 0;
}

/* ========================================================================
 * Block length 128 or 32, float32 or binary16 scales, 8-bit weights with a
 * zero point in the packed signed form.
 *
 * Source: the page "ONNX Runtime" (SpaceMiT X60), "How we got there":
 * item 3 (AMD's Qwen2.5-0.5B export uses block_size = 128; a BlkLen = 128
 * CompInt8 path with int8 activations), item 4 (8-bit weights packed as
 * signed B' = B - 128 with flat scales, and a per-block correction
 * -scale * (zp - 128) that vanishes when the zero point is 128 or absent),
 * item 5 (panels with float16 scales).  What the method computes is the
 * plain product of the dequantised blocks: per block b of row r,
 *   sumi = sum_i w_i * a_i,  w_i = n_i - 8 (4-bit, symmetric)  or
 *                            w_i = B_i - zp_b = B'_i + 128 - zp_b (8-bit),
 *   y[r] += ((float)sumi * scale_b) * dx_b   in float32, blocks in order.
 * The signed-offset correction reaches the same int32 sumi exactly:
 * sum (B' + 128 - zp) a = sum B' a + (128 - zp) sum a; the oracle forms
 * sumi from w_i directly.  Readings taken where the page is silent:
 *   - 4-bit blocks of `blk` elements pack element j in the low nibble and
 *     element j + blk/2 in the high nibble of byte j (the Q4_0 order, which
 *     it equals for blk = 32); 4-bit weights have no zero points;
 *   - 8-bit weights are stored as B' (int8) with one uint8 zero point per
 *     block (NULL: 128 for every block);
 *   - scales are one per block, float32 or IEEE 754 binary16 (converted to
 *     float32 exactly, below, from the binary16 definition);
 *   - activations are quantised per `blk` elements with the Q8_0 rule (one
 *     float32 scale per block), plus the int32 sum of each block's quants.
 * ====================================================================== */

/* IEEE 754 binary16 -> float (every binary16 value is a float32 value):
 * sign bit 15, exponent bits 14..10 (bias 15), fraction bits 9..0;
 * exponent 0: subnormal (fraction * 2^-24); exponent 31: inf or NaN. */
float mlqo_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    float v;
    if (e == 0)       v = ldexpf((float)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else              v = ldexpf((float)(f + 1024), e - 25);
    return sign ? -v : v;
}

int mlqo_quantize_blk(int8_t *q, float *d, int32_t *bsums, const float *x, int k, int blk)
{
    if (blk <= 0 || k <= 0 || k % blk != 0) return -1;
    for (int b = 0; b < k / blk; ++b) {
        quantize_span(q + (size_t)b * blk, d + b, x + (size_t)b * blk, blk);
        int32_t t = 0;
        for (int i = 0; i < blk; ++i) t += q[(size_t)b * blk + i];
        bsums[b] = t;
    }
    return 0;
}

/* Weight element i of block b of row r (n - 8, or B' + 128 - zp). */
static int32_t nbits_weight(const uint8_t *wq, const uint8_t *zp, int bits, int blk, int cols,
                            int r, int b, int i)
{
    const size_t nb = (size_t)(cols / blk);
    if (bits == 4) {
        const uint8_t *blkb = wq + ((size_t)r * nb + b) * (blk / 2);
        const int n = i < blk / 2 ? (blkb[i] & 0x0F) : (blkb[i - blk / 2] >> 4);
        return n - 8;
    }
    const int8_t bp = (int8_t)wq[((size_t)r * nb + b) * blk + i];
    const int z = zp ? zp[(size_t)r * nb + b] : 128;
    return (int32_t)bp + 128 - z;
}

int mlqo_block_sumi_nbits(int32_t *sumi, const uint8_t *wq, const uint8_t *zp, int rows, int cols,
                          int bits, int blk, const int8_t *xq, int r0, int r1)
{
    if ((bits != 4 && bits != 8) || (blk != 32 && blk != 128) || cols <= 0 || cols % blk != 0) return -1;
    if (bits == 4 && zp != NULL) return -1;
    if (r0 < 0 || r1 > rows || r0 > r1) return -1;
    const int nb = cols / blk;
    for (int r = r0; r < r1; ++r)
        for (int b = 0; b < nb; ++b) {
            int32_t s = 0;
            for (int i = 0; i < blk; ++i)
                s += nbits_weight(wq, zp, bits, blk, cols, r, b, i) * (int32_t)xq[(size_t)b * blk + i];
            sumi[(size_t)(r - r0) * nb + b] = s;
        }
    return 0;
}

/* scales: float32 (scale_f16 = 0) or binary16 bit patterns (scale_f16 = 1). */
int mlqo_matvec_nbits(float *y, const uint8_t *wq, const void *scales, int scale_f16,
                      const uint8_t *zp, int rows, int cols, int bits, int blk, const int8_t *xq,
                      const float *xd, int r0, int r1)
{
    if ((bits != 4 && bits != 8) || (blk != 32 && blk != 128) || cols <= 0 || cols % blk != 0) return -1;
    if (bits == 4 && zp != NULL) return -1;
    if (r0 < 0 || r1 > rows || r0 > r1) return -1;
    const int nb = cols / blk;
    for (int r = r0; r < r1; ++r) {
        float acc = 0.0f;
        for (int b = 0; b < nb; ++b) {
            int32_t s = 0;
            for (int i = 0; i < blk; ++i)
                s += nbits_weight(wq, zp, bits, blk, cols, r, b, i) * (int32_t)xq[(size_t)b * blk + i];
            const size_t si = (size_t)r * nb + b;
            const float sc = scale_f16 ? mlqo_half_to_float(((const uint16_t *)scales)[si])
                                       : ((const float *)scales)[si];
            const float t = (float)s * sc;
            acc = acc + t * xd[b];
        }
        y[r] = acc;
    }
    return 0;
}
