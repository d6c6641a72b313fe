/*
 * mlq.h -- C ABI of the GB300 (sm_103a) block-quantized decode library.
 *
 * The operations follow the page "Legacy-ISA ML Inference Runtime -- Design
 * Spec":
 *   Sec. 4 (Quantization Formats) fixes the data: blocks of QK = 32
 *     elements; Q8_0 = int8 quants clamped to [-127, 127] plus one float32
 *     scale per block; Q4_0 = 16 bytes per block (low nibble = element
 *     0..15, high nibble = element 16..31, value = nibble - 8) plus one
 *     float32 scale; quants and scales of a tensor are two separate arrays;
 *     per block sumi = sum(qw*qx) is an int32 and the output accumulates
 *     (float)sumi * dw * dx in float32.
 *   Sec. 5 (Kernel Interface) fixes the calls: matvec over a row range
 *     [r0, r1) of W, and quantize_q8 with
 *     q = trunc(x*id + copysign(0.5, x)), id = 127/amax, d = amax/127.
 *   Sec. 6 (Error handling) fixes the convention: every call returns a
 *     status, nothing aborts.
 * The small-M product (M independent activation rows against one weight
 * matrix) is the batched-decode case of the page "ONNX Runtime", section
 * "6. Panel loop (pre-TCM)" (M = 4 rows of 4096 x 11008).
 *
 * Memory and layout (all pointers inside the structs are DEVICE pointers;
 * the structs themselves may live in host memory and are read during the
 * call only):
 *   W->q  Q4_0: rows * cols/2 bytes; block b of row r is the 16 bytes at
 *              offset (r*nb + b)*16, nb = cols/32.
 *         Q8_0: rows * cols int8; block b of row r at offset (r*nb + b)*32.
 *   W->d  rows * nb float32; scale of block (r, b) at index r*nb + b.
 *   x->q  m rows of n int8 (row i at x->q + i*n); x->d m rows of n/32 floats.
 *   y     float32 indexed by absolute row: y[r] for r in [r0, r1).  Entries
 *         outside [r0, r1) are never written.
 * Every q and d pointer must be 16-byte aligned (torch allocations are).
 * n (= cols) must be a positive multiple of 32 and at most MLQ_MAX_COLS.
 *
 * Ownership: the caller owns every buffer.  No call allocates device memory
 * or keeps a pointer after it returns.
 *
 * Launch: every compute call is asynchronous on `stream` (a cudaStream_t
 * passed as void*; NULL = the legacy default stream) and returns as soon
 * as the work is queued.  A status other than MLQ_OK means nothing was
 * queued.  Device-side problems (a bounded wait that gave up) are reported
 * by mlq_last_device_error() after the work has finished.
 *
 * Kernels are launched with programmatic dependent launch: a kernel may
 * start while the previous kernel on the stream is finishing and prefetch
 * weight bytes into L2 (always safe: L2 is the point of coherence), but it
 * reads and writes nothing through the caches before that previous kernel
 * has completed.  Set the environment variable MLQ_PDL=0 to launch plainly.
 * MLQ_STATIC_WEIGHTS=1 additionally lets the products issue their first
 * weight loads before that previous kernel has finished; set it only when
 * no work queued earlier on the stream writes the weight arrays (true for
 * inference weights loaded once; mlq_matvec_fused takes the same promise
 * per call through MLQ_F_STATIC_WEIGHTS).  MLQ_FUSED_L2_PREFETCH=1 makes
 * the register-pipelined mlq_matvec_fused kernel hint its whole weight
 * range into L2 first.  Both are off by default.
 *
 * Diagnostics: with MLQ_DIAG=1 every entry point reports on stderr, once per
 * distinct line, which kernel it launched for the shape it was given and
 * how (grid, threads, dynamic shared memory, cluster size, dependent launch,
 * and the launcher's own geometry: rows per CTA, K-chunks, ring stages ...),
 * e.g.
 *   mlq diag: mlq_matvec_q4 rows=11008 cols=4096 r=[0,11008) ->
 *     mlq::phase_ring_kernel<1, 16> grid=152 block=544 smem=... route=phase
 *     ring: products=1 rows=11008 K=4096 rows/CTA<=96 chunks=2 ...
 * (one line).  Off by default; when off it costs one predictable branch
 * per call.
 */
#ifndef MLQ_H
#define MLQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLQ_QK 32
#define MLQ_MAX_COLS 65536
#define MLQ_MAX_M 16
#define MLQ_MAX_SEQ 32768
#define MLQ_MAX_HEAD_DIM 256
#define MLQ_MAX_PREFETCH_RANGES 32
#define MLQ_FUSED_MAX_PRODUCTS 8
#define MLQ_CHAIN_MAX_PRODUCTS 32
#define MLQ_CHAIN_MAX_PHASES 24
#define MLQ_CHAIN_STATIC_MAX_PHASES 24

typedef enum {
    MLQ_OK = 0,
    MLQ_E_SHAPE = 1,   /* cols % 32 != 0, cols > MLQ_MAX_COLS, r0/r1 outside
                          0 <= r0 <= r1 <= rows, x->n != W->cols, M outside
                          1..16, x->m != M, ldy < r1, k != out->n           */
    MLQ_E_ALIGN = 2,   /* a q or d pointer is not 16-byte aligned          */
    MLQ_E_TYPE = 3,    /* W->type does not match the entry point           */
    MLQ_E_NULL = 4,    /* a required pointer is NULL                       */
    MLQ_E_ARCH = 5,    /* no CUDA device, or it is not compute capability
                          10.3 (the library is built for sm_103a only)     */
    MLQ_E_CUDA = 6,    /* a CUDA runtime call (launch, copy) failed        */
    MLQ_E_TIMEOUT = 7, /* a bounded device-side wait gave up; results of
                          that work are undefined                          */
    MLQ_E_BOUNDS = 8   /* bounds-checking build only (MLQ_CHECK_BOUNDS): a
                          kernel found an index outside the buffer it was
                          about to access and skipped that access; results
                          of that work are undefined                       */
} mlq_status;

enum { MLQ_Q8_0 = 0, MLQ_Q4_0 = 1 };

/* Weight tensor (Design Spec Sec. 4, ml_qtensor).  type is MLQ_Q8_0 or
 * MLQ_Q4_0; q holds raw bytes (int8 for Q8_0, packed nibbles for Q4_0). */
typedef struct {
    void *q;
    float *d;
    int rows, cols;
    uint8_t type;
} mlq_qtensor;

/* Q8_0 activations (Design Spec Sec. 4, ml_qact) extended to m rows of n. */
typedef struct {
    int8_t *q;
    float *d;
    int n;
    int m;
} mlq_qact;

/* Check that device 0.. the current device is compute capability 10.3 and
 * cache its SM count.  Called implicitly by every entry point; returns
 * MLQ_E_ARCH without a suitable device.  Idempotent, thread-safe. */
mlq_status mlq_init(void);

/* Design Spec Sec. 4 "Q8 quantization" and Sec. 5 quantize_q8: quantise
 * out->m rows of k float32 (x, device, row-major m x k) into out->q
 * (m x k int8) and out->d (m x k/32 float32).  Per block of 32:
 * amax = max|x|, d = amax/127 (IEEE division), id = 127/amax (0 when
 * amax = 0), q = trunc(x*id + copysign(0.5, x)) with the product and the
 * sum each rounded to float32 (no fused multiply-add), clamped to
 * [-127, 127]; a NaN (0 * inf when 127/amax overflows) stores 0.  Results
 * are bit-identical to that definition.  Requires out->n == k and
 * out->m >= 1. */
mlq_status mlq_quantize_q8(mlq_qact *out, const float *x, int k, void *stream);

/* Design Spec Sec. 5 matvec_q4: for r in [r0, r1)
 *   y[r] = sum_b (float)sumi(r, b) * W->d[r*nb + b] * x->d[b],
 *   sumi(r, b) = sum_j (nibble(r, b, j) - 8) * x->q[32b + j]   (exact int32).
 * W->type must be MLQ_Q4_0; x->m must be 1.  The float32 sum is taken in
 * an order other than b = 0, 1, ...; it agrees with the in-order sum within
 * 1e-5 * sum_b |term_b| per row. */
mlq_status mlq_matvec_q4(float *y, const mlq_qtensor *W, const mlq_qact *x,
                         int r0, int r1, void *stream);

/* Design Spec Sec. 5 matvec_q8: as mlq_matvec_q4 with int8 weights
 * (W->type == MLQ_Q8_0). */
mlq_status mlq_matvec_q8(float *y, const mlq_qtensor *W, const mlq_qact *X,
                         int r0, int r1, void *stream);

/* Batched small-M decode (ONNX Runtime page, "6. Panel loop"): M activation
 * rows X (X->m == M, each quantised per row) against one Q4_0 matrix:
 *   Y[m*ldy + r] = sum_b (float)sumi(m, r, b) * W->d[r*nb + b] * X->d[m*nb + b]
 * for m < M, r in [r0, r1).  1 <= M <= 16; ldy >= r1.  Same tolerance as
 * the M = 1 calls, per (m, r). */
mlq_status mlq_gemm_q4_small_m(float *Y, int ldy, const mlq_qtensor *W, const mlq_qact *X,
                               int M, int r0, int r1, void *stream);

/* Test hook (Design Spec Sec. 7: per-block int32 sums are checked exactly):
 * sumi[(r - r0)*nb + b] for r in [r0, r1), b < nb, computed by the same
 * block-dot code as the matvec of W->type (Q4_0 or Q8_0); x->m must be 1. */
mlq_status mlq_block_sumi(int32_t *sumi, const mlq_qtensor *W, const mlq_qact *x,
                          int r0, int r1, void *stream);

/* ---- Q4_K-style super-blocks ------------------------------------------- */
/* Page "SKaiNET-native-kernels", section "Proving an optimization is safe
 * before writing it": 4-bit nibbles n in [0, 15], 32-element sub-blocks
 * with a 6-bit scale s_b and a 6-bit minimum m_b, 8 sub-blocks per
 * 256-element super-block with a float32 scale d and a float32 scale of the
 * minima dmin; element value d*s_b*n - dmin*m_b.  The sub-block scales are
 * folded in the integer domain: per super-block the int32 sums
 *   ISUM = sum_b s_b * sum_i a_i n_i,   MSUM = sum_b m_b * sum_i a_i
 * (|ISUM| <= 8*63*32*127*15 = 3.07e7; with any byte values, 8*255*32*127*15
 * still fits int32) are converted to float once.
 * Layout (the page gives none; rows row-major, all device pointers):
 *   q:    rows x cols/2 bytes, 16 per 32-element sub-block in the Q4_0
 *         order (byte j: element j in the low nibble, j + 16 in the high);
 *   s:    rows x cols/256 x 16 bytes: per super-block the 8 sub-block
 *         scales, then the 8 sub-block minima;
 *   d, dmin: rows x cols/256 float32.
 * cols a positive multiple of 256, at most MLQ_MAX_COLS; q and s 16-byte
 * aligned, d and dmin 4-byte aligned. */
typedef struct {
    const void *q;
    const void *s;
    const float *d;
    const float *dmin;
    int rows, cols;
} mlq_q4k_tensor;

/* Activations for Q4_K products: n int8 quants q, n/256 float32 scales d
 * (one per 256 elements) and n/32 int32 sums of the quants per 32 elements
 * (bsums).  q, d and bsums 16-byte aligned device pointers. */
typedef struct {
    int8_t *q;
    float *d;
    int32_t *bsums;
    int n;
} mlq_q8k_act;

/* Quantise k float32 (x, device, 16-byte aligned) per 256 elements with the
 * rule of mlq_quantize_q8 (amax over the 256, d = amax/127, id = 127/amax,
 * q = trunc(x*id + copysign(0.5, x)) without fused multiply-add, clamp to
 * [-127, 127], NaN -> 0), and write the per-32 sums of the quants.
 * Bit-identical to that definition.  Requires out->n == k, k a positive
 * multiple of 256, at most MLQ_MAX_COLS. */
mlq_status mlq_quantize_q8k(mlq_q8k_act *out, const float *x, int k, void *stream);

/* For r in [r0, r1):
 *   y[r] = sum_B ((float)ISUM(r, B) * W->d[r*nsb + B]
 *                 - (float)MSUM(r, B) * W->dmin[r*nsb + B]) * x->d[B],
 * nsb = cols/256, each term in float32 in that order; the sum over B is
 * taken in an order other than B = 0, 1, ... and agrees with the in-order
 * sum within 1e-5 * sum_B |term_B| per row.  x->n == W->cols. */
mlq_status mlq_matvec_q4k(float *y, const mlq_q4k_tensor *W, const mlq_q8k_act *x, int r0, int r1,
                          void *stream);

/* Test hook: isum[(r - r0)*nsb + B] = ISUM(r, B), msum[...] = MSUM(r, B)
 * for r in [r0, r1), computed by the same code as mlq_matvec_q4k. */
mlq_status mlq_block_sums_q4k(int32_t *isum, int32_t *msum, const mlq_q4k_tensor *W,
                              const mlq_q8k_act *x, int r0, int r1, void *stream);

/* A Q4_K-style decode phase (the phase of mlq_decode_phase, Design Spec
 * Sec. 6 "Forward pass": products that read one activation): for each of
 * the nproducts (1..4) products, y_j = W_j * Q8K(x), every row of W_j,
 * where Q8K(x) is exactly what mlq_quantize_q8k writes for x and the
 * product is computed as mlq_matvec_q4k computes it.  One launch: every
 * CTA quantises x itself, so no quantiser launch precedes it.
 * x: k float32, device, 16-byte aligned; every W_j->cols == k (a positive
 * multiple of 256, at most MLQ_MAX_COLS); y_j: W_j->rows float32, 4-byte
 * aligned, owned by the caller.  Tensors as for mlq_matvec_q4k.  flags: 0
 * or MLQ_F_STATIC_INPUT (x is not written by work queued earlier on the
 * stream: the launch reads and quantises it before that work has
 * finished; its outputs still wait); anything else: MLQ_E_SHAPE. */
typedef struct {
    mlq_q4k_tensor W;
    float *y;
} mlq_q4k_product;
mlq_status mlq_q4k_phase(const float *x, int k, const mlq_q4k_product *products, int nproducts,
                         unsigned flags, void *stream);

/* ---- block length 32 / 128, float16 scales, signed-offset 8-bit -------- */
/* Page "ONNX Runtime" (SpaceMiT X60), "How we got there": item 3 (AMD's
 * Qwen2.5-0.5B export uses block_size 128; int8 activations), item 4
 * (8-bit weights packed as B' = B - 128 with flat scales and a per-block
 * zero-point correction that vanishes for zp = 128), item 5 (float16
 * scales).  Per block b of `blk` weights of row r:
 *   sumi = sum_i w_i * a_i,  w = nibble - 8 (bits 4) or B' + 128 - zp_b (bits 8),
 *   y[r] += ((float)sumi * scale_b) * x->d[b]   (float32, in this order);
 * the kernel forms sumi as sum B' a + (128 - zp) * sum a (or sum n a -
 * 8 * sum a) in int32, exactly.  Layout (the page gives none; rows
 * row-major, device pointers, all 16-byte aligned):
 *   q:      bits 4: rows x cols/2 bytes, block b's byte j holding element j
 *           (low nibble) and element j + blk/2 (high nibble);
 *           bits 8: rows x cols int8 B' = B - 128;
 *   scales: rows x scale_ld, float32 (scale_f16 = 0) or IEEE binary16
 *           (scale_f16 = 1); scale_ld >= cols/blk with scale_ld * (4 or 2)
 *           a multiple of 16 bytes;
 *   zp:     bits 8 only (NULL for bits 4): rows x zp_ld uint8 zero points
 *           of B, zp_ld >= cols/blk a multiple of 16; NULL means 128.
 * blk is 32 or 128; cols a positive multiple of blk, at most MLQ_MAX_COLS. */
typedef struct {
    const void *q;
    const void *scales;
    const uint8_t *zp;
    int rows, cols;
    int bits, blk;
    int scale_f16;
    int scale_ld, zp_ld;
} mlq_nbits_tensor;

/* Activations quantised per block of blk (32 or 128) elements: n int8
 * quants q (16-byte aligned), n/blk float32 scales d and n/blk int32 quant
 * sums bsums (4-byte aligned). */
typedef struct {
    int8_t *q;
    float *d;
    int32_t *bsums;
    int n;
    int blk;
} mlq_blk_act;

/* Quantise k float32 (x, device, 16-byte aligned) per out->blk elements
 * with the rule of mlq_quantize_q8 (bit-identical), and write each block's
 * quant sum.  out->n == k, k a positive multiple of out->blk, at most
 * MLQ_MAX_COLS; out->blk is 32 or 128. */
mlq_status mlq_quantize_blk(mlq_blk_act *out, const float *x, int k, void *stream);

/* A block-length decode phase (the phase of mlq_decode_phase, Design Spec
 * Sec. 6 "Forward pass"): for each of the nproducts (1..4) products,
 * y_j = W_j * Qblk(x), every row of W_j, where Qblk(x) is exactly what
 * mlq_quantize_blk writes for x with the products' block length, and the
 * product is computed as mlq_matvec_nbits computes it.  One launch: every
 * CTA quantises x itself.  All W_j share bits, blk, scale_f16, scale_ld,
 * zp_ld and whether zp is NULL (else MLQ_E_TYPE / MLQ_E_SHAPE); every
 * W_j->cols == k.  x: k float32, device, 16-byte aligned; y_j: W_j->rows
 * float32, 4-byte aligned, owned by the caller.  flags: 0 or
 * MLQ_F_STATIC_INPUT, as for mlq_q4k_phase. */
typedef struct {
    mlq_nbits_tensor W;
    float *y;
} mlq_nbits_product;
mlq_status mlq_nbits_phase(const float *x, int k, const mlq_nbits_product *products, int nproducts,
                           unsigned flags, void *stream);

/* y[r] for r in [r0, r1) as above; the sum over blocks is taken in another
 * order than b = 0, 1, ... and agrees with the in-order sum within
 * 1e-5 * sum_b |term_b| per row.  x->n == W->cols, x->blk == W->blk. */
mlq_status mlq_matvec_nbits(float *y, const mlq_nbits_tensor *W, const mlq_blk_act *x, int r0,
                            int r1, void *stream);

/* Test hook: sumi[(r - r0)*(cols/blk) + b] for r in [r0, r1), by the same
 * code as mlq_matvec_nbits. */
mlq_status mlq_block_sumi_nbits(int32_t *sumi, const mlq_nbits_tensor *W, const mlq_blk_act *x,
                                int r0, int r1, void *stream);

/* ---- the floating-point steps of a decode layer ------------------------ */
/* Page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 5 (ml_k_rmsnorm,
 * ml_k_softmax, ml_k_rope, ml_k_silu_mul, ml_k_add, ml_k_dot_f32,
 * ml_k_axpy_f32) and Sec. 6 (forward pass per token, GQA).  All arrays are
 * float32 on the device, 4-byte aligned; an optional Q8_0 output (one row,
 * ->n equal to the vector length, a multiple of 32, q and d 16-byte
 * aligned) receives exactly the bytes mlq_quantize_q8 would give for the
 * float32 result.  Float results match the definitions within relative
 * error 1e-5 (Sec. 7); sums are taken in a fixed order (deterministic).
 * Errors: MLQ_E_NULL for a missing pointer, MLQ_E_SHAPE for sizes out of
 * range, MLQ_E_ALIGN, MLQ_E_ARCH, MLQ_E_CUDA.  Calls are asynchronous on
 * `stream`; the caller owns every buffer. */

/* o = w * x / sqrt(mean(x^2) + eps), n elements; o (float) and/or oq (Q8_0)
 * may be NULL but not both.  o may alias x. */
mlq_status mlq_rmsnorm(float *o, const float *x, const float *w, int n, float eps, mlq_qact *oq,
                       void *stream);

/* The residual step of the forward pass followed by the next rmsnorm: x += y
 * (x is written back), then o = rmsnorm(x) as mlq_rmsnorm. */
mlq_status mlq_add_rmsnorm(float *x, const float *y, const float *w, int n, float eps, float *o,
                           mlq_qact *oq, void *stream);

/* y += x, n elements. */
mlq_status mlq_add(float *y, const float *x, int n, void *stream);

/* x = exp(x - max) / sum(exp(x - max)) in place, n elements. */
mlq_status mlq_softmax(float *x, int n, void *stream);

/* g = g / (1 + exp(-g)) * u in place, n elements; gq (Q8_0 of the result) or
 * NULL. */
mlq_status mlq_silu_mul(float *g, const float *u, int n, mlq_qact *gq, void *stream);

/* RoPE tables [max_seq][head_dim/2]: cos and sin of pos * theta^(-2i/head_dim)
 * (computed in double, rounded to float). */
mlq_status mlq_rope_tables(float *cos_t, float *sin_t, int max_seq, int head_dim, float theta,
                           void *stream);

/* Rotate the interleaved pairs (2i, 2i+1) of every head of q (n_heads x
 * head_dim) and k (n_kv_heads x head_dim) by the angles of one position:
 * cos_row / sin_row are that row of the tables.  q is rotated in place; the
 * rotated k goes to k_out (a KV cache row) or, if k_out is NULL, back to k.
 * v, v_out: NULL, or v (n_kv_heads x head_dim) is copied to v_out (the V
 * cache row).  n_heads % n_kv_heads == 0, head_dim even and <= 256. */
mlq_status mlq_rope(float *q, float *k, const float *cos_row, const float *sin_row, int head_dim,
                    int n_heads, int n_kv_heads, float *k_out, const float *v, float *v_out,
                    void *stream);

/* Attention of one token over n_pos cached positions: for query head h and
 * its KV head g = h / (n_heads / n_kv_heads), s_t = dot(q_h, K[t][g]) /
 * sqrt(head_dim) for t < n_pos, p = softmax(s), o_h = sum_t p_t V[t][g].
 * K and V caches: row t holds the n_kv_heads heads of position t, one after
 * another (row length n_kv_heads * head_dim).  oq: NULL, or the Q8_0 of o
 * (n_heads * head_dim elements; head_dim a multiple of 32).
 * 1 <= n_pos <= MLQ_MAX_SEQ. */
mlq_status mlq_attention(float *o, mlq_qact *oq, const float *q, const float *k_cache,
                         const float *v_cache, int n_pos, int head_dim, int n_heads, int n_kv_heads,
                         void *stream);

/* ---- decode chains: a whole decode step in one launch ------------------ */

/* One product of a chain: y[r] = sum_b (float)sumi(r, b) * W.d[r*nb+b] * dx_b
 * for every r < W.rows (Design Spec Sec. 5 matvec), x being its phase's
 * quantised input.  y is a device pointer.  A product with W.rows == 0 may
 * have NULL pointers (nothing is read or written). */
typedef struct {
    mlq_qtensor W;
    float *y;
} mlq_chain_product;

/* One phase: quantise x (n float32, device) to Q8_0 exactly as
 * mlq_quantize_q8 does, then run products[first .. first+count), all of
 * width n.  x may be the output y of a product of an EARLIER phase (the
 * chain runs phase by phase); it must not overlap an output of its own
 * phase.  xq_out / xd_out (both NULL, or n bytes and n/32 floats, 16-byte
 * aligned) receive the phase's quantised input, for inspection. */
typedef struct {
    const float *x;
    int n;
    int first, count;
    int8_t *xq_out;
    float *xd_out;
} mlq_chain_phase;

/* mlq_decode_chain for callers that cannot allocate device memory.
 *
 * Some callers may not call cudaMalloc (or any allocator) once they are
 * running: a decode loop that, like the Design Spec's runtime, sets up all
 * of its memory at load time and allocates nothing afterwards; code whose
 * device allocator belongs to another framework; code that runs while a
 * stream is being captured, where an allocation would break the capture.
 * mlq_decode_chain needs a small caller-allocated workspace for its grid
 * barriers; this variant takes none.  Its barrier counters live in a fixed
 * array of 64 words (256 bytes) inside the library, which every device that
 * loads the library keeps until the process exits.
 *
 * Arguments, requirements and results are those of mlq_decode_chain, with
 * at most MLQ_CHAIN_STATIC_MAX_PHASES phases (MLQ_E_SHAPE beyond).  The
 * caller still passes every input and output buffer.  Each call clears the
 * counters on `stream` before its kernel (cudaMemsetAsync, which allocates
 * nothing).  All calls on a device share the one array, so two calls whose
 * work overlaps on the GPU (different streams, or different host threads)
 * race and give wrong results or MLQ_E_TIMEOUT: serialise them.  The first
 * call on each device looks up the array's device address (once, with that
 * device current); make that first call before any stream capture.  The
 * address is kept for the life of the process: after cudaDeviceReset the
 * library's device state (this array, like the per-device status word and
 * properties that every entry point caches) is gone, so do not call into the
 * library on that device again in the same process.
 * Nothing on the pages corresponds to this entry point. */
mlq_status mlq_decode_chain_static(const mlq_chain_phase *phases, int nphases,
                                   const mlq_chain_product *products, int nproducts,
                                   void *stream);

/* One decode phase in one launch (Design Spec Sec. 6 "Forward pass": a
 * quantised activation feeds one or more products, e.g. Wq|Wk|Wv):
 * quantise x (n float32, device, 16-byte aligned) to Q8_0 exactly as
 * mlq_quantize_q8 does, then for each of the nproducts products
 * (1..MLQ_FUSED_MAX_PRODUCTS, same type, W.cols == n, n a multiple of 32
 * and at most MLQ_MAX_COLS) write y[r] for every r < W.rows, within the
 * tolerance of mlq_matvec_q4/_q8.  xq_out / xd_out (both NULL, or n bytes
 * and n/32 floats, 16-byte aligned) receive the quantised x.  The outputs
 * must not overlap x.  Built for chains of such calls under programmatic
 * dependent launch.  When a CTA's share of the weights fits in shared
 * memory, the kernel copies that share there in pieces and reduces rows as
 * they land.  flags: 0 or MLQ_F_STATIC_WEIGHTS (anything else:
 * MLQ_E_SHAPE).  MLQ_F_STATIC_WEIGHTS promises that no work queued earlier
 * on the stream writes any W.q or W.d of this call (true for inference
 * weights loaded once); the kernel may then start reading its weights
 * while the previous kernel is still running.
 * No counterpart on the pages: a GPU fusion of quantize_q8 and matvec. */
#define MLQ_F_STATIC_WEIGHTS 1u
/* mlq_decode_phase: the float input x is not written by work queued earlier
 * on the stream (a step's own input, copied in before its first launch): the
 * launch may read and quantise x before that work has finished.  Its writes
 * (xq_out / xd_out, the outputs) still wait.  Ignored for a Q8_0 input. */
#define MLQ_F_STATIC_INPUT 2u
mlq_status mlq_matvec_fused(const float *x, int n, const mlq_chain_product *products,
                            int nproducts, int8_t *xq_out, float *xd_out, unsigned flags,
                            void *stream);

/* One product of mlq_decode_phase: y = W * (the phase input), and, when yq
 * is not NULL, y quantised to Q8_0 in the same launch (yq: W.rows int8,
 * yd: W.rows/32 floats, both 16-byte aligned, W.rows a multiple of 32),
 * bytes identical to mlq_quantize_q8 applied to the stored y. */
typedef struct {
    mlq_qtensor W;
    float *y;
    int8_t *yq;
    float *yd;
} mlq_phase_product;

/* The input of mlq_decode_phase: either float x (xq, xd NULL), quantised
 * in the launch exactly as mlq_quantize_q8 does -- xq_out / xd_out (both
 * NULL, or n bytes and n/32 floats) then receive that quantisation -- or,
 * with x NULL, an input already in Q8_0 (xq: n int8, xd: n/32 floats),
 * typically the yq / yd of a product of the previous phase; xq_out / xd_out
 * must be NULL then.  All pointers device, 16-byte aligned. */
typedef struct {
    const float *x;
    const int8_t *xq;
    const float *xd;
    int n;
    int8_t *xq_out;
    float *xd_out;
} mlq_phase_input;

/* One decode phase of the Design Spec's forward pass (Sec. 6: a quantised
 * activation feeds one or more products -- Wq|Wk|Wv, gate|up -- and a
 * product's output is quantised as the next product's input) in ONE launch:
 * for each of the nproducts products (1..MLQ_FUSED_MAX_PRODUCTS, all of one
 * type, W.cols == n, n a positive multiple of 32 and at most MLQ_MAX_COLS)
 * y[r] for every r < W.rows, within the tolerance of mlq_matvec_q4/_q8, and
 * each requested Q8_0 copy of y.  If any product has yq, every product's
 * W.rows must be a multiple of 32 (MLQ_E_SHAPE otherwise).  Outputs must
 * not overlap the input or each other.  flags: 0, MLQ_F_STATIC_WEIGHTS (as
 * for mlq_matvec_fused) and/or MLQ_F_STATIC_INPUT (anything else:
 * MLQ_E_SHAPE).  A chain of such calls, each taking the
 * previous one's yq / yd, runs a decode step with no separate quantize
 * launches: each phase quantises its outputs while they are still on chip.
 * prefetch / prefetch_bytes (host arrays of nprefetch <= MLQ_PHASE_MAX_PREFETCH
 * device ranges, read during the call; NULL when nprefetch == 0): a pure
 * hint, typically the weights of the phase after next.  Once the launch has
 * read its own input, its CTAs hint those ranges into L2, so that a chain
 * streams the next weights from HBM while its phases run, behind no
 * critical-path read (an SM serves its reads in order: a prefetch issued
 * earlier would delay them).  Unaligned range ends are trimmed to 16 bytes.
 * A CTA's share of the weights is held whole in shared memory when it fits,
 * else streamed through a ring of shared-memory stages (K <= 16384); the
 * ring launch ignores the hint (its SMs' reads are its own stream: L2
 * hints there measured slower on GB300).  Other
 * shapes (K not a multiple of 128, longer rows) get the same work as several
 * launches (products, then quantize, then the prefetch).
 * No counterpart on the pages: a GPU fusion of their quantize_q8 and
 * matvec calls. */
#define MLQ_PHASE_MAX_PREFETCH 16
mlq_status mlq_decode_phase(const mlq_phase_input *in, const mlq_phase_product *products,
                            int nproducts, const void *const *prefetch,
                            const size_t *prefetch_bytes, int nprefetch, unsigned flags,
                            void *stream);

/* Bytes of workspace mlq_decode_chain needs for `nphases` phases. */
size_t mlq_chain_workspace_bytes(int nphases);

/* Run a chain of phases (Design Spec Sec. 6 "Forward pass": per layer, a
 * norm/activation output is quantised and multiplied by one or more
 * matrices, whose output feeds the next quantisation) in ONE cooperative
 * launch: one CTA per SM streams the weights of every phase back to back
 * while the phases run in order, separated by grid-wide barriers.
 * Requirements: 1 <= nphases <= MLQ_CHAIN_MAX_PHASES, 1 <= nproducts <=
 * MLQ_CHAIN_MAX_PRODUCTS; every product of the same type (Q4_0 or Q8_0);
 * cols a multiple of 128 and at most MLQ_MAX_COLS; W.q, W.d, x 16-byte
 * aligned.  Results: identical quantisation; products within the same
 * tolerance as mlq_matvec_q4/_q8.
 * workspace: device memory of at least mlq_chain_workspace_bytes(nphases)
 * bytes, 4-byte aligned, owned by the caller, ZERO-FILLED before its first
 * use; every call leaves it zero again (also after MLQ_E_TIMEOUT).  Calls
 * that share a workspace must not overlap on the GPU.  No counterpart on
 * the pages: a GPU scheduling of their decode step. */
mlq_status mlq_decode_chain(const mlq_chain_phase *phases, int nphases,
                            const mlq_chain_product *products, int nproducts,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Hint n byte ranges (device pointers ptrs[i], lengths bytes[i]; the two
 * arrays live in host memory and are read during the call) into L2, e.g.
 * the weights of the next products of a decode step, so that their HBM
 * reads overlap earlier work.  Queues one short kernel that issues bulk L2
 * prefetches and exits; the data keeps arriving after it finishes.  Pure
 * hint: it changes no memory, never waits for earlier work on the stream
 * and never makes later work read stale data (L2 is the device's point of
 * coherence).  Unaligned range ends are trimmed to 16-byte boundaries.
 * 0 <= n <= MLQ_MAX_PREFETCH_RANGES.  No counterpart on the pages: an
 * addition for GPU decode chains. */
mlq_status mlq_prefetch_l2(const void *const *ptrs, const size_t *bytes, int n, void *stream);

/* Synchronise `stream`, then report and clear the library's device status
 * word: MLQ_E_TIMEOUT if any kernel since the last call gave up a bounded
 * wait, MLQ_E_CUDA if the stream reported an error, else MLQ_OK. */
mlq_status mlq_last_device_error(void *stream);

/* Test hook: limit, in nanoseconds, of every device-side wait (default
 * 1e9 = one second).  0 makes every wait give up at once, which exercises
 * the timeout path without any real hang: the kernel then records
 * MLQ_E_TIMEOUT, drains its own copies in flight with the default limit
 * and returns.  Affects launches made after the call. */
mlq_status mlq_debug_set_wait_limit_ns(uint64_t limit_ns);

/* Test hook, host only (no device work, pointers not dereferenced): the
 * plan mlq_decode_chain's streaming kernel would use for these arguments
 * on num_sms CTAs, written to info (int32):
 *   info[0] 1 if the streaming kernel takes the chain, 0 if the legacy
 *           kernel would (then only info[0..3 + 8*nphases] are written, 0);
 *   info[1] CTAs; info[2] ring bytes; info[3] dynamic shared memory bytes;
 *   info[4 + 8p ..]: phase p's K-chunks C, blocks per chunk, warps per
 *           chunk G, rows per warp RW, rows per stage R, input read as
 *           Q8_0 from an earlier phase (0/1), some output written as Q8_0
 *           in-chain (0/1), bit mask of the phase's products that do;
 *   info[4 + 8*nphases + p*(CTAs + 1) + b]: the first row (phase
 *           numbering) of CTA b in phase p, b = 0..CTAs.
 * Arguments are validated as by mlq_decode_chain.  MLQ_E_SHAPE when
 * info_len is too small or num_sms < 1.  Nothing on the pages corresponds
 * to this entry point. */
mlq_status mlq_debug_chain_plan(const mlq_chain_phase *phases, int nphases,
                                const mlq_chain_product *products, int nproducts, int num_sms,
                                int32_t *info, int info_len);

/* Human-readable name of a status. Never NULL. */
const char *mlq_status_str(mlq_status s);

#ifdef __cplusplus
}
#endif

#endif /* MLQ_H */
