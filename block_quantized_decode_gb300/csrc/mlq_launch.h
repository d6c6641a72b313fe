// mlq_launch.h -- host-side declarations shared by the C-ABI shim and the
// kernel translation units of libmlq (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "diag.h"

namespace mlq {

// Everything a launcher needs besides the operands.
struct LaunchCtx {
  cudaStream_t stream;
  bool pdl;                     // launch with programmatic stream serialization
  int num_sms;                  // SMs of the current device
  int *status;                  // device status word (MLQ_E_TIMEOUT on a bounded-wait give-up)
  unsigned long long wait_ns;   // limit of every device-side wait
  bool early_weights;           // weights are not written by earlier queued work:
                                // their first loads may precede the dependency wait
};

// Kernels of a dependent decode chain (quantize, M = 1 products, fused
// phases) ask for the largest shared-memory carveout.  An SM's L1/shared
// split can only change while it is idle, so kernels of one chain with
// different preferences could not share an SM; with one common split the
// next kernel of a chain can become resident while the previous one is
// still running.  (The small-M kernels keep the default: they read their
// activations through L1.)  Done once per kernel.
void prefer_max_shared_impl(const void *kern);
template <typename K>
inline void prefer_max_shared(K kern) {
  prefer_max_shared_impl(reinterpret_cast<const void *>(kern));
}

// Launch `kern` with cudaLaunchKernelEx, optionally with programmatic
// dependent launch, on ctx.stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          const LaunchCtx &ctx, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ctx.pdl ? 1 : 0;
  if (diag_on()) diag_launch(reinterpret_cast<const void *>(kern), grid, block, smem, 1, ctx.pdl);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// prefetch.cu: up to kMaxPrefetchRanges byte ranges to hint into L2.
constexpr int kMaxPrefetchRanges = 32;
struct PrefetchList {
  const void *ptr[kMaxPrefetchRanges];
  size_t bytes[kMaxPrefetchRanges];
  int n;
};
cudaError_t launch_prefetch_l2(const LaunchCtx &ctx, const PrefetchList &list);

// quantize.cu: m rows of k floats -> Q8_0 (q, d).
cudaError_t launch_quantize_q8(const LaunchCtx &ctx, const float *x, int8_t *q, float *d, int m,
                               int k);

// matvec.cu: M = 1 product over rows [r0, r1).  qtype 0 = Q8_0, 1 = Q4_0.
// Exactly one of y / sumi is non-null (sumi = per-block int32 test hook).
cudaError_t launch_matvec_m1(const LaunchCtx &ctx, int qtype, const void *wq, const float *wd,
                             int nb, const int8_t *xq, const float *xd, float *y, int32_t *sumi,
                             int r0, int r1);

// matvec_tma.cu: the bulk-copy ring version of launch_matvec_m1; returns
// cudaErrorNotSupported without launching when the shape does not suit it.
cudaError_t launch_matvec_m1_tma(const LaunchCtx &ctx, int qtype, const void *wq, const float *wd,
                                 int nb, const int8_t *xq, const float *xd, float *y,
                                 int32_t *sumi, int r0, int r1);

// chain.cu: a decode step of dependent products in one persistent launch.
constexpr int kChainMaxProducts = 32;
constexpr int kChainMaxPhases = 24;
struct ChainProductDev {
  const uint8_t *wq;
  const float *wd;
  float *y;
  int rows;
};
struct ChainPhaseDev {
  const float *x;
  int8_t *xq_out;
  float *xd_out;
  int nb;
  int first, count;
};
struct ChainArgs {
  ChainProductDev prod[kChainMaxProducts];
  ChainPhaseDev phase[kChainMaxPhases];
  int nphases;
  int kmax;             // largest phase width
  unsigned *counters;   // nphases + 1 words of caller workspace, zero on entry and exit
  int *status;
  unsigned long long wait_ns;
  int ns, stage_bytes, xbuf_bytes;  // ring geometry (set by the launcher)
};
cudaError_t launch_decode_chain(const LaunchCtx &ctx, int qtype, const ChainArgs &a);
// stream.cu: the same chain with the weight stream running ahead across
// phases and in-chain Q8_0 hand-offs; cudaErrorNotSupported (nothing
// launched) when a phase is wider than its consumer warps can hold.
cudaError_t launch_decode_stream(const LaunchCtx &ctx, int qtype, const ChainArgs &a);
// The streaming kernel's plan for `a` on `num_sms` CTAs, as integers (the
// layout of mlq_debug_chain_plan); host only.  Returns -1 when info_len is
// too small, 0 when the chain does not suit the kernel, 1 otherwise.
int describe_decode_stream(int num_sms, int qtype, const ChainArgs &a, int32_t *info, int info_len);
// Same chain with its barrier counters in a fixed device array of chain.cu
// (no workspace, no allocation); at most kStaticChainWords - 1 phases.
constexpr int kStaticChainWords = 64;
cudaError_t launch_decode_chain_static(const LaunchCtx &ctx, int device, int qtype,
                                       const ChainArgs &a);

// fused.cu: quantise x and run up to kFusedMaxProducts products of its width.
constexpr int kFusedMaxProducts = 8;
constexpr int kPhaseMaxPrefetch = 16;
struct FusedProduct {
  const uint8_t *wq;
  const float *wd;
  float *y;
  int rows;
  int8_t *yq;   // optional Q8_0 copy of y, written in the same launch (rows % 32 == 0)
  float *yd;
};
struct FusedArgs {
  FusedProduct prod[kFusedMaxProducts];
  int nproducts;
  const float *x;         // float input, quantised in the prologue; or nullptr and ...
  const int8_t *xq_in;    // ... the input already in Q8_0 (written by an earlier launch)
  const float *xd_in;
  int nb;
  int8_t *xq_out;   // optional copy of the quantised x (written by CTA 0)
  float *xd_out;
  int any_yq;       // some product quantises its output: rows are split in 32-row atoms there
  int total_rows;   // set by the launcher
  int nchunks;      // set by the launcher
  int chunk_blocks; // set by the launcher (phase kernel: blocks of K per warp chunk)
  unsigned smem_part, smem_w, smem_wd;  // set by the launcher (phase kernel: smem offsets)
  int ring_rows, ring_slots;            // set by the launcher (ring phase kernel: stage geometry)
  unsigned ring_stage, ring_dq;         //   stage bytes; offset of a stage's scales
  int early;        // first weight loads before the dependency wait (static weights)
  int early_input;  // the float input x is read and quantised before the dependency wait (static input)
  int input_bulk;   // set by the launcher (ring phase kernel): the Q8_0 input lands by bulk copies
  int input_issue_release;  // set by the launcher (ring): the producer goes on once the input's copies are issued
  int hint_partner;         // set by the launcher (ring): k > 0: CTAs b < grid / k hint a late CTA's first stage
  int hint_stages;          // set by the launcher (ring): stages of the late CTA hinted
  int prefetch;     // set by the launcher: hint the CTA's weights into L2 first
  int *status;      // set by the launcher
  unsigned long long wait_ns;
  // byte ranges to hint into L2 once the input has been read (phase kernel)
  const void *pf_ptr[kPhaseMaxPrefetch];
  size_t pf_bytes[kPhaseMaxPrefetch];
  int npf;
};
// Every launch of a phase: the phase kernel when the CTA slices fit in
// shared memory, else the streaming kernel of fused.cu (float input, no
// quantised outputs) or, for the other cases, matvec + quantize launches.
cudaError_t launch_matvec_fused(const LaunchCtx &ctx, int qtype, const FusedArgs &a);
// phase.cu: the shared-memory phase kernel, else the ring phase kernel;
// returns cudaErrorNotSupported without launching when neither suits.
cudaError_t launch_phase(const LaunchCtx &ctx, int qtype, const FusedArgs &a);
// phase_ring.cu: the ring phase kernel alone (same contract).
cudaError_t launch_phase_ring(const LaunchCtx &ctx, int qtype, const FusedArgs &a);

// gemm_mma.cu: M activation rows (2..16) against a Q4_0 matrix on the
// tensor cores (fp16 mma.sync, exact block sums).
cudaError_t launch_gemm_q4_mma(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                               const int8_t *xq, const float *xd, int M, float *Y, int ldy,
                               int r0, int r1);

// gemm_mma_cluster.cu: the same product streaming the weights through
// per-warp TMA rings, K split over a thread-block cluster.  `rows` is the
// row count of W (the tensor copies describe the whole matrix).
// cudaErrorNotSupported when K is above 16384, nb is not a multiple of 4,
// or the device cannot hold one cluster.
cudaError_t launch_gemm_q4_mma_cluster(const LaunchCtx &ctx, const void *wq, const float *wd,
                                       int nb, const int8_t *xq, const float *xd, int M, float *Y,
                                       int ldy, int r0, int r1, int rows);

// gemm_ring.cu: M <= 4 activation rows against a Q4_0 matrix, the
// activations in registers, whole weight rows streamed through a shared-
// memory ring.  cudaErrorNotSupported when M > 4, nb is not a multiple of 4
// or K needs more than 16 chunks of 32 (M > 2) or 64 (M <= 2) blocks.
cudaError_t launch_gemm_q4_ring(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                                const int8_t *xq, const float *xd, int M, float *Y, int ldy, int r0,
                                int r1);

// gemm_umma.cu: the same product on the tcgen05 tensor cores, the weights
// and the block sums in tensor memory, K split over a thread-block cluster.
// cudaErrorNotSupported when K is above 16384, nb is not a multiple of 4,
// or the device cannot hold one cluster.
cudaError_t launch_gemm_q4_umma(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                                const int8_t *xq, const float *xd, int M, float *Y, int ldy, int r0,
                                int r1, int rows);

// q4k.cu: Q4_K-style super-blocks (per-256 activation quantiser; M = 1
// product with the sub-block scales folded in int32; isum/msum non-null
// selects the integer-sums test hook instead of y).
cudaError_t launch_quantize_q8k(const LaunchCtx &ctx, const float *x, int8_t *q, float *d,
                                int32_t *bsums, int k);
cudaError_t launch_matvec_q4k(const LaunchCtx &ctx, const void *wq, const void *ws, const float *wd,
                              const float *wdmin, int nsb, const int8_t *xq, const float *xd,
                              const int32_t *xbs, float *y, int32_t *isum, int32_t *msum, int r0,
                              int r1);
// A Q4_K-style phase: up to 4 products sharing the float input x (nsb
// super-blocks), every CTA quantising x itself; product j writes rows
// 0 .. rows_j of y_j.
struct Q4KProductDev {
  const void *q, *s;
  const float *d, *dmin;
  float *y;
  int rows;
};
// early_input: x is not written by earlier work (read and quantised before
// the dependency wait).
cudaError_t launch_phase_q4k(const LaunchCtx &ctx, const float *x, int nsb, const Q4KProductDev *p,
                             int np, bool early_input);

// nbits.cu: blocks of 32 or 128, float32 / binary16 scales, 4-bit or
// signed-offset 8-bit weights (sumi non-null: the integer test hook).
cudaError_t launch_quantize_blk(const LaunchCtx &ctx, const float *x, int8_t *q, float *d,
                                int32_t *bsums, int k, int blk);
cudaError_t launch_matvec_nbits(const LaunchCtx &ctx, int bits, int blk, const void *wq, const void *sc,
                                int sc_f16, int sc_ld, const uint8_t *zp, int zp_ld, int cols,
                                const int8_t *xq, const float *xd, const int32_t *xbs, float *y,
                                int32_t *sumi, int r0, int r1);
// A block-length phase: up to 4 products of one format sharing the float
// input x (cols elements), every CTA quantising x itself; product j writes
// rows 0 .. rows_j of y_j.
struct NBitsProductDev {
  const void *q, *scales;
  const uint8_t *zp;
  float *y;
  int rows;
};
cudaError_t launch_phase_nbits(const LaunchCtx &ctx, int bits, int blk, int sc_f16, int sc_ld, int zp_ld,
                               int cols, const float *x, const NBitsProductDev *p, int np, bool early_input);

// layer.cu: the floating-point steps of a decode layer (each one launch).
cudaError_t launch_rmsnorm_q8(const LaunchCtx &ctx, float *x, const float *y, const float *w,
                              float *h, int8_t *hq, float *hd, int n, float eps);
cudaError_t launch_add(const LaunchCtx &ctx, float *y, const float *x, int n);
cudaError_t launch_softmax(const LaunchCtx &ctx, float *x, int n);
cudaError_t launch_silu_mul_q8(const LaunchCtx &ctx, float *g, const float *u, int n, int8_t *gq,
                               float *gd);
cudaError_t launch_rope_tables(const LaunchCtx &ctx, float *cos_t, float *sin_t, int max_seq,
                               int head_dim, float theta);
struct RopeArgs;
struct AttnArgs;
cudaError_t launch_rope_call(const LaunchCtx &ctx, float *q, float *k, float *k_out, const float *v,
                             float *v_out, const float *cos_t, const float *sin_t, int head_dim,
                             int n_heads, int n_kv_heads);
cudaError_t launch_attention_call(const LaunchCtx &ctx, float *o, int8_t *oq, float *od,
                                  const float *q, const float *kc, const float *vc, int n_pos,
                                  int head_dim, int n_heads, int n_kv_heads);

// gemm_small_m.cu: M activation rows (1..16) against a Q4_0 matrix.
cudaError_t launch_gemm_q4_small_m(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                                   const int8_t *xq, const float *xd, int M, float *Y, int ldy,
                                   int r0, int r1,
                                   int rows);

}  // namespace mlq
