// matvec.cu -- M = 1 block-quantized matrix-vector product on sm_103a.
//
// Computes, for rows r in [r0, r1) (page "Legacy-ISA ML Inference Runtime --
// Design Spec", Sec. 4 "Integer dot per block" and Sec. 5 matvec_q4 /
// matvec_q8):
//   sumi(r, b) = sum_{j<32} qw(r, b, j) * qx(32b + j)          (exact int32)
//   y[r]       = sum_b ((float)sumi(r, b) * dw(r, b)) * dx(b)  (float32)
// Q4_0: qw = nibble - 8, low nibble of byte j = element j, high nibble =
// element j + 16.  Q8_0: qw = int8.
//
// Design (GB300-first; the pages' SIMD designs are CPU prior art):
//  * HBM streaming: each CTA owns a contiguous, balanced range of rows, so
//    its weight bytes are one contiguous stretch of q and one of d.  Every
//    lane reads 16 B of q per load (a whole Q4_0 block, or half a Q8_0
//    block) with a read-only 128-bit load that does not allocate in L1 and
//    is marked evict-first in L2; consecutive lanes read consecutive 16 B,
//    so every warp-wide load is a fully used 512 B stretch.  Scales are read
//    with coalesced 32-bit loads of the same units.
//  * Memory-level parallelism: a warp works on tasks = (row, K-chunk of
//    32*U units) and software-pipelines them (the next task's loads are in
//    flight while the current one is reduced), eight warps per CTA, several
//    CTAs per SM.  At kernel start one thread bulk-prefetches the first
//    64 KiB of the CTA's weight bytes into L2 (cp.async.bulk.prefetch), which
//    also runs before the wait on the previous kernel under programmatic
//    dependent launch.
//  * Activations: the Q8_0 vector (K bytes of q, K/32 floats of d) is staged
//    once per CTA in shared memory by a 1-D bulk copy (TMA) completing on an
//    mbarrier; the wait is bounded (see mlq_device.cuh).
//  * Integer dot: __dp4a on four packed int8 at a time.  For Q4_0 the
//    nibbles are used as unsigned 0..15 and the -8 offset is folded into a
//    per-block correction: sum (n-8) qx = sum n qx - 8 * sum qx, where
//    sum qx of every activation block is computed once per CTA in the
//    prologue.  For Q8_0 two adjacent lanes hold the two halves of a block
//    and combine their int32 partial sums with one shuffle, so sumi is
//    formed exactly before it is converted to float.
//  * Reduction: per-lane float partials, a warp-shuffle tree per task, and
//    (when a row spans several chunks) a fixed-order sum of the per-chunk
//    partials in shared memory: deterministic, no atomics.
#include <cstdlib>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

struct MatvecArgs {
  const uint8_t *wq;
  const float *wd;
  const int8_t *xq;
  const float *xd;
  float *y;          // output (null when sumi is set)
  int32_t *sumi;     // per-block sums test hook (null for the product)
  int nb;            // blocks per row
  int r0, r1;        // row range
  int nchunks;       // tasks per row
  int early;         // 1: first weight loads may precede the dependency wait
  int *status;
  unsigned long long wait_ns;
};

constexpr size_t kPrefetchBytes = 64 * 1024;
constexpr int kWarps = 8;

template <int U>
struct WRegs {
  uint4 q[U];
  float d[U];
};

// Units: Q4_0 -> one unit = one 16-byte block; Q8_0 -> one unit = one
// 16-byte half block (two units per block).
template <int QT, int U>
__device__ __forceinline__ void load_task(WRegs<U> &r, const MatvecArgs &a, int row, int base,
                                          int lane, int upr) {
  const size_t rowq = static_cast<size_t>(a.nb) * (QT == 1 ? 16 : 32);
  const uint8_t *qrow = a.wq + static_cast<size_t>(row) * rowq;
  const float *drow = a.wd + static_cast<size_t>(row) * a.nb;
  const uint64_t pol = l2_policy_evict_first();
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int unit = base + lane + 32 * u;
    if (unit < upr) {
      r.q[u] = ld_stream_v4(qrow + static_cast<size_t>(unit) * 16, pol);
      r.d[u] = ld_stream_f32(drow + (QT == 1 ? unit : (unit >> 1)), pol);
    } else {
      r.q[u] = make_uint4(0u, 0u, 0u, 0u);
      r.d[u] = 0.0f;
    }
  }
}

// Q4_0 block dot with the -8 fold: nibbles as unsigned bytes, then
// subtract 8 * sum(qx) of the activation block.
__device__ __forceinline__ int q4_block_dot(const uint4 w, const int4 xa, const int4 xb,
                                            int sx) {
  constexpr uint32_t kLo = 0x0F0F0F0Fu;
  int s = __dp4a(static_cast<int>(w.x & kLo), xa.x, 0);         // elements 0..3
  s = __dp4a(static_cast<int>(w.y & kLo), xa.y, s);             // 4..7
  s = __dp4a(static_cast<int>(w.z & kLo), xa.z, s);             // 8..11
  s = __dp4a(static_cast<int>(w.w & kLo), xa.w, s);             // 12..15
  s = __dp4a(static_cast<int>((w.x >> 4) & kLo), xb.x, s);      // 16..19
  s = __dp4a(static_cast<int>((w.y >> 4) & kLo), xb.y, s);      // 20..23
  s = __dp4a(static_cast<int>((w.z >> 4) & kLo), xb.z, s);      // 24..27
  s = __dp4a(static_cast<int>((w.w >> 4) & kLo), xb.w, s);      // 28..31
  return s - 8 * sx;
}

template <bool SUMI, int U>
__device__ __forceinline__ float compute_q4(const WRegs<U> &r, const int8_t *xq_s,
                                            const float *xd_s, const int *sx_s, int base,
                                            int lane, int nb, int32_t *sumi_row) {
  float acc = 0.0f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int b = base + lane + 32 * u;
    if (b < nb) {
      const int4 xa = *reinterpret_cast<const int4 *>(xq_s + b * kQK);
      const int4 xb = *reinterpret_cast<const int4 *>(xq_s + b * kQK + 16);
      const int s = q4_block_dot(r.q[u], xa, xb, sx_s[b]);
      if (SUMI) {
        sumi_row[b] = s;
      } else {
        acc = __fmaf_rn(__fmul_rn(__int2float_rn(s), r.d[u]), xd_s[b], acc);
      }
    }
  }
  return acc;
}

template <bool SUMI, int U>
__device__ __forceinline__ float compute_q8(const WRegs<U> &r, const int8_t *xq_s,
                                            const float *xd_s, int base, int lane, int upr,
                                            int32_t *sumi_row) {
  float acc = 0.0f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int h = base + lane + 32 * u;  // half-block index; pairs never straddle upr
    const bool valid = h < upr;
    int s = 0;
    if (valid) {
      const int4 xa = *reinterpret_cast<const int4 *>(xq_s + h * 16);
      const uint4 w = r.q[u];
      s = __dp4a(static_cast<int>(w.x), xa.x, 0);
      s = __dp4a(static_cast<int>(w.y), xa.y, s);
      s = __dp4a(static_cast<int>(w.z), xa.z, s);
      s = __dp4a(static_cast<int>(w.w), xa.w, s);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);  // the other half of the block
    if (valid && !(lane & 1)) {
      const int b = h >> 1;
      if (SUMI) {
        sumi_row[b] = s;
      } else {
        acc = __fmaf_rn(__fmul_rn(__int2float_rn(s), r.d[u]), xd_s[b], acc);
      }
    }
  }
  return acc;
}

// Shared memory: [K bytes qx][nb floats dx][nb ints sum(qx)][partials].
template <int QT, int U, bool SUMI>
__global__ void __launch_bounds__(kWarps * 32) matvec_m1_kernel(const MatvecArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_storage;
  const int nb = a.nb;
  const int K = nb * kQK;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + K);
  int *sx_s = reinterpret_cast<int *>(smem + K + 4 * nb);
  float *part_s = reinterpret_cast<float *>(smem + K + 8 * nb);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.r1 - a.r0;
  const int ra = a.r0 + static_cast<int>(static_cast<long long>(n) * blockIdx.x / gridDim.x);
  const int rb =
      a.r0 + static_cast<int>(static_cast<long long>(n) * (blockIdx.x + 1) / gridDim.x);
  const int nr = rb - ra;
  const int upr = QT == 1 ? nb : 2 * nb;
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  const uint32_t bar = smem_addr(&bar_storage);

  if (tid == 0) {
    if (nr > 0) {
      prefetch_range_l2(a.wq + static_cast<size_t>(ra) * rowq, static_cast<size_t>(nr) * rowq,
                        kPrefetchBytes);
      prefetch_range_l2(a.wd + static_cast<size_t>(ra) * nb, static_cast<size_t>(nr) * nb * 4,
                        kPrefetchBytes / 4);
    }
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  const int nch = a.nchunks;
  const int tasks = nr * nch;
  int t = warp;
  WRegs<U> cur;
  bool loaded = false;
  if (a.early && t < tasks) {  // weights are static: start streaming before the wait
    const int rl = t / nch;
    load_task<QT, U>(cur, a, ra + rl, (t - rl * nch) * 32 * U, lane, upr);
    loaded = true;
  }
  griddep_wait();  // x (and anything else we read) may come from the previous kernel
  griddep_launch_dependents();
  __syncthreads();

  const bool bulk_xd = (nb & 3) == 0;  // the bulk engine copies multiples of 16 B
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(K + (bulk_xd ? 4 * nb : 0)));
    bulk_copy_g2s(smem_addr(xq_s), a.xq, static_cast<uint32_t>(K), bar);
    if (bulk_xd) bulk_copy_g2s(smem_addr(xd_s), a.xd, static_cast<uint32_t>(4 * nb), bar);
  }
  if (!bulk_xd) {
    for (int i = tid; i < nb; i += kWarps * 32) xd_s[i] = a.xd[i];
  }

  if (!loaded && t < tasks) {
    const int rl = t / nch;
    load_task<QT, U>(cur, a, ra + rl, (t - rl * nch) * 32 * U, lane, upr);
  }

  bool ok = mbar_wait_warp(bar, 0, a.wait_ns);
  ok = __syncthreads_and(ok) != 0;
  if (!ok) {
    if (tid == 0) set_status(a.status, kStatusTimeout);
    mbar_wait_bounded(bar, 0, kDrainWaitNs);  // our own copy must land before we exit
    return;
  }
  if (QT == 1) {
    for (int b = tid; b < nb; b += kWarps * 32) {
      const int *w = reinterpret_cast<const int *>(xq_s + b * kQK);
      int s = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) s = __dp4a(w[i], 0x01010101, s);
      sx_s[b] = s;
    }
  }
  __syncthreads();

  for (; t < tasks; t += kWarps) {
    const int rl = t / nch;
    const int c = t - rl * nch;
    const int tn = t + kWarps;
    WRegs<U> nxt;
    if (tn < tasks) {
      const int rln = tn / nch;
      load_task<QT, U>(nxt, a, ra + rln, (tn - rln * nch) * 32 * U, lane, upr);
    }
    const int row = ra + rl;
    int32_t *srow = SUMI ? a.sumi + static_cast<size_t>(row - a.r0) * nb : nullptr;
    float acc;
    if (QT == 1) {
      acc = compute_q4<SUMI, U>(cur, xq_s, xd_s, sx_s, c * 32 * U, lane, nb, srow);
    } else {
      acc = compute_q8<SUMI, U>(cur, xq_s, xd_s, c * 32 * U, lane, upr, srow);
    }
    if (!SUMI) {
      acc = warp_sum(acc);
      if (lane == 0) {
        if (nch == 1) {
          if (in_bounds(row >= a.r0 && row < a.r1, a.status)) a.y[row] = acc;
        } else {
          part_s[rl * nch + c] = acc;
        }
      }
    }
    if (tn < tasks) cur = nxt;
  }
  if (!SUMI && nch > 1) {
    __syncthreads();
    for (int rl = tid; rl < nr; rl += kWarps * 32) {
      float s = 0.0f;
      for (int c = 0; c < nch; ++c) s += part_s[rl * nch + c];
      if (in_bounds(ra + rl >= a.r0 && ra + rl < a.r1, a.status)) a.y[ra + rl] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
constexpr int kCtasPerSm = 4;
constexpr size_t kSmemBudget = 200 * 1024;

template <int QT, int U, bool SUMI>
static cudaError_t launch_variant(const LaunchCtx &ctx, MatvecArgs a) {
  auto kern = matvec_m1_kernel<QT, U, SUMI>;
  prefer_max_shared(kern);
  const int n = a.r1 - a.r0;
  const size_t base = static_cast<size_t>(a.nb) * kQK + 8 * static_cast<size_t>(a.nb);
  long long grid = static_cast<long long>(ctx.num_sms) * kCtasPerSm;
  if (grid > n) grid = n;
  size_t smem = base;
  if (!SUMI && a.nchunks > 1) {
    long long rows_max = (n + grid - 1) / grid;
    const long long fit = static_cast<long long>((kSmemBudget - base) / (4 * a.nchunks));
    if (rows_max > fit) {
      grid = (n + fit - 1) / fit;
      rows_max = (n + grid - 1) / grid;
    }
    smem += static_cast<size_t>(rows_max) * a.nchunks * 4;
  }
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kWarps * 32), smem, ctx, a);
}

template <int QT, bool SUMI>
static cudaError_t launch_qt(const LaunchCtx &ctx, MatvecArgs a, int upr) {
  if (upr <= 32) {
    a.nchunks = 1;
    return launch_variant<QT, 1, SUMI>(ctx, a);
  }
  if (upr <= 64) {
    a.nchunks = 1;
    return launch_variant<QT, 2, SUMI>(ctx, a);
  }
  a.nchunks = (upr + 127) / 128;
  return launch_variant<QT, 4, SUMI>(ctx, a);
}

// Kernel choice.  A product y[r0, r1) of at least kPhaseMinBytes of
// weights runs as a one-product decode phase (phase.cu: the CTA's rows whole
// in shared memory; phase_ring.cu: streamed through a ring of bulk-copy
// stages), the kernels the decode phases use, wherever they take the shape
// (K a multiple of 128, at most 16384).  Measured on GB300, back-to-back
// launches with static weights: 4096 x 11008 Q4_0 7.35 us (9.32 us on the
// register kernel), Q8_0 9.73 us (14.11), 151936 x 896 Q8_0 24.3 us (34.1 on
// the ring kernel of matvec_tma.cu).  Smaller products stay on the kernels
// of this file: at 2.6 MB and below they are 0.2-0.4 us faster back to back,
// and chained behind quantize launches the TinyLlama layer's 7.2 MB products
// cost more as phases (the layer's calls step: 34.9 us with its gate, up and
// down as phases, 25.9 us without).  The per-block sums of the test hook,
// and the other shapes, take
// the register-pipelined kernel above for rows of 2048 or more elements or
// the bulk-copy ring kernel for very many short rows.
// MLQ_MATVEC_KERNEL=phase|ldg|tma overrides the choice (A/B timing, tests).
constexpr size_t kPhaseMinBytes = 16u << 20;
static int kernel_override() {
  static const int v = [] {
    const char *e = std::getenv("MLQ_MATVEC_KERNEL");
    if (e == nullptr) return 0;
    if (e[0] == 'l') return 1;
    if (e[0] == 't') return 2;
    if (e[0] == 'p') return 3;
    return 0;
  }();
  return v;
}

static bool prefer_tma(int nb, int rows, int num_sms) {
  const int o = kernel_override();
  if (o == 1 || o == 2) return o == 2;
  return nb <= 32 && rows >= 64 * num_sms;
}

cudaError_t launch_matvec_m1(const LaunchCtx &ctx, int qtype, const void *wq, const float *wd,
                             int nb, const int8_t *xq, const float *xd, float *y, int32_t *sumi,
                             int r0, int r1) {
  if (r1 <= r0) return cudaSuccess;
  const int o = kernel_override();
  const size_t rowq = static_cast<size_t>(nb) * (qtype == 1 ? 16 : 32);
  const size_t wbytes = static_cast<size_t>(r1 - r0) * (rowq + static_cast<size_t>(nb) * 4);
  if (y != nullptr && (o == 3 || (o == 0 && wbytes >= kPhaseMinBytes))) {
    // rows [r0, r1) as a one-product phase on the Q8_0 input
    FusedArgs f = {};
    f.prod[0].wq = static_cast<const uint8_t *>(wq) + static_cast<size_t>(r0) * rowq;
    f.prod[0].wd = wd + static_cast<size_t>(r0) * nb;
    f.prod[0].y = y + r0;
    f.prod[0].rows = r1 - r0;
    f.nproducts = 1;
    f.xq_in = xq;
    f.xd_in = xd;
    f.nb = nb;
    f.total_rows = r1 - r0;
    f.nchunks = 1;
    f.early = ctx.early_weights ? 1 : 0;
    f.status = ctx.status;
    f.wait_ns = ctx.wait_ns;
    diag_note("route=phase");
    const cudaError_t e = launch_phase(ctx, qtype, f);
    if (e != cudaErrorNotSupported) return e;
  }
  diag_note("route=%s", prefer_tma(nb, r1 - r0, ctx.num_sms) ? "ring" : "ldg");
  if (prefer_tma(nb, r1 - r0, ctx.num_sms)) {
    const cudaError_t e = launch_matvec_m1_tma(ctx, qtype, wq, wd, nb, xq, xd, y, sumi, r0, r1);
    if (e != cudaErrorNotSupported) return e;
  }
  MatvecArgs a;
  a.wq = static_cast<const uint8_t *>(wq);
  a.wd = wd;
  a.xq = xq;
  a.xd = xd;
  a.y = y;
  a.sumi = sumi;
  a.nb = nb;
  a.r0 = r0;
  a.r1 = r1;
  a.nchunks = 1;
  a.early = ctx.early_weights ? 1 : 0;
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  const int upr = qtype == 1 ? nb : 2 * nb;
  if (qtype == 1) {
    return sumi ? launch_qt<1, true>(ctx, a, upr) : launch_qt<1, false>(ctx, a, upr);
  }
  return sumi ? launch_qt<0, true>(ctx, a, upr) : launch_qt<0, false>(ctx, a, upr);
}

}  // namespace mlq
