// fused.cu -- one decode "phase" in one launch, streaming variant: quantise
// a float32 vector to Q8_0 and multiply it with one or more weight matrices
// of that width (e.g. Wq|Wk|Wv, or gate|up).  Definitions: page "Legacy-ISA
// ML Inference Runtime -- Design Spec", Sec. 4 (formats, block dot), Sec. 5
// (quantize_q8 rounding, matvec), Sec. 6 "Forward pass" (a quantised
// activation feeds several products).
//
// launch_matvec_fused() (end of file) is the dispatcher of every phase
// launch: the shared-memory phase kernel of phase.cu wherever a CTA's share
// of the weights fits on chip, else the streaming kernel below (float input,
// no quantised outputs), else separate matvec / quantize launches.
//
// The streaming kernel, for chains of dependent launches (PDL):
//  * one CTA of 16 warps per SM, at most 64 registers per thread, so the
//    next phase's CTA fits on the same SM while this one runs;
//  * with static weights the first weight loads of each warp are issued
//    before the wait on the previous kernel; with MLQ_FUSED_L2_PREFETCH=1
//    the CTA also hints its whole weight range into L2 first;
//  * after the wait it quantises x into shared memory (same element
//    arithmetic as quantize.cu: identical bytes), and streams its rows with
//    128-bit evict-first loads, one task = (row, K-chunk of 32*U 16-byte
//    units) per warp, software-pipelined;
//  * block dot: dp4a; Q4_0 -8 folded via sum(qx) per block; Q8_0 halves
//    joined with one shuffle; fixed-order reductions (deterministic).
#include <cstdlib>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

constexpr int kFusedWarps = 16;
constexpr int kFusedThreads = kFusedWarps * 32;

// Q4_0 activation layout in shared memory: block b at b*32, its 16-byte
// halves swapped when bit 2 of b is set, so the eight lanes of a quarter
// warp reading consecutive blocks hit distinct banks.
__device__ __forceinline__ int fused_half_offset(int b, int half) {
  return b * 32 + ((half ^ ((b >> 2) & 1)) << 4);
}

template <int U>
struct FRegs {
  uint4 q[U];
  float d[U];
};

// The product holding concatenated row `g` and the row inside it.
__device__ __forceinline__ int find_product(const FusedArgs &a, int g, int *local) {
  int j = 0;
  int off = 0;
  while (j + 1 < a.nproducts && g >= off + a.prod[j].rows) {
    off += a.prod[j].rows;
    ++j;
  }
  *local = g - off;
  return j;
}

template <int QT, int U>
__device__ __forceinline__ void fused_load(FRegs<U> &r, const FusedArgs &a, int g, int base,
                                           int lane, int upr, uint64_t pol) {
  int lr;
  const int j = find_product(a, g, &lr);
  const size_t rowq = static_cast<size_t>(a.nb) * (QT == 1 ? 16 : 32);
  const uint8_t *qrow = a.prod[j].wq + static_cast<size_t>(lr) * rowq;
  const float *drow = a.prod[j].wd + static_cast<size_t>(lr) * a.nb;
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

template <int QT, int U>
__device__ __forceinline__ float fused_compute(const FRegs<U> &r, const int8_t *xq_s,
                                               const float *xd_s, const int *sx_s, int base,
                                               int lane, int upr) {
  float acc = 0.0f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int unit = base + lane + 32 * u;
    const bool valid = unit < upr;
    if (QT == 1) {
      if (valid) {
        const int4 xa = *reinterpret_cast<const int4 *>(xq_s + fused_half_offset(unit, 0));
        const int4 xb = *reinterpret_cast<const int4 *>(xq_s + fused_half_offset(unit, 1));
        const uint4 w = r.q[u];
        constexpr uint32_t kLo = 0x0F0F0F0Fu;
        int s = __dp4a(static_cast<int>(w.x & kLo), xa.x, 0);
        s = __dp4a(static_cast<int>(w.y & kLo), xa.y, s);
        s = __dp4a(static_cast<int>(w.z & kLo), xa.z, s);
        s = __dp4a(static_cast<int>(w.w & kLo), xa.w, s);
        s = __dp4a(static_cast<int>((w.x >> 4) & kLo), xb.x, s);
        s = __dp4a(static_cast<int>((w.y >> 4) & kLo), xb.y, s);
        s = __dp4a(static_cast<int>((w.z >> 4) & kLo), xb.z, s);
        s = __dp4a(static_cast<int>((w.w >> 4) & kLo), xb.w, s);
        s -= 8 * sx_s[unit];
        acc = __fmaf_rn(__fmul_rn(__int2float_rn(s), r.d[u]), xd_s[unit], acc);
      }
    } else {
      int s = 0;
      if (valid) {
        const int4 xa = *reinterpret_cast<const int4 *>(xq_s + unit * 16);
        const uint4 w = r.q[u];
        s = __dp4a(static_cast<int>(w.x), xa.x, 0);
        s = __dp4a(static_cast<int>(w.y), xa.y, s);
        s = __dp4a(static_cast<int>(w.z), xa.z, s);
        s = __dp4a(static_cast<int>(w.w), xa.w, s);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      if (valid && !(lane & 1)) acc = __fmaf_rn(__fmul_rn(__int2float_rn(s), r.d[u]), xd_s[unit >> 1], acc);
    }
  }
  return acc;
}

// Quantise x (nb blocks of 32 floats) into shared memory, eight lanes per
// block; every thread of the CTA takes part.  All global loads of x are
// issued before any block is reduced (up to kQPass passes of the CTA), so
// the prologue costs one memory round trip, not one per pass.
constexpr int kQPass = 8;

template <int QT>
__device__ __forceinline__ void fused_quantize(const FusedArgs &a, int8_t *xq_s, float *xd_s,
                                               int *sx_s, int tid) {
  const int nb = a.nb;
  const int part = tid & 7;
  const bool writer = blockIdx.x == 0 && a.xq_out != nullptr;
  constexpr int kPer = kFusedThreads / 8;  // blocks per pass
  // Every CTA reads all of x; start each CTA at a different block so that
  // the CTAs do not all request the same L2 lines at the same moment.
  const int rot = static_cast<int>((static_cast<long long>(blockIdx.x) * 37) % nb);
  for (int base0 = 0; base0 < nb; base0 += kPer * kQPass) {
    float4 v[kQPass];
#pragma unroll
    for (int p = 0; p < kQPass; ++p) {
      const int i = base0 + p * kPer + (tid >> 3);
      const int b = i + rot < nb ? i + rot : i + rot - nb;
      v[p] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nb) v[p] = *reinterpret_cast<const float4 *>(a.x + static_cast<size_t>(b) * kQK + part * 4);
    }
#pragma unroll
    for (int p = 0; p < kQPass; ++p) {
      const int i = base0 + p * kPer + (tid >> 3);
      const int b = i + rot < nb ? i + rot : i + rot - nb;
      if (base0 + p * kPer >= nb) break;  // uniform across the CTA
      const bool valid = i < nb;
      uint32_t m = max(max(__float_as_uint(fabsf(v[p].x)), __float_as_uint(fabsf(v[p].y))),
                       max(__float_as_uint(fabsf(v[p].z)), __float_as_uint(fabsf(v[p].w))));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      const float amax = __uint_as_float(m);
      const float dd = amax / 127.0f;
      const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
      const int q0 = quant_one(v[p].x, id), q1 = quant_one(v[p].y, id), q2 = quant_one(v[p].z, id),
                q3 = quant_one(v[p].w, id);
      const uint32_t packed = (q0 & 0xff) | ((q1 & 0xff) << 8) | ((q2 & 0xff) << 16) |
                              (static_cast<uint32_t>(q3 & 0xff) << 24);
      int s4 = q0 + q1 + q2 + q3;
      s4 += __shfl_xor_sync(0xffffffffu, s4, 4);
      s4 += __shfl_xor_sync(0xffffffffu, s4, 2);
      s4 += __shfl_xor_sync(0xffffffffu, s4, 1);
      if (valid) {
        const int off = QT == 1 ? fused_half_offset(b, part >> 2) + (part & 3) * 4 : b * kQK + part * 4;
        *reinterpret_cast<uint32_t *>(xq_s + off) = packed;
        if (part == 0) {
          xd_s[b] = dd;
          sx_s[b] = s4;
        }
        if (writer) {
          *reinterpret_cast<uint32_t *>(a.xq_out + static_cast<size_t>(b) * kQK + part * 4) = packed;
          if (part == 0) a.xd_out[b] = dd;
        }
      }
    }
  }
}

template <int QT, int U>
__global__ void __launch_bounds__(kFusedThreads, 2) matvec_fused_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nb = a.nb;
  const int K = nb * kQK;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + K);
  int *sx_s = reinterpret_cast<int *>(smem + K + 4 * nb);
  float *part_s = reinterpret_cast<float *>(smem + K + 8 * nb);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.total_rows;
  const int ra = static_cast<int>(static_cast<long long>(n) * blockIdx.x / gridDim.x);
  const int rb = static_cast<int>(static_cast<long long>(n) * (blockIdx.x + 1) / gridDim.x);
  const int nr = rb - ra;
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  const int upr = QT == 1 ? nb : 2 * nb;

  if (tid == 0 && nr > 0 && a.prefetch) {  // hint this CTA's whole weight range into L2
    int off = 0;
    for (int j = 0; j < a.nproducts; ++j) {
      const int lo = max(ra, off) - off, hi = min(rb, off + a.prod[j].rows) - off;
      if (hi > lo) {
        prefetch_range_l2(a.prod[j].wq + static_cast<size_t>(lo) * rowq,
                          static_cast<size_t>(hi - lo) * rowq, static_cast<size_t>(1) << 30);
        prefetch_range_l2(a.prod[j].wd + static_cast<size_t>(lo) * nb,
                          static_cast<size_t>(hi - lo) * nb * 4, static_cast<size_t>(1) << 30);
      }
      off += a.prod[j].rows;
    }
  }
  const int nch = a.nchunks;
  const int tasks = nr * nch;
  const uint64_t pol = l2_policy_evict_first();
  int t = warp;
  FRegs<U> cur;
  bool loaded = false;
  if (a.early && t < tasks) {  // weights are static: start streaming before the wait
    const int rl = t / nch;
    fused_load<QT, U>(cur, a, ra + rl, (t - rl * nch) * 32 * U, lane, upr, pol);
    loaded = true;
  }
  griddep_launch_dependents();
  griddep_wait();  // x may be the previous kernel's output

  fused_quantize<QT>(a, xq_s, xd_s, sx_s, tid);
  __syncthreads();

  // ---- products: tasks (row, chunk), software-pipelined per warp ----
  if (!loaded && t < tasks) {
    const int rl = t / nch;
    fused_load<QT, U>(cur, a, ra + rl, (t - rl * nch) * 32 * U, lane, upr, pol);
  }
  for (; t < tasks; t += kFusedWarps) {
    const int rl = t / nch;
    const int c = t - rl * nch;
    const int tn = t + kFusedWarps;
    FRegs<U> nxt;
    if (tn < tasks) {
      const int rln = tn / nch;
      fused_load<QT, U>(nxt, a, ra + rln, (tn - rln * nch) * 32 * U, lane, upr, pol);
    }
    float acc = fused_compute<QT, U>(cur, xq_s, xd_s, sx_s, c * 32 * U, lane, upr);
    acc = warp_sum(acc);
    if (lane == 0) {
      if (nch == 1) {
        int lr;
        const int j = find_product(a, ra + rl, &lr);
        a.prod[j].y[lr] = acc;
      } else {
        part_s[rl * nch + c] = acc;
      }
    }
    if (tn < tasks) cur = nxt;
  }
  if (nch > 1) {
    __syncthreads();
    for (int rl = tid; rl < nr; rl += kFusedThreads) {
      float s = 0.0f;
      for (int c = 0; c < nch; ++c) s += part_s[rl * nch + c];
      int lr;
      const int j = find_product(a, ra + rl, &lr);
      a.prod[j].y[lr] = s;
    }
  }
}

template <int QT, int U>
static cudaError_t launch_fused_variant(const LaunchCtx &ctx, FusedArgs a) {
  auto kern = matvec_fused_kernel<QT, U>;
  prefer_max_shared(kern);
  const int n = a.total_rows;
  const size_t base = static_cast<size_t>(a.nb) * kQK + 8 * static_cast<size_t>(a.nb);
  long long grid = ctx.num_sms;
  if (grid > n) grid = n > 0 ? n : 1;
  size_t smem = base;
  if (a.nchunks > 1 && n > 0) {
    long long rows_max = (n + grid - 1) / grid;
    constexpr size_t kBudget = 96 * 1024;  // two CTAs of this kernel must fit on one SM
    const long long fit = static_cast<long long>((kBudget - base) / (4 * a.nchunks));
    if (rows_max > fit) {
      grid = (n + fit - 1) / fit;
      rows_max = (n + grid - 1) / grid;
    }
    smem += static_cast<size_t>(rows_max) * a.nchunks * 4;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kFusedThreads), smem, ctx, a);
}

template <int QT>
static cudaError_t launch_fused_qt(const LaunchCtx &ctx, FusedArgs a) {
  const int upr = QT == 1 ? a.nb : 2 * a.nb;
  if (upr <= 32) {
    a.nchunks = 1;
    return launch_fused_variant<QT, 1>(ctx, a);
  }
  if (upr <= 64) {
    a.nchunks = 1;
    return launch_fused_variant<QT, 2>(ctx, a);
  }
  a.nchunks = (upr + 127) / 128;
  return launch_fused_variant<QT, 4>(ctx, a);
}

cudaError_t launch_matvec_fused(const LaunchCtx &ctx, int qtype, const FusedArgs &args) {
  FusedArgs a = args;
  long long total = 0;
  for (int j = 0; j < a.nproducts; ++j) total += a.prod[j].rows;
  if (total > 0x7fffffff) return cudaErrorInvalidValue;
  if (total == 0 && a.xq_out == nullptr) return cudaSuccess;  // nothing to do
  a.total_rows = static_cast<int>(total);  // 0: one CTA only quantises x for xq_out
  a.early = (ctx.early_weights || a.early) ? 1 : 0;
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  static const int pf = [] {
    const char *e = std::getenv("MLQ_FUSED_L2_PREFETCH");
    return e != nullptr && e[0] == '1' ? 1 : 0;
  }();
  a.prefetch = pf;
  // MLQ_FUSED_KERNEL=phase|ldg picks the kernel for a float input without
  // quantised outputs or L2 hints (A/B timing); the default is the phase
  // kernel (phase.cu) wherever the CTA slices fit in shared memory.
  static const int mode = [] {
    const char *e = std::getenv("MLQ_FUSED_KERNEL");
    return e != nullptr && e[0] == 'l' ? 1 : 0;
  }();
  const bool plain = a.x != nullptr && !a.any_yq && a.npf == 0;
  if (!plain || mode == 0) {
    const cudaError_t e = launch_phase(ctx, qtype, a);
    if (e != cudaErrorNotSupported) return e;
  }
  // The phase kernel does not take this shape (or the streaming kernel was
  // asked for): the same results from other launches -- the products, then
  // the quantised outputs, then the L2 hints.
  cudaError_t e = cudaSuccess;
  if (a.x != nullptr) {
    e = qtype == 1 ? launch_fused_qt<1>(ctx, a) : launch_fused_qt<0>(ctx, a);
  } else {
    for (int j = 0; j < a.nproducts && e == cudaSuccess; ++j) {
      if (a.prod[j].rows > 0)
        e = launch_matvec_m1(ctx, qtype, a.prod[j].wq, a.prod[j].wd, a.nb, a.xq_in, a.xd_in,
                             a.prod[j].y, nullptr, 0, a.prod[j].rows);
    }
  }
  for (int j = 0; j < a.nproducts && e == cudaSuccess; ++j) {
    if (a.prod[j].yq != nullptr && a.prod[j].rows > 0)
      e = launch_quantize_q8(ctx, a.prod[j].y, a.prod[j].yq, a.prod[j].yd, 1, a.prod[j].rows);
  }
  if (e == cudaSuccess && a.npf > 0) {
    PrefetchList pl;
    pl.n = 0;
    for (int i = 0; i < a.npf && pl.n < kMaxPrefetchRanges; ++i) {
      pl.ptr[pl.n] = a.pf_ptr[i];
      pl.bytes[pl.n++] = a.pf_bytes[i];
    }
    e = launch_prefetch_l2(ctx, pl);
  }
  return e;
}

}  // namespace mlq
