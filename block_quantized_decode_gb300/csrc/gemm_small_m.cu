// gemm_small_m.cu -- batched small-M decode: M (1..16) Q8_0 activation rows
// against one Q4_0 weight matrix (page "ONNX Runtime", section "6. Panel
// loop (pre-TCM)": M >= 4 batched decode of 4096 x 11008; definitions of
// the page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 4):
//   Y[m*ldy + r] = sum_b ((float)sumi(m, r, b) * dw(r, b)) * dx(m, b),
//   sumi(m, r, b) = sum_j (nibble - 8) * qx(m, 32b + j)  (exact int32).
//
// dp4a design: a warp task is one weight row x one K-chunk; each lane holds
// one 16-byte Q4_0 block of the row (one 128-bit streaming load) and reuses
// it for all M activation rows, so the weight bytes are read from HBM once
// for the whole batch.  The nibbles are placed in the high half of each
// byte and offset by 0x80, which makes every byte the signed value
// 16*(nibble - 8); dp4a against int8 activations then yields 16*sumi
// exactly (|16*sumi| <= 16*32*8*127 < 2^31) and an arithmetic shift
// recovers sumi with no per-block correction term.  Activation blocks are
// read through L1 (they are shared by every warp of the SM).
#include <cstdlib>
#include <cstring>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

struct GemmArgs {
  const uint8_t *wq;
  const float *wd;
  const int8_t *xq;
  const float *xd;
  float *Y;
  int ldy;
  int nb;
  int M;
  int r0, r1;
  int nchunks;
};

constexpr int kGemmWarps = 8;

__device__ __forceinline__ int4 ld_nc_v4i(const void *p) {
  int4 v;
  asm("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

template <int MM, int U>
__global__ void __launch_bounds__(kGemmWarps * 32) gemm_q4_small_m_dp4a_kernel(const GemmArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float *part_s = reinterpret_cast<float *>(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = a.nb;
  const int K = nb * kQK;
  const int n = a.r1 - a.r0;
  const int ra = a.r0 + static_cast<int>(static_cast<long long>(n) * blockIdx.x / gridDim.x);
  const int rb =
      a.r0 + static_cast<int>(static_cast<long long>(n) * (blockIdx.x + 1) / gridDim.x);
  const int nr = rb - ra;
  const size_t rowq = static_cast<size_t>(nb) * 16;
  if (tid == 0 && nr > 0) {
    prefetch_range_l2(a.wq + static_cast<size_t>(ra) * rowq, static_cast<size_t>(nr) * rowq,
                      64 * 1024);
  }
  griddep_wait();
  griddep_launch_dependents();

  const int nch = a.nchunks;
  const int tasks = nr * nch;
  const uint64_t pol = l2_policy_evict_first();
  for (int t = warp; t < tasks; t += kGemmWarps) {
    const int rl = t / nch;
    const int c = t - rl * nch;
    const int row = ra + rl;
    const uint8_t *qrow = a.wq + static_cast<size_t>(row) * rowq;
    const float *drow = a.wd + static_cast<size_t>(row) * nb;
    uint4 w[U];
    float dw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = c * 32 * U + lane + 32 * u;
      if (b < nb) {
        w[u] = ld_stream_v4(qrow + static_cast<size_t>(b) * 16, pol);
        dw[u] = ld_stream_f32(drow + b, pol);
      } else {
        w[u] = make_uint4(0u, 0u, 0u, 0u);
        dw[u] = 0.0f;
      }
    }
    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = c * 32 * U + lane + 32 * u;
      if (b < nb) {
        constexpr uint32_t kHi = 0xF0F0F0F0u, kBias = 0x80808080u;
        const int l0 = static_cast<int>(((w[u].x << 4) & kHi) ^ kBias);
        const int l1 = static_cast<int>(((w[u].y << 4) & kHi) ^ kBias);
        const int l2 = static_cast<int>(((w[u].z << 4) & kHi) ^ kBias);
        const int l3 = static_cast<int>(((w[u].w << 4) & kHi) ^ kBias);
        const int h0 = static_cast<int>((w[u].x & kHi) ^ kBias);
        const int h1 = static_cast<int>((w[u].y & kHi) ^ kBias);
        const int h2 = static_cast<int>((w[u].z & kHi) ^ kBias);
        const int h3 = static_cast<int>((w[u].w & kHi) ^ kBias);
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          if (m < a.M) {
            const int8_t *xb = a.xq + static_cast<size_t>(m) * K + static_cast<size_t>(b) * kQK;
            const int4 xa = ld_nc_v4i(xb);
            const int4 xc = ld_nc_v4i(xb + 16);
            int s = __dp4a(l0, xa.x, 0);
            s = __dp4a(l1, xa.y, s);
            s = __dp4a(l2, xa.z, s);
            s = __dp4a(l3, xa.w, s);
            s = __dp4a(h0, xc.x, s);
            s = __dp4a(h1, xc.y, s);
            s = __dp4a(h2, xc.z, s);
            s = __dp4a(h3, xc.w, s);
            const int sumi = s >> 4;  // exact: s is 16 * sumi
            const float dx = __ldg(a.xd + static_cast<size_t>(m) * nb + b);
            acc[m] = __fmaf_rn(__fmul_rn(__int2float_rn(sumi), dw[u]), dx, acc[m]);
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      if (m < a.M) {
        const float v = warp_sum(acc[m]);
        if (lane == 0) {
          if (nch == 1) {
            a.Y[static_cast<size_t>(m) * a.ldy + row] = v;
          } else {
            part_s[(rl * nch + c) * MM + m] = v;
          }
        }
      }
    }
  }
  if (nch > 1) {
    __syncthreads();
    for (int i = tid; i < nr * a.M; i += kGemmWarps * 32) {
      const int rl = i / a.M, m = i - rl * a.M;
      float s = 0.0f;
      for (int c = 0; c < nch; ++c) s += part_s[(rl * nch + c) * MM + m];
      a.Y[static_cast<size_t>(m) * a.ldy + ra + rl] = s;
    }
  }
}

template <int MM, int U>
static cudaError_t launch_gemm_variant(const LaunchCtx &ctx, GemmArgs a) {
  auto kern = gemm_q4_small_m_dp4a_kernel<MM, U>;
  const int n = a.r1 - a.r0;
  long long grid = static_cast<long long>(ctx.num_sms) * 4;
  if (grid > n) grid = n;
  size_t smem = 0;
  if (a.nchunks > 1) {
    long long rows_max = (n + grid - 1) / grid;
    const long long fit = static_cast<long long>((160 * 1024) / (4 * a.nchunks * MM));
    if (rows_max > fit) {
      grid = (n + fit - 1) / fit;
      rows_max = (n + grid - 1) / grid;
    }
    smem = static_cast<size_t>(rows_max) * a.nchunks * MM * 4;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kGemmWarps * 32), smem, ctx,
                       a);
}

template <int MM>
static cudaError_t launch_gemm_mm(const LaunchCtx &ctx, GemmArgs a) {
  if (a.nb <= 32) {
    a.nchunks = 1;
    return launch_gemm_variant<MM, 1>(ctx, a);
  }
  if (a.nb <= 64) {
    a.nchunks = 1;
    return launch_gemm_variant<MM, 2>(ctx, a);
  }
  a.nchunks = (a.nb + 127) / 128;
  return launch_gemm_variant<MM, 4>(ctx, a);
}

// Kernel choice, measured on GB300 (11008 x 4096 and 4096 x 11008 Q4_0):
// the tensor-core kernels win from M = 8 on, this dp4a kernel below at
// small M (M = 2: 11 us vs 19-24 us).  Of the tensor-core kernels the
// cluster kernel (gemm_mma_cluster.cu) is the default; the register-load
// kernel (gemm_mma.cu) serves the shapes it does not take (K above 16384).
// The tcgen05 kernel (gemm_umma.cu) is exact and tested but slower on these
// shapes (28-34 us at M = 16): each of its N = 16 MMAs costs the full
// instruction latency.
// Below M = 8 the ring kernel (gemm_ring.cu: activations in registers,
// whole weight rows through a shared-memory ring) comes first for M <= 4.
// At M = 6 and 7 the cluster kernel comes first too: its time stays flat in
// M while this kernel's grows by about 3 us a row (per product, back to
// back: 11008 x 4096 / 4096 x 11008 at M = 7 20.3 / 22.1 us against
// 26.8 / 26.0, at M = 6 20.1 / 22.2 against 24.0 / 22.9; at M = 5 20.3 /
// 22.4 against 20.8 / 20.1, where this kernel stays).  This dp4a kernel
// takes M = 5 and the shapes the others decline.
// MLQ_GEMM_KERNEL=dp4a|mma|mma_ldg|umma|ring overrides (A/B timing, tests).
static int gemm_override() {
  static const int v = [] {
    const char *e = std::getenv("MLQ_GEMM_KERNEL");
    if (e == nullptr) return 0;
    if (std::strcmp(e, "dp4a") == 0) return 1;
    if (std::strcmp(e, "mma") == 0) return 2;
    if (std::strcmp(e, "mma_ldg") == 0) return 3;
    if (std::strcmp(e, "umma") == 0) return 4;
    if (std::strcmp(e, "ring") == 0) return 5;
    return 0;
  }();
  return v;
}

cudaError_t launch_gemm_q4_small_m(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                                   const int8_t *xq, const float *xd, int M, float *Y, int ldy,
                                   int r0, int r1,
                                   int rows) {
  if (r1 <= r0 || M <= 0) return cudaSuccess;
  const int o = gemm_override();
  if (o == 3) return launch_gemm_q4_mma(ctx, wq, wd, nb, xq, xd, M, Y, ldy, r0, r1);
  if (o == 4) {
    const cudaError_t e = launch_gemm_q4_umma(ctx, wq, wd, nb, xq, xd, M, Y, ldy, r0, r1, rows);
    if (e != cudaErrorNotSupported) return e;
    return launch_gemm_q4_mma(ctx, wq, wd, nb, xq, xd, M, Y, ldy, r0, r1);
  }
  constexpr int kClusterMinM = 6;  // the cluster kernel from this M on (above)
  if (o == 2 || (o == 0 && M >= kClusterMinM)) {
    const cudaError_t e = launch_gemm_q4_mma_cluster(ctx, wq, wd, nb, xq, xd, M, Y, ldy, r0, r1, rows);
    if (e != cudaErrorNotSupported) return e;
    if (o == 2 || M >= 8) return launch_gemm_q4_mma(ctx, wq, wd, nb, xq, xd, M, Y, ldy, r0, r1);
  }
  if ((o == 0 || o == 5) && M <= 4) {
    const cudaError_t e = launch_gemm_q4_ring(ctx, wq, wd, nb, xq, xd, M, Y, ldy, r0, r1);
    if (e != cudaErrorNotSupported) return e;
  }
  GemmArgs a;
  a.wq = static_cast<const uint8_t *>(wq);
  a.wd = wd;
  a.xq = xq;
  a.xd = xd;
  a.Y = Y;
  a.ldy = ldy;
  a.nb = nb;
  a.M = M;
  a.r0 = r0;
  a.r1 = r1;
  a.nchunks = 1;
  if (M <= 4) return launch_gemm_mm<4>(ctx, a);
  if (M <= 8) return launch_gemm_mm<8>(ctx, a);
  return launch_gemm_mm<16>(ctx, a);
}

}  // namespace mlq
