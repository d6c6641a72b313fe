// gemm_ring.cu -- batched small-M decode for M up to 4: the activation rows
// held in registers, the Q4_0 weights streamed through a shared-memory ring.
//
// Computes (page "ONNX Runtime", "6. Panel loop (pre-TCM)": M >= 4 batched
// decode of 4096 x 11008; definitions of the page "Legacy-ISA ML Inference
// Runtime -- Design Spec", Sec. 4):
//   Y[m*ldy + r] = sum_b ((float)sumi(m, r, b) * dw(r, b)) * dx(m, b),
//   sumi(m, r, b) = sum_j (nibble(r, b, j) - 8) * qx(m, 32b + j)  (exact int32).
//
// The M = 1 phase kernels' design with M activation rows.  Per CTA (one per
// SM, its rows an even share of [r0, r1)):
//  * a producer thread copies stages of R whole rows (quants, then scales)
//    with 1-D bulk copies into a ring of up to 216 KB; with static weights it
//    starts before the dependency wait;
//  * consumer warp (chunk c, group g) holds K-chunk c of all M activation
//    rows in registers (one 32-element block per lane; two for M <= 2 when
//    K is above 16384) with
//    their scales and the dp4a start values, and per stage reduces rows g,
//    g + G, g + 2G, g + 3G: per block one 128-bit weight load serves all M
//    rows, the nibbles are masked once, and each (row, m) block sum is exact
//    in int32 (low nibbles with the -8 fold in the start value, high nibbles
//    as 16 n) and turned into float through the exponent bias;
//  * the 4 M partial sums of a stage are added across the warp's lanes by
//    one transposed butterfly, the K-chunks of a row in a fixed order at
//    the end.
// One 128-bit load per block per row, reused M times, keeps the activation
// traffic in registers: the earlier dp4a kernel re-read the M activation
// blocks through L1 for every weight block (128 bytes per 16 weight bytes
// at M = 4) and reached 8 GB/s per SM.
#include "phase_common.cuh"

#include <cstdlib>

namespace mlq {

constexpr int kGrWarps = 16;                    // consumer warps
constexpr int kGrMaxSlots = 8;
constexpr size_t kGrBudget = 216 * 1024;        // dynamic shared memory (one CTA per SM)
constexpr size_t kGrStageCap = 48 * 1024;       // a stage holds at most this many bytes (4 rows at least)

struct GrArgs {
  const uint8_t *wq;
  const float *wd;
  const int8_t *xq;
  const float *xd;
  float *Y;
  int *status;
  unsigned long long wait_ns;
  int ldy;
  int nb;
  int M;
  int r0, r1;
  int C;            // K-chunks (of 32 * NBL blocks)
  int G;            // row groups: C * G consumer warps work, R = 4 G rows per stage
  int ns;           // ring slots
  int stage_bytes;  // bytes of a slot (R rows of quants, then their scales), 128-aligned
  int part;         // offset of the partial sums
  int early;        // weights are not written by earlier queued work: copy before the wait
};

__device__ __forceinline__ bool gr_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
                                        unsigned long long limit_ns) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = sm_cycles(), lim = limit_cycles(limit_ns);
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (sm_cycles() - t0 > lim) return false;
  }
}

__device__ __forceinline__ void gr_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Transposed butterfly: afterwards lane l holds the warp-wide sum of
// v[l / (32 / N)] (v is consumed).  N - 1 + log2(32 / N) shuffles for N sums.
template <int N>
__device__ __forceinline__ float reduce_t(float (&v)[N], int lane) {
  static_assert(N == 8 || N == 16, "8 or 16 values");
#pragma unroll
  for (int lvl = 0; (1 << lvl) < N; ++lvl) {
    const int o = 16 >> lvl, h = N >> (lvl + 1);
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float keep = up ? v[i + h] : v[i];
      const float send = up ? v[i] : v[i + h];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float k = v[0];
#pragma unroll
  for (int o = 16 / N; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
  return k;
}

template <int MM, int NBL>
__global__ void __launch_bounds__((kGrWarps + 1) * 32, 1) gemm_q4_ring_kernel(const GrArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kGrMaxSlots];
  __shared__ __align__(8) uint64_t empty_bar[kGrMaxSlots];
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = a.nb;
  const int n_all = a.r1 - a.r0;
  const int ra = a.r0 + static_cast<int>(static_cast<long long>(n_all) * blockIdx.x / gridDim.x);
  const int rb = a.r0 + static_cast<int>(static_cast<long long>(n_all) * (blockIdx.x + 1) / gridDim.x);
  const int nr = rb - ra;
  const size_t rowq = static_cast<size_t>(nb) * 16;
  const int C = a.C, G = a.G, R = 4 * a.G, ns = a.ns;
  const int active = C * G;
  const size_t dq = static_cast<size_t>(R) * rowq;  // scales after the stage's R rows of quants
  uint8_t *ring = smem;
  float *part_s = reinterpret_cast<float *>(smem + a.part);
  const int nstages = (nr + R - 1) / R;

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), active);  // one arrival per working consumer warp
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The next kernel may be scheduled now (it waits for this grid to
  // complete before it reads anything we write).
  griddep_launch_dependents();

  if (warp == kGrWarps) {
    // ------------------------------ producer ------------------------------
    if (lane != 0 || nr == 0) return;
    if (!a.early) griddep_wait();  // weights written by earlier work: wait for it first
    int s = 0;
    for (; s < nstages; ++s) {
      const int slot = s % ns;
      if (s >= ns && !gr_wait(smem_addr(&empty_bar[slot]), ((s / ns) - 1) & 1, abort_v, a.wait_ns)) {
        if (atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        break;
      }
      if (*abort_v) break;
      const int row0 = ra + s * R, n = min(R, rb - row0);
      const uint32_t qb = static_cast<uint32_t>(n * rowq), db = static_cast<uint32_t>(n) * nb * 4;
      uint8_t *dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
      const uint32_t fb = smem_addr(&full_bar[slot]);
      mbar_arrive_expect_tx(fb, qb + db);
      bulk_copy_g2s(smem_addr(dst), a.wq + static_cast<size_t>(row0) * rowq, qb, fb);
      bulk_copy_g2s(smem_addr(dst + dq), a.wd + static_cast<size_t>(row0) * nb, db, fb);
    }
    if (*abort_v) {  // copies may still be landing: the last ns issued stages (bounded)
      for (int t = s > ns ? s - ns : 0; t < s; ++t)
        mbar_wait_bounded(smem_addr(&full_bar[t % ns]), (t / ns) & 1, kDrainWaitNs);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  griddep_wait();  // the activations may come from the previous kernel
  if (nr == 0) return;
  const bool act = warp < active;
  const int c = warp % C, g = warp / C;
  // lane's blocks u_k = 32 NBL c + lane + 32 k of all M rows, in registers
  int4 xl[NBL][MM], xh[NBL][MM];
  float xs[NBL][MM];
  int adj[NBL][MM];
  bool vk[NBL];
  int uk[NBL];
#pragma unroll
  for (int k = 0; k < NBL; ++k) {
    uk[k] = 32 * NBL * c + lane + 32 * k;
    vk[k] = act && uk[k] < nb;
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      xl[k][m] = xh[k][m] = make_int4(0, 0, 0, 0);
      xs[k][m] = 0.0f;
      adj[k][m] = kMagicBits;
      if (vk[k] && m < a.M) {
        const int4 *src = reinterpret_cast<const int4 *>(a.xq + (static_cast<size_t>(m) * nb + uk[k]) * kQK);
        xl[k][m] = src[0];
        xh[k][m] = src[1];
        xs[k][m] = a.xd[static_cast<size_t>(m) * nb + uk[k]];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < NBL; ++k)
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      constexpr int kOnes = 0x01010101;
      int sx = __dp4a(xl[k][m].x, kOnes, 0);
      sx = __dp4a(xl[k][m].y, kOnes, sx);
      sx = __dp4a(xl[k][m].z, kOnes, sx);
      sx = __dp4a(xl[k][m].w, kOnes, sx);
      sx = __dp4a(xh[k][m].x, kOnes, sx);
      sx = __dp4a(xh[k][m].y, kOnes, sx);
      sx = __dp4a(xh[k][m].z, kOnes, sx);
      sx = __dp4a(xh[k][m].w, kOnes, sx);
      adj[k][m] = kMagicBits - 8 * sx;  // the -8 of every nibble, folded into the start value
    }

  for (int s = 0; s < nstages && act; ++s) {
    const int slot = s % ns;
    const int row0 = s * R, n = min(R, nr - row0);
    if (!warp_wait([&] { return gr_wait(smem_addr(&full_bar[slot]), (s / ns) & 1, abort_v, a.wait_ns); })) {
      if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      break;
    }
    const uint8_t *wq_s = ring + static_cast<size_t>(slot) * a.stage_bytes;
    const float *wd_s = reinterpret_cast<const float *>(wq_s + dq);
    float acc[4 * MM];
#pragma unroll
    for (int i = 0; i < 4 * MM; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = min(g + G * j, n - 1);  // rows past the stage repeat its last row (discarded)
#pragma unroll
      for (int k = 0; k < NBL; ++k) {
        if (!vk[k]) continue;
        const uint4 q = *reinterpret_cast<const uint4 *>(wq_s + static_cast<size_t>(row) * rowq + uk[k] * 16);
        const float dw = wd_s[static_cast<size_t>(row) * nb + uk[k]];
        constexpr uint32_t kLo = 0x0F0F0F0Fu, kHi = 0xF0F0F0F0u;
        const int l0 = static_cast<int>(q.x & kLo), l1 = static_cast<int>(q.y & kLo);
        const int l2 = static_cast<int>(q.z & kLo), l3 = static_cast<int>(q.w & kLo);
        const uint32_t h0 = q.x & kHi, h1 = q.y & kHi, h2 = q.z & kHi, h3 = q.w & kHi;
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          int lo = __dp4a(l0, xl[k][m].x, adj[k][m]);
          int hi = dp4a_us(h0, xh[k][m].x, 0);  // 16 * (high nibble) per byte: exact multiple of 16
          lo = __dp4a(l1, xl[k][m].y, lo);
          hi = dp4a_us(h1, xh[k][m].y, hi);
          lo = __dp4a(l2, xl[k][m].z, lo);
          hi = dp4a_us(h2, xh[k][m].z, hi);
          lo = __dp4a(l3, xl[k][m].w, lo);
          hi = dp4a_us(h3, xh[k][m].w, hi);
          const float sumi = __fsub_rn(__int_as_float(lo + (hi >> 4)), kMagic);
          acc[j * MM + m] = __fmaf_rn(__fmul_rn(sumi, dw), xs[k][m], acc[j * MM + m]);
        }
      }
    }
    const float v = reduce_t<4 * MM>(acc, lane);
    constexpr int kSpan = 32 / (4 * MM);  // lanes holding each sum
    const int idx = lane / kSpan, j = idx / MM, m = idx % MM, row = g + G * j;
    if (lane % kSpan == 0 && row < n && m < a.M) part_s[((row0 + row) * C + c) * MM + m] = v;
    __syncwarp();
    if (lane == 0) gr_arrive(smem_addr(&empty_bar[slot]));
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kGrWarps * 32) : "memory");  // consumers only
  if (*abort_v) return;
  // Y: the K-chunks of each (row, m) added in chunk order
  for (int i = tid; i < nr * a.M; i += kGrWarps * 32) {
    const int row = i / a.M, m = i - row * a.M;
    float sum = 0.0f;
    for (int cc = 0; cc < C; ++cc) sum += part_s[(row * C + cc) * MM + m];
    if (in_bounds(m < a.M && ra + row >= a.r0 && ra + row < a.r1, a.status))
      a.Y[static_cast<size_t>(m) * a.ldy + ra + row] = sum;
  }
}

template <int MM, int NBL>
static cudaError_t launch_ring_mm(const LaunchCtx &ctx, GrArgs a) {
  const int chunk = 32 * NBL;
  a.C = (a.nb + chunk - 1) / chunk;
  if (a.C > kGrWarps || a.nb % 4 != 0) return cudaErrorNotSupported;
  const size_t rowq = static_cast<size_t>(a.nb) * 16, rowb = rowq + static_cast<size_t>(a.nb) * 4;
  // row groups: every warp busy, stages of at most kGrStageCap bytes
  int G = kGrWarps / a.C;
  const int g_cap = static_cast<int>(kGrStageCap / (4 * rowb));
  G = G < g_cap ? G : (g_cap > 0 ? g_cap : 1);
  a.G = G;
  const int R = 4 * G;
  const int n = a.r1 - a.r0;
  const int grid = ctx.num_sms < n ? ctx.num_sms : n;
  const int rows_max = (n + grid - 1) / grid;
  const size_t stage = (static_cast<size_t>(R) * rowb + 127) / 128 * 128;
  const size_t part = (static_cast<size_t>(rows_max) * a.C * MM * 4 + 127) / 128 * 128;
  if (stage + part > kGrBudget) return cudaErrorNotSupported;
  int ns = static_cast<int>((kGrBudget - part) / stage);
  const int nstages_max = (rows_max + R - 1) / R;
  ns = ns < kGrMaxSlots ? ns : kGrMaxSlots;
  ns = ns < nstages_max ? ns : nstages_max;
  a.ns = ns;
  a.stage_bytes = static_cast<int>(stage);
  a.part = static_cast<int>(static_cast<size_t>(ns) * stage);
  const size_t smem = static_cast<size_t>(ns) * stage + part;
  diag_note("ring: M=%d rows/CTA<=%d chunks=%d rows/stage=%d slots=%d stage=%zuB", a.M, rows_max, a.C, R, ns,
            stage);
  auto kern = gemm_q4_ring_kernel<MM, NBL>;
  static const cudaError_t attr = [&] {
    prefer_max_shared(kern);
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kGrBudget));
  }();
  if (attr != cudaSuccess) return attr;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3((kGrWarps + 1) * 32), smem, ctx, a);
}

cudaError_t launch_gemm_q4_ring(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                                const int8_t *xq, const float *xd, int M, float *Y, int ldy, int r0,
                                int r1) {
  if (r1 <= r0 || M <= 0) return cudaSuccess;
  if (M > 4) return cudaErrorNotSupported;
  GrArgs a;
  a.wq = static_cast<const uint8_t *>(wq);
  a.wd = wd;
  a.xq = xq;
  a.xd = xd;
  a.Y = Y;
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  a.ldy = ldy;
  a.nb = nb;
  a.M = M;
  a.r0 = r0;
  a.r1 = r1;
  a.early = ctx.early_weights ? 1 : 0;
  // one block per lane keeps the most warps busy; two per lane only where
  // K needs more than 16 chunks of 32 blocks (M <= 2)
  if (M <= 2) return (nb + 31) / 32 <= kGrWarps ? launch_ring_mm<2, 1>(ctx, a) : launch_ring_mm<2, 2>(ctx, a);
  return launch_ring_mm<4, 1>(ctx, a);
}

}  // namespace mlq
