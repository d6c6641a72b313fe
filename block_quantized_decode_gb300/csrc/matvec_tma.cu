// matvec_tma.cu -- M = 1 block-quantized matrix-vector product, bulk-copy
// (TMA) ring version for sm_103a.
//
// Same result as matvec.cu (page "Legacy-ISA ML Inference Runtime -- Design
// Spec", Sec. 4 "Integer dot per block", Sec. 5 matvec_q4 / matvec_q8):
//   y[r] = sum_b ((float)sumi(r, b) * dw(r, b)) * dx(b),  r in [r0, r1).
//
// Why a second kernel: the weight stream is the whole cost, and a warp that
// keeps its loads in registers can only hold a few KB in flight, so one
// round trip per task serialises.  Here one CTA per SM owns a contiguous,
// balanced range of rows; a producer warp streams that range (q bytes and
// d scales, both contiguous) into a ring of shared-memory stages with 1-D
// bulk copies (cp.async.bulk, completion on an mbarrier per stage), so
// up to ~200 KB per SM are in flight from the first microsecond.  Consumer
// warps own a fixed K-slice of every row: each lane keeps the activation
// blocks of its slice in registers for the whole kernel (loaded once from
// the shared-memory copy of x), reads weight blocks from the stage with
// conflict-free 16-byte shared loads, and releases the stage to the
// producer through a second mbarrier.  Block dot as in matvec.cu: dp4a;
// Q4_0 -8 fold via the per-block sum of qx; Q8_0 half blocks combined with
// one shuffle before the int32 -> float conversion.  Rows whose K-slices are
// spread over several warps are summed in a fixed order through shared
// memory: deterministic, no atomics.
//
// Requirements (else the launcher declines and matvec.cu runs): cols a
// multiple of 128 (so every stage's scale range is 16-byte aligned), one row
// fits a stage, and x fits next to the ring.  Every wait is bounded; on a
// give-up the CTA records MLQ_E_TIMEOUT, stops issuing, waits (bounded) for
// its own copies in flight and returns.
#include <cstdlib>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

struct TmaArgs {
  const uint8_t *wq;
  const float *wd;
  const int8_t *xq;
  const float *xd;
  float *y;
  int32_t *sumi;
  int nb;
  int r0, r1;
  int rs;     // rows per stage
  int ns;     // ring slots
  int pre;    // rows to hint into L2 before the dependency wait
  int S;      // consumer warps per row (K-slices)
  int G;      // row groups (consumer warps = S * G)
  int *status;
  unsigned long long wait_ns;
};

constexpr int kMaxSlots = 8;
constexpr int kMaxConsumerWarps = 16;
constexpr size_t kTmaSmemBudget = 220 * 1024;
constexpr size_t kStageTarget = 48 * 1024;

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait that also gives up when another warp of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              const volatile int *abort_flag,
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

template <int BL>
struct XRegs {
  int4 lo[BL];   // Q4_0: qx elements 0..15 of the block; Q8_0: the unit's 16 qx
  int4 hi[BL];   // Q4_0: qx elements 16..31 (unused for Q8_0)
  float dx[BL];
  int sx[BL];    // Q4_0: sum of the block's 32 qx (the -8 fold)
};

template <int QT, int BL, bool SUMI>
__global__ void __launch_bounds__((kMaxConsumerWarps + 1) * 32, 1)
    matvec_tma_kernel(const TmaArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxSlots];
  __shared__ __align__(8) uint64_t empty_bar[kMaxSlots];
  __shared__ __align__(8) uint64_t x_bar;
  __shared__ int abort_flag;

  const int nb = a.nb;
  const int K = nb * kQK;
  const int upr = QT == 1 ? nb : 2 * nb;  // 16-byte units per row
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  const int NC = a.S * a.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int n = a.r1 - a.r0;
  const int ra = a.r0 + static_cast<int>(static_cast<long long>(n) * blockIdx.x / gridDim.x);
  const int rb =
      a.r0 + static_cast<int>(static_cast<long long>(n) * (blockIdx.x + 1) / gridDim.x);
  const int nr = rb - ra;
  const int nstages = (nr + a.rs - 1) / a.rs;

  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + K);
  const size_t xbytes = align_up(static_cast<size_t>(K) + 4 * nb, 128);
  const size_t stage_q = static_cast<size_t>(a.rs) * rowq;
  const size_t stage_bytes = align_up(stage_q + static_cast<size_t>(a.rs) * nb * 4, 128);
  uint8_t *stages = smem + xbytes;
  float *part_s = reinterpret_cast<float *>(stages + a.ns * stage_bytes);
  volatile int *abort_v = &abort_flag;

  if (tid == 0) {
    if (nr > 0) {  // L2 hint for the first ring's worth: safe before the dependency wait
      const size_t pre = static_cast<size_t>(a.pre);
      const size_t rows_pre = pre < static_cast<size_t>(nr) ? pre : static_cast<size_t>(nr);
      prefetch_range_l2(a.wq + static_cast<size_t>(ra) * rowq, rows_pre * rowq, 1u << 30);
      prefetch_range_l2(a.wd + static_cast<size_t>(ra) * nb, rows_pre * nb * 4, 1u << 30);
    }
    for (int s = 0; s < a.ns; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), static_cast<uint32_t>(NC));
    }
    mbar_init(smem_addr(&x_bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  griddep_wait();  // x (and anything else we read) may come from the previous kernel
  griddep_launch_dependents();
  __syncthreads();

  int issued = 0;  // producer lane only
  if (warp == NC) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      const uint32_t xb = smem_addr(&x_bar);
      mbar_arrive_expect_tx(xb, static_cast<uint32_t>(K + 4 * nb));
      bulk_copy_g2s(smem_addr(xq_s), a.xq, static_cast<uint32_t>(K), xb);
      bulk_copy_g2s(smem_addr(xd_s), a.xd, static_cast<uint32_t>(4 * nb), xb);
      for (int st = 0; st < nstages; ++st) {
        const int slot = st % a.ns;
        if (st >= a.ns &&
            !wait_or_abort(smem_addr(&empty_bar[slot]), ((st / a.ns) - 1) & 1, abort_v, a.wait_ns)) {
          if (!*abort_v) set_status(a.status, kStatusTimeout);
          *abort_v = 1;
          break;
        }
        const int row0 = ra + st * a.rs;
        const int rows = min(a.rs, rb - row0);
        const uint32_t qb = static_cast<uint32_t>(rows * rowq);
        const uint32_t db = static_cast<uint32_t>(rows * nb * 4);
        uint8_t *dst = stages + slot * stage_bytes;
        const uint32_t fb = smem_addr(&full_bar[slot]);
        mbar_arrive_expect_tx(fb, qb + db);
        bulk_copy_g2s(smem_addr(dst), a.wq + static_cast<size_t>(row0) * rowq, qb, fb);
        bulk_copy_g2s(smem_addr(dst + stage_q), a.wd + static_cast<size_t>(row0) * nb, db, fb);
        issued = st + 1;
      }
    }
  } else if (warp < NC) {
    // ------------------------------ consumers ------------------------------
    const int g = warp / a.S;
    const int s = warp - g * a.S;
    bool ok = warp_wait([&] { return wait_or_abort(smem_addr(&x_bar), 0, abort_v, a.wait_ns); });
    XRegs<BL> xr;
    int unit[BL];
#pragma unroll
    for (int j = 0; j < BL; ++j) {
      unit[j] = s * 32 * BL + lane + 32 * j;
      xr.lo[j] = make_int4(0, 0, 0, 0);
      xr.hi[j] = make_int4(0, 0, 0, 0);
      xr.dx[j] = 0.0f;
      xr.sx[j] = 0;
      if (ok && unit[j] < upr) {
        if (QT == 1) {
          xr.lo[j] = *reinterpret_cast<const int4 *>(xq_s + unit[j] * 32);
          xr.hi[j] = *reinterpret_cast<const int4 *>(xq_s + unit[j] * 32 + 16);
          xr.dx[j] = xd_s[unit[j]];
          int t = __dp4a(xr.lo[j].x, 0x01010101, 0);
          t = __dp4a(xr.lo[j].y, 0x01010101, t);
          t = __dp4a(xr.lo[j].z, 0x01010101, t);
          t = __dp4a(xr.lo[j].w, 0x01010101, t);
          t = __dp4a(xr.hi[j].x, 0x01010101, t);
          t = __dp4a(xr.hi[j].y, 0x01010101, t);
          t = __dp4a(xr.hi[j].z, 0x01010101, t);
          t = __dp4a(xr.hi[j].w, 0x01010101, t);
          xr.sx[j] = t;
        } else {
          xr.lo[j] = *reinterpret_cast<const int4 *>(xq_s + unit[j] * 16);
          xr.dx[j] = xd_s[unit[j] >> 1];
        }
      }
    }
    if (!ok) {
      if (!*abort_v) set_status(a.status, kStatusTimeout);
      *abort_v = 1;
    }
    for (int st = 0; ok && st < nstages; ++st) {
      const int slot = st % a.ns;
      if (!warp_wait([&] { return wait_or_abort(smem_addr(&full_bar[slot]), (st / a.ns) & 1, abort_v,
                                                a.wait_ns); })) {
        if (!*abort_v) set_status(a.status, kStatusTimeout);
        *abort_v = 1;
        break;
      }
      const uint8_t *sq = stages + slot * stage_bytes;
      const float *sd = reinterpret_cast<const float *>(sq + stage_q);
      const int rows = min(a.rs, nr - st * a.rs);
      for (int i = g; i < rows; i += a.G) {
        const int row = ra + st * a.rs + i;
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < BL; ++j) {
          const bool valid = unit[j] < upr;
          if (QT == 1) {
            if (valid) {
              const uint4 w = *reinterpret_cast<const uint4 *>(sq + i * rowq + unit[j] * 16);
              const float dw = sd[i * nb + unit[j]];
              constexpr uint32_t kLo = 0x0F0F0F0Fu;
              int sm = __dp4a(static_cast<int>(w.x & kLo), xr.lo[j].x, 0);
              sm = __dp4a(static_cast<int>(w.y & kLo), xr.lo[j].y, sm);
              sm = __dp4a(static_cast<int>(w.z & kLo), xr.lo[j].z, sm);
              sm = __dp4a(static_cast<int>(w.w & kLo), xr.lo[j].w, sm);
              sm = __dp4a(static_cast<int>((w.x >> 4) & kLo), xr.hi[j].x, sm);
              sm = __dp4a(static_cast<int>((w.y >> 4) & kLo), xr.hi[j].y, sm);
              sm = __dp4a(static_cast<int>((w.z >> 4) & kLo), xr.hi[j].z, sm);
              sm = __dp4a(static_cast<int>((w.w >> 4) & kLo), xr.hi[j].w, sm);
              sm -= 8 * xr.sx[j];
              if (SUMI) {
                a.sumi[static_cast<size_t>(row - a.r0) * nb + unit[j]] = sm;
              } else {
                acc = __fmaf_rn(__fmul_rn(__int2float_rn(sm), dw), xr.dx[j], acc);
              }
            }
          } else {
            int sm = 0;
            float dw = 0.0f;
            if (valid) {
              const uint4 w = *reinterpret_cast<const uint4 *>(sq + i * rowq + unit[j] * 16);
              dw = sd[i * nb + (unit[j] >> 1)];
              sm = __dp4a(static_cast<int>(w.x), xr.lo[j].x, 0);
              sm = __dp4a(static_cast<int>(w.y), xr.lo[j].y, sm);
              sm = __dp4a(static_cast<int>(w.z), xr.lo[j].z, sm);
              sm = __dp4a(static_cast<int>(w.w), xr.lo[j].w, sm);
            }
            sm += __shfl_xor_sync(0xffffffffu, sm, 1);  // the block's other half
            if (valid && !(lane & 1)) {
              if (SUMI) {
                a.sumi[static_cast<size_t>(row - a.r0) * nb + (unit[j] >> 1)] = sm;
              } else {
                acc = __fmaf_rn(__fmul_rn(__int2float_rn(sm), dw), xr.dx[j], acc);
              }
            }
          }
        }
        if (!SUMI) {
          acc = warp_sum(acc);
          if (lane == 0) {
            if (a.S == 1) {
              a.y[row] = acc;
            } else {
              part_s[(row - ra) * a.S + s] = acc;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[slot]));
    }
  }

  __syncthreads();
  if (!SUMI && a.S > 1 && !*abort_v) {
    for (int rl = tid; rl < nr; rl += blockDim.x) {
      float sum = 0.0f;
      for (int q = 0; q < a.S; ++q) sum += part_s[rl * a.S + q];
      a.y[ra + rl] = sum;
    }
  }
  if (warp == NC && lane == 0 && *abort_v) {
    // Copies this CTA issued may still be landing in its shared memory:
    // wait (bounded) for the last use of every slot before exiting.
    for (int slot = 0; slot < a.ns && slot < issued; ++slot) {
      const int last = slot + ((issued - 1 - slot) / a.ns) * a.ns;
      mbar_wait_bounded(smem_addr(&full_bar[slot]), (last / a.ns) & 1, kDrainWaitNs);
    }
    mbar_wait_bounded(smem_addr(&x_bar), 0, kDrainWaitNs);
  }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
static size_t env_size(const char *name, size_t dflt) {
  const char *e = std::getenv(name);
  if (e == nullptr || *e == 0) return dflt;
  return static_cast<size_t>(std::strtoull(e, nullptr, 10));
}

template <int QT, int BL, bool SUMI>
static cudaError_t launch_tma_variant(const LaunchCtx &ctx, const TmaArgs &a, int grid,
                                      size_t smem) {
  auto kern = matvec_tma_kernel<QT, BL, SUMI>;
  prefer_max_shared(kern);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)),
                       dim3(static_cast<unsigned>((a.S * a.G + 1) * 32)), smem, ctx, a);
}

// Returns cudaErrorNotSupported (without launching) when the shape does not
// suit this kernel.
cudaError_t launch_matvec_m1_tma(const LaunchCtx &ctx, int qtype, const void *wq, const float *wd,
                                 int nb, const int8_t *xq, const float *xd, float *y,
                                 int32_t *sumi, int r0, int r1) {
  if (nb % 4 != 0) return cudaErrorNotSupported;
  const int n = r1 - r0;
  if (n <= 0) return cudaSuccess;
  const int upr = qtype == 1 ? nb : 2 * nb;
  const size_t rowq = static_cast<size_t>(nb) * (qtype == 1 ? 16 : 32);
  const size_t rowbytes = rowq + static_cast<size_t>(nb) * 4;
  const int BL = upr <= 32 ? 1 : (upr <= 512 ? 2 : 4);
  const int S = (upr + 32 * BL - 1) / (32 * BL);
  if (S > kMaxConsumerWarps) return cudaErrorNotSupported;
  int G = kMaxConsumerWarps / S;
  const size_t xbytes = align_up(static_cast<size_t>(nb) * kQK + 4 * static_cast<size_t>(nb), 128);

  long long grid = ctx.num_sms;
  if (grid > n) grid = n;
  long long rows_cta = (n + grid - 1) / grid;
  size_t part = (S > 1 && sumi == nullptr) ? align_up(static_cast<size_t>(rows_cta) * S * 4, 128) : 0;
  if (part > 48 * 1024) {  // very many rows: use more, smaller CTAs
    grid = (static_cast<long long>(n) * S * 4 + 48 * 1024 - 1) / (48 * 1024);
    rows_cta = (n + grid - 1) / grid;
    part = align_up(static_cast<size_t>(rows_cta) * S * 4, 128);
  }
  static const size_t stage_target = env_size("MLQ_TMA_STAGE_KB", kStageTarget / 1024) * 1024;
  // ring slots: at most kMaxSlots (the barrier arrays' size), at least 2
  static const int max_slots = [] {
    const size_t v = env_size("MLQ_TMA_SLOTS", 4);
    return static_cast<int>(v < 2 ? 2 : (v > static_cast<size_t>(kMaxSlots) ? kMaxSlots : v));
  }();
  static const int pre_stages = static_cast<int>(env_size("MLQ_TMA_PREFETCH_STAGES", 8));
  int rs = static_cast<int>(stage_target / rowbytes);
  if (rs < 1) rs = 1;
  if (rs > rows_cta) rs = static_cast<int>(rows_cta);
  if (G > rs) G = rs;               // no row group without a row in a stage
  rs = rs / G * G;
  const size_t stage_bytes = align_up(static_cast<size_t>(rs) * rowbytes, 128);
  if (xbytes + part + 2 * stage_bytes > kTmaSmemBudget) return cudaErrorNotSupported;
  int ns = static_cast<int>((kTmaSmemBudget - xbytes - part) / stage_bytes);
  if (ns > max_slots) ns = max_slots;
  const long long stages_cta = (rows_cta + rs - 1) / rs;
  if (ns > stages_cta) ns = static_cast<int>(stages_cta < 2 ? 2 : stages_cta);
  const size_t smem = xbytes + ns * stage_bytes + part;

  TmaArgs a;
  a.wq = static_cast<const uint8_t *>(wq);
  a.wd = wd;
  a.xq = xq;
  a.xd = xd;
  a.y = y;
  a.sumi = sumi;
  a.nb = nb;
  a.r0 = r0;
  a.r1 = r1;
  a.rs = rs;
  a.ns = ns;
  a.pre = rs * pre_stages;
  a.S = S;
  a.G = G;
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  const int g = static_cast<int>(grid);
  const bool s = sumi != nullptr;
  if (qtype == 1) {
    if (BL == 1) return s ? launch_tma_variant<1, 1, true>(ctx, a, g, smem) : launch_tma_variant<1, 1, false>(ctx, a, g, smem);
    if (BL == 2) return s ? launch_tma_variant<1, 2, true>(ctx, a, g, smem) : launch_tma_variant<1, 2, false>(ctx, a, g, smem);
    return s ? launch_tma_variant<1, 4, true>(ctx, a, g, smem) : launch_tma_variant<1, 4, false>(ctx, a, g, smem);
  }
  if (BL == 1) return s ? launch_tma_variant<0, 1, true>(ctx, a, g, smem) : launch_tma_variant<0, 1, false>(ctx, a, g, smem);
  if (BL == 2) return s ? launch_tma_variant<0, 2, true>(ctx, a, g, smem) : launch_tma_variant<0, 2, false>(ctx, a, g, smem);
  return s ? launch_tma_variant<0, 4, true>(ctx, a, g, smem) : launch_tma_variant<0, 4, false>(ctx, a, g, smem);
}

}  // namespace mlq
