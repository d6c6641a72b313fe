// q4k.cu -- Q4_K-style super-block weights: the per-256 activation
// quantiser and the M = 1 product with the sub-block scales folded in the
// integer domain.
//
// Definitions: page "SKaiNET-native-kernels", section "Proving an
// optimization is safe before writing it": 4-bit weight nibbles n in
// [0, 15], 32 elements per sub-block, 6-bit sub-block scales s_b, 8
// sub-blocks per block, int8 activations, and per-32 asymmetric minima m_b.
// Because |sum_b s_b sum_i a_i n_i| <= 8*63*32*127*15 = 3.07e7 < 2^31, the
// scaled sub-block sums are added in int32 and converted to float once per
// 256-element super-block.  Layout (rows row-major): q = 16 nibble bytes
// per sub-block in the Q4_0 order (byte j: element j low, j + 16 high);
// s = 16 bytes per super-block, the 8 scales then the 8 minima; d, dmin =
// float32 per super-block.  Element value d*s_b*n - dmin*m_b.  Activations:
// Q8_0 rounding with one scale per 256 and int32 sums per 32.  For each
// super-block B of row r (the same float operations, in the same order, as
// the plain definition):
//   ISUM = sum_b s_b * sum_i a_i n_i,   MSUM = sum_b m_b * bsum_b,
//   y[r] += ((float)ISUM * d - (float)MSUM * dmin) * dx_B.
// (Even 8-bit scales and minima stay inside int32: 8*255*32*127*15 < 2^31.)
//
// The product streams weights like the other M = 1 kernels: a CTA per SM
// (two fit on an SM, so that under programmatic dependent launch the next
// product's CTA streams its weights while this one finishes; with static
// weights its producer starts before the dependency wait), a producer warp
// filling a ring of shared-memory stages of R
// rows -- the nibbles and the scale/minimum bytes by bulk copies (their row
// strides are multiples of 16 bytes), d and dmin by 4-byte asynchronous
// copies (their row stride need not be), all completing on the stage's
// full barrier -- and 16 consumer warps.  A stage's rows go to the warps
// whole, or, when a stage holds fewer rows than warps, each row is split in
// P parts over its columns of 64 sub-blocks (part p takes columns p, p + P,
// ...; the parts' float sums are added in part order at the end).  Within
// a part, lane l works on sub-block l (+32, ...), 8 lanes per super-block; the
// lane's scaled integer dot and minimum term are added across its 8 lanes
// with integer shuffles (two sub-block columns at a time, so that two
// shuffle chains overlap), and the group's first lane does the float
// arithmetic of the super-block.
#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

constexpr int kQKK = 256;
constexpr int kKSubs = kQKK / kQK;                 // sub-blocks per super-block
constexpr int kKWarps = 16;                        // consumer warps (17 warps: at most 96 registers)
constexpr int kKThreads = (kKWarps + 1) * 32;      // + the producer warp
constexpr int kKSlots = 8;
constexpr size_t kKBudget = 110 * 1024;        // two CTAs per SM: the next launch's CTA can stream
                                                // its weights while this one finishes
constexpr size_t kKBudgetWide = 220 * 1024;    // one CTA per SM (very long rows)
constexpr size_t kKStageTarget = 32 * 1024;

// ---- quantiser ------------------------------------------------------------
// One warp per 256-element block; lane l holds elements 8l .. 8l + 7, and
// the four lanes of each 32-element sub-block add their quants for bsums.
// Returns the lane's 8 quants; *d = the block's scale; *sum = its sub-block's
// quant sum (in every lane).  Used by the quantiser kernel and by the phase
// kernel's in-CTA quantisation alike.
__device__ __forceinline__ uint2 q8k_block(const float *xb, int lane, float *d, int *sum_out) {
  const float4 *src = reinterpret_cast<const float4 *>(xb + lane * 8);
  const float4 a = src[0], b = src[1];
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, __float_as_uint(fabsf(v[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float amax = __uint_as_float(m);
  const float dd = amax / 127.0f;
  const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
  int qs[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    qs[i] = quant_one(v[i], id);
    sum += qs[i];
  }
  uint2 packed;
  packed.x = (qs[0] & 0xff) | ((qs[1] & 0xff) << 8) | ((qs[2] & 0xff) << 16) |
             (static_cast<uint32_t>(qs[3] & 0xff) << 24);
  packed.y = (qs[4] & 0xff) | ((qs[5] & 0xff) << 8) | ((qs[6] & 0xff) << 16) |
             (static_cast<uint32_t>(qs[7] & 0xff) << 24);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  *d = dd;
  *sum_out = sum;
  return packed;
}

__global__ void __launch_bounds__(256) quantize_q8k_kernel(const float *__restrict__ x, int8_t *q,
                                                           float *d, int32_t *bsums, int nblocks) {
  const int blk = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  griddep_wait();
  if (blk >= nblocks) return;
  float dd;
  int sum;
  const uint2 packed = q8k_block(x + static_cast<size_t>(blk) * kQKK, lane, &dd, &sum);
  *reinterpret_cast<uint2 *>(q + static_cast<size_t>(blk) * kQKK + lane * 8) = packed;
  if ((lane & 3) == 0) bsums[static_cast<size_t>(blk) * kKSubs + (lane >> 2)] = sum;
  if (lane == 0) d[blk] = dd;
}

cudaError_t launch_quantize_q8k(const LaunchCtx &ctx, const float *x, int8_t *q, float *d,
                                int32_t *bsums, int k) {
  const int nblocks = k / kQKK;
  if (nblocks <= 0) return cudaSuccess;
  const int per = 256 / 32;
  return launch_kernel(quantize_q8k_kernel, dim3(static_cast<unsigned>((nblocks + per - 1) / per)),
                       dim3(256), 0, ctx, x, q, d, bsums, nblocks);
}

// ---- product ----------------------------------------------------------------
constexpr int kKMaxProducts = 4;
// The launch's rows: products j = 0 .. nprod-1, rows rbase[j] .. rbase[j] +
// rows[j] of each, one after another ([0, total) over all of them); every
// product reads the same input.
struct Q4KArgs {
  const uint8_t *wq[kKMaxProducts], *ws[kKMaxProducts];
  const float *wd[kKMaxProducts], *wdmin[kKMaxProducts];
  float *y[kKMaxProducts];
  int rbase[kKMaxProducts], rows[kKMaxProducts];
  int nprod, total;
  const float *xf;       // float input quantised in each CTA (a phase), or null:
  const int8_t *xq;      // the quantised input (quants, scales, sub-block sums)
  const float *xd;
  const int32_t *xbs;
  int32_t *isum, *msum;  // test hook (one product): per-super-block integer sums instead of y
  int nsb;
  int R, ns;                                    // rows per stage, ring slots
  int P;                                        // parts per row (P > 1: partial sums in smem_part)
  int early;                                    // weights not written by earlier work
  int early_input;                              // xf not written by earlier work: quantised before the wait
  unsigned smem_part;
  unsigned stage_bytes, stage_s, stage_d;       // stage size; offsets of s and of d, dmin
  unsigned smem_ring;
  int *status;
  unsigned long long wait_ns;
};

__device__ __forceinline__ void k_consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kKWarps * 32) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
// The stage's full barrier counts one arrival per producer lane once that
// lane's earlier 4-byte copies have landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool k_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
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

// The stage of at most R rows that starts at row r of [0, total) and ends
// before rb and before the end of r's product: returns its row count, with
// *j its product and *lrow its first row in that product.
__device__ __forceinline__ int k_stage(const Q4KArgs &a, int r, int rb, int R, int *j, int *lrow) {
  int jj = 0, off = 0;
  while (jj + 1 < a.nprod && r >= off + a.rows[jj]) {
    off += a.rows[jj];
    ++jj;
  }
  *j = jj;
  *lrow = a.rbase[jj] + (r - off);
  return min(R, min(rb, off + a.rows[jj]) - r);
}

template <bool SUMS>
__global__ void __launch_bounds__(kKThreads, 2) matvec_q4k_kernel(const __grid_constant__ Q4KArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kKSlots];
  __shared__ __align__(8) uint64_t empty_bar[kKSlots];
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nsb = a.nsb, nsub = nsb * kKSubs, K = nsb * kQKK;
  const size_t rowq = static_cast<size_t>(nsb) * (kQKK / 2), rows_s = static_cast<size_t>(nsb) * 16;
  const int n_all = a.total;
  const int ra = static_cast<int>(static_cast<long long>(n_all) * blockIdx.x / gridDim.x);
  const int rb = static_cast<int>(static_cast<long long>(n_all) * (blockIdx.x + 1) / gridDim.x);
  const int R = a.R, ns = a.ns;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  int32_t *xbs_s = reinterpret_cast<int32_t *>(smem + K);
  float *xd_s = reinterpret_cast<float *>(smem + K + 4 * nsub);
  uint8_t *ring = smem + a.smem_ring;
  float *part_s = reinterpret_cast<float *>(smem + a.smem_part);
  const int P = a.P;

  if (tid == 0) {
    for (int k = 0; k < ns; ++k) {
      mbar_init(smem_addr(&full_bar[k]), 1 + 32);  // the bulk-copy arrival + 32 producer lanes
      mbar_init(smem_addr(&empty_bar[k]), kKWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kKWarps) {
    // ------------------------------ producer ------------------------------
    if (!a.early) griddep_wait();  // weights written by earlier work: wait for it first
    int s = 0, n = 0;
    for (int r = ra; r < rb; r += n, ++s) {
      int j, lrow;
      n = k_stage(a, r, rb, R, &j, &lrow);
      const int slot = s % ns;
      if (s >= ns && !warp_wait([&] {
            return k_wait(smem_addr(&empty_bar[slot]), ((s / ns) - 1) & 1, abort_v, a.wait_ns);
          })) {
        if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        break;
      }
      if (*abort_v) break;
      uint8_t *dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
      const uint32_t fb = smem_addr(&full_bar[slot]);
      if (lane == 0) {
        const uint32_t qb = static_cast<uint32_t>(n * rowq), sb = static_cast<uint32_t>(n * rows_s);
        mbar_arrive_expect_tx(fb, qb + sb);
        bulk_copy_g2s(smem_addr(dst), a.wq[j] + static_cast<size_t>(lrow) * rowq, qb, fb);
        bulk_copy_g2s(smem_addr(dst + a.stage_s), a.ws[j] + static_cast<size_t>(lrow) * rows_s, sb, fb);
      }
      float *dd = reinterpret_cast<float *>(dst + a.stage_d);
      float *dm = dd + static_cast<size_t>(R) * nsb;
      for (int e = lane; e < n * nsb; e += 32) {
        cp_async4(dd + e, a.wd[j] + static_cast<size_t>(lrow) * nsb + e);
        cp_async4(dm + e, a.wdmin[j] + static_cast<size_t>(lrow) * nsb + e);
      }
      cp_async_arrive(fb);
    }
    if (*abort_v && lane == 0) {  // copies may still be landing: the last issued stages (bounded)
      for (int t = s > ns ? s - ns : 0; t < s; ++t)
        mbar_wait_bounded(smem_addr(&full_bar[t % ns]), (t / ns) & 1, kDrainWaitNs);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  // x may come from the previous kernel; a static float input is quantised
  // before the wait (the outputs are written only after it)
  const bool early_in = a.xf != nullptr && a.early_input != 0;
  if (!early_in) griddep_wait();
  if (rb <= ra) return;
  // The activation quants in shared memory: sub-block u at u*32, its two
  // 16-byte halves swapped when bit 2 of u is set, so that the 8 lanes of a
  // quarter warp (sub-blocks u .. u+7) read distinct banks.
  if (a.xf != nullptr) {
    // a phase: every CTA quantises the float input itself, one warp per
    // 256-element block, with the quantiser kernel's own arithmetic
    for (int blk = warp; blk < nsb; blk += kKWarps) {
      float dd;
      int sum;
      const uint2 packed = q8k_block(a.xf + static_cast<size_t>(blk) * kQKK, lane, &dd, &sum);
      const int u = blk * 16 + (lane >> 1);  // the lane's 16-byte unit, placed as in the loads below
      *reinterpret_cast<uint2 *>(xq_s + (u ^ ((u >> 3) & 1)) * 16 + (lane & 1) * 8) = packed;
      if ((lane & 3) == 0) xbs_s[blk * kKSubs + (lane >> 2)] = sum;
      if (lane == 0) xd_s[blk] = dd;
    }
  } else {  // all loads before any store
    const int uq = K / 16, ub = nsub / 4;
    for (int base = 0; base < uq + ub; base += 2 * kKWarps * 32) {
      int4 v[2];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int u = base + p * kKWarps * 32 + tid;
        if (u < uq) v[p] = __ldg(reinterpret_cast<const int4 *>(a.xq) + u);
        else if (u < uq + ub) v[p] = __ldg(reinterpret_cast<const int4 *>(a.xbs) + (u - uq));
      }
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int u = base + p * kKWarps * 32 + tid;
        if (u < uq) reinterpret_cast<int4 *>(xq_s)[u ^ ((u >> 3) & 1)] = v[p];  // 16-byte unit u: sub-block u/2
        else if (u < uq + ub) reinterpret_cast<int4 *>(xbs_s)[u - uq] = v[p];
      }
    }
    for (int u = tid; u < nsb; u += kKWarps * 32) xd_s[u] = __ldg(a.xd + u);
  }
  k_consumers_sync();
  if (early_in) griddep_wait();

  int s = 0, n = 0;
  for (int r = ra; r < rb; r += n, ++s) {
    int j, lrow;
    n = k_stage(a, r, rb, R, &j, &lrow);
    const int slot = s % ns;
    if (!warp_wait([&] { return k_wait(smem_addr(&full_bar[slot]), (s / ns) & 1, abort_v, a.wait_ns); })) {
      if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      break;  // every consumer warp still reaches the final sync
    }
    const uint8_t *stq = ring + static_cast<size_t>(slot) * a.stage_bytes;
    const uint8_t *sts = stq + a.stage_s;
    const float *std_ = reinterpret_cast<const float *>(stq + a.stage_d);
    const float *stm = std_ + static_cast<size_t>(R) * nsb;
    for (int task = warp; task < n * P; task += kKWarps) {
      const int i = task % n, part = task / n;
      const uint8_t *wrow = stq + static_cast<size_t>(i) * rowq;
      const uint8_t *srow = sts + static_cast<size_t>(i) * rows_s;
      float acc = 0.0f;
      for (int u0 = 64 * part; u0 < nsub; u0 += 64 * P) {
        int is[2], ms[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int u = u0 + 32 * h + lane;
          is[h] = 0;
          ms[h] = 0;
          if (u < nsub) {  // whole groups of 8 lanes (nsub is a multiple of 8)
            const uint4 w = *reinterpret_cast<const uint4 *>(wrow + static_cast<size_t>(u) * 16);
            const int hs = (u >> 2) & 1;  // the swapped halves (see the staging above)
            const int4 xa = *reinterpret_cast<const int4 *>(xq_s + static_cast<size_t>(u) * kQK + 16 * hs);
            const int4 xb = *reinterpret_cast<const int4 *>(xq_s + static_cast<size_t>(u) * kQK + 16 * (hs ^ 1));
            const int B = u >> 3, j = u & 7;
            constexpr uint32_t kLo = 0x0F0F0F0Fu;
            int dot = 0;
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"(w.x & kLo), "r"(xa.x));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"(w.y & kLo), "r"(xa.y));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"(w.z & kLo), "r"(xa.z));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"(w.w & kLo), "r"(xa.w));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"((w.x >> 4) & kLo), "r"(xb.x));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"((w.y >> 4) & kLo), "r"(xb.y));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"((w.z >> 4) & kLo), "r"(xb.z));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(dot) : "r"((w.w >> 4) & kLo), "r"(xb.w));
            is[h] = static_cast<int>(srow[B * 16 + j]) * dot;
            ms[h] = static_cast<int>(srow[B * 16 + 8 + j]) * xbs_s[u];
          }
        }
        // each super-block's 8 sub-blocks: integer sums, exact
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            is[h] += __shfl_xor_sync(0xffffffffu, is[h], o);
            ms[h] += __shfl_xor_sync(0xffffffffu, ms[h], o);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int u = u0 + 32 * h + lane;
          if (u < nsub && (lane & 7) == 0) {
            const int B = u >> 3;
            if (SUMS) {
              a.isum[static_cast<size_t>(lrow + i - a.rbase[0]) * nsb + B] = is[h];
              a.msum[static_cast<size_t>(lrow + i - a.rbase[0]) * nsb + B] = ms[h];
            } else {
              const float t = __fmul_rn(__int2float_rn(is[h]), std_[static_cast<size_t>(i) * nsb + B]);
              const float um = __fmul_rn(__int2float_rn(ms[h]), stm[static_cast<size_t>(i) * nsb + B]);
              acc = __fadd_rn(acc, __fmul_rn(__fsub_rn(t, um), xd_s[B]));
            }
          }
        }
      }
      if (!SUMS) {
        acc += __shfl_xor_sync(0xffffffffu, acc, 8);
        acc += __shfl_xor_sync(0xffffffffu, acc, 16);
        if (lane == 0) {
          if (P == 1) a.y[j][lrow + i] = acc;
          else part_s[static_cast<size_t>(r + i - ra) * P + part] = acc;
        }
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[slot])) : "memory");
  }
  if (!SUMS && P > 1) {  // the parts of each row, added in part order
    k_consumers_sync();
    if (*abort_v) return;
    for (int i = tid; i < rb - ra; i += kKWarps * 32) {
      float v = part_s[static_cast<size_t>(i) * P];
      for (int p = 1; p < P; ++p) v = __fadd_rn(v, part_s[static_cast<size_t>(i) * P + p]);
      int j, lrow;
      k_stage(a, ra + i, rb, 1, &j, &lrow);
      a.y[j][lrow] = v;
    }
  }
}

// Geometry of a launch over a.total rows of a.nsb super-blocks (a's products
// and input already filled), then the launch.
static cudaError_t launch_q4k_common(const LaunchCtx &ctx, Q4KArgs &a, bool sums) {
  const int n = a.total;
  const int nsb = a.nsb;
  if (n <= 0) return cudaSuccess;
  auto up = [](size_t v, size_t al) { return (v + al - 1) / al * al; };
  const size_t K = static_cast<size_t>(nsb) * kQKK;
  const size_t rowq = static_cast<size_t>(nsb) * (kQKK / 2), rows_s = static_cast<size_t>(nsb) * 16;
  const size_t rowbytes = rowq + rows_s + 8 * static_cast<size_t>(nsb);
  const size_t xs = up(K + 4 * (K / kQK) + 4 * static_cast<size_t>(nsb), 128);
  int R = static_cast<int>(kKStageTarget / rowbytes);
  if (R < 1) R = 1;
  const int per_sm = (n + ctx.num_sms - 1) / ctx.num_sms;  // spread the rows over every SM
  if (R > per_sm) R = per_sm;
  int grid = ctx.num_sms;
  if (grid > (n + R - 1) / R) grid = (n + R - 1) / R;
  const int rows_cta = (n + grid - 1) / grid;
  if (R > rows_cta) R = rows_cta;
  // parts per row: enough that every warp has work when a stage holds few rows
  const int cols64 = (nsb * kKSubs + 63) / 64;
  int P = R >= kKWarps ? 1 : kKWarps / R;
  if (P > cols64) P = cols64;
  if (P < 1) P = 1;
  size_t part = sums || P == 1 ? 0 : up(static_cast<size_t>(rows_cta) * P * 4, 128);
  if (part > 32 * 1024) {  // very many rows per CTA: whole rows per warp
    P = 1;
    part = 0;
  }
  const size_t stage_s = R * rowq;                       // multiple of 128
  const size_t stage_d = stage_s + R * rows_s;           // multiple of 16
  const size_t stage = up(stage_d + 8 * static_cast<size_t>(R) * nsb, 128);
  const size_t budget = xs + part + 2 * stage <= kKBudget ? kKBudget : kKBudgetWide;
  if (xs + part + 2 * stage > budget) return cudaErrorNotSupported;
  int ns = static_cast<int>((budget - xs - part) / stage);
  if (ns > kKSlots) ns = kKSlots;
  // stages per CTA, counted with the breaks at product boundaries
  const int stages_cta = (rows_cta + R - 1) / R + a.nprod - 1;
  if (ns > stages_cta) ns = stages_cta < 2 ? 2 : stages_cta;
  a.R = R;
  a.ns = ns;
  a.stage_bytes = static_cast<unsigned>(stage);
  a.stage_s = static_cast<unsigned>(stage_s);
  a.stage_d = static_cast<unsigned>(stage_d);
  a.P = P;
  a.early = ctx.early_weights ? 1 : 0;
  a.smem_part = static_cast<unsigned>(xs);
  a.smem_ring = static_cast<unsigned>(xs + part);
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  const size_t smem = xs + part + static_cast<size_t>(ns) * stage;
  auto kern = sums ? matvec_q4k_kernel<true> : matvec_q4k_kernel<false>;
  prefer_max_shared(kern);
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kKThreads), smem, ctx, a);
}

cudaError_t launch_matvec_q4k(const LaunchCtx &ctx, const void *wq, const void *ws, const float *wd,
                              const float *wdmin, int nsb, const int8_t *xq, const float *xd,
                              const int32_t *xbs, float *y, int32_t *isum, int32_t *msum, int r0,
                              int r1) {
  Q4KArgs a = {};
  a.wq[0] = static_cast<const uint8_t *>(wq);
  a.ws[0] = static_cast<const uint8_t *>(ws);
  a.wd[0] = wd;
  a.wdmin[0] = wdmin;
  a.y[0] = y;
  a.rbase[0] = r0;
  a.rows[0] = r1 - r0;
  a.nprod = 1;
  a.total = r1 - r0;
  a.xf = nullptr;
  a.xq = xq;
  a.xd = xd;
  a.xbs = xbs;
  a.isum = isum;
  a.msum = msum;
  a.nsb = nsb;
  return launch_q4k_common(ctx, a, isum != nullptr);
}

cudaError_t launch_phase_q4k(const LaunchCtx &ctx, const float *x, int nsb, const Q4KProductDev *p,
                             int np, bool early_input) {
  if (np < 1 || np > kKMaxProducts) return cudaErrorInvalidValue;
  Q4KArgs a = {};
  a.total = 0;
  for (int j = 0; j < np; ++j) {
    a.wq[j] = static_cast<const uint8_t *>(p[j].q);
    a.ws[j] = static_cast<const uint8_t *>(p[j].s);
    a.wd[j] = p[j].d;
    a.wdmin[j] = p[j].dmin;
    a.y[j] = p[j].y;
    a.rbase[j] = 0;
    a.rows[j] = p[j].rows;
    a.total += p[j].rows;
  }
  a.nprod = np;
  a.xf = x;
  a.nsb = nsb;
  a.early_input = early_input ? 1 : 0;
  return launch_q4k_common(ctx, a, false);
}

}  // namespace mlq
