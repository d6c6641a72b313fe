// nbits.cu -- M = 1 products on blocks of 32 or 128 weights with float32
// or binary16 scales, 4-bit (nibble - 8) or 8-bit weights in the packed
// signed form with per-block zero points, and the per-block activation
// quantiser they read.
//
// Definitions: page "ONNX Runtime" (SpaceMiT X60), "How we got there":
// item 3 (block_size 128 with int8 activations), item 4 (8-bit weights
// packed as B' = B - 128, flat scales, the correction -scale * (zp - 128)
// that vanishes for zp = 128), item 5 (float16 scales).  Per block b of
// row r:
//   sumi = sum_i w_i a_i,  w = n - 8 (4-bit) or B' + 128 - zp_b (8-bit),
//   y[r] += ((float)sumi * scale_b) * dx_b            (float32, this order).
// The kernel forms sumi with the signed-offset correction in the integer
// domain -- sum B' a + (128 - zp) * sum a, or sum n a - 8 * sum a -- which
// equals the definition exactly, with the per-block activation quant sums.
// Layout: 4-bit blocks pack element j in the low nibble and element
// j + blk/2 in the high nibble of byte j; scale and zero-point rows have a
// caller-given stride padded to 16 bytes, so that every per-row array is
// bulk-copied.
//
// Streaming as in q4k.cu: a producer warp fills a ring of shared-memory
// stages of R rows (weights, scales, zero points: bulk copies on one full
// barrier), 16 consumer warps take rows (split in column parts when a stage
// holds fewer rows than warps), lane l takes 16-byte unit l (+32, ...) of
// the row, the units of a block add their dp4a sums with integer shuffles,
// and the block's first lane applies the correction and the two float
// multiplications.  Two CTAs fit on an SM.
#include <cuda_fp16.h>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

constexpr int kNWarps = 16;
constexpr int kNThreads = (kNWarps + 1) * 32;
constexpr int kNSlots = 8;
constexpr size_t kNBudget = 110 * 1024;
constexpr size_t kNBudgetWide = 220 * 1024;
constexpr size_t kNStageTarget = 32 * 1024;

// ---- per-block activation quantiser ------------------------------------------
// One warp per block of `blk` (32 or 128) elements; lane l holds elements
// l*E .. l*E + E - 1 (E = blk / 32).
// Returns the lane's E quants packed in bytes; *d = the block's scale;
// *sum_out = the block's quant sum (every lane).  Used by the quantiser
// kernel and by the phase kernel's in-CTA quantisation alike.
template <int E>
__device__ __forceinline__ uint32_t blk_quant(const float *xb, int lane, float *d, int *sum_out) {
  float v[E];
  const float *src = xb + lane * E;
  if (E == 4) {
    const float4 t = *reinterpret_cast<const float4 *>(src);
    v[0] = t.x;
    v[1 % E] = t.y;
    v[2 % E] = t.z;
    v[3 % E] = t.w;
  } else {
    v[0] = src[0];
  }
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) m = max(m, __float_as_uint(fabsf(v[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float amax = __uint_as_float(m);
  const float dd = amax / 127.0f;
  const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
  int sum = 0;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int qq = quant_one(v[i], id);
    sum += qq;
    packed |= static_cast<uint32_t>(qq & 0xff) << (8 * i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  *d = dd;
  *sum_out = sum;
  return packed;
}

template <int E>
__global__ void __launch_bounds__(256) quantize_blk_kernel(const float *__restrict__ x, int8_t *q,
                                                           float *d, int32_t *bsums, int nblocks) {
  const int blk = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  griddep_wait();
  if (blk >= nblocks) return;
  float dd;
  int sum;
  const uint32_t packed = blk_quant<E>(x + static_cast<size_t>(blk) * (32 * E), lane, &dd, &sum);
  int8_t *dst = q + static_cast<size_t>(blk) * (32 * E) + lane * E;
  if (E == 4) *reinterpret_cast<uint32_t *>(dst) = packed;
  else *dst = static_cast<int8_t>(packed & 0xff);
  if (lane == 0) {
    d[blk] = dd;
    bsums[blk] = sum;
  }
}

cudaError_t launch_quantize_blk(const LaunchCtx &ctx, const float *x, int8_t *q, float *d,
                                int32_t *bsums, int k, int blk) {
  const int nblocks = k / blk;
  if (nblocks <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((nblocks + 7) / 8));
  if (blk == 128) return launch_kernel(quantize_blk_kernel<4>, grid, dim3(256), 0, ctx, x, q, d, bsums, nblocks);
  return launch_kernel(quantize_blk_kernel<1>, grid, dim3(256), 0, ctx, x, q, d, bsums, nblocks);
}

// ---- product ------------------------------------------------------------------
constexpr int kNMaxProducts = 4;
// The launch's rows: products j = 0 .. nprod-1 (one format, scale and zero-
// point row strides), rows rbase[j] .. rbase[j] + rows[j] of each, one after
// another ([0, total) over all of them); every product reads the same input.
struct NBitsArgs {
  const uint8_t *wq[kNMaxProducts];
  const void *sc[kNMaxProducts];
  const uint8_t *zp[kNMaxProducts];  // 8-bit: zero points (nullptr: 128), all or none
  float *y[kNMaxProducts];
  int rbase[kNMaxProducts], rows[kNMaxProducts];
  int nprod, total;
  const float *xf;    // float input quantised in each CTA (a phase), or null:
  const int8_t *xq;   // the quantised input (quants, scales, block sums)
  const float *xd;
  const int32_t *xbs;
  int32_t *sumi;      // test hook (one product): per-block int32 sums instead of y
  int cols, blk, nb, f16, sc_ld, zp_ld;
  int R, ns, P, early;
  int early_input;  // xf not written by earlier work: quantised before the dependency wait
  unsigned rowq, row_sc, row_zp;          // bytes per row of each array
  unsigned stage_bytes, stage_sc, stage_zp, smem_part, smem_ring;
  int *status;
  unsigned long long wait_ns;
};

__device__ __forceinline__ void n_consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kNWarps * 32) : "memory");
}
__device__ __forceinline__ bool n_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
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
__device__ __forceinline__ int n_stage(const NBitsArgs &a, int r, int rb, int R, int *j, int *lrow) {
  int jj = 0, off = 0;
  while (jj + 1 < a.nprod && r >= off + a.rows[jj]) {
    off += a.rows[jj];
    ++jj;
  }
  *j = jj;
  *lrow = a.rbase[jj] + (r - off);
  return min(R, min(rb, off + a.rows[jj]) - r);
}

template <int BITS, bool SUMS>
__global__ void __launch_bounds__(kNThreads, 2) matvec_nbits_kernel(const __grid_constant__ NBitsArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kNSlots];
  __shared__ __align__(8) uint64_t empty_bar[kNSlots];
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.cols, blk = a.blk, nb = a.nb;
  const size_t rowq = a.rowq, row_sc = a.row_sc, row_zp = a.row_zp;
  const int n_all = a.total;
  const int ra = static_cast<int>(static_cast<long long>(n_all) * blockIdx.x / gridDim.x);
  const int rb = static_cast<int>(static_cast<long long>(n_all) * (blockIdx.x + 1) / gridDim.x);
  const int R = a.R, ns = a.ns, P = a.P;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + K);
  int32_t *xbs_s = reinterpret_cast<int32_t *>(smem + K + 4 * nb);
  float *part_s = reinterpret_cast<float *>(smem + a.smem_part);
  uint8_t *ring = smem + a.smem_ring;

  if (tid == 0) {
    for (int k = 0; k < ns; ++k) {
      mbar_init(smem_addr(&full_bar[k]), 1);
      mbar_init(smem_addr(&empty_bar[k]), kNWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kNWarps) {
    // ------------------------------ producer ------------------------------
    if (lane != 0) return;
    if (!a.early) griddep_wait();  // weights written by earlier work: wait for it first
    int s = 0, n = 0;
    for (int r = ra; r < rb; r += n, ++s) {
      int j, lrow;
      n = n_stage(a, r, rb, R, &j, &lrow);
      const int slot = s % ns;
      if (s >= ns && !n_wait(smem_addr(&empty_bar[slot]), ((s / ns) - 1) & 1, abort_v, a.wait_ns)) {
        if (atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        break;
      }
      if (*abort_v) break;
      uint8_t *dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
      const uint32_t fb = smem_addr(&full_bar[slot]);
      const uint32_t qb = static_cast<uint32_t>(n * rowq), sb = static_cast<uint32_t>(n * row_sc);
      const uint32_t zb = a.zp[j] != nullptr ? static_cast<uint32_t>(n * row_zp) : 0u;
      mbar_arrive_expect_tx(fb, qb + sb + zb);
      bulk_copy_g2s(smem_addr(dst), a.wq[j] + static_cast<size_t>(lrow) * rowq, qb, fb);
      bulk_copy_g2s(smem_addr(dst + a.stage_sc),
                    static_cast<const uint8_t *>(a.sc[j]) + static_cast<size_t>(lrow) * row_sc, sb, fb);
      if (zb) bulk_copy_g2s(smem_addr(dst + a.stage_zp), a.zp[j] + static_cast<size_t>(lrow) * row_zp, zb, fb);
    }
    if (*abort_v) {  // copies may still be landing: the last issued stages (bounded)
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
  if (a.xf != nullptr) {
    // a phase: every CTA quantises the float input itself, one warp per
    // block, with the quantiser kernel's own arithmetic
    for (int b = warp; b < nb; b += kNWarps) {
      float dd;
      int sum;
      if (blk == 128) {
        const uint32_t packed = blk_quant<4>(a.xf + static_cast<size_t>(b) * 128, lane, &dd, &sum);
        *reinterpret_cast<uint32_t *>(xq_s + b * 128 + lane * 4) = packed;
      } else {
        const uint32_t packed = blk_quant<1>(a.xf + static_cast<size_t>(b) * 32, lane, &dd, &sum);
        xq_s[b * 32 + lane] = static_cast<int8_t>(packed & 0xff);
      }
      if (lane == 0) {
        xd_s[b] = dd;
        xbs_s[b] = sum;
      }
    }
  } else {  // the activations into shared memory, all loads before any store
    const int uq = K / 16;
    for (int base = 0; base < uq; base += 2 * kNWarps * 32) {
      int4 v[2];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int u = base + p * kNWarps * 32 + tid;
        if (u < uq) v[p] = __ldg(reinterpret_cast<const int4 *>(a.xq) + u);
      }
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int u = base + p * kNWarps * 32 + tid;
        if (u < uq) reinterpret_cast<int4 *>(xq_s)[u] = v[p];
      }
    }
    for (int b = tid; b < nb; b += kNWarps * 32) {
      xd_s[b] = __ldg(a.xd + b);
      xbs_s[b] = __ldg(a.xbs + b);
    }
  }
  n_consumers_sync();
  if (early_in) griddep_wait();

  // A row is U 16-byte units; UPB units per block (a power of two).
  const int U = static_cast<int>(rowq / 16);
  const int upb = BITS == 4 ? blk / 32 : blk / 16;
  int s = 0, n = 0;
  for (int r = ra; r < rb; r += n, ++s) {
    int j, lrow;
    n = n_stage(a, r, rb, R, &j, &lrow);
    const int slot = s % ns;
    if (!warp_wait([&] { return n_wait(smem_addr(&full_bar[slot]), (s / ns) & 1, abort_v, a.wait_ns); })) {
      if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      break;  // every consumer warp still reaches the final sync
    }
    const uint8_t *stq = ring + static_cast<size_t>(slot) * a.stage_bytes;
    const uint8_t *sts = stq + a.stage_sc;
    const uint8_t *stz = stq + a.stage_zp;
    for (int task = warp; task < n * P; task += kNWarps) {
      const int i = task % n, part = task / n;
      const uint8_t *wrow = stq + static_cast<size_t>(i) * rowq;
      float acc = 0.0f;
      for (int u0 = 32 * part; u0 < U; u0 += 32 * P) {
        const int u = u0 + lane;
        int sacc = 0;
        const int b = u / upb, p = u % upb;
        if (u < U) {
          const uint4 w = *reinterpret_cast<const uint4 *>(wrow + static_cast<size_t>(u) * 16);
          if (BITS == 4) {
            const int e0 = b * blk + 16 * p;  // low nibbles: elements e0 .. e0 + 15; high: + blk/2
            const int4 xa = *reinterpret_cast<const int4 *>(xq_s + e0);
            const int4 xb = *reinterpret_cast<const int4 *>(xq_s + e0 + blk / 2);
            constexpr uint32_t kLo = 0x0F0F0F0Fu;
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"(w.x & kLo), "r"(xa.x));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"(w.y & kLo), "r"(xa.y));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"(w.z & kLo), "r"(xa.z));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"(w.w & kLo), "r"(xa.w));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"((w.x >> 4) & kLo), "r"(xb.x));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"((w.y >> 4) & kLo), "r"(xb.y));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"((w.z >> 4) & kLo), "r"(xb.z));
            asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(sacc) : "r"((w.w >> 4) & kLo), "r"(xb.w));
          } else {
            const int4 xa = *reinterpret_cast<const int4 *>(xq_s + b * blk + 16 * p);
            sacc = __dp4a(static_cast<int>(w.x), xa.x, sacc);
            sacc = __dp4a(static_cast<int>(w.y), xa.y, sacc);
            sacc = __dp4a(static_cast<int>(w.z), xa.z, sacc);
            sacc = __dp4a(static_cast<int>(w.w), xa.w, sacc);
          }
        }
        // the block's units: integer sums, exact (upb lanes, aligned groups)
        for (int o = 1; o < upb; o <<= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, o);
        if (u < U && p == 0) {
          int corr;
          if (BITS == 4) {
            corr = -8;
          } else {
            corr = 128 - (a.zp[j] != nullptr ? static_cast<int>(stz[static_cast<size_t>(i) * row_zp + b]) : 128);
          }
          const int sumi = sacc + corr * xbs_s[b];
          if (SUMS) {
            a.sumi[static_cast<size_t>(lrow + i - a.rbase[0]) * nb + b] = sumi;
          } else {
            const float sc = a.f16 ? __half2float(reinterpret_cast<const __half *>(sts + static_cast<size_t>(i) * row_sc)[b])
                                   : reinterpret_cast<const float *>(sts + static_cast<size_t>(i) * row_sc)[b];
            acc = __fadd_rn(acc, __fmul_rn(__fmul_rn(__int2float_rn(sumi), sc), xd_s[b]));
          }
        }
      }
      if (!SUMS) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
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
    n_consumers_sync();
    if (*abort_v) return;
    for (int i = tid; i < rb - ra; i += kNWarps * 32) {
      float v = part_s[static_cast<size_t>(i) * P];
      for (int p = 1; p < P; ++p) v = __fadd_rn(v, part_s[static_cast<size_t>(i) * P + p]);
      int j, lrow;
      n_stage(a, ra + i, rb, 1, &j, &lrow);
      a.y[j][lrow] = v;
    }
  }
}

// Geometry of a launch over a.total rows (a's format, products and input
// already filled), then the launch.
static cudaError_t launch_nbits_common(const LaunchCtx &ctx, NBitsArgs &a, int bits, bool sums) {
  const int n = a.total;
  if (n <= 0) return cudaSuccess;
  auto up = [](size_t v, size_t al) { return (v + al - 1) / al * al; };
  const int cols = a.cols, blk = a.blk, nb = cols / blk;
  const size_t rowq = static_cast<size_t>(cols) * bits / 8;
  const size_t row_sc = static_cast<size_t>(a.sc_ld) * (a.f16 ? 2 : 4);
  const size_t row_zp = a.zp[0] != nullptr ? static_cast<size_t>(a.zp_ld) : 0;
  const size_t rowbytes = rowq + row_sc + row_zp;
  const size_t xs = up(static_cast<size_t>(cols) + 8 * static_cast<size_t>(nb), 128);
  int R = static_cast<int>(kNStageTarget / rowbytes);
  if (R < 1) R = 1;
  const int per_sm = (n + ctx.num_sms - 1) / ctx.num_sms;  // spread the rows over every SM
  if (R > per_sm) R = per_sm;
  int grid = ctx.num_sms;
  if (grid > (n + R - 1) / R) grid = (n + R - 1) / R;
  const int rows_cta = (n + grid - 1) / grid;
  if (R > rows_cta) R = rows_cta;
  const int units = static_cast<int>(rowq / 16);
  const int cols32 = (units + 31) / 32;
  int P = R >= kNWarps ? 1 : kNWarps / R;
  if (P > cols32) P = cols32;
  if (P < 1) P = 1;
  size_t part = sums || P == 1 ? 0 : up(static_cast<size_t>(rows_cta) * P * 4, 128);
  if (part > 32 * 1024) {
    P = 1;
    part = 0;
  }
  const size_t stage_sc = up(R * rowq, 16);
  const size_t stage_zp = up(stage_sc + R * row_sc, 16);
  const size_t stage = up(stage_zp + R * row_zp, 128);
  const size_t budget = xs + part + 2 * stage <= kNBudget ? kNBudget : kNBudgetWide;
  if (xs + part + 2 * stage > budget) return cudaErrorNotSupported;
  int ns = static_cast<int>((budget - xs - part) / stage);
  if (ns > kNSlots) ns = kNSlots;
  // stages per CTA, counted with the breaks at product boundaries
  const int stages_cta = (rows_cta + R - 1) / R + a.nprod - 1;
  if (ns > stages_cta) ns = stages_cta < 2 ? 2 : stages_cta;
  a.nb = nb;
  a.R = R;
  a.ns = ns;
  a.P = P;
  a.early = ctx.early_weights ? 1 : 0;
  a.rowq = static_cast<unsigned>(rowq);
  a.row_sc = static_cast<unsigned>(row_sc);
  a.row_zp = static_cast<unsigned>(row_zp);
  a.stage_bytes = static_cast<unsigned>(stage);
  a.stage_sc = static_cast<unsigned>(stage_sc);
  a.stage_zp = static_cast<unsigned>(stage_zp);
  a.smem_part = static_cast<unsigned>(xs);
  a.smem_ring = static_cast<unsigned>(xs + part);
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  const size_t smem = xs + part + static_cast<size_t>(ns) * stage;
  auto kern = bits == 4 ? (sums ? matvec_nbits_kernel<4, true> : matvec_nbits_kernel<4, false>)
                        : (sums ? matvec_nbits_kernel<8, true> : matvec_nbits_kernel<8, false>);
  prefer_max_shared(kern);
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kNThreads), smem, ctx, a);
}

cudaError_t launch_matvec_nbits(const LaunchCtx &ctx, int bits, int blk, const void *wq, const void *sc,
                                int sc_f16, int sc_ld, const uint8_t *zp, int zp_ld, int cols,
                                const int8_t *xq, const float *xd, const int32_t *xbs, float *y,
                                int32_t *sumi, int r0, int r1) {
  NBitsArgs a = {};
  a.wq[0] = static_cast<const uint8_t *>(wq);
  a.sc[0] = sc;
  a.zp[0] = zp;
  a.y[0] = y;
  a.rbase[0] = r0;
  a.rows[0] = r1 - r0;
  a.nprod = 1;
  a.total = r1 - r0;
  a.xf = nullptr;
  a.xq = xq;
  a.xd = xd;
  a.xbs = xbs;
  a.sumi = sumi;
  a.cols = cols;
  a.blk = blk;
  a.f16 = sc_f16;
  a.sc_ld = sc_ld;
  a.zp_ld = zp_ld;
  return launch_nbits_common(ctx, a, bits, sumi != nullptr);
}

cudaError_t launch_phase_nbits(const LaunchCtx &ctx, int bits, int blk, int sc_f16, int sc_ld, int zp_ld,
                               int cols, const float *x, const NBitsProductDev *p, int np, bool early_input) {
  if (np < 1 || np > kNMaxProducts) return cudaErrorInvalidValue;
  NBitsArgs a = {};
  a.total = 0;
  for (int j = 0; j < np; ++j) {
    a.wq[j] = static_cast<const uint8_t *>(p[j].q);
    a.sc[j] = p[j].scales;
    a.zp[j] = p[j].zp;
    a.y[j] = p[j].y;
    a.rbase[j] = 0;
    a.rows[j] = p[j].rows;
    a.total += p[j].rows;
  }
  a.nprod = np;
  a.xf = x;
  a.cols = cols;
  a.blk = blk;
  a.f16 = sc_f16;
  a.sc_ld = sc_ld;
  a.zp_ld = zp_ld;
  a.early_input = early_input ? 1 : 0;
  return launch_nbits_common(ctx, a, bits, false);
}

}  // namespace mlq
