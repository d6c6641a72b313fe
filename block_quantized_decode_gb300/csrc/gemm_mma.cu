// gemm_mma.cu -- batched small-M decode on the tensor cores: M (2..16)
// Q8_0 activation rows against one Q4_0 weight matrix.
//
// Computes (page "ONNX Runtime", "6. Panel loop (pre-TCM)": batched decode,
// M rows against 4096 x 11008; definitions of the page "Legacy-ISA ML
// Inference Runtime -- Design Spec", Sec. 4):
//   Y[m*ldy + r] = sum_b ((float)sumi(m, r, b) * dw(r, b)) * dx(m, b),
//   sumi(m, r, b) = sum_j (nibble(r, b, j) - 8) * qx(m, 32b + j).
//
// At M = 16 the product does about 51 integer operations per weight byte,
// too many for dp4a at HBM speed.  GB300's legacy warp MMA runs fp16 at
// about four times its int8 rate (measured: 603 vs 151 TOPS), and fp16 is
// exact here: nibble - 8 and int8 activations are small integers, every
// product is exact in the fp32 accumulator and a 32-term block sum (at most
// 32*8*127 in magnitude) stays far below 2^24.  So one block of 32 is two
// mma.m16n8k16 steps per 8 activation rows, started from zero: the result
// IS the block's int32 sum, exactly.  The per-block scales are then applied
// in fp32 ((sumi * dw) * dx, accumulated with a fused multiply-add, as in the
// M = 1 kernels), two elements at a time with packed f32x2 instructions.
//
// Operand staging.  Both operands use the same permutation of the 32 k
// positions of a block, chosen so that lane (g, t) of the warp needs exactly
// 32-bit word t of its weight rows' 16-byte blocks: the low nibbles of that
// word are elements 4t..4t+3 and the high nibbles 16+4t..16+4t+3.  MMA step
// 0 takes elements {4t, 4t+2} in k-slots {2t, 2t+1} and {4t+1, 4t+3} in
// {2t+8, 2t+9}; step 1 the same plus 16.  Nibbles become fp16 by OR-ing them
// into the mantissa of 1024.0 and subtracting 1032.0 (= 1024 + 8); int8
// activations by biasing to unsigned, OR-ing into 1024.0 and subtracting
// 1152.0.  Both conversions are exact.
//
// Work split: a warp task is (16-row tile, K-slice); the S slices of a tile
// live in the same CTA and are summed in a fixed order through shared
// memory (deterministic).
#include <cuda_fp16.h>

#include "mlq_device.cuh"
#include "mlq_launch.h"
#include "mma_frag.cuh"

namespace mlq {

struct MmaArgs {
  const uint8_t *wq;
  const float *wd;
  const int8_t *xq;
  const float *xd;
  float *Y;
  int ldy;
  int nb;
  int M;
  int r0, r1;
  int S;      // K-slices per tile (warps per tile)
  int tpc;    // tiles per CTA (warps per CTA = S * tpc)
};

constexpr int kMmaWarps = 8;  // at most, per CTA

__device__ __forceinline__ uint32_t ldg_u32(const void *p) {
  uint32_t v;
  asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

template <int NT>
__global__ void __launch_bounds__(kMmaWarps * 32) gemm_q4_mma_kernel(const MmaArgs a) {
  __shared__ float red[kMmaWarps][16][16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tpc = a.tpc;
  const int tile = blockIdx.x * tpc + warp / a.S;
  const int s = warp % a.S;
  const int nb = a.nb;
  const int K = nb * kQK;
  const size_t rowq = static_cast<size_t>(nb) * 16;
  const int row_lo = a.r0 + tile * 16 + g;
  const int row_hi = row_lo + 8;
  const bool v_lo = row_lo < a.r1, v_hi = row_hi < a.r1;
  const int b0 = static_cast<int>(static_cast<long long>(nb) * s / a.S);
  const int b1 = static_cast<int>(static_cast<long long>(nb) * (s + 1) / a.S);

  griddep_wait();  // the activations may come from the previous kernel
  griddep_launch_dependents();

  const uint8_t *wlo = a.wq + static_cast<size_t>(v_lo ? row_lo : 0) * rowq + 4 * t;
  const uint8_t *whi = a.wq + static_cast<size_t>(v_hi ? row_hi : 0) * rowq + 4 * t;
  const float *dlo = a.wd + static_cast<size_t>(v_lo ? row_lo : 0) * nb;
  const float *dhi = a.wd + static_cast<size_t>(v_hi ? row_hi : 0) * nb;
  // activation rows this lane feeds into the MMA (n = g) and scales it needs (m = 2t, 2t+1)
  const int8_t *xrow[NT];
  bool xv[NT];
  const float *dxrow[NT][2];
  bool dv[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = nt * 8 + g;
    xv[nt] = m < a.M;
    xrow[nt] = a.xq + static_cast<size_t>(xv[nt] ? m : 0) * K + 4 * t;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int mc = nt * 8 + 2 * t + c;
      dv[nt][c] = mc < a.M;
      dxrow[nt][c] = a.xd + static_cast<size_t>(dv[nt][c] ? mc : 0) * nb;
    }
  }

  unsigned long long acc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0ull;

  // Four blocks per step: every load of the step is issued before any of
  // its data is used, so a warp keeps ~4x more loads in flight.
  constexpr int kB = 4;
  for (int bb = b0; bb < b1; bb += kB) {
    uint32_t wl[kB], wh[kB], xa[NT][kB], xb[NT][kB];
    float sl[kB], sh[kB], dx0[NT][kB], dx1[NT][kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int b = bb + j;
      const bool in = b < b1;
      wl[j] = (v_lo && in) ? ldg_u32(wlo + static_cast<size_t>(b) * 16) : 0x88888888u;
      wh[j] = (v_hi && in) ? ldg_u32(whi + static_cast<size_t>(b) * 16) : 0x88888888u;
      sl[j] = (v_lo && in) ? __ldg(dlo + b) : 0.0f;
      sh[j] = (v_hi && in) ? __ldg(dhi + b) : 0.0f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        xa[nt][j] = (xv[nt] && in) ? ldg_u32(xrow[nt] + static_cast<size_t>(b) * kQK) : 0u;
        xb[nt][j] = (xv[nt] && in) ? ldg_u32(xrow[nt] + static_cast<size_t>(b) * kQK + 16) : 0u;
        dx0[nt][j] = (dv[nt][0] && in) ? __ldg(dxrow[nt][0] + b) : 0.0f;
        dx1[nt][j] = (dv[nt][1] && in) ? __ldg(dxrow[nt][1] + b) : 0.0f;
      }
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      // A fragments, step 0 (low nibbles) and step 1 (high nibbles)
      uint32_t A0[4], A1[4];
      A0[0] = nib_to_h2(wl[j]);
      A0[1] = nib_to_h2(wh[j]);
      A0[2] = nib_to_h2(wl[j] >> 8);
      A0[3] = nib_to_h2(wh[j] >> 8);
      A1[0] = nib_to_h2(wl[j] >> 4);
      A1[1] = nib_to_h2(wh[j] >> 4);
      A1[2] = nib_to_h2(wl[j] >> 12);
      A1[3] = nib_to_h2(wh[j] >> 12);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t ba = xa[nt][j] ^ 0x80808080u, bbits = xb[nt][j] ^ 0x80808080u;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(d, A0, s8_to_h2(ba, 0x4240u), s8_to_h2(ba, 0x4341u));
        mma16816(d, A1, s8_to_h2(bbits, 0x4240u), s8_to_h2(bbits, 0x4341u));
        const unsigned long long x2 = pack2(dx0[nt][j], dx1[nt][j]);
        scale_acc2(acc[nt][0], d[0], d[1], sl[j], x2);
        scale_acc2(acc[nt][1], d[2], d[3], sh[j], x2);
      }
    }
  }

  // fixed-order sum over the S slices of each tile
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float a0, a1, a2, a3;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc[nt][0]));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a2), "=f"(a3) : "l"(acc[nt][1]));
    red[warp][g][nt * 8 + 2 * t] = a0;
    red[warp][g][nt * 8 + 2 * t + 1] = a1;
    red[warp][g + 8][nt * 8 + 2 * t] = a2;
    red[warp][g + 8][nt * 8 + 2 * t + 1] = a3;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < tpc * 16 * 16; i += blockDim.x) {
    const int tl = i / 256, rr = (i / 16) % 16, m = i % 16;
    const int row = a.r0 + (blockIdx.x * tpc + tl) * 16 + rr;
    if (row < a.r1 && m < a.M && m < NT * 8) {
      float v = 0.0f;
      for (int q = 0; q < a.S; ++q) v += red[tl * a.S + q][rr][m];
      a.Y[static_cast<size_t>(m) * a.ldy + row] = v;
    }
  }
}

static long long ctas_limit_sms(const LaunchCtx &ctx) { return ctx.num_sms; }

cudaError_t launch_gemm_q4_mma(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                               const int8_t *xq, const float *xd, int M, float *Y, int ldy,
                               int r0, int r1) {
  const int n = r1 - r0;
  if (n <= 0 || M <= 0) return cudaSuccess;
  MmaArgs a;
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
  const long long tiles = (n + 15) / 16;
  // Pick the K-slice count S (warps per 16-row tile) that gives the most
  // warps while the whole grid stays resident in one wave; a second,
  // mostly empty wave costs more than the extra parallelism gains.
  auto kern = M <= 8 ? gemm_q4_mma_kernel<1> : gemm_q4_mma_kernel<2>;
  int bestS = 1, best_tpc = 4;
  long long best_warps = -1, best_waves = 1LL << 40;
  for (int S = 1; S <= kMmaWarps; S *= 2) {
    if (S > 1 && nb / S < 8) break;
    const int warps = S >= 4 ? S : 4;
    const int tpc = warps / S;
    const long long ctas = (tiles + tpc - 1) / tpc;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, warps * 32, 0) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    const long long resident = static_cast<long long>(per_sm) * ctas_limit_sms(ctx);
    const long long waves = (ctas + resident - 1) / resident;
    const long long total_warps = tiles * S;
    if (waves < best_waves || (waves == best_waves && total_warps > best_warps)) {
      best_waves = waves;
      best_warps = total_warps;
      bestS = S;
      best_tpc = tpc;
    }
  }
  a.S = bestS;
  a.tpc = best_tpc;
  const long long grid = (tiles + best_tpc - 1) / best_tpc;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(bestS * best_tpc * 32), 0, ctx, a);
}

}  // namespace mlq
