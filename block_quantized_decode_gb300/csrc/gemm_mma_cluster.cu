// gemm_mma_cluster.cu -- batched small-M decode (M up to 16) on the tensor
// cores, built to stream the Q4_0 weights at memory speed.
//
// Computes (page "ONNX Runtime", "6. Panel loop (pre-TCM)": batched decode,
// M rows against 4096 x 11008; definitions of the page "Legacy-ISA ML
// Inference Runtime -- Design Spec", Sec. 4):
//   Y[m*ldy + r] = sum_b ((float)sumi(m, r, b) * dw(r, b)) * dx(m, b),
//   sumi(m, r, b) = sum_j (nibble(r, b, j) - 8) * qx(m, 32b + j).
//
// Operand roles.  The (up to 16) activation rows are the A operand of
// mma.m16n8k16 and eight weight rows its B operand, so the activations of
// a block serve every 8-row weight tile.  The CTA copies its K-part of the
// activations into shared memory with one tensor copy and lays it out
// there in fragment order, in one of two forms, next to two 16-byte quads
// per block and row group: the scale pairs (dx_g, dx_g, dx_g+8, dx_g+8) and
// the start values of the block sums.
//  * fp16 A fragments, 1 KB per block of 32 columns, converted once;
//  * int8 words, 512 bytes per block (lane (g, t) holds words t and t + 4
//    of rows g and g + 8, biased to unsigned), which each warp turns into
//    its fp16 A fragments when it takes the block of a stage (byte permutes
//    and one fp16 subtract or multiply-add per pair, all exact).
// The int8 form holds 96 blocks per CTA instead of 64, so a long row needs
// fewer K-parts (4096 x 11008: clusters of 4 in one round of rows instead
// of clusters of 6 in two; measured 26.1 -> 22.2 us).  Where the K-parts
// stay the same its per-stage conversion only adds work (11008 x 4096:
// 18.0-19.3 -> 19.1-20.2 us), so it is taken only where it needs fewer.
//
// Exact block sums without a per-weight subtraction.  A weight word turns
// into B fragments with bit operations only: a low nibble n becomes the
// fp16 value 1024 + n (n in the mantissa of 1024) and a high nibble, left in
// place, 1024 + 16 n.  The first MMA step (low nibbles) multiplies them by
// the activations x, the second (high nibbles) by x / 16, which fp16 holds
// exactly; the sum then carries 1024 * Sx_lo + 64 * Sx_hi on top of
// sum n * x, where Sx_lo, Sx_hi are the block's activation sums over its two
// halves.  Starting the accumulator at -(1032 Sx_lo + 72 Sx_hi) instead of
// zero leaves exactly sum (n - 8) * x = sumi: every product and partial sum
// is an integer below 2^23, which fp32 holds exactly.  The block sums are
// then scaled in fp32 as (sumi * dw) * dx and accumulated with a fused
// multiply-add, as in every other kernel.
//
// Weights.  Thread 0 streams the CTA's share through a ring of 4-8 stages
// with TMA tensor copies, all but one in flight: a stage is the cluster's rows (up to 160)
// x 8 blocks, one weight box (128 bytes per row) and one scale box, both
// completing on the stage's mbarrier.  Measured on GB300, the copy engine
// spends about 150 ns per copy whatever its size below 8 KB, so stages are
// made of few large boxes.  The weight box lands with the 128-byte swizzle:
// block b of row r sits at 16-byte position b ^ (r % 8), so one ldmatrix.x2
// (eight rows of one block per matrix, no bank conflicts) hands lane (g, t)
// the 32-bit word t of weight rows g and g + 8 of a 16-row tile: exactly
// the bytes of its B fragments for both 8-row halves.  Both operands use
// one permutation of the 32 k positions of a block: in MMA step 0, k slots
// 2t, 2t+1 hold elements 4t, 4t+2 (low nibbles of bytes 0 and 2 of word t)
// and slots 2t+8, 2t+9 hold 4t+1, 4t+3 (bytes 1 and 3); step 1 the same
// elements plus 16 (the high nibbles).
//
// Consumers.  Consumer warp w takes block w % 8 of every stage, for the
// tiles of parity w / 8: it loads that block's activation fragments once
// per stage and reuses them for each of its (up to 5) tiles, whose
// accumulators stay in registers across the stages.  K-parts and stages
// are whole 8-block chunks, so a stage only runs past its part at the end
// of a row, where the copy reads zeros and the fragments are zero.
//
// K-split.  For large K the activations of a whole row do not fit in shared
// memory as fp16 fragments, so K is cut into P parts (P <= 8) and the P CTAs
// of a thread-block cluster take one part each of the same row range.  At
// the end of a round of stages each warp leaves one partial per tile, the
// CTA sums the 8 partials of a tile in block order, and after a cluster
// barrier CTA p adds the P CTAs' tile sums, in rank order, for the tiles
// with index = p mod P, reading the others through distributed shared
// memory.  The summation order is fixed by the launch shape: deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstdlib>

#include "mlq_device.cuh"
#include "mlq_launch.h"
#include "mma_frag.cuh"

namespace mlq {

constexpr int kMcConsumers = 16;                 // warps
constexpr int kMcThreads = kMcConsumers * 32;
constexpr int kMcMaxSlots = 12;                  // stages in the ring, at most (at least 4)
constexpr int kMcFirst = 4;                      // stages copied before the activations are staged (<= 4 slots)
constexpr int kMcChunk = 8;                      // blocks per stage (128 bytes of a Q4_0 row)
constexpr int kMcMaxRows = 160;                  // rows per round (tensor box height)
constexpr int kMcMaxTpw = kMcMaxRows / 32;       // tiles of one parity in a round
constexpr int kMcMaxPartF16 = 64;                // blocks of activations per CTA: fp16 fragments
constexpr int kMcMaxPart = 96;                   //   int8 words
// bytes of one block's activations, and blocks per CTA, of each form
template <bool I8> __host__ __device__ constexpr int mc_xblock() { return I8 ? 512 : 1024; }
template <bool I8> __host__ __device__ constexpr int mc_max_part() { return I8 ? kMcMaxPart : kMcMaxPartF16; }
constexpr int kMcXdBlock = 128;                  // (dx_g, dx_g, dx_g+8, dx_g+8) for g < 8
constexpr int kMcXcBlock = 128;                  // -(C_g, C_g, C_g+8, C_g+8) for g < 8
constexpr int kMcXRaw = 16 * (kQK + 4);          // raw activation bytes and scale per block
constexpr int kMcTileBytes = 1024;               // one warp's partial (or sum) of one tile
constexpr int kMcMaxCluster = 8;
constexpr int kMcSmemLimit = 227 * 1024 - 256;   // dynamic shared memory, leaving room for the barriers
static_assert(kMcConsumers == 2 * kMcChunk, "two warps per block of a stage");

struct McArgs {
  float *Y;
  int *status;
  unsigned long long wait_ns;
  int ldy;
  int nb;
  int M;
  int r0, r1;
  int P;         // K-parts = CTAs per cluster
  int G;         // clusters
  int units;     // 8-row units in [r0, r1), split over the clusters
  int H;         // rows per round = tensor box height (multiple of 8, <= kMcMaxRows)
  int xblocks;   // activation blocks held per CTA (largest part, whole chunks)
  int slot_q;    // bytes of a stage's weight box, 1024-aligned
  int slot_d;    // bytes of a stage's scale box, 128-aligned
  int slots;     // stages in the ring
  int ring;      // bytes of the ring area
  int xraw;      // offset of the raw activations: in ring slots kMcFirst.. or after the fragments
  int parts;     // offset of the partials and tile sums: 0 (they reuse the ring) or their own area
  int early;     // weights are not written by earlier queued work: copy before the wait
  int refill_lag;  // 0: refill the previous stage's slot before computing a stage; 1: the one before
};

struct McParams {
  CUtensorMap wq;  // Q4_0 bytes: rows x (nb * 16), box H rows x 128 B, 128-byte swizzle
  CUtensorMap wd;  // scales: rows x nb floats, box H rows x 8
  CUtensorMap xq;  // activations: M rows x nb blocks x 4 8-byte elements, box 16 x one part x 4
  CUtensorMap xd;  // their scales: M x nb floats, box 16 rows x one part
  McArgs a;
};

// ---- cluster, copy and shared-memory helpers --------------------------------
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return static_cast<int>(r);
}
// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it are visible to reads after it, cluster-wide.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The same without ordering: only that every thread of the cluster got here.
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile(
      "barrier.cluster.arrive.relaxed.aligned;\n\t"
      "barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local, int rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}
// 2-D tensor copy global -> shared, completion counted in bytes on `bar`.
// x is the innermost coordinate (bytes for the weight map, floats for the
// scale map; 16-byte aligned in both), y the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 3-D tensor copy global -> shared: coordinates (x innermost, y, z).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses (and
// those made visible to it) before its later tensor copies.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
// Bounded wait that also gives up once another warp of the CTA has aborted.
__device__ __forceinline__ bool mc_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
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

// d = A * B + C (C a quad of start values) and d += A * B.
__device__ __forceinline__ void mma_from(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1,
                                         const float4 &c) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z),
        "f"(c.w));
}
__device__ __forceinline__ void mma_acc(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// The lane's A fragments of one block from its four biased int8 words
// (row g: words t, t + 4; row g + 8: words t, t + 4): step 0 holds x, step 1
// x / 16.  A biased byte u = x + 128 placed in the mantissa of 1024 is the
// fp16 value 1024 + u; subtracting 1152 gives x, and (1024 + u) / 16 - 72 =
// x / 16 in one fused multiply-add -- (1024 + u) / 16 has 1/16 steps below
// 80, which fp16 holds, so both are exact.
__device__ __forceinline__ void raw_to_frags(const uint4 &w, uint4 &f0, uint4 &f1) {
  const __half2 sixteenth = __half2half2(__ushort_as_half(0x2C00));
  const __half2 m72 = __half2half2(__ushort_as_half(0xD480));  // -72
  auto place = [](uint32_t biased, uint32_t sel) {
    uint32_t v;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(v) : "r"(biased), "r"(0x64646464u), "r"(sel));
    return v;
  };
  auto lo = [&](uint32_t biased, uint32_t sel) {  // x
    const uint32_t v = place(biased, sel);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&v), __half2half2(__ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t *>(&r);
  };
  auto hi = [&](uint32_t biased, uint32_t sel) {  // x / 16
    const uint32_t v = place(biased, sel);
    const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&v), sixteenth, m72);
    return *reinterpret_cast<const uint32_t *>(&r);
  };
  f0.x = lo(w.x, 0x4240u);  // row g,     elements 4t, 4t+2
  f0.y = lo(w.z, 0x4240u);  // row g + 8
  f0.z = lo(w.x, 0x4341u);  // row g,     elements 4t+1, 4t+3
  f0.w = lo(w.z, 0x4341u);  // row g + 8
  f1.x = hi(w.y, 0x4240u);  // the same, elements + 16, over 16
  f1.y = hi(w.w, 0x4240u);
  f1.z = hi(w.y, 0x4341u);
  f1.w = hi(w.w, 0x4341u);
}

// The B fragments of one weight word (see the header comment): step 0,
// the low nibbles of bytes {0, 2} and {1, 3} as 1024 + n; step 1, the high
// nibbles in place as 1024 + 16 n.
__device__ __forceinline__ void word_to_frags(uint32_t w, uint32_t (&s0)[2], uint32_t (&s1)[2]) {
  const uint32_t w8 = w >> 8;
  s0[0] = (w & 0x000F000Fu) | 0x64006400u;
  s0[1] = (w8 & 0x000F000Fu) | 0x64006400u;
  s1[0] = (w & 0x00F000F0u) | 0x64006400u;
  s1[1] = (w8 & 0x00F000F0u) | 0x64006400u;
}

// acc(2) += (d(2) * dw(2)) * dx(2), each product rounded as in the
// definition ((sumi * dw) * dx), the accumulate fused.
__device__ __forceinline__ void scale_acc_pair(unsigned long long &acc, float d0, float d1, float dw0,
                                               float dw1, unsigned long long dx2) {
  unsigned long long t;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(pack2(d0, d1)), "l"(pack2(dw0, dw1)));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(t), "l"(dx2));
}

// One stage of a warp: block jw of the stage for its NT tiles 2i + par.
template <int NT>
__device__ __forceinline__ void stage_tiles(unsigned long long (&acc)[kMcMaxTpw][2][2], uint32_t sq,
                                            const float *sd, int jw, int par, int lane, int t,
                                            const uint4 &xa, const uint4 &xb, const ulonglong2 &dx,
                                            const float4 &cc) {
  const int lrow = lane & 15;  // ldmatrix rows: lane i < 16 -> row i of the tile (half i / 8)
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int tau = 2 * i + par;
    const int row = tau * 16 + lrow;
    uint32_t w[2];
    ldmatrix_x2(w, sq + row * 128 + ((jw ^ (row & 7)) << 4));
    const float *sr = sd + (tau * 16 + 2 * t) * kMcChunk + jw;
    const float dw[4] = {sr[0], sr[kMcChunk], sr[8 * kMcChunk], sr[9 * kMcChunk]};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t s0[2], s1[2];
      word_to_frags(w[h], s0, s1);
      float d[4];
      mma_from(d, xa, s0[0], s0[1], cc);
      mma_acc(d, xb, s1[0], s1[1]);
      scale_acc_pair(acc[i][h][0], d[0], d[1], dw[2 * h], dw[2 * h + 1], dx.x);
      scale_acc_pair(acc[i][h][1], d[2], d[3], dw[2 * h], dw[2 * h + 1], dx.y);
    }
  }
}

template <bool I8>
__global__ void __launch_bounds__(kMcThreads, 1)
    gemm_q4_mma_cluster_kernel(const __grid_constant__ McParams prm) {
  constexpr int kMcXfBlock = mc_xblock<I8>();
  constexpr int kMcXTasks = mc_max_part<I8>() * 32 / (kMcConsumers * 32);
  const McArgs &a = prm.a;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMcMaxSlots];
  __shared__ __align__(8) uint64_t empty_bar[kMcMaxSlots];
  __shared__ __align__(8) uint64_t x_bar;
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int p = cluster_rank();
  const int c = cluster_index();
  // K-part: whole 8-block chunks [C p / P, C (p + 1) / P) of the C chunks
  const int nchunks = (a.nb + kMcChunk - 1) / kMcChunk;
  const int c0 = nchunks * p / a.P, c1 = nchunks * (p + 1) / a.P;
  const int kb0 = c0 * kMcChunk;
  const int cp = c1 - c0;  // stages per round
  // this cluster's rows: [row_lo, row_hi), cut at 8-row units
  const int row_lo = a.r0 + 8 * static_cast<int>(static_cast<long long>(a.units) * c / a.G);
  const int row_hi =
      min(a.r1, a.r0 + 8 * static_cast<int>(static_cast<long long>(a.units) * (c + 1) / a.G));
  const int rounds = (row_hi - row_lo + a.H - 1) / a.H;

  // shared memory: [ring (weight boxes, then scale boxes) | fragments | scale pairs | start
  // values | (raw activations and scales, unless in ring slots kMcFirst..) | (partials)]
  const int S = a.slots;
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringq_s = base_s, ringd_s = base_s + S * a.slot_q;
  const float *ringd = reinterpret_cast<const float *>(base + S * a.slot_q);
  uint8_t *xf = base + a.ring;
  uint8_t *xdx = xf + static_cast<size_t>(a.xblocks) * kMcXfBlock;
  uint8_t *xcc = xdx + static_cast<size_t>(a.xblocks) * kMcXdBlock;
  uint8_t *xraw = base + a.xraw;  // 16 rows x xblocks x 32 B
  const float *xdraw = reinterpret_cast<const float *>(xraw + 16 * a.xblocks * kQK);  // 16 x xblocks

  if (rounds <= 0) return;  // the whole cluster has no rows

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kMcConsumers);
    }
    mbar_init(smem_addr(&x_bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // Thread 0 copies the stages in order: stage n is stage k = n % cp of round
  // n / cp (rows y..y+H, blocks kb0 + 8k).  A slot is refilled once all
  // warps released the stage it held.  With a separate partials area the
  // copies run ahead into the next round while this one is reduced.
  const int total = rounds * cp;
  uint32_t issued = 0;  // stages copied (thread 0)
  auto issue = [&](int k, int y) -> bool {
    const int slot = issued % S;
    if (static_cast<int>(issued) >= S) {
      const uint32_t n = issued - S;  // the stage that held this slot
      if (!mc_wait(smem_addr(&empty_bar[slot]), (n / S) & 1u, abort_v, a.wait_ns)) {
        if (atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        return false;
      }
    }
    const uint32_t bar = smem_addr(&full_bar[slot]);
    const int x = kb0 + k * kMcChunk;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(a.H * kMcChunk * (16 + 4)));  // both boxes
    tma_load_2d(ringq_s + slot * a.slot_q, &prm.wq, x * 16, y, bar);
    tma_load_2d(ringd_s + slot * a.slot_d, &prm.wd, x, y, bar);
    ++issued;
    return true;
  };
  auto issue_next = [&]() -> bool {
    return issue(static_cast<int>(issued) % cp, row_lo + static_cast<int>(issued) / cp * a.H);
  };
  // Stages 0..kMcFirst-1 go first (slots kMcFirst.. may hold the raw
  // activations until they are converted), the rest of the ring after.
  if (tid == 0 && a.early)  // static weights: before the dependency wait
    while (static_cast<int>(issued) < min(total, kMcFirst) && issue_next()) {
    }

  griddep_wait();  // the activations (and, unless static, the weights) come from earlier work
  griddep_launch_dependents();

  if (tid == 0) {
    // the activations first: an SM serves its reads in order
    const uint32_t xb = smem_addr(&x_bar);
    mbar_arrive_expect_tx(xb, static_cast<uint32_t>(16 * a.xblocks * (kQK + 4)));
    tma_load_3d(smem_addr(xraw), &prm.xq, 0, kb0, 0, xb);  // lands as [16 rows][xblocks][32 bytes]
    tma_load_2d(smem_addr(xdraw), &prm.xd, kb0, 0, xb);
    while (static_cast<int>(issued) < min(total, kMcFirst) && issue_next()) {
    }
  }
  if (!warp_wait([&] { return mc_wait(smem_addr(&x_bar), 0, abort_v, a.wait_ns); })) {
    if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
  }
  if (!*abort_v) {
    // Activations -> fragment order.  Task (block j, lane (gg, tt)): words
    // tt and tt + 4 of rows gg and gg + 8, biased to unsigned, are the
    // lane's a0..a3 of both MMA steps: kept as int8 words (I8; raw_to_frags
    // converts them per stage) or converted now.  The four lanes of a row
    // group add up the block halves for the start values.  Rows past M and
    // blocks past the row end were copied as zeros.
#pragma unroll
    for (int q = 0; q < kMcXTasks; ++q) {
      const int i = tid + q * kMcThreads, j = i >> 5, ln = i & 31, gg = ln >> 2, tt = ln & 3;
      const int jj = j < a.xblocks ? j : 0;  // whole warps share j: the shuffles stay converged
      const uint8_t *r0 = xraw + static_cast<size_t>(gg) * a.xblocks * kQK + jj * kQK + 4 * tt;
      const uint8_t *r1 = r0 + static_cast<size_t>(8) * a.xblocks * kQK;
      const uint32_t lo0 = *reinterpret_cast<const uint32_t *>(r0);
      const uint32_t hi0 = *reinterpret_cast<const uint32_t *>(r0 + 16);
      const uint32_t lo1 = *reinterpret_cast<const uint32_t *>(r1);
      const uint32_t hi1 = *reinterpret_cast<const uint32_t *>(r1 + 16);
      int sl0 = __dp4a(static_cast<int>(lo0), 0x01010101, 0), sh0 = __dp4a(static_cast<int>(hi0), 0x01010101, 0);
      int sl1 = __dp4a(static_cast<int>(lo1), 0x01010101, 0), sh1 = __dp4a(static_cast<int>(hi1), 0x01010101, 0);
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        sl0 += __shfl_xor_sync(0xffffffffu, sl0, o);
        sh0 += __shfl_xor_sync(0xffffffffu, sh0, o);
        sl1 += __shfl_xor_sync(0xffffffffu, sl1, o);
        sh1 += __shfl_xor_sync(0xffffffffu, sh1, o);
      }
      if (j < a.xblocks) {
        const uint4 words =
            make_uint4(lo0 ^ 0x80808080u, hi0 ^ 0x80808080u, lo1 ^ 0x80808080u, hi1 ^ 0x80808080u);
        uint8_t *dst = xf + static_cast<size_t>(j) * kMcXfBlock + ln * 16;
        if (I8) {
          *reinterpret_cast<uint4 *>(dst) = words;
        } else {
          uint4 f0, f1;
          raw_to_frags(words, f0, f1);
          *reinterpret_cast<uint4 *>(dst) = f0;
          *reinterpret_cast<uint4 *>(dst + 512) = f1;
        }
        if (tt == 0) {
          const float d0 = xdraw[gg * a.xblocks + j], d1 = xdraw[(gg + 8) * a.xblocks + j];
          *reinterpret_cast<float4 *>(xdx + static_cast<size_t>(j) * kMcXdBlock + gg * 16) =
              make_float4(d0, d0, d1, d1);
          const float n0 = -static_cast<float>(1032 * sl0 + 72 * sh0);
          const float n1 = -static_cast<float>(1032 * sl1 + 72 * sh1);
          *reinterpret_cast<float4 *>(xcc + static_cast<size_t>(j) * kMcXcBlock + gg * 16) =
              make_float4(n0, n0, n1, n1);
        }
      }
    }
  }
  __syncthreads();

  uint32_t used = 0;  // stages consumed, over all rounds
  const int par = warp >> 3, jw = warp & 7;

  for (int r = 0; r < rounds; ++r) {
    const int rlo = row_lo + r * a.H;
    const int rhi = min(row_hi, rlo + a.H);  // rows of this round
    const int tiles = (rhi - rlo + 15) / 16;
    // copies may run up to this stage (exclusive), S - 1 ahead of the one consumed
    const int limit = a.parts != 0 ? total : (r + 1) * cp;
    if (tid == 0 && (r == 0 || a.parts == 0)) {
      if (r > 0) fence_proxy_async();  // the ring held partials and tile sums last round
      while (static_cast<int>(issued) < min(limit, r * cp + S - 1) && !*abort_v && issue_next()) {
      }
    }

    // acc[i][h][e]: tile 2i + (warp / 8), rows 2t, 2t+1 of half h, m = g + 8e
    unsigned long long acc[kMcMaxTpw][2][2];
#pragma unroll
    for (int i = 0; i < kMcMaxTpw; ++i) acc[i][0][0] = acc[i][0][1] = acc[i][1][0] = acc[i][1][1] = 0ull;
    const int nt = (tiles - par + 1) / 2;  // this warp's tiles
    for (int k = 0; k < cp; ++k, ++used) {
      const int slot = used % S;
      if (*abort_v) continue;
      const uint32_t fb = smem_addr(&full_bar[slot]);
      const uint32_t ph = (used / S) & 1u;
      if (!warp_wait([&] { return mc_wait(fb, ph, abort_v, a.wait_ns); })) {
        if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        continue;
      }
      // refill the slot of the stage before the previous one (all warps
      // have released it) before this one is computed: S - 2 stages stay in
      // flight (S - 1 with refill_lag = 0: the previous stage's slot)
      if (tid == 0 && static_cast<int>(issued) < min(limit, static_cast<int>(used) + S - a.refill_lag) &&
          !*abort_v)
        issue_next();
      const int jb = k * kMcChunk + jw;  // part-local block
      uint4 xa, xb;
      if (I8) {
        raw_to_frags(*reinterpret_cast<const uint4 *>(xf + static_cast<size_t>(jb) * kMcXfBlock + lane * 16), xa,
                     xb);
      } else {
        xa = *reinterpret_cast<const uint4 *>(xf + static_cast<size_t>(jb) * kMcXfBlock + lane * 16);
        xb = *reinterpret_cast<const uint4 *>(xf + static_cast<size_t>(jb) * kMcXfBlock + 512 + lane * 16);
      }
      const ulonglong2 dx =
          *reinterpret_cast<const ulonglong2 *>(xdx + static_cast<size_t>(jb) * kMcXdBlock + g * 16);
      const float4 cc = *reinterpret_cast<const float4 *>(xcc + static_cast<size_t>(jb) * kMcXcBlock + g * 16);
      const uint32_t sq = ringq_s + slot * a.slot_q;
      const float *sd = ringd + slot * (a.slot_d / 4);
      switch (nt) {
        case 5: stage_tiles<5>(acc, sq, sd, jw, par, lane, t, xa, xb, dx, cc); break;
        case 4: stage_tiles<4>(acc, sq, sd, jw, par, lane, t, xa, xb, dx, cc); break;
        case 3: stage_tiles<3>(acc, sq, sd, jw, par, lane, t, xa, xb, dx, cc); break;
        case 2: stage_tiles<2>(acc, sq, sd, jw, par, lane, t, xa, xb, dx, cc); break;
        case 1: stage_tiles<1>(acc, sq, sd, jw, par, lane, t, xa, xb, dx, cc); break;
        default: break;
      }
      __syncwarp();  // every lane is done with the stage
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[slot]));
    }
    if (tid == 0 && *abort_v) {
      // copies still landing after an abort (bounded)
      for (uint32_t n = static_cast<int>(issued) > S ? issued - S : 0; n < issued; ++n)
        mbar_wait_bounded(smem_addr(&full_bar[n % S]), (n / S) & 1u, kDrainWaitNs);
      mbar_wait_bounded(smem_addr(&x_bar), 0, kDrainWaitNs);
    }
    __syncthreads();
    if (*abort_v) used = issued = 0;  // results are void; keep the counters simple

    // Partials: warp w, tile slot i -> 1 KB at (w * tpw + i), in the ring
    // or their own area.
    const int tpw = (tiles + 1) / 2;
    uint8_t *parts = base + a.parts;
#pragma unroll
    for (int i = 0; i < kMcMaxTpw; ++i) {
      if (i < nt) {
        float v[8];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            asm("mov.b64 {%0, %1}, %2;" : "=f"(v[4 * h + 2 * e]), "=f"(v[4 * h + 2 * e + 1]) : "l"(acc[i][h][e]));
        float4 *dst = reinterpret_cast<float4 *>(parts + (warp * tpw + i) * kMcTileBytes + lane * 32);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
    __syncthreads();

    // Per tile: the 8 partials (blocks 0..7 of each stage), in block order.
    float4 sum[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int idx = tid + q * kMcThreads, tau = idx >> 6, f = idx & 63;
      sum[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (tau < tiles) {
        const int w0 = (tau & 1) * kMcChunk, i = tau >> 1;
#pragma unroll
        for (int j = 0; j < kMcChunk; ++j) {
          const float4 v = *reinterpret_cast<const float4 *>(parts + ((w0 + j) * tpw + i) * kMcTileBytes + f * 16);
          sum[q].x += v.x;
          sum[q].y += v.y;
          sum[q].z += v.z;
          sum[q].w += v.w;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int idx = tid + q * kMcThreads;
      if ((idx >> 6) < tiles) *reinterpret_cast<float4 *>(parts + idx * 16) = sum[q];
    }
    cluster_sync();

    // Tiles tau = p mod P: the P CTAs' sums in rank order, then the stores.
    // Tile sum layout: lane (gg, tt) -> 8 floats, half h, m = gg + 8e,
    // rows 8h + 2tt + {0, 1}.
    for (int tau = p + a.P * (tid >> 6); tau < tiles; tau += a.P * (kMcThreads / 64)) {
      const int f = tid & 63, idx = tau * 64 + f;
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int q = 0; q < a.P; ++q) {
        const float4 u = ld_cluster_f4(base_s + a.parts + idx * 16, q);
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
      }
      const int ln = f >> 1, h = f & 1, gg = ln >> 2, tt = ln & 3;
      const int row = rlo + tau * 16 + 8 * h + 2 * tt;
      const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = gg + 8 * (e >> 1), rw = row + (e & 1);
        if (m < a.M && rw < rhi && in_bounds(rw >= a.r0 && rw < a.r1, a.status))
          a.Y[static_cast<size_t>(m) * a.ldy + rw] = vals[e];
      }
    }
    cluster_sync_relaxed();  // no CTA reuses the area of its tile sums while others read them
  }
}

// ---- host side ---------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

static bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *ptr, uint64_t inner,
                      uint64_t rows, uint64_t stride, uint32_t box_inner, uint32_t box_rows,
                      CUtensorMapSwizzle swz) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {stride};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(map, type, 2, const_cast<void *>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The activations as M rows x nb blocks x 4 8-byte elements, box 16 rows x
// xblocks x 4: the part lands densely as [16][xblocks][32 bytes], the
// layout of a 2-D box of one row part, while every box dimension stays
// within the 256-element limit of a tensor copy (a 2-D box of xblocks * 4
// elements would exceed it beyond 64 blocks).  Rows past M read as zeros.
static bool encode_act_3d(CUtensorMap *map, const void *xq, int nb, int M, int xblocks) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {kQK / 8, static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[2] = {kQK, static_cast<cuuint64_t>(nb) * kQK};
  const cuuint32_t box[3] = {kQK / 8, static_cast<cuuint32_t>(xblocks), 16};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(xq), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of P CTAs that fit on the device at once, by (P, activation chunks).
static std::atomic<int> g_mc_clusters[2][kMcMaxCluster + 1][kMcMaxPart / kMcChunk + 1];

// Shared-memory layout of a launch (byte offsets from the 1024-aligned base).
struct McLayout {
  int slots, ring, xraw, parts;
  size_t bytes;  // dynamic shared memory, alignment slack included
};
static bool mc_layout(int H, int xblocks, int xblock_bytes, bool multi_round, McLayout *L) {
  const int slot_q = (H * kMcChunk * 16 + 1023) / 1024 * 1024;
  const int slot_d = (H * kMcChunk * 4 + 127) / 128 * 128;
  const int tiles = (H + 15) / 16;
  const int parts = kMcConsumers * ((tiles + 1) / 2) * kMcTileBytes;
  const int xfixed = xblocks * (xblock_bytes + kMcXdBlock + kMcXcBlock);
  const int raw = xblocks * kMcXRaw;
  // most slots first; partials in their own area (several rounds) when it fits
  for (int own = multi_round ? 1 : 0; own >= 0; --own) {
    for (int S = kMcMaxSlots; S >= 4; --S) {
      const bool alias = (S - kMcFirst) * slot_q >= raw;
      const int stages = S * (slot_q + slot_d);
      const int ring = own ? stages : (stages > parts ? stages : parts);
      const size_t bytes = 1024 + static_cast<size_t>(ring) + xfixed + (alias ? 0 : raw) + (own ? parts : 0);
      if (bytes > static_cast<size_t>(kMcSmemLimit)) continue;
      L->slots = S;
      L->ring = ring;
      L->xraw = alias ? kMcFirst * slot_q : ring + xfixed;
      L->parts = own ? ring + xfixed + (alias ? 0 : raw) : 0;
      L->bytes = bytes;
      return true;
    }
  }
  return false;
}

cudaError_t launch_gemm_q4_mma_cluster(const LaunchCtx &ctx, const void *wq, const float *wd,
                                       int nb, const int8_t *xq, const float *xd, int M, float *Y,
                                       int ldy, int r0, int r1, int rows) {
  const int n = r1 - r0;
  if (n <= 0 || M <= 0) return cudaSuccess;
  const int nchunks = (nb + kMcChunk - 1) / kMcChunk;
  // the fewest K-parts whose activations fit (MLQ_MMA_CLUSTER=P asks for more: A/B timing)
  static const int p_env = [] {
    const char *e = std::getenv("MLQ_MMA_CLUSTER");
    return e != nullptr ? std::atoi(e) : 0;
  }();
  // the int8 form only where it needs fewer K-parts than fp16 fragments
  // (MLQ_MMA_I8=1 / 0 forces one form: A/B timing)
  static const int i8_env = [] {
    const char *e = std::getenv("MLQ_MMA_I8");
    return e == nullptr ? -1 : (e[0] == '1' ? 1 : 0);
  }();
  const int p_f16 = (nchunks * kMcChunk + kMcMaxPartF16 - 1) / kMcMaxPartF16;
  const int p_i8 = (nchunks * kMcChunk + kMcMaxPart - 1) / kMcMaxPart;
  const bool i8 = i8_env >= 0 ? i8_env == 1 : p_i8 < p_f16;
  const int p_min = i8 ? p_i8 : p_f16;
  const int P = p_env > p_min && p_env <= kMcMaxCluster && p_env <= nchunks ? p_env : p_min;
  // the scale map needs 16-byte row strides
  if (M > 16 || P > kMcMaxCluster || nb % 4 != 0) return cudaErrorNotSupported;
  McParams prm;
  McArgs &a = prm.a;
  a.Y = Y;
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  a.ldy = ldy;
  a.nb = nb;
  a.M = M;
  a.r0 = r0;
  a.r1 = r1;
  a.P = P;
  a.early = ctx.early_weights ? 1 : 0;
  // Thread 0 computes too: refilling the slot of the stage before the
  // previous one, rather than of the previous one, spares it a wait for the
  // slowest warp (11008 x 4096 M = 16: 19.6 -> 19.3 us); MLQ_MMA_REFILL_LAG=0
  // refills the previous stage's slot.
  static const int lag_env = [] {
    const char *e = std::getenv("MLQ_MMA_REFILL_LAG");
    return e != nullptr && e[0] == '0' ? 0 : 1;
  }();
  a.refill_lag = lag_env;
  const int part_chunks = (nchunks + P - 1) / P;
  a.xblocks = part_chunks * kMcChunk;
  a.units = (n + 7) / 8;
  auto kern = i8 ? gemm_q4_mma_cluster_kernel<true> : gemm_q4_mma_cluster_kernel<false>;
  static const cudaError_t attr = [] {
    const cudaError_t e0 = cudaFuncSetAttribute(gemm_q4_mma_cluster_kernel<false>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMcSmemLimit);
    const cudaError_t e1 = cudaFuncSetAttribute(gemm_q4_mma_cluster_kernel<true>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMcSmemLimit);
    return e0 != cudaSuccess ? e0 : e1;
  }();
  if (attr != cudaSuccess) return attr;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(P);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kMcThreads);
  cfg.stream = ctx.stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;

  int clusters = g_mc_clusters[i8][P][part_chunks].load(std::memory_order_relaxed);
  if (clusters == 0) {
    // with the most shared memory a launch may take
    cfg.gridDim = dim3(static_cast<unsigned>(P * ctx.num_sms));
    cfg.dynamicSmemBytes = kMcSmemLimit;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      return cudaErrorNotSupported;
    }
    g_mc_clusters[i8][P][part_chunks].store(clusters, std::memory_order_relaxed);
  }
  a.G = clusters < a.units ? clusters : a.units;
  // rows per round: a cluster's share in the fewest rounds of equal height
  const int per_cluster = 8 * ((a.units + a.G - 1) / a.G);
  const int nrounds = (per_cluster + kMcMaxRows - 1) / kMcMaxRows;
  a.H = 8 * ((per_cluster / 8 + nrounds - 1) / nrounds);
  a.slot_q = (a.H * kMcChunk * 16 + 1023) / 1024 * 1024;
  a.slot_d = (a.H * kMcChunk * 4 + 127) / 128 * 128;
  // with several rounds, partials in their own area when it fits: the next
  // round's copies then overlap this round's reduction
  McLayout L;
  if (!mc_layout(a.H, a.xblocks, i8 ? mc_xblock<true>() : mc_xblock<false>(), nrounds > 1, &L))
    return cudaErrorNotSupported;
  a.slots = L.slots;
  a.ring = L.ring;
  a.xraw = L.xraw;
  a.parts = L.parts;
  const size_t rowq = static_cast<size_t>(nb) * 16;
  if (!encode_2d(&prm.wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, rowq, static_cast<uint64_t>(rows), rowq,
                 kMcChunk * 16, static_cast<uint32_t>(a.H), CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&prm.wd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, wd, static_cast<uint64_t>(nb),
                 static_cast<uint64_t>(rows), static_cast<uint64_t>(nb) * 4, kMcChunk,
                 static_cast<uint32_t>(a.H), CU_TENSOR_MAP_SWIZZLE_NONE) ||
      // activations: a part of 16 rows (rows past M read as zeros), 8-byte elements
      !encode_act_3d(&prm.xq, xq, nb, M, a.xblocks) ||
      !encode_2d(&prm.xd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xd, static_cast<uint64_t>(nb),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(nb) * 4,
                 static_cast<uint32_t>(a.xblocks), 16, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorNotSupported;
  cfg.gridDim = dim3(static_cast<unsigned>(a.G * P));
  cfg.dynamicSmemBytes = L.bytes;
  cfg.numAttrs = ctx.pdl ? 2 : 1;
  diag_note("mma_cluster: M=%d K-parts=%d clusters=%d rows/round=%d rounds=%d slots=%d activations=%s", M, P,
            a.G, a.H, nrounds, a.slots, i8 ? "int8" : "fp16");
  diag_launch_cfg(reinterpret_cast<const void *>(kern), cfg);
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace mlq
