// gemm_umma.cu -- batched small-M decode (M up to 16) on the fifth-generation
// tensor cores: tcgen05.mma with the weights and the block sums in tensor
// memory (TMEM).
//
// Computes (page "ONNX Runtime", "6. Panel loop (pre-TCM)": batched decode,
// M rows against 4096 x 11008; definitions of the page "Legacy-ISA ML
// Inference Runtime -- Design Spec", Sec. 4):
//   Y[m*ldy + r] = sum_b ((float)sumi(m, r, b) * dw(r, b)) * dx(m, b),
//   sumi(m, r, b) = sum_j (nibble(r, b, j) - 8) * qx(m, 32b + j).
//
// Operand roles.  The MMA's M dimension (128 TMEM lanes) is up to 128 weight
// rows, N = 16 the activation rows, K = 16 per instruction, fp16 operands and
// fp32 accumulators (kind::f16; sm_103a has no int8 kind).  A block of 32
// columns takes two instructions into its own 16-column accumulator, so the
// per-block sums stay separate and are scaled one by one as the definition
// asks.
//
// Exact block sums.  A converter thread owns one weight row (one TMEM lane)
// and turns each 32-bit word of nibbles into four fp16 pairs with bit
// operations only: a low nibble n becomes 1024 + n, a high nibble, left in
// place, 1024 + 16 n.  The activations (the B operand, staged once per CTA
// in shared memory) hold x at the low-nibble positions and x / 16 at the
// high ones, both exact in fp16, permuted the same way as the weight words.
// The accumulator then holds sum n*x + 1024*Sx_lo + 64*Sx_hi, an integer
// below 2^23 (Sx_lo, Sx_hi: the block's activation sums over its two
// halves), and sumi = acc - (1032*Sx_lo + 72*Sx_hi) exactly, subtracted in
// fp32 before the scaling.
//
// Pipeline (576 threads, one CTA per SM, all 512 TMEM columns).  A stage of
// the shared-memory ring is (up to 128 rows) x 8 blocks; each half of it
// (4 blocks, a sub-stage) goes through one of four TMEM buffers, each 64
// columns of A (fp16 weights) and 64 columns of D (block sums):
//  * warp 16, one thread: tensor copies of the stage's weights (128-byte
//    swizzle) and scales into the ring;
//  * warps 0-7 (converters): warp w owns TMEM lanes 32 (w % 4) .. + 31 and
//    half w / 4 of every stage: it reads its rows' words and scales, frees
//    the ring slot, and stores the fp16 weights into the sub-stage's A;
//  * warp 17 (MMA): 8 MMAs per sub-stage, ordered so that consecutive ones
//    write different accumulators, then one commit;
//  * warps 8-15 (epilogue): per sub-stage, the 4 block sums of each row,
//    ((acc - C) * dw) * dx accumulated with fused multiply-adds in
//    registers, one row and one half of the blocks per thread.
// While the first stages stream in, the epilogue and MMA warps stage the
// activations from global memory (the B operand, C, dx), so the converters
// and the copies do not wait for them.
//
// Measured on GB300 (globaltimer stamps per role): an M = 128, N = 16,
// K = 16 MMA with A in TMEM completes about 125 cycles after the previous
// one, whether or not the two write the same accumulator, so a stage's 16
// MMAs take about 1 us and the kernel streams 12-20 GB/s per SM: 28-34 us
// for the 11008 x 4096 and 4096 x 11008 Q4_0 products at M = 16, against
// 18-26 us for the mma.sync cluster kernel.  N = 16 (the activation rows)
// leaves the tensor cores mostly idle while each instruction still pays
// its full latency.  The dispatcher therefore takes this kernel only when
// asked (MLQ_GEMM_KERNEL=umma).
//
// K-split.  The 16 activation rows of a whole row of K do not fit in shared
// memory as fp16 for large K, so K is cut into P parts and the P CTAs of a
// thread-block cluster take one part each of the same rows.  Each epilogue
// thread leaves its row's 16 partial sums of every round (the cluster's
// rows, up to 128 per round) in shared memory; at the end the P CTAs
// signal each other through mbarriers in distributed shared memory, and
// CTA p adds the 2P partials (rank by rank, half by half) of the rows
// i with i mod P == p.  The summation order is fixed by the launch shape:
// deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstdlib>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

constexpr int kUmConvWarps = 8;                  // two per TMEM lane quarter
constexpr int kUmEpiWarps = 8;
constexpr int kUmProdWarp = 16;
constexpr int kUmMmaWarp = 17;
constexpr int kUmThreads = 576;
constexpr int kUmStageThreads = kUmEpiWarps * 32 + 32;  // stage the activations: epilogue + MMA warps
constexpr int kUmChunk = 8;                      // blocks per stage (128 bytes of a Q4_0 row)
constexpr int kUmSub = 4;                        // blocks per sub-stage
constexpr int kUmBufs = 4;                       // TMEM buffers
constexpr int kUmRows = 128;                     // rows per round: the TMEM lanes
constexpr int kUmMaxSlots = 16;
constexpr int kUmMaxPart = 64;                   // blocks of activations per CTA
constexpr int kUmBBlock = 1024;                  // B operand of one block: 2 K-steps x 16 rows x 16 fp16
constexpr int kUmCBlock = 64;                    // -(1032 Sx_lo + 72 Sx_hi) of the 16 rows
constexpr int kUmXdBlock = 64;                   // dx of the 16 rows
constexpr int kUmMaxCluster = 8;
constexpr int kUmSmemLimit = 227 * 1024 - 512;   // dynamic, leaving room for the static barriers
constexpr uint32_t kUmTmemCols = 512;            // A of buffer b at 64 b, D of buffer b at 256 + 64 b
// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A
// and B fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kUmIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
static_assert(kUmConvWarps == 8 && kUmEpiWarps == 8 && kUmChunk == 2 * kUmSub, "two halves per stage");
static_assert(kUmBufs * kUmSub * 16 * 2 == static_cast<int>(kUmTmemCols), "TMEM budget");

struct UmArgs {
  float *Y;
  const int8_t *xq;  // activations: M rows of nb * 32 bytes
  const float *xd;   // their scales: M rows of nb floats
  int *status;
  unsigned long long wait_ns;
  int ldy;
  int nb;
  int M;
  int r0, r1;
  int P;         // K-parts = CTAs per cluster
  int G;         // clusters
  int units;     // 8-row units in [r0, r1), split over the clusters
  int H;         // rows per round = tensor box height (multiple of 8, <= 128)
  int rounds;    // rounds of the busiest cluster (partials area)
  int xblocks;   // activation blocks held per CTA (largest part, whole chunks)
  int slot_q;    // bytes of a stage's weight box, 1024-aligned
  int slot_d;    // bytes of a stage's scale box, 128-aligned
  int slots;     // stages in the ring
  int ring;      // bytes of the ring area
  int early;     // weights are not written by earlier queued work: copy before the wait
  uint32_t lbo;  // B operand: byte offset between core matrices along K
  uint32_t sbo;  // B operand: byte offset between core matrices along N
};

struct UmParams {
  CUtensorMap wq;  // Q4_0 bytes: rows x (nb * 16), box H rows x 128 B, 128-byte swizzle
  CUtensorMap wd;  // scales: rows x nb floats, box H rows x 8
  UmArgs a;
};

// ---- cluster, copy and tensor-memory helpers ---------------------------------
__device__ __forceinline__ int um_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int um_cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ void um_cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t um_mapa(uint32_t local, int rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
__device__ __forceinline__ float4 um_ld_cluster_f4(uint32_t local, int rank) {
  const uint32_t remote = um_mapa(local, rank);
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}
// Arrive, with release at cluster scope, on the mbarrier at the same offset
// in the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ void um_arrive_remote(uint32_t local_bar, int rank) {
  const uint32_t remote = um_mapa(local_bar, rank);
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}
__device__ __forceinline__ bool um_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void um_tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void um_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Bounded wait (cluster-scope acquire when `cluster`) that also gives up once
// another warp of the CTA has aborted.
__device__ __forceinline__ bool um_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
                                        unsigned long long limit_ns, bool cluster = false) {
  if (limit_ns == 0) return false;
  auto probe = [&] { return cluster ? um_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (probe()) return true;
  const uint64_t t0 = sm_cycles(), lim = limit_cycles(limit_ns);
  for (;;) {
    if (probe()) return true;
    if (*abort_flag) return false;
    if (sm_cycles() - t0 > lim) return false;
  }
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (the tensor cores' operand reads).
__device__ __forceinline__ void fence_proxy_async_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive TMEM columns of the warp's 32 lanes (one lane per thread).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]),
      "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
      "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Load and wait in one statement: the registers are only read after the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// Shared-memory matrix descriptor: start address, the two core-matrix
// strides, the fixed version bits (46-48 = 0b001), no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// D[tmem] (+)= A[tmem] * B[smem]^T, 128 x 16 x 16, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(accumulate), "r"(kUmIdesc)
      : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ unsigned long long um_pack(uint32_t a, uint32_t b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ bool um_elect() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__global__ void __launch_bounds__(kUmThreads, 1)
    gemm_q4_umma_kernel(const __grid_constant__ UmParams prm) {
  const UmArgs &a = prm.a;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kUmMaxSlots];
  __shared__ __align__(8) uint64_t empty_bar[kUmMaxSlots];
  __shared__ __align__(8) uint64_t a_full[kUmBufs];    // converters stored sub-stage u's A (and dw)
  __shared__ __align__(8) uint64_t mma_done[kUmBufs];  // sub-stage u's MMAs completed
  __shared__ __align__(8) uint64_t d_empty[kUmBufs];   // the epilogue read sub-stage u's D (and dw)
  __shared__ __align__(8) uint64_t parts_ready;         // all P CTAs of the cluster left their partials
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p = um_cluster_rank();
  const int c = um_cluster_index();
  // K-part: whole 8-block chunks [C p / P, C (p + 1) / P) of the C chunks
  const int nchunks = (a.nb + kUmChunk - 1) / kUmChunk;
  const int c0 = nchunks * p / a.P, c1 = nchunks * (p + 1) / a.P;
  const int kb0 = c0 * kUmChunk;
  const int cp = c1 - c0;  // stages per round
  // this cluster's rows: [row_lo, row_hi), cut at 8-row units
  const int row_lo = a.r0 + 8 * static_cast<int>(static_cast<long long>(a.units) * c / a.G);
  const int row_hi =
      min(a.r1, a.r0 + 8 * static_cast<int>(static_cast<long long>(a.units) * (c + 1) / a.G));
  const int rounds = (row_hi - row_lo + a.H - 1) / a.H;
  if (rounds <= 0 || cp <= 0) return;  // the same for every CTA of the cluster

  // shared memory: [ring (weight boxes, then scale boxes) | B operand | -C | dx | dw of the
  // TMEM buffers | partials of every round and half]
  const int S = a.slots;
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringq_s = base_s, ringd_s = base_s + S * a.slot_q;
  const uint8_t *ringq = base;
  const float *ringd = reinterpret_cast<const float *>(base + S * a.slot_q);
  const uint32_t xb_s = base_s + a.ring;
  uint8_t *xbm = base + a.ring;
  float *negc = reinterpret_cast<float *>(xbm + static_cast<size_t>(a.xblocks) * kUmBBlock);
  float *dxs = negc + a.xblocks * 16;
  float *dwbuf = dxs + a.xblocks * 16;            // [kUmBufs][H][kUmSub]
  float *parts = dwbuf + kUmBufs * a.H * kUmSub;  // [rounds][2][H][16]
  const uint32_t parts_s = smem_addr(parts);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kUmConvWarps);
    }
    for (int b = 0; b < kUmBufs; ++b) {
      mbar_init(smem_addr(&a_full[b]), kUmConvWarps / 2);  // the four warps of one half
      mbar_init(smem_addr(&mma_done[b]), 1);
      mbar_init(smem_addr(&d_empty[b]), kUmEpiWarps / 2);
    }
    mbar_init(smem_addr(&parts_ready), kUmEpiWarps * a.P);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base_s)),
                 "r"(kUmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  um_cluster_sync();  // barriers initialised cluster-wide, TMEM address published
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  auto fail = [&] {
    if (atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
  };
  auto aborted = [&] { return __shfl_sync(0xffffffffu, *abort_v, 0) != 0; };  // warp-uniform

  // The producer copies stage n = (round n / cp, chunk n % cp) into slot
  // n % S once the converters freed the stage that held it.
  const int total = rounds * cp;
  const bool producer = warp == kUmProdWarp && lane == 0;
  uint32_t issued = 0;
  auto issue_next = [&]() -> bool {
    const int slot = issued % S;
    if (static_cast<int>(issued) >= S) {
      const uint32_t n = issued - S;
      if (!um_wait(smem_addr(&empty_bar[slot]), (n / S) & 1u, abort_v, a.wait_ns)) {
        fail();
        return false;
      }
    }
    const int k = static_cast<int>(issued) % cp;
    const int y = row_lo + static_cast<int>(issued) / cp * a.H;
    const int x = kb0 + k * kUmChunk;
    const uint32_t bar = smem_addr(&full_bar[slot]);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(a.H * kUmChunk * (16 + 4)));
    um_tma_2d(ringq_s + slot * a.slot_q, &prm.wq, x * 16, y, bar);
    um_tma_2d(ringd_s + slot * a.slot_d, &prm.wd, x, y, bar);
    ++issued;
    return true;
  };
  if (producer && a.early)  // static weights: before the dependency wait
    while (static_cast<int>(issued) < min(total, S) && issue_next()) {
    }

  griddep_wait();  // the activations (and, unless static, the weights) come from earlier work
  griddep_launch_dependents();

  // The B operand, -C and dx of this CTA's K-part, from global memory, by
  // the epilogue and MMA warps (thread ts of kUmStageThreads).  B task
  // (block j, row n, step s, K-core kc): the 16 bytes of k = 8kc..8kc+7,
  // i.e. elements 16s + 8kc + {0, 2, 1, 3, 4, 6, 5, 7} of the block (the
  // order of the converted weight words), as fp16, over 16 for s = 1.
  // Core matrix (kc, n / 8) of step s sits at 512 s + 128 kc + 256 (n / 8),
  // row n % 8 at 16 (n % 8) within it.  Rows past M and blocks past the
  // row end are zeros.
  auto stage_activations = [&](int ts) {
    // all of a thread's loads are issued before any is used: one memory
    // latency, not one per task
    constexpr int kQB = (kUmMaxPart * 64 + kUmStageThreads - 1) / kUmStageThreads;
    constexpr int kQC = (kUmMaxPart * 16 + kUmStageThreads - 1) / kUmStageThreads;
    const int nblk = cp * kUmChunk;
    uint2 raw[kQB];
#pragma unroll
    for (int qb = 0; qb < kQB; ++qb) {
      const int t = ts + qb * kUmStageThreads;
      const int n = ((t >> 5) & 1) * 8 + (t & 7), kc = (t >> 3) & 1, s = (t >> 4) & 1, kb = kb0 + (t >> 6);
      raw[qb] = make_uint2(0u, 0u);
      if (t < nblk * 64 && n < a.M && kb < a.nb)
        raw[qb] = *reinterpret_cast<const uint2 *>(a.xq + (static_cast<size_t>(n) * a.nb + kb) * kQK +
                                                   16 * s + 8 * kc);
    }
    int4 clo[kQC], chi[kQC];
    float cdx[kQC];
#pragma unroll
    for (int qc = 0; qc < kQC; ++qc) {
      const int t = ts + qc * kUmStageThreads;
      const int n = t & 15, kb = kb0 + (t >> 4);
      clo[qc] = chi[qc] = make_int4(0, 0, 0, 0);
      cdx[qc] = 0.0f;
      if (t < nblk * 16 && n < a.M && kb < a.nb) {
        const int4 *src = reinterpret_cast<const int4 *>(a.xq + (static_cast<size_t>(n) * a.nb + kb) * kQK);
        clo[qc] = src[0];
        chi[qc] = src[1];
        cdx[qc] = a.xd[static_cast<size_t>(n) * a.nb + kb];
      }
    }
#pragma unroll
    for (int qb = 0; qb < kQB; ++qb) {
      const int t = ts + qb * kUmStageThreads;
      if (t < nblk * 64) {
        const int n8 = t & 7, kc = (t >> 3) & 1, s = (t >> 4) & 1, ng = (t >> 5) & 1, j = t >> 6;
        const int8_t *e = reinterpret_cast<const int8_t *>(&raw[qb]);
        const float sc = s ? 0.0625f : 1.0f;
        const __half2 h0 = __floats2half2_rn(static_cast<float>(e[0]) * sc, static_cast<float>(e[2]) * sc);
        const __half2 h1 = __floats2half2_rn(static_cast<float>(e[1]) * sc, static_cast<float>(e[3]) * sc);
        const __half2 h2 = __floats2half2_rn(static_cast<float>(e[4]) * sc, static_cast<float>(e[6]) * sc);
        const __half2 h3 = __floats2half2_rn(static_cast<float>(e[5]) * sc, static_cast<float>(e[7]) * sc);
        *reinterpret_cast<uint4 *>(xbm + static_cast<size_t>(j) * kUmBBlock + 512 * s + 128 * kc + 256 * ng +
                                   16 * n8) =
            make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                       *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
      }
    }
#pragma unroll
    for (int qc = 0; qc < kQC; ++qc) {
      const int t = ts + qc * kUmStageThreads;
      if (t < nblk * 16) {
        const int n = t & 15, j = t >> 4;
        int slo = __dp4a(clo[qc].x, 0x01010101, 0), shi = __dp4a(chi[qc].x, 0x01010101, 0);
        slo = __dp4a(clo[qc].y, 0x01010101, slo);
        slo = __dp4a(clo[qc].z, 0x01010101, slo);
        slo = __dp4a(clo[qc].w, 0x01010101, slo);
        shi = __dp4a(chi[qc].y, 0x01010101, shi);
        shi = __dp4a(chi[qc].z, 0x01010101, shi);
        shi = __dp4a(chi[qc].w, 0x01010101, shi);
        negc[j * 16 + n] = -static_cast<float>(1032 * slo + 72 * shi);
        dxs[j * 16 + n] = cdx[qc];
      }
    }
    fence_proxy_async_cta();  // the B operand is read by the tensor cores (async proxy)
    asm volatile("bar.sync 1, %0;" ::"r"(kUmStageThreads) : "memory");
  };

  if (warp < kUmConvWarps) {
    // ---- converters: row i = TMEM lane 32 q + lane, blocks 4h..4h+3 of each stage ----
    const int q = warp & 3, h = warp >> 2;
    const int i = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    for (int n = 0; n < total; ++n) {
      if (aborted()) break;
      const int slot = n % S, u = 2 * n + h, buf = u % kUmBufs;
      const int rlo = row_lo + (n / cp) * a.H;
      const int nrows = min(row_hi, rlo + a.H) - rlo;
      if (!warp_wait([&] { return um_wait(smem_addr(&full_bar[slot]), (n / S) & 1u, abort_v, a.wait_ns); })) {
        if (lane == 0) fail();
        break;
      }
      if (u >= kUmBufs && !warp_wait([&] {
            return um_wait(smem_addr(&d_empty[buf]), ((u / kUmBufs) - 1) & 1u, abort_v, a.wait_ns);
          })) {
        if (lane == 0) fail();
        break;
      }
      uint4 w[kUmSub];
      if (i < nrows) {
        const uint8_t *row = ringq + static_cast<size_t>(slot) * a.slot_q + i * 128;
#pragma unroll
        for (int b = 0; b < kUmSub; ++b)
          w[b] = *reinterpret_cast<const uint4 *>(row + (((kUmSub * h + b) ^ (i & 7)) << 4));
        *reinterpret_cast<float4 *>(dwbuf + (buf * a.H + i) * kUmSub) =
            *reinterpret_cast<const float4 *>(ringd + slot * (a.slot_d / 4) + i * kUmChunk + kUmSub * h);
      } else {
#pragma unroll
        for (int b = 0; b < kUmSub; ++b) w[b] = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
      if (lane == 0) um_arrive(smem_addr(&empty_bar[slot]));
      // block b of the sub-stage -> columns 16 b .. 16 b + 15 of its A buffer:
      // step 0 (low nibbles as 1024 + n) in the first 8, step 1 (high, 1024 + 16 n) after
#pragma unroll
      for (int bp = 0; bp < kUmSub / 2; ++bp) {
        uint32_t v[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint4 &wb = w[2 * bp + hh];
          const uint32_t wd[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint32_t x = wd[qq], x8 = x >> 8;
            v[16 * hh + 2 * qq] = (x & 0x000F000Fu) | 0x64006400u;
            v[16 * hh + 2 * qq + 1] = (x8 & 0x000F000Fu) | 0x64006400u;
            v[16 * hh + 8 + 2 * qq] = (x & 0x00F000F0u) | 0x64006400u;
            v[16 * hh + 8 + 2 * qq + 1] = (x8 & 0x00F000F0u) | 0x64006400u;
          }
        }
        tmem_st32(tmem + lane_base + static_cast<uint32_t>(buf * kUmSub * 16 + bp * 32), v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) um_arrive(smem_addr(&a_full[buf]));
    }
    tmem_wait_st();
  } else if (warp < kUmConvWarps + kUmEpiWarps) {
    // ---- epilogue: row i = TMEM lane 32 q + lane, blocks 4h..4h+3 of each stage ----
    const int ew = warp - kUmConvWarps, q = ew & 3, h = ew >> 2;
    const int i = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int te = tid - kUmConvWarps * 32;  // 0 .. 255
    stage_activations(te);
    unsigned long long acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0ull;
    for (int n = 0; n < total; ++n) {
      if (aborted()) break;
      const int k = n % cp, r = n / cp, u = 2 * n + h, buf = u % kUmBufs;
      const int rlo = row_lo + r * a.H;
      const int nrows = min(row_hi, rlo + a.H) - rlo;
      const uint32_t ph = (u / kUmBufs) & 1u;
      if (!warp_wait([&] {
            return um_wait(smem_addr(&mma_done[buf]), ph, abort_v, a.wait_ns) &&
                   um_wait(smem_addr(&a_full[buf]), ph, abort_v, a.wait_ns);
          })) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      float4 dw = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (i < nrows) dw = *reinterpret_cast<const float4 *>(dwbuf + (buf * a.H + i) * kUmSub);
      const float dws[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
      for (int bp = 0; bp < kUmSub / 2; ++bp) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(256 + buf * kUmSub * 16 + bp * 32), v);
        if (i < nrows) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int j = k * kUmChunk + kUmSub * h + 2 * bp + hh;  // part-local block
            const ulonglong2 *nc = reinterpret_cast<const ulonglong2 *>(negc + j * 16);
            const ulonglong2 *xs = reinterpret_cast<const ulonglong2 *>(dxs + j * 16);
            const float wv = dws[2 * bp + hh];
            const unsigned long long w2 = um_pack(__float_as_uint(wv), __float_as_uint(wv));
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const ulonglong2 cq = nc[qq], xq = xs[qq];
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const int e = 2 * qq + e2;  // m = 2e, 2e + 1
                const unsigned long long cc = e2 ? cq.y : cq.x, xx = e2 ? xq.y : xq.x;
                unsigned long long s2, t2;
                asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s2) : "l"(um_pack(v[16 * hh + 2 * e], v[16 * hh + 2 * e + 1])), "l"(cc));
                asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t2) : "l"(s2), "l"(w2));
                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc[e]) : "l"(t2), "l"(xx));
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) um_arrive(smem_addr(&d_empty[buf]));
      if (k == cp - 1) {  // the round's partial sums of this row and half
        if (i < nrows) {
          ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(parts + ((r * 2 + h) * a.H + i) * 16);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) dst[qq] = make_ulonglong2(acc[2 * qq], acc[2 * qq + 1]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0ull;
      }
    }
    // The cluster's sums: rows i = p mod P of every round, the 2P partials
    // added rank by rank, half by half.
    if (!aborted()) {
      __syncwarp();
      if (lane == 0)
        for (int rk = 0; rk < a.P; ++rk) um_arrive_remote(smem_addr(&parts_ready), rk);
      if (!warp_wait([&] { return um_wait(smem_addr(&parts_ready), 0, abort_v, a.wait_ns, true); })) {
        if (lane == 0) fail();
      } else {
        for (int r = 0; r < rounds; ++r) {
          const int rlo = row_lo + r * a.H;
          const int nrows = min(row_hi, rlo + a.H) - rlo;
          const int mine = nrows > p ? (nrows - p + a.P - 1) / a.P : 0;
          for (int t = te; t < mine * 4; t += kUmEpiWarps * 32) {
            const int ii = p + (t >> 2) * a.P, mq = t & 3;
            float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int rk = 0; rk < a.P; ++rk) {
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t off =
                    parts_s + static_cast<uint32_t>((((r * 2 + hh) * a.H + ii) * 16 + 4 * mq) * 4);
                const float4 v = um_ld_cluster_f4(off, rk);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
              }
            }
            const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 4 * mq + e;
              if (m < a.M) a.Y[static_cast<size_t>(m) * a.ldy + rlo + ii] = vals[e];
            }
          }
        }
      }
    }
  } else if (warp == kUmMmaWarp) {
    // ---- MMA warp: one elected thread issues each sub-stage's MMAs ----
    stage_activations(kUmEpiWarps * 32 + lane);
    int committed = 0;
    for (int u = 0; u < 2 * total; ++u) {
      if (aborted()) break;
      const int buf = u % kUmBufs, n = u >> 1, hh = u & 1, k = n % cp;
      if (!warp_wait([&] { return um_wait(smem_addr(&a_full[buf]), (u / kUmBufs) & 1u, abort_v, a.wait_ns); })) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      if (um_elect()) {
        // step 0 of the four blocks, then step 1: consecutive MMAs write
        // different accumulators
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int bb = 0; bb < kUmSub; ++bb) {
            const int j = k * kUmChunk + kUmSub * hh + bb;
            umma_f16(tmem + static_cast<uint32_t>(256 + buf * kUmSub * 16 + bb * 16),
                     tmem + static_cast<uint32_t>(buf * kUmSub * 16 + bb * 16 + 8 * s),
                     umma_desc(xb_s + static_cast<uint32_t>(j * kUmBBlock + 512 * s), a.lbo, a.sbo),
                     static_cast<uint32_t>(s));
          }
        umma_commit(smem_addr(&mma_done[buf]));
      }
      __syncwarp();
      ++committed;
    }
    if (lane == 0 && committed > 0) {  // nothing in flight at the end, even after an abort
      const int last = committed - 1;
      mbar_wait_bounded(smem_addr(&mma_done[last % kUmBufs]), (last / kUmBufs) & 1u, kDrainWaitNs);
    }
    __syncwarp();
  } else {
    // ---- the producer: the rest of the stages ----
    if (producer) {
      while (static_cast<int>(issued) < total && !*abort_v && issue_next()) {
      }
      if (*abort_v)  // copies still landing after an abort (bounded)
        for (uint32_t n = static_cast<int>(issued) > S ? issued - S : 0; n < issued; ++n)
          mbar_wait_bounded(smem_addr(&full_bar[n % S]), (n / S) & 1u, kDrainWaitNs);
    }
    __syncwarp();
  }

  // No CTA leaves while a peer may still read its partials; TMEM is freed
  // once every MMA and every tensor-memory access of the CTA is done.
  tc_fence_before();
  um_cluster_sync();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kUmTmemCols)
                 : "memory");
}

// ---- host side ---------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 um_tensor_map_encoder() {
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

static bool um_encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *ptr, uint64_t inner,
                         uint64_t rows, uint64_t stride, uint32_t box_inner, uint32_t box_rows,
                         CUtensorMapSwizzle swz) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = um_tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {stride};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(map, type, 2, const_cast<void *>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of P CTAs that fit on the device at once.
static std::atomic<int> g_um_clusters[kUmMaxCluster + 1];

// Shared-memory bytes (alignment slack included) of a launch with S ring slots.
static size_t um_bytes(int S, int H, int rounds, int xblocks, int slot_q, int slot_d) {
  const size_t fixed = static_cast<size_t>(xblocks) * (kUmBBlock + kUmCBlock + kUmXdBlock) +
                       static_cast<size_t>(kUmBufs) * H * kUmSub * 4 + static_cast<size_t>(rounds) * 2 * H * 16 * 4;
  return 1024 + static_cast<size_t>(S) * (slot_q + slot_d) + fixed;
}

cudaError_t launch_gemm_q4_umma(const LaunchCtx &ctx, const void *wq, const float *wd, int nb,
                                const int8_t *xq, const float *xd, int M, float *Y, int ldy, int r0,
                                int r1, int rows) {
  const int n = r1 - r0;
  if (n <= 0 || M <= 0) return cudaSuccess;
  const int nchunks = (nb + kUmChunk - 1) / kUmChunk;
  // the fewest K-parts whose activations fit (MLQ_UMMA_CLUSTER=P asks for more: A/B timing)
  static const int p_env = [] {
    const char *e = std::getenv("MLQ_UMMA_CLUSTER");
    return e != nullptr ? std::atoi(e) : 0;
  }();
  const int p_min = (nchunks * kUmChunk + kUmMaxPart - 1) / kUmMaxPart;
  const int P = p_env > p_min && p_env <= kUmMaxCluster && p_env <= nchunks ? p_env : p_min;
  // the scale map needs 16-byte row strides
  if (M > 16 || P > kUmMaxCluster || nb % 4 != 0) return cudaErrorNotSupported;
  UmParams prm;
  UmArgs &a = prm.a;
  a.Y = Y;
  a.xq = xq;
  a.xd = xd;
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  a.ldy = ldy;
  a.nb = nb;
  a.M = M;
  a.r0 = r0;
  a.r1 = r1;
  a.P = P;
  a.early = ctx.early_weights ? 1 : 0;
  // core-matrix strides of the B operand as staged by the kernel: 128 bytes
  // along K, 256 along N
  a.lbo = 128u;
  a.sbo = 256u;
  const int part_chunks = (nchunks + P - 1) / P;
  a.xblocks = part_chunks * kUmChunk;
  a.units = (n + 7) / 8;
  auto kern = gemm_q4_umma_kernel;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kUmSmemLimit);
  if (attr != cudaSuccess) return attr;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(P);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kUmThreads);
  cfg.stream = ctx.stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // Every launch takes the whole shared memory: one CTA per SM, so no two
  // CTAs ever compete for the SM's tensor memory.
  cfg.dynamicSmemBytes = kUmSmemLimit;

  int clusters = g_um_clusters[P].load(std::memory_order_relaxed);
  if (clusters == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(P * ctx.num_sms));
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      return cudaErrorNotSupported;
    }
    g_um_clusters[P].store(clusters, std::memory_order_relaxed);
  }
  a.G = clusters < a.units ? clusters : a.units;
  // rows per round: a cluster's share in the fewest rounds of equal height
  const int per_cluster = 8 * ((a.units + a.G - 1) / a.G);
  a.rounds = (per_cluster + kUmRows - 1) / kUmRows;
  a.H = 8 * ((per_cluster / 8 + a.rounds - 1) / a.rounds);
  a.slot_q = (a.H * kUmChunk * 16 + 1023) / 1024 * 1024;
  a.slot_d = (a.H * kUmChunk * 4 + 127) / 128 * 128;
  a.slots = 0;
  for (int S = kUmMaxSlots; S >= 4 && a.slots == 0; --S)
    if (um_bytes(S, a.H, a.rounds, a.xblocks, a.slot_q, a.slot_d) <= static_cast<size_t>(kUmSmemLimit))
      a.slots = S;
  if (a.slots == 0) return cudaErrorNotSupported;
  a.ring = a.slots * (a.slot_q + a.slot_d);
  const size_t rowq = static_cast<size_t>(nb) * 16;
  if (!um_encode_2d(&prm.wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, rowq, static_cast<uint64_t>(rows), rowq,
                    kUmChunk * 16, static_cast<uint32_t>(a.H), CU_TENSOR_MAP_SWIZZLE_128B) ||
      !um_encode_2d(&prm.wd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, wd, static_cast<uint64_t>(nb),
                    static_cast<uint64_t>(rows), static_cast<uint64_t>(nb) * 4, kUmChunk,
                    static_cast<uint32_t>(a.H), CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorNotSupported;
  cfg.gridDim = dim3(static_cast<unsigned>(a.G * P));
  cfg.numAttrs = ctx.pdl ? 2 : 1;
  diag_launch_cfg(reinterpret_cast<const void *>(kern), cfg);
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace mlq
