// phase_ring.cu -- one decode phase per launch for weight slices too large
// to hold in shared memory (the Llama-7B-sized products, the lm_head): the
// same phase as phase.cu -- products sharing one input, float or Q8_0
// input, optional Q8_0 outputs in whole 32-row blocks -- with the CTA's
// rows streamed through a ring of shared-memory stages.  Definitions: page
// "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 4 (Q4_0 / Q8_0
// blocks, block dot), Sec. 5 (quantize_q8 rounding, matvec), Sec. 6
// "Forward pass".
//
// Per CTA (one per SM; for slices below 128 KB two fit on an SM, so the
// next phase's CTA is already resident while this one runs; larger slices
// take a 216 KB ring and 16 consumer warps with the SM to themselves):
//  * a producer warp copies the CTA's rows, stage by stage, with 1-D bulk
//    copies (rows of one product per stage, quants then scales), completion
//    on a full mbarrier per ring slot; with static weights it starts before
//    the dependency wait, so the ring is full when the phase begins and the
//    HBM stream continues across the launch boundary;
//  * 8 (16) consumer warps read the input (as phase.cu: the Q8_0 input loaded
//    once per CTA, or float x quantised in the CTA), keep their K-chunk of it
//    in registers, reduce each stage -- warp (chunk c, group g) takes one
//    four-row group per stage -- and free the slot on an empty mbarrier;
//  * per-chunk partial sums are added in a fixed order, y is stored, and the
//    32-row blocks of products with a quantised output are quantised from
//    exactly the stored floats.
// Consumer-only synchronisation uses a named barrier (the producer never
// joins it).  Every wait is bounded; on a give-up the CTA records
// MLQ_E_TIMEOUT and its copies in flight are drained before it exits.
#include "phase_common.cuh"

#include <cstdlib>

namespace mlq {

// consumer warps: 8 with two CTAs per SM, 16 with the SM to itself (both
// at 96 registers: an SM sub-partition holds at most 5 warps of either)
constexpr int kRingWarps = 8;
constexpr int kRingWarpsWide = 16;
constexpr int kRingMaxSlots = 8;
constexpr size_t kRingBudget = 110 * 1024;      // two CTAs per SM
constexpr size_t kRingBudgetWide = 216 * 1024;  // one CTA per SM (very long rows, large slices)
constexpr size_t kRingWideSlice = 128 * 1024;    // CTA slices from this size take the wide ring
constexpr int kRingInputBulkDefault = 1;        // a Q8_0 input by bulk copies unless forced off

template <int NW>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait that also gives up once another warp of the CTA has aborted.
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
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

// Bounded wait for phase `parity` of `bar` or for *flag to become nonzero,
// whichever comes first; false on a give-up or once the CTA has aborted.
__device__ __forceinline__ bool ring_wait_either(uint32_t bar, uint32_t parity, const volatile int *flag,
                                                 const volatile int *abort_flag,
                                                 unsigned long long limit_ns) {
  if (limit_ns == 0) return false;
  if (*flag || mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = sm_cycles(), lim = limit_cycles(limit_ns);
  for (;;) {
    if (*flag || mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (sm_cycles() - t0 > lim) return false;
  }
}

// Row r's K-chunk partial sums added in chunk order (C <= kRingWarps): all
// loads issued before the additions.
__device__ __forceinline__ float chunk_sum(const float *part_s, int prow, int r, int C) {
  float p[kRingWarps];
#pragma unroll
  for (int cc = 0; cc < kRingWarps; ++cc) p[cc] = cc < C ? part_s[cc * prow + r] : 0.0f;
  float v = p[0];
#pragma unroll
  for (int cc = 1; cc < kRingWarps; ++cc)
    if (cc < C) v += p[cc];
  return v;
}

// The CTA's stages: runs of at most R rows of [ra, rb), never spanning two
// products.  Producer and consumers walk them in the same order.
struct StageIter {
  int j, off, r;  // current product, its first row, next row (concatenated numbering)
};
__device__ __forceinline__ int stage_next(StageIter &it, const FusedArgs &a, int rb, int R,
                                          int *j, int *lrow) {
  while (it.r < rb && it.r >= it.off + a.prod[it.j].rows) {
    it.off += a.prod[it.j].rows;
    ++it.j;
  }
  if (it.r >= rb) return 0;
  const int end = min(rb, it.off + a.prod[it.j].rows);
  const int n = min(R, end - it.r);
  *j = it.j;
  *lrow = it.r - it.off;
  it.r += n;
  return n;
}

template <int QT, int NW>
__global__ void __launch_bounds__((NW + 1) * 32, NW == kRingWarps ? 2 : 1)
    phase_ring_kernel(const __grid_constant__ PhaseArgs pa) {
  const FusedArgs &a = pa.a;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kRingMaxSlots];
  __shared__ __align__(8) uint64_t empty_bar[kRingMaxSlots];
  __shared__ __align__(8) uint64_t in_bar;  // the Q8_0 input's bulk copies
  __shared__ int abort_flag;
  __shared__ int input_ready;
  volatile int *abort_v = &abort_flag;
  volatile int *input_v = &input_ready;
  const int IN = a.x == nullptr ? 1 : 0;
  const int nb = a.nb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ra = pa.bounds[blockIdx.x];
  const int rb = pa.bounds[blockIdx.x + 1];
  const int nr = rb - ra;
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  const int C = a.nchunks, cblk = a.chunk_blocks;
  const int G = NW / C;  // warps per chunk; a stage has R = 4 * G rows
  const int R = a.ring_rows, ns = a.ring_slots;
  const size_t stage_bytes = a.ring_stage, dq = a.ring_dq;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + static_cast<size_t>(nb) * kQK);
  // per-chunk partial sums: chunk c of the CTA's row r at part_s[c * prow + r]
  // (the epilogue's lanes then read consecutive words)
  float *part_s = reinterpret_cast<float *>(smem + a.smem_part);
  const int part_cap = static_cast<int>((a.smem_w - a.smem_part) / 4);  // floats of part_s
  const int prow = part_cap / C;  // >= the CTA's rows
  uint8_t *ring = smem + a.smem_w;

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), NW);  // one arrival per consumer warp
    }
    mbar_init(smem_addr(&in_bar), 1);
    abort_flag = 0;
    input_ready = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The next phase's kernel may be scheduled now (it waits for this grid to
  // complete before it reads anything we write).
  griddep_launch_dependents();

  if (warp == NW) {
    // ------------------------------ producer ------------------------------
    if (lane != 0 || nr == 0) return;
    if (!a.early) griddep_wait();  // weights written by earlier work: wait for it first
    StageIter it{0, 0, ra};
    int s = 0, j, lrow, n;
    // CTAs start in index order as SMs free up, so the last ones meet a
    // loaded memory system with their first stage.  With hint_partner = k,
    // CTA b < grid / k hints into L2 the first hint_stages stages of CTA
    // b + grid - grid / k (static weights only), in the tail of the previous
    // launch.
    const int nh = a.hint_partner > 0 ? static_cast<int>(gridDim.x) / a.hint_partner : 0;  // CTAs hinted
    const int partner = static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - nh;
    const bool hint = a.early && nh > 0 && static_cast<int>(blockIdx.x) < nh && partner < static_cast<int>(gridDim.x);
    while ((n = stage_next(it, a, rb, R, &j, &lrow)) > 0) {
      const int slot = s % ns;
      if (s >= ns && !ring_wait(smem_addr(&empty_bar[slot]), ((s / ns) - 1) & 1, abort_v, a.wait_ns)) {
        if (atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        break;
      }
      // Until the consumers hold the phase input (or, with bulk copies, have
      // issued its copies), keep at most one stage in flight: an SM serves
      // its reads in order, so the input read would otherwise wait behind
      // the whole ring (measured: 4-6 us behind 216 KB under load).  Once
      // stage s - 1 has landed, or the input is in, go on.
      if (s > 0 && !*input_v &&
          !ring_wait_either(smem_addr(&full_bar[(s - 1) % ns]), ((s - 1) / ns) & 1, input_v, abort_v,
                            a.wait_ns)) {
        if (atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
        break;
      }
      if (*abort_v) break;
      const uint32_t qb = static_cast<uint32_t>(n * rowq), db = static_cast<uint32_t>(n) * nb * 4;
      uint8_t *dst = ring + static_cast<size_t>(slot) * stage_bytes;
      const uint32_t fb = smem_addr(&full_bar[slot]);
      // the stage fits its slot, and its rows are rows of product j
      if (!in_bounds(n <= R && qb <= dq && dq + db <= stage_bytes && lrow + n <= a.prod[j].rows, a.status)) {
        mbar_arrive_expect_tx(fb, 0);  // complete the slot empty: the consumers do not wait
        ++s;
        continue;
      }
      mbar_arrive_expect_tx(fb, qb + db);
      bulk_copy_g2s(smem_addr(dst), a.prod[j].wq + static_cast<size_t>(lrow) * rowq, qb, fb);
      bulk_copy_g2s(smem_addr(dst + dq), a.prod[j].wd + static_cast<size_t>(lrow) * nb, db, fb);
      if (s == 0 && hint) {
        StageIter pit{0, 0, pa.bounds[partner]};
        int pj, plrow, pn;
        for (int ps = 0; ps < a.hint_stages && (pn = stage_next(pit, a, pa.bounds[partner + 1], R, &pj, &plrow)) > 0;
             ++ps) {
          prefetch_range_l2(a.prod[pj].wq + static_cast<size_t>(plrow) * rowq, static_cast<size_t>(pn) * rowq,
                            static_cast<size_t>(pn) * rowq);
          prefetch_range_l2(a.prod[pj].wd + static_cast<size_t>(plrow) * nb, static_cast<size_t>(pn) * nb * 4,
                            static_cast<size_t>(pn) * nb * 4);
        }
      }
      ++s;
    }
    if (*abort_v) {  // copies may still be landing: the last ns issued stages (bounded)
      for (int t = s > ns ? s - ns : 0; t < s; ++t)
        mbar_wait_bounded(smem_addr(&full_bar[t % ns]), (t / ns) & 1, kDrainWaitNs);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  // A static float input (no earlier work writes it) is read and quantised
  // before the dependency wait: off the critical path of a CTA that starts
  // early, and ahead of the ring's copies for one that starts late.
  const bool early_in = IN == 0 && a.early_input != 0;
  const bool writer = blockIdx.x == 0 && a.xq_out != nullptr;
  if (early_in) {
    if (nr > 0 || writer) quantize_input<NW>(a.x, nb, nullptr, nullptr, false, xq_s, xd_s, tid);
    consumers_sync<NW>();
    if (tid == 0) *input_v = 1;  // the producer may fill the ring now
  }
  griddep_wait();  // the input may come from the previous kernel
  if (IN == 0) {
    if (!early_in) {
      if (nr > 0 || writer) phase_quantize<NW>(a, xq_s, xd_s, tid);
    } else if (writer) {
      store_input_copy(xq_s, xd_s, nb, a.xq_out, a.xd_out, tid, NW * 32);
    }
  } else if (nr > 0 && a.input_bulk) {
    // the Q8_0 input by two bulk copies (quants, scales) on one barrier
    const uint32_t ib = smem_addr(&in_bar);
    if (tid == 0) {
      mbar_arrive_expect_tx(ib, static_cast<uint32_t>(nb) * (kQK + 4));
      bulk_copy_g2s(smem_addr(xq_s), a.xq_in, static_cast<uint32_t>(nb) * kQK, ib);
      bulk_copy_g2s(smem_addr(xd_s), a.xd_in, static_cast<uint32_t>(nb) * 4, ib);
      // the producer may go on now: its copies queue behind the input's
      if (a.input_issue_release) *input_v = 1;
    }
    if (!warp_wait([&] { return ring_wait(ib, 0, abort_v, a.wait_ns); })) {
      if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      if (tid == 0) mbar_wait_bounded(ib, 0, kDrainWaitNs);  // the copies may still be landing
    }
  } else if (nr > 0) {
    const int uq = nb * 2, nu = nb * 2 + nb / 4;
    for (int base = 0; base < nu; base += 4 * NW * 32) {  // all loads before any store
      int4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int u = base + q * NW * 32 + tid;
        if (u < nu)
          v[q] = u < uq ? __ldcg(reinterpret_cast<const int4 *>(a.xq_in) + u)
                        : __ldcg(reinterpret_cast<const int4 *>(a.xd_in) + (u - uq));
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int u = base + q * NW * 32 + tid;
        if (u < uq) reinterpret_cast<int4 *>(xq_s)[u] = v[q];
        else if (u < nu) reinterpret_cast<int4 *>(xd_s)[u - uq] = v[q];
      }
    }
  }
  consumers_sync<NW>();
  if (tid == 0) *input_v = 1;  // the producer may fill the ring now
  if (nr == 0) return;

  const int c = warp & (C - 1), g = warp / C;
  const int u0 = c * cblk + lane;
  XChunk xc;
  load_chunk<QT>(xc, xq_s, xd_s, nb, c * cblk, cblk, lane);
  bool ok = true;
  StageIter it{0, 0, ra};
  int s = 0, j, lrow, n;
  while ((n = stage_next(it, a, rb, R, &j, &lrow)) > 0) {
    const int slot = s % ns;
    const int srow = it.r - n - ra;  // the stage's first row in the CTA's slice
    ok = warp_wait([&] { return ring_wait(smem_addr(&full_bar[slot]), (s / ns) & 1, abort_v, a.wait_ns); });
    if (!ok) {
      if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      break;
    }
    const uint8_t *wq_s = ring + static_cast<size_t>(slot) * stage_bytes;
    const float *wd_s = reinterpret_cast<const float *>(wq_s + dq);
    float acc[4];
    if (QT == 1) {
      rows4_q4(acc, wq_s, wd_s, rowq, nb, g, G, n, xc, u0);
    } else {
      rows4_q8(acc, wq_s, wd_s, rowq, nb, g, G, n, xc, u0, lane);
    }
    const float v = reduce4(acc[0], acc[1], acc[2], acc[3], lane);
    const int row = g + G * (lane >> 3);
    const int pi = c * prow + srow + row;
    if ((lane & 7) == 0 && row < n && in_bounds(srow + row < prow, a.status)) part_s[pi] = v;
    __syncwarp();
    if (lane == 0) mbar_arrive1(smem_addr(&empty_bar[slot]));
    ++s;
  }
  consumers_sync<NW>();
  if (*abort_v) return;

  // y.  A product without a quantised output: one row per consumer thread,
  // the K-chunk partial sums added in a fixed order.  A product with one: y
  // and its Q8_0 blocks in one pass, warp w taking every NW-th of the CTA's
  // 32-row blocks of it, one row per lane, the block quantised from exactly
  // the floats stored -- its maximum by one warp reduction on the float bit
  // patterns (non-negative floats order as unsigned integers).
  int t = 0;
  for (int jj = 0, off = 0; jj < a.nproducts; off += a.prod[jj].rows, ++jj) {
    const int lo = max(ra, off), hi = min(rb, off + a.prod[jj].rows);
    int8_t *yq = a.prod[jj].yq;
    if (yq == nullptr) {
      for (int gr = lo + tid; gr < hi; gr += NW * 32) {
        const int r = gr - ra;
        if (!in_bounds(r < prow && gr - off < a.prod[jj].rows, a.status)) continue;
        a.prod[jj].y[gr - off] = chunk_sum(part_s, prow, r, C);
      }
      continue;
    }
    for (int g0 = lo; g0 < hi; g0 += kQK, ++t) {  // whole 32-row blocks here
      if ((t & (NW - 1)) != warp) continue;
      const int gr = g0 + lane;
      const int r = gr - ra;
      const bool ok = in_bounds(r < prow && gr - off >= 0 && gr - off < a.prod[jj].rows, a.status);
      float v = 0.0f;
      if (ok) {
        v = chunk_sum(part_s, prow, r, C);
        a.prod[jj].y[gr - off] = v;
      }
      const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
      const float dd = amax / 127.0f;
      const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
      if (ok) yq[gr - off] = static_cast<int8_t>(quant_one(v, id));
      if (lane == 0 && ok) a.prod[jj].yd[(gr - off) / kQK] = dd;
    }
  }
}

template <int QT>
static cudaError_t launch_ring_t(const LaunchCtx &ctx, const FusedArgs &args) {
  PhaseArgs pa;
  pa.a = args;
  FusedArgs &a = pa.a;
  const int nb = a.nb;
  if (a.total_rows <= 0 || nb % 4 != 0) return cudaErrorNotSupported;
  int grid = ctx.num_sms < a.total_rows ? ctx.num_sms : a.total_rows;
  grid = grid < kPhMaxGrid ? grid : kPhMaxGrid;
  // Q4_0 phases leave a few SMs free, on which the next launch's first CTAs
  // start (and stream) before this one ends: the Q4_0 stack 103.5 -> 102.9 /
  // 102.55 / 102.65 / 103.9 us with 148 / 144 / 140 / 128 of 152 SMs.  Q8_0
  // phases, twice as long, lose more streaming than they gain (174.9 ->
  // 177.7 us with 144).  MLQ_RING_GRID=n sets the grid (A/B timing).
  constexpr int kRingSpareSmsQ4 = 8;
  static const int grid_env = [] {
    const char *e = std::getenv("MLQ_RING_GRID");
    return e != nullptr ? std::atoi(e) : 0;
  }();
  if (grid_env > 0) {
    grid = grid_env < grid ? grid_env : grid;
  } else if (QT == 1 && grid == ctx.num_sms && grid > 2 * kRingSpareSmsQ4) {
    grid -= kRingSpareSmsQ4;
  }
  // Front-heavy split: the CTAs that start first (lowest index) take the
  // larger shares (the 11008-row product: the 40 CTAs with three 32-row
  // blocks start first instead of last).  MLQ_RING_FRONT=0 turns it off
  // (A/B timing).
  static const bool front_env = [] {
    const char *e = std::getenv("MLQ_RING_FRONT");
    return e == nullptr || e[0] != '0';
  }();
  const int rows_max = plan_rows(a, a.total_rows, grid, pa.bounds, front_env);
  // A Q8_0 input by bulk copies (16-byte aligned source) or by the
  // consumers' 16-byte loads; MLQ_RING_INPUT=ldg / bulk forces one (A/B timing).
  static const int input_env = [] {
    const char *e = std::getenv("MLQ_RING_INPUT");
    return e == nullptr ? -1 : (e[0] == 'b' ? 1 : 0);
  }();
  const bool aligned = a.x == nullptr && (reinterpret_cast<uintptr_t>(a.xq_in) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.xd_in) & 15) == 0;
  a.input_bulk = aligned && input_env != 0 ? (input_env == 1 ? 1 : kRingInputBulkDefault) : 0;
  // With bulk copies, the producer may go on once the input's copies are
  // issued instead of landed (Q4_0 stack 107.3 -> 106.3 us, Q8_0 + lm_head
  // 175.9 -> 174.8 us); MLQ_RING_ISSUE_RELEASE=0 waits for the landing.
  static const int release_env = [] {
    const char *e = std::getenv("MLQ_RING_ISSUE_RELEASE");
    return e != nullptr && e[0] == '0' ? 0 : 1;
  }();
  a.input_issue_release = release_env;
  // Late CTAs' first stages hinted into L2 by early ones: the Q4_0 stack
  // 106.6 -> 105.35 us with half the CTAs hinting (a quarter: 105.9), while
  // every fraction slowed the Q8_0 stack with its larger stages (175.2 ->
  // 176.2-179.9 us): on for Q4_0 only.  MLQ_RING_HINT_PARTNER=k (0: off)
  // sets the fraction 1/k for both.
  static const int hint_env = [] {
    const char *e = std::getenv("MLQ_RING_HINT_PARTNER");
    return e != nullptr ? std::atoi(e) : -1;
  }();
  a.hint_partner = hint_env >= 0 ? hint_env : (QT == 1 ? 2 : 0);
  static const int hint_stages_env = [] {
    const char *e = std::getenv("MLQ_RING_HINT_STAGES");
    return e != nullptr ? std::atoi(e) : 2;
  }();
  a.hint_stages = hint_stages_env > 0 ? hint_stages_env : 2;  // two: 103.5 -> 103.2 us (Q4_0 stack)
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  auto up128 = [](size_t v) { return (v + 127) / 128 * 128; };
  const size_t xs = up128(static_cast<size_t>(nb) * (kQK + 4));
  // Geometry: the fewest K-chunks (a power of two, at most 64 blocks each,
  // at most one per consumer warp) whose ring of >= 2 stages of R = 4 * G
  // rows fits the budget; two CTAs per SM if possible, else one.
  // Ring size.  Two CTAs per SM (110 KB each, 8 consumer warps) let the
  // next phase's CTA stream its first stages while this one finishes; a CTA
  // alone on its SM (216 KB, 16 consumer warps) keeps twice the bytes in
  // flight and reduces a landed stage twice as fast.  For slices beyond
  // the small ring the wide one wins (measured: the 7B Q4_0 stack, 185 KB
  // per CTA, 129.5 -> 115.6 us; the Q8_0 stack with the lm_head, 330 KB and
  // 1 MB per CTA, 228 -> 192 us).  MLQ_RING_WIDE=1 / 0 forces one order
  // (A/B timing).
  static const int wide_env = [] {
    const char *e = std::getenv("MLQ_RING_WIDE");
    return e == nullptr ? -1 : (e[0] == '1' ? 1 : 0);
  }();
  const size_t slice = static_cast<size_t>(rows_max) * (rowq + static_cast<size_t>(nb) * 4);
  const bool wide_first = wide_env >= 0 ? wide_env == 1 : slice >= kRingWideSlice;
  const size_t budgets[2] = {wide_first ? kRingBudgetWide : kRingBudget,
                             wide_first ? kRingBudget : kRingBudgetWide};
  for (size_t budget : budgets) {
    const int NW = budget == kRingBudgetWide ? kRingWarpsWide : kRingWarps;
    for (int C = 1; C <= NW && C <= kRingWarps; C *= 2) {
      if (C * kPhChunk < nb) continue;
      const int R = 4 * (NW / C);
      const size_t dq = up128(static_cast<size_t>(R) * rowq);
      const size_t stage = up128(dq + static_cast<size_t>(R) * nb * 4);
      const size_t ps = up128(static_cast<size_t>(rows_max) * C * 4);
      const size_t fixed = xs + ps;
      if (fixed + 2 * stage > budget) continue;
      int ns = static_cast<int>((budget - fixed) / stage);
      ns = ns < kRingMaxSlots ? ns : kRingMaxSlots;
      a.nchunks = C;
      a.chunk_blocks = (nb + C - 1) / C;
      a.ring_rows = R;
      a.ring_slots = ns;
      a.ring_stage = static_cast<unsigned>(stage);
      a.ring_dq = static_cast<unsigned>(dq);
      a.smem_part = static_cast<unsigned>(xs);
      a.smem_w = static_cast<unsigned>(fixed);
      const size_t smem = fixed + static_cast<size_t>(ns) * stage;
      diag_note("ring: products=%d rows=%d K=%d rows/CTA<=%d chunks=%d rows/stage=%d slots=%d stage=%zuB "
                "input=%s q8_out=%d early=%d", a.nproducts, a.total_rows, nb * kQK, rows_max, C, R, ns, stage,
                a.x != nullptr ? "f32" : (a.input_bulk ? "q8 bulk" : "q8 ldg"), a.any_yq, a.early);
      auto kern = NW == kRingWarps ? phase_ring_kernel<QT, kRingWarps> : phase_ring_kernel<QT, kRingWarpsWide>;
      prefer_max_shared(kern);
      if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
      }
      return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3((NW + 1) * 32), smem, ctx, pa);
    }
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_phase_ring(const LaunchCtx &ctx, int qtype, const FusedArgs &a) {
  return qtype == 1 ? launch_ring_t<1>(ctx, a) : launch_ring_t<0>(ctx, a);
}

}  // namespace mlq
