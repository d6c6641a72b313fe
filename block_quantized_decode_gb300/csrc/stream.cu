// stream.cu -- a decode chain (mlq_decode_chain) as one persistent launch
// whose weight stream never stops at a phase boundary.
//
// What it computes is what chain.cu computes: phase p quantises its input
// x_p to Q8_0 and multiplies it with the phase's weight matrices; x_p may
// be the output of an earlier phase.  Definitions: page "Legacy-ISA ML
// Inference Runtime -- Design Spec", Sec. 4 (Q4_0 / Q8_0 blocks, block
// dot), Sec. 5 (quantize_q8 rounding, matvec), Sec. 6 "Forward pass".
//
// Why it is built this way.  An M = 1 product reads every weight byte once,
// so a decode step is bound by HBM, and an SM's share of the bandwidth is
// set by the bytes it keeps in flight (about 160 KB per SM are needed to
// approach the copy rate).  One CTA per SM (cooperative launch) keeps about
// 200 KB of weight stages in flight in a byte ring of shared memory:
//  * the stages are 1-D bulk copies of the CTA's rows, phase after phase,
//    issued in order by a producer warp whenever ring space and a stage
//    descriptor are free.  Weights never depend on activations, so issuing
//    runs ahead across phase boundaries: while the consumers wait at a grid
//    barrier, the ring fills with the next phase's rows;
//  * stages differ in size from phase to phase (R rows of the phase's row
//    length), so the ring is addressed in bytes: a stage starts where the
//    previous one ended, or at offset 0 if it would cross the end, and is
//    issued once every stage it overlaps has been consumed;
//  * 12 consumer warps (13 warps in all keep 128 registers per thread: an
//    SM sub-partition then holds at most four warps), warp (K-chunk c, row
//    group g) holding its chunk of the Q8_0 input in registers, take RW
//    rows of each stage (R = RW * G rows, no warp idle), reduce each row
//    across the warp, write per-chunk partial sums, and release the stage
//    (one arrival per warp);
//  * the phase input: when x_p is the output of a product of an earlier
//    phase whose rows are whole 32-row blocks, that product also writes its
//    output in Q8_0 (into the phase's xq_out / xd_out: bytes identical to
//    quantising the stored floats), and every CTA loads those int8 bytes
//    and scales, all loads in flight at once; otherwise every CTA quantises
//    the float x itself (CTA 0 writes xq_out / xd_out);
//  * per-chunk partial sums are added in a fixed order, y is stored, and
//    the 32-row blocks of products with an in-chain Q8_0 output are
//    quantised from exactly the stored floats.
// Rows are split over the CTAs on the host, phase by phase, so that the
// bytes each CTA has streamed up to the end of every phase are as even as
// the row granularity allows (32-row atoms where the output is quantised).
//
// Grid barrier: after a phase the consumers sync, one thread fences and
// adds 1 to that phase's counter in the caller's workspace; the next phase
// starts when the counter reaches gridDim.x (acquire loads, bounded wait).
// The last CTA out resets every counter.  Every wait is bounded: a give-up
// records MLQ_E_TIMEOUT, the CTA stops issuing copies and drains its own
// copies in flight (bounded) before it exits.
#include "phase_common.cuh"

#include <algorithm>
#include <cstdlib>
#include <numeric>
#include <vector>

namespace mlq {

constexpr int kStWarps = 12;                   // consumer warps
constexpr int kStThreads = (kStWarps + 1) * 32;  // + the producer warp
constexpr int kStConsumers = kStWarps * 32;
constexpr int kStSlots = 16;                   // stage descriptors (stages in flight)
constexpr size_t kStStageMax = 40 * 1024;      // preferred largest stage
constexpr size_t kStBudget = 226 * 1024;       // dynamic shared memory of the CTA

struct StreamPhaseDev {
  int C, cblk, G, RW, R;  // K-chunks, blocks per chunk, warps per chunk, rows per warp, rows per stage
  int qin;                // input read as Q8_0 from xq_out / xd_out (written by an earlier phase)
  int any_out;            // some product of the phase writes an in-chain Q8_0 output
};
struct StreamOutDev {
  int8_t *yq;
  float *yd;
};
struct StreamArgs {
  ChainArgs c;
  StreamPhaseDev ph[kChainMaxPhases];
  StreamOutDev out[kChainMaxProducts];
  int bounds[kChainMaxPhases][kPhMaxGrid + 1];  // rows [bounds[p][b], bounds[p][b+1]) of phase p: CTA b
  unsigned smem_part, smem_ring, ring_bytes;
};

// A stage as the producer placed it (read by the consumers after the
// stage's full barrier completes, which orders the write before the read).
struct StDesc {
  unsigned off;  // byte offset in the ring
  int prow;      // first row, in the phase's concatenated numbering
  int n;         // rows
  int pad;
};

__device__ __forceinline__ void st_sync() {  // consumer warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kStConsumers) : "memory");
}
__device__ __forceinline__ void st_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ unsigned st_ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct StShared {
  uint64_t full_bar[kStSlots];
  uint64_t empty_bar[kStSlots];
  unsigned long long vstart[kStSlots];  // virtual start of the stage in each descriptor (producer only)
  StDesc desc[kStSlots];
  int abort_flag;
};

// Bounded wait that also gives up once another warp of the CTA has aborted.
__device__ __forceinline__ bool st_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
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

// The producer (one thread): every stage of every phase of the CTA, in
// order.  A stage of `bytes` is placed at virtual byte position v (the end
// of the previous stage, or the start of the next lap of the ring if it
// would cross the end); it may be issued once a descriptor is free and the
// oldest unreleased stage starts at least one ring length before v + bytes.
// Returns the number of stages issued.
template <int QT>
__device__ __forceinline__ int st_produce(const StreamArgs &sa, StShared &sh, uint8_t *ring) {
  const ChainArgs &a = sa.c;
  const volatile int *abort_v = &sh.abort_flag;
  const unsigned long long RB = sa.ring_bytes;
  unsigned long long *vstart = sh.vstart;
  unsigned long long vhead = 0;
  int t = 0, tail = 0;
  for (int p = 0; p < a.nphases; ++p) {
    const int nb = a.phase[p].nb;
    const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
    const int R = sa.ph[p].R;
    const int ra = sa.bounds[p][blockIdx.x], rb = sa.bounds[p][blockIdx.x + 1];
    for (int j = a.phase[p].first, off = 0; j < a.phase[p].first + a.phase[p].count; off += a.prod[j].rows, ++j) {
      const int lo = max(ra, off), hi = min(rb, off + a.prod[j].rows);
      for (int r = lo; r < hi; r += R) {
        const int n = min(R, hi - r);
        const unsigned qb = static_cast<unsigned>(n * rowq), db = static_cast<unsigned>(n) * nb * 4;
        const unsigned bytes = qb + db;
        unsigned long long v = vhead;
        const unsigned long long pos = v % RB;
        if (pos + bytes > RB) v += RB - pos;
        while (tail < t && (t - tail >= kStSlots || v + bytes > vstart[tail % kStSlots] + RB)) {
          if (!st_wait(smem_addr(&sh.empty_bar[tail % kStSlots]), (tail / kStSlots) & 1, abort_v, a.wait_ns)) {
            if (atomicExch(&sh.abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
            return t;
          }
          ++tail;
        }
        if (*abort_v) return t;
        const int slot = t % kStSlots;
        const unsigned o = static_cast<unsigned>(v % RB);
        sh.desc[slot] = StDesc{o, r, n, 0};
        vstart[slot] = v;
        const uint32_t fb = smem_addr(&sh.full_bar[slot]);
        const int lrow = r - off;
        mbar_arrive_expect_tx(fb, bytes);
        bulk_copy_g2s(smem_addr(ring + o), a.prod[j].wq + static_cast<size_t>(lrow) * rowq, qb, fb);
        bulk_copy_g2s(smem_addr(ring + o + qb), a.prod[j].wd + static_cast<size_t>(lrow) * nb, db, fb);
        vhead = v + bytes;
        ++t;
      }
    }
  }
  return t;
}

// Stages of phase p that fall to this CTA.
__device__ __forceinline__ int st_stage_count(const StreamArgs &sa, int p) {
  const ChainArgs &a = sa.c;
  const int ra = sa.bounds[p][blockIdx.x], rb = sa.bounds[p][blockIdx.x + 1];
  const int R = sa.ph[p].R;
  int cnt = 0;
  for (int j = a.phase[p].first, off = 0; j < a.phase[p].first + a.phase[p].count; off += a.prod[j].rows, ++j) {
    const int lo = max(ra, off), hi = min(rb, off + a.prod[j].rows);
    if (hi > lo) cnt += (hi - lo + R - 1) / R;
  }
  return cnt;
}

// Q4_0: RW rows of the stage (rows g, g + G, ...), the lane's (at most
// two) blocks of the warp's K-chunk; the RW rows' loads of a block are
// issued before any of its arithmetic.  Rows past n contribute 0.
template <int RW>
__device__ __forceinline__ void rows_q4(float acc[RW], const uint8_t *wq_s, const float *wd_s, size_t rowq,
                                        int nb, int g, int G, int n, const XChunk &c, int u0) {
  const uint8_t *wr[RW];
  const float *dr[RW];
#pragma unroll
  for (int q = 0; q < RW; ++q) {
    const int row = min(g + G * q, n - 1);
    wr[q] = wq_s + static_cast<size_t>(row) * rowq;
    dr[q] = wd_s + static_cast<size_t>(row) * nb;
    acc[q] = 0.0f;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (!c.v[k]) continue;
    const int u = u0 + 32 * k;
    uint4 w[RW];
    float dw[RW];
#pragma unroll
    for (int q = 0; q < RW; ++q) {
      w[q] = *reinterpret_cast<const uint4 *>(wr[q] + u * 16);
      dw[q] = dr[q][u];
    }
    constexpr uint32_t kLo = 0x0F0F0F0Fu, kHi = 0xF0F0F0F0u;
    const int4 xa = c.x[k][0], xb = c.x[k][1];
#pragma unroll
    for (int q = 0; q < RW; ++q) {
      const uint4 t = w[q];
      int lo = __dp4a(static_cast<int>(t.x & kLo), xa.x, c.adj[k]);
      int hi = dp4a_us(t.x & kHi, xb.x, 0);  // 16 * (high nibble) per byte: exact multiple of 16
      lo = __dp4a(static_cast<int>(t.y & kLo), xa.y, lo);
      hi = dp4a_us(t.y & kHi, xb.y, hi);
      lo = __dp4a(static_cast<int>(t.z & kLo), xa.z, lo);
      hi = dp4a_us(t.z & kHi, xb.z, hi);
      lo = __dp4a(static_cast<int>(t.w & kLo), xa.w, lo);
      hi = dp4a_us(t.w & kHi, xb.w, hi);
      const float sumi = __fsub_rn(__int_as_float(lo + (hi >> 4)), kMagic);
      acc[q] = __fmaf_rn(__fmul_rn(sumi, dw[q]), c.d[k], acc[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < RW; ++q) acc[q] = g + G * q < n ? acc[q] : 0.0f;
}

// N per-lane partial sums -> N warp sums (N = 1, 2, 4, 8), fixed order:
// at each of the first log2(N) butterfly levels a lane keeps half of its
// values and adds the partner's other half, then the remaining levels add
// plain.  Lane l returns the sum of value l / (32 / N).
template <int N>
__device__ __forceinline__ float reduce_n(float v[N], int lane) {
#pragma unroll
  for (int half = N / 2, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[i + half] : v[i];
      const float send = up ? v[i] : v[i + half];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
  float k = v[0];
#pragma unroll
  for (int bit = 16 / N; bit >= 1; bit >>= 1) k += __shfl_xor_sync(0xffffffffu, k, bit);
  return k;
}

// RW rows (g, g + G, ...) of one stage into acc[0, RW).
template <int QT, int RW>
__device__ __forceinline__ void st_stage_rows(float *acc, const uint8_t *ring, const StDesc &d, size_t rowq,
                                              int nb, int g, int G, const XChunk &xc, int u0, int lane) {
  const uint8_t *wq_s = ring + d.off;
  const float *wd_s = reinterpret_cast<const float *>(wq_s + static_cast<size_t>(d.n) * rowq);
  if (QT == 1) {
    rows_q4<RW>(acc, wq_s, wd_s, rowq, nb, g, G, d.n, xc, u0);
  } else {
#pragma unroll
    for (int q = 0; q < RW; ++q) {
      const int row = g + G * q;
      acc[q] = row < d.n ? row_part<QT>(wq_s + static_cast<size_t>(row) * rowq,
                                        wd_s + static_cast<size_t>(row) * nb, xc, u0, lane)
                         : 0.0f;
    }
  }
}

// The CTA's stages of phase p, in order: wait for the stage, RW rows of
// the warp's K-chunk, one warp reduction, partial sums to shared memory,
// release (one arrival per warp).
template <int QT, int RW>
__device__ __forceinline__ bool st_phase_stages(const StreamArgs &sa, int p, StShared &sh, uint8_t *ring,
                                                float *part_s, const XChunk &xc, int &s, int warp, int lane,
                                                int ra, int count) {
  const ChainArgs &a = sa.c;
  const StreamPhaseDev &sp = sa.ph[p];
  const int nb = a.phase[p].nb;
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  const int C = sp.C, G = sp.G;
  const int c = warp % C, g = warp / C;
  const int u0 = c * sp.cblk + lane;
  for (int i = 0; i < count; ++i, ++s) {
    const int slot = s % kStSlots;
    if (!warp_wait([&] {
          return st_wait(smem_addr(&sh.full_bar[slot]), (s / kStSlots) & 1, &sh.abort_flag, a.wait_ns);
        })) {
      if (lane == 0 && atomicExch(&sh.abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      return false;
    }
    const StDesc d = sh.desc[slot];
    float acc[RW];
    st_stage_rows<QT, RW>(acc, ring, d, rowq, nb, g, G, xc, u0, lane);
    const float v = reduce_n<RW>(acc, lane);
    const int q = lane / (32 / RW);
    const int row = g + G * q;
    if (lane % (32 / RW) == 0 && row < d.n) part_s[(d.prow - ra + row) * C + c] = v;
    __syncwarp();
    if (lane == 0) st_arrive(smem_addr(&sh.empty_bar[slot]));
  }
  return true;
}

template <int QT>
__global__ void __launch_bounds__(kStThreads, 1) decode_stream_kernel(const __grid_constant__ StreamArgs sa) {
  const ChainArgs &a = sa.c;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) StShared sh;
  volatile int *abort_v = &sh.abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + a.kmax);
  float *part_s = reinterpret_cast<float *>(smem + sa.smem_part);
  uint8_t *ring = smem + sa.smem_ring;

  if (tid == 0) {
    for (int k = 0; k < kStSlots; ++k) {
      mbar_init(smem_addr(&sh.full_bar[k]), 1);
      mbar_init(smem_addr(&sh.empty_bar[k]), kStWarps);  // one arrival per consumer warp
    }
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kStWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      const int issued = st_produce<QT>(sa, sh, ring);
      if (*abort_v) {  // copies may still be landing: the last issued stages (bounded)
        for (int u = issued > kStSlots ? issued - kStSlots : 0; u < issued; ++u)
          mbar_wait_bounded(smem_addr(&sh.full_bar[u % kStSlots]), (u / kStSlots) & 1, kDrainWaitNs);
      }
    }
    __syncwarp();
  } else {
  // ------------------------------ consumers ------------------------------
  int s = 0;  // stages consumed so far
  for (int p = 0; p < a.nphases; ++p) {
    const ChainPhaseDev &ph = a.phase[p];
    const StreamPhaseDev &sp = sa.ph[p];
    const int nb = ph.nb;
    if (p > 0) {  // every CTA has written the outputs of phases < p
      if (tid == 0) {
        bool ok = a.wait_ns != 0;
        const uint64_t t0 = sm_cycles(), lim = limit_cycles(a.wait_ns);
        while (ok && st_ld_acquire(a.counters + (p - 1)) < gridDim.x) {
          if (*abort_v || sm_cycles() - t0 > lim) ok = false;
        }
        if (!ok && atomicExch(&sh.abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
      }
      st_sync();
      if (*abort_v) break;
    }
    const int ra = sa.bounds[p][blockIdx.x], rb = sa.bounds[p][blockIdx.x + 1];
    // ---- the phase input into shared memory ----
    if (sp.qin) {
      if (rb > ra) {
        const int uq = nb * 2, nu = nb * 2 + nb / 4;  // int4 units: quants, then scales
        for (int base = 0; base < nu; base += 2 * kStConsumers) {  // all loads before any store
          int4 v[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int u = base + q * kStConsumers + tid;
            if (u < nu)
              v[q] = u < uq ? __ldcg(reinterpret_cast<const int4 *>(ph.xq_out) + u)
                            : __ldcg(reinterpret_cast<const int4 *>(ph.xd_out) + (u - uq));
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int u = base + q * kStConsumers + tid;
            if (u < uq) reinterpret_cast<int4 *>(xq_s)[u] = v[q];
            else if (u < nu) reinterpret_cast<int4 *>(xd_s)[u - uq] = v[q];
          }
        }
      }
    } else {
      const bool writer = blockIdx.x == 0 && ph.xq_out != nullptr;
      if (rb > ra || writer) quantize_input<kStWarps>(ph.x, nb, ph.xq_out, ph.xd_out, writer, xq_s, xd_s, tid);
    }
    st_sync();

    if (rb > ra) {
      // ---- the CTA's rows of the phase, stage by stage ----
      const int C = sp.C;
      XChunk xc;
      load_chunk<QT>(xc, xq_s, xd_s, nb, (warp % C) * sp.cblk, sp.cblk, lane);
      const int count = st_stage_count(sa, p);
      if (sp.RW == 4) st_phase_stages<QT, 4>(sa, p, sh, ring, part_s, xc, s, warp, lane, ra, count);
      else if (sp.RW == 2) st_phase_stages<QT, 2>(sa, p, sh, ring, part_s, xc, s, warp, lane, ra, count);
      else st_phase_stages<QT, 1>(sa, p, sh, ring, part_s, xc, s, warp, lane, ra, count);
      st_sync();
      if (*abort_v) break;

      // ---- y: the K-chunks of each row added in a fixed order ----
      for (int jj = ph.first, off = 0; jj < ph.first + ph.count; off += a.prod[jj].rows, ++jj) {
        const int lo = max(ra, off), hi = min(rb, off + a.prod[jj].rows);
        for (int gr = lo + tid; gr < hi; gr += kStConsumers) {
          const int r = gr - ra;
          float v = part_s[r * C];
          for (int cc = 1; cc < C; ++cc) v += part_s[r * C + cc];
          a.prod[jj].y[gr - off] = v;
          part_s[r * C] = v;
        }
      }
      if (sp.any_out) {
        st_sync();
        // each whole 32-row block of a product with an in-chain Q8_0
        // output, from exactly the stored floats; one warp per block
        int t = 0;
        for (int jj = ph.first, off = 0; jj < ph.first + ph.count; off += a.prod[jj].rows, ++jj) {
          const int lo = max(ra, off), hi = min(rb, off + a.prod[jj].rows);
          int8_t *yq = sa.out[jj].yq;
          if (yq == nullptr || hi <= lo) continue;
          for (int gr = lo; gr < hi; gr += kQK, ++t) {
            if ((t % kStWarps) != warp) continue;
            const float v = part_s[(gr - ra + lane) * C];
            uint32_t m = __float_as_uint(fabsf(v));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float amax = __uint_as_float(m);
            const float dd = amax / 127.0f;
            const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
            yq[gr - off + lane] = static_cast<int8_t>(quant_one(v, id));
            if (lane == 0) sa.out[jj].yd[(gr - off) / kQK] = dd;
          }
        }
      }
    }
    st_sync();  // every output of this CTA for phase p written
    if (tid == 0) {  // release: orders the CTA's output writes (joined by the sync) before it
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.counters + p) : "memory");
    }
  }
  }

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned done = atomicAdd(a.counters + a.nphases, 1u);
    if (done == gridDim.x - 1) {  // last CTA out: leave the workspace zeroed
      for (int p = 0; p <= a.nphases; ++p) atomicExch(a.counters + p, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side: in-chain Q8_0 hand-offs, geometry, row split, launch.
// ---------------------------------------------------------------------------
namespace {

// The row split of every phase.  Phase by phase, rows go out in atoms (32
// rows where an output is quantised in-chain, else 1); each CTA gets
// floor(atoms / grid) atoms, and the remaining ones go to the CTAs that
// have streamed the fewest bytes so far (ties: lower index).  A CTA's rows
// are contiguous and CTAs take them in index order.
void plan_stream_rows(StreamArgs &sa, int grid, const size_t *row_bytes, int *rows_max) {
  const ChainArgs &a = sa.c;
  std::vector<double> cum(grid, 0.0);
  std::vector<int> order(grid), take(grid);
  for (int p = 0; p < a.nphases; ++p) {
    long long total = 0;
    for (int j = a.phase[p].first; j < a.phase[p].first + a.phase[p].count; ++j) total += a.prod[j].rows;
    const int atom = sa.ph[p].any_out ? kQK : 1;
    const long long atoms = total / atom;
    const long long base = atoms / grid;
    const int extra = static_cast<int>(atoms % grid);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cum[x] < cum[y]; });
    for (int b = 0; b < grid; ++b) take[b] = static_cast<int>(base);
    for (int e = 0; e < extra; ++e) ++take[order[e]];
    int pos = 0;
    rows_max[p] = 0;
    sa.bounds[p][0] = 0;
    for (int b = 0; b < grid; ++b) {
      const int rows = take[b] * atom;
      pos += rows;
      sa.bounds[p][b + 1] = pos;
      cum[b] += static_cast<double>(rows) * static_cast<double>(row_bytes[p]);
      rows_max[p] = rows > rows_max[p] ? rows : rows_max[p];
    }
  }
}

}  // namespace

// Everything but the launch: the kernel arguments and the dynamic shared
// memory of a chain on `num_sms` CTAs.  cudaErrorNotSupported when the
// chain does not suit the kernel.
cudaError_t plan_decode_stream(int num_sms, int qtype, const ChainArgs &args, StreamArgs &sa,
                               size_t *smem_out, int *grid_out) {
  sa.c = args;
  ChainArgs &a = sa.c;
  const int grid = num_sms < kPhMaxGrid ? num_sms : kPhMaxGrid;
  if (grid < 1 || a.nphases < 1 || a.nphases > kChainMaxPhases) return cudaErrorNotSupported;
  const char *qin_env = std::getenv("MLQ_CHAIN_QIN");
  const bool allow_qin = qin_env == nullptr || qin_env[0] != '0';

  // In-chain Q8_0 hand-offs: phase p reads the Q8_0 output of the product
  // of an earlier phase whose y is x_p, when that phase's rows are whole
  // 32-row blocks and x_p's quantisation has a home (xq_out / xd_out) that
  // no other phase writes.
  for (int j = 0; j < kChainMaxProducts; ++j) sa.out[j] = StreamOutDev{nullptr, nullptr};
  for (int p = 0; p < a.nphases; ++p) {
    sa.ph[p].qin = 0;
    sa.ph[p].any_out = 0;
  }
  auto overlaps = [](const void *x, size_t nx, const void *y, size_t ny) {
    const char *a0 = static_cast<const char *>(x), *b0 = static_cast<const char *>(y);
    return a0 < b0 + ny && b0 < a0 + nx;
  };
  for (int p = 1; p < a.nphases && allow_qin; ++p) {
    const ChainPhaseDev &ph = a.phase[p];
    if (ph.xq_out == nullptr) continue;
    bool shared = false;
    for (int r = 0; r < a.nphases; ++r) {
      const ChainPhaseDev &pr = a.phase[r];
      if (r == p || pr.xq_out == nullptr) continue;
      shared = shared || overlaps(ph.xq_out, static_cast<size_t>(ph.nb) * kQK, pr.xq_out,
                                  static_cast<size_t>(pr.nb) * kQK) ||
               overlaps(ph.xd_out, static_cast<size_t>(ph.nb) * 4, pr.xd_out,
                        static_cast<size_t>(pr.nb) * 4);
    }
    if (shared) continue;
    for (int q = 0; q < p && !sa.ph[p].qin; ++q) {
      const ChainPhaseDev &pq = a.phase[q];
      bool whole = true;
      for (int j = pq.first; j < pq.first + pq.count; ++j) whole = whole && a.prod[j].rows % kQK == 0;
      if (!whole) continue;
      for (int j = pq.first; j < pq.first + pq.count; ++j) {
        if (a.prod[j].y == ph.x && a.prod[j].rows == ph.nb * kQK && sa.out[j].yq == nullptr) {
          sa.out[j] = StreamOutDev{ph.xq_out, ph.xd_out};
          sa.ph[p].qin = 1;
          sa.ph[q].any_out = 1;
          break;
        }
      }
    }
  }

  // Geometry per phase: C K-chunks (a divisor of the 12 consumer warps, at
  // most 64 blocks each: two per lane), G = 12 / C row groups, RW rows per
  // warp per stage, R = RW * G rows per stage.  Of the choices whose stage
  // is at most kStStageMax (or the smallest stage, for very long rows), take
  // the one with the fewest idle lanes, then the larger stage, then fewer
  // chunks.
  size_t row_bytes[kChainMaxPhases];
  size_t stage_max = 0;
  for (int p = 0; p < a.nphases; ++p) {
    const int nb = a.phase[p].nb;
    if (nb % 4 != 0) return cudaErrorNotSupported;
    row_bytes[p] = static_cast<size_t>(nb) * (qtype == 1 ? 16 : 32) + static_cast<size_t>(nb) * 4;
    double best_util = -1.0;
    size_t best_bytes = 0;
    int best_c = 0, best_rw = 0;
    for (int C = 1; C <= kStWarps; ++C) {
      if (kStWarps % C != 0 || C * kPhChunk < nb) continue;
      const int cblk = (nb + C - 1) / C;
      const int passes = (cblk + 31) / 32;
      const double util = static_cast<double>(nb) / (static_cast<double>(C) * 32.0 * passes);
      for (int RW : {1, 2, 4}) {
        const int R = RW * (kStWarps / C);
        const size_t bytes = static_cast<size_t>(R) * row_bytes[p];
        const bool fits = bytes <= kStStageMax;
        const bool better =
            best_rw == 0 ||
            (fits && (best_bytes > kStStageMax || util > best_util + 1e-9 ||
                      (util > best_util - 1e-9 && bytes > best_bytes))) ||
            (!fits && best_bytes > kStStageMax && bytes < best_bytes);
        if (better) {
          best_util = util;
          best_bytes = bytes;
          best_c = C;
          best_rw = RW;
        }
      }
    }
    if (best_rw == 0) return cudaErrorNotSupported;  // wider than 12 chunks of 64 blocks
    StreamPhaseDev &sp = sa.ph[p];
    sp.C = best_c;
    sp.cblk = (nb + best_c - 1) / best_c;
    sp.G = kStWarps / best_c;
    sp.RW = best_rw;
    sp.R = best_rw * sp.G;
    stage_max = best_bytes > stage_max ? best_bytes : stage_max;
  }
  int rows_max[kChainMaxPhases];
  plan_stream_rows(sa, grid, row_bytes, rows_max);
  size_t part = 0;
  for (int p = 0; p < a.nphases; ++p) {
    const size_t v = static_cast<size_t>(rows_max[p]) * sa.ph[p].C * 4;
    part = v > part ? v : part;
  }
  auto up128 = [](size_t v) { return (v + 127) / 128 * 128; };
  const size_t xs = up128(static_cast<size_t>(a.kmax) + 4 * (static_cast<size_t>(a.kmax) / kQK));
  const size_t fixed = xs + up128(part);
  if (fixed + 2 * stage_max > kStBudget) return cudaErrorNotSupported;
  sa.ring_bytes = static_cast<unsigned>((kStBudget - fixed) / 16 * 16);
  sa.smem_part = static_cast<unsigned>(xs);
  sa.smem_ring = static_cast<unsigned>(fixed);
  *smem_out = fixed + sa.ring_bytes;
  *grid_out = grid;
  return cudaSuccess;
}

int describe_decode_stream(int num_sms, int qtype, const ChainArgs &args, int32_t *info, int info_len) {
  StreamArgs *sap = new StreamArgs();
  struct Free {
    StreamArgs *p;
    ~Free() { delete p; }
  } guard{sap};
  StreamArgs &sa = *sap;
  size_t smem = 0;
  int grid = 0;
  const cudaError_t e = plan_decode_stream(num_sms, qtype, args, sa, &smem, &grid);
  const int np = args.nphases;
  const int need = 4 + 8 * np + (e == cudaSuccess ? np * (grid + 1) : 0);
  if (info_len < need) return -1;
  for (int i = 0; i < need; ++i) info[i] = 0;
  if (e != cudaSuccess) return 0;  // info[0] = 0: the chain takes the other kernel
  info[0] = 1;
  info[1] = grid;
  info[2] = static_cast<int32_t>(sa.ring_bytes);
  info[3] = static_cast<int32_t>(smem);
  for (int p = 0; p < np; ++p) {
    const StreamPhaseDev &sp = sa.ph[p];
    int32_t *o = info + 4 + 8 * p;
    o[0] = sp.C;
    o[1] = sp.cblk;
    o[2] = sp.G;
    o[3] = sp.RW;
    o[4] = sp.R;
    o[5] = sp.qin;
    o[6] = sp.any_out;
    int out = 0;
    for (int j = args.phase[p].first; j < args.phase[p].first + args.phase[p].count; ++j)
      out |= sa.out[j].yq != nullptr ? 1 << (j - args.phase[p].first) : 0;
    o[7] = out;  // bit i: product first + i writes an in-chain Q8_0 output
    for (int b = 0; b <= grid; ++b) info[4 + 8 * np + p * (grid + 1) + b] = sa.bounds[p][b];
  }
  return 1;
}

cudaError_t launch_decode_stream(const LaunchCtx &ctx, int qtype, const ChainArgs &args) {
  StreamArgs *sap = new StreamArgs();  // ~19 KB: keep it off the host stack
  struct Free {
    StreamArgs *p;
    ~Free() { delete p; }
  } guard{sap};
  StreamArgs &sa = *sap;
  size_t smem = 0;
  int grid = 0;
  cudaError_t e = plan_decode_stream(ctx.num_sms, qtype, args, sa, &smem, &grid);
  if (e != cudaSuccess) return e;
  sa.c.status = ctx.status;
  sa.c.wait_ns = ctx.wait_ns;
  auto kern = qtype == 1 ? decode_stream_kernel<1> : decode_stream_kernel<0>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kStThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  diag_note("stream: phases=%d ring=%uB grid=%d", sa.c.nphases, sa.ring_bytes, grid);
  diag_launch_cfg(reinterpret_cast<const void *>(kern), cfg);
  return cudaLaunchKernelEx(&cfg, kern, sa);
}

}  // namespace mlq
