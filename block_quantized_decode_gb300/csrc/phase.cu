// phase.cu -- one decode "phase" per launch: y_j = W_j x for the products
// that share one input (Wq|Wk|Wv, gate|up, ...), for chains of dependent
// launches under programmatic dependent launch (PDL).  Definitions: page
// "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 4 (Q4_0 / Q8_0
// blocks, block dot), Sec. 5 (quantize_q8 rounding, matvec), Sec. 6
// "Forward pass" (one quantised activation feeds several products, and each
// product's output is quantised again as the next product's input).
//
// Design, per CTA (one per SM, 16 warps, <= 64 registers: the next phase's
// CTA fits on the same SM while this one runs):
//  * the CTA owns a slice of rows, held whole in shared memory, copied by
//    1-D bulk copies in up to 16 pieces that each complete on their own
//    mbarrier.  With static weights the copies are issued BEFORE the wait
//    on the previous kernel, so the weights of the next phases stream from
//    HBM while this one computes;
//  * the input is either float x (quantised in the prologue by the whole
//    CTA, same element arithmetic as quantize.cu) or already Q8_0 -- the
//    previous phase wrote it -- and then the CTA loads it once into shared
//    memory (every CTA reads the same few L2 lines: one request per line
//    and CTA, not one per warp);
//  * warp w owns one K-chunk of at most 64 blocks (two per lane), keeps that
//    chunk of x in registers and runs down its rows four at a time: per
//    block one 16-byte shared load of weights, dp4a, the int32 block sum
//    turned into float exactly, ((float)sumi * dw) * dx accumulated; the
//    four rows are reduced together by a transposed butterfly;
//  * a product may also write its output quantised to Q8_0 (for the next
//    phase): its rows are then split between CTAs in whole 32-row blocks,
//    and each block is quantised from the float values that were stored.
//    The host splits the rows so that the largest CTA share is as small as
//    those block boundaries allow.
#include "phase_common.cuh"

#include <cstdlib>

namespace mlq {

struct PieceTable {
  int n;
  int start[kPhPieces];  // first slice row
  int cnt[kPhPieces];
  int prod[kPhPieces];
  int lrow[kPhPieces];   // first row inside the product
};

template <int QT, int NW>
__global__ void __launch_bounds__(NW * 32, 32 / NW) phase_kernel(const __grid_constant__ PhaseArgs pa) {
  // one code image for both input kinds (float x, or Q8_0 from an earlier phase)
  const int IN = pa.a.x == nullptr ? 1 : 0;
  constexpr int kPhWarps = NW;
  constexpr int kPhThreads = NW * 32;
  const FusedArgs &a = pa.a;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kPhPieces];
  __shared__ PieceTable pt;
  __shared__ int abort_flag;
  __shared__ int slice_ok;
  const int nb = a.nb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ra = pa.bounds[blockIdx.x];
  const int rb = pa.bounds[blockIdx.x + 1];
  const int nr = rb - ra;
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  uint8_t *wq_s = smem + a.smem_w;
  float *wd_s = reinterpret_cast<float *>(smem + a.smem_wd);
  const int part_cap = static_cast<int>((a.smem_w - a.smem_part) / 4);  // floats of part_s

  if (tid == 0) {
    // pieces of at most ceil(nr / 8) rows, never spanning two products
    const int rpp = nr > 0 ? (nr + kPhPieces / 2 - 1) / (kPhPieces / 2) : 1;
    int np = 0, off = 0;
    for (int j = 0; j < a.nproducts; ++j) {
      const int lo = max(ra, off) - off, hi = min(rb, off + a.prod[j].rows) - off;
      for (int r = lo; r < hi; r += rpp) {
        if (!in_bounds(np < kPhPieces, a.status)) break;
        pt.start[np] = off + r - ra;
        pt.cnt[np] = min(rpp, hi - r);
        pt.prod[np] = j;
        pt.lrow[np] = r;
        mbar_init(smem_addr(&bars[np]), 1);  // one arrival, with the piece's byte count
        ++np;
      }
      off += a.prod[j].rows;
    }
    pt.n = np;
    abort_flag = 0;
    slice_ok = 1;
    fence_mbar_init();
  }
  __syncthreads();
  const int np = pt.n;
  // Bulk copies of the slice, one piece per lane of warp 0.  With static
  // weights they are issued before the dependency wait and land while the
  // previous kernel runs: then the whole slice completes on ONE mbarrier,
  // checked once per warp (each barrier check costs a few hundred cycles on
  // an SM whose barrier unit is busy with other CTAs' incoming copies).
  // Otherwise they are issued once the input has been read and each piece
  // completes on its own mbarrier, so rows are reduced as pieces land.
  const bool one_bar = a.early != 0;
  auto issue_slice = [&]() {
    if (warp != 0) return;
    if (one_bar && lane == 0 && np > 0)
      mbar_arrive_expect_tx(smem_addr(&bars[0]),
                            static_cast<uint32_t>(nr) * static_cast<uint32_t>(rowq + 4u * nb));
    __syncwarp();
    // the piece lies inside the slice area (rows_cap rows of quants, then scales)
    const size_t rows_cap = rowq > 0 ? (a.smem_wd - a.smem_w) / rowq : 0;
    if (lane < np && in_bounds(static_cast<size_t>(pt.start[lane]) + pt.cnt[lane] <= rows_cap, a.status)) {
      const int p = lane;
      const FusedProduct &pr = a.prod[pt.prod[p]];
      const uint32_t qb = static_cast<uint32_t>(pt.cnt[p] * rowq);
      const uint32_t db = static_cast<uint32_t>(pt.cnt[p]) * nb * 4;
      const uint32_t bar = smem_addr(&bars[one_bar ? 0 : p]);
      if (!one_bar) mbar_arrive_expect_tx(bar, qb + db);
      bulk_copy_g2s(smem_addr(wq_s + static_cast<size_t>(pt.start[p]) * rowq),
                    pr.wq + static_cast<size_t>(pt.lrow[p]) * rowq, qb, bar);
      bulk_copy_g2s(smem_addr(wd_s + static_cast<size_t>(pt.start[p]) * nb),
                    pr.wd + static_cast<size_t>(pt.lrow[p]) * nb, db, bar);
    }
  };
  if (a.early) issue_slice();
  // Let the next phase's kernel be scheduled now: it still waits for this
  // grid to complete before it reads anything we write.
  griddep_launch_dependents();
  if (one_bar && np > 0 && warp == kPhWarps - 1) {
    // One warp checks the slice while the previous kernel still runs; the
    // CTA barrier after the input publishes the result (and orders the
    // slice's bytes) for every warp, so no warp checks it again.
    if (!mbar_wait_warp(smem_addr(&bars[0]), 0, a.wait_ns) && lane == 0) slice_ok = 0;
  }
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + static_cast<size_t>(nb) * kQK);
  // A static float input (no earlier work writes it) is read and quantised
  // before the dependency wait; CTA 0 writes xq_out / xd_out after it.
  const bool early_in = IN == 0 && a.early_input != 0;
  const bool writer = blockIdx.x == 0 && a.xq_out != nullptr;
  if (early_in && (nr > 0 || writer)) quantize_input<NW>(a.x, nb, nullptr, nullptr, false, xq_s, xd_s, tid);
  griddep_wait();  // the input (and, without static weights, W) may come from the previous kernel

  bool ok = true;
  if (IN == 0) {
    if (!early_in) {
      if (nr > 0 || writer) phase_quantize<NW>(a, xq_s, xd_s, tid);
    } else if (writer) {
      __syncthreads();
      store_input_copy(xq_s, xd_s, nb, a.xq_out, a.xd_out, tid, kPhThreads);
    }
    __syncthreads();
  } else if (nr > 0) {
    // The Q8_0 input (n bytes + n/32 scales): one 16-byte load per thread
    // and unit, into shared memory; each CTA reads each line once.
    const int uq = nb * 2, nu = nb * 2 + nb / 4;
    for (int base = 0; base < nu; base += 4 * kPhThreads) {  // all loads before any store
      int4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = base + j * kPhThreads + tid;
        if (u < nu)
          v[j] = u < uq ? __ldcg(reinterpret_cast<const int4 *>(a.xq_in) + u)
                        : __ldcg(reinterpret_cast<const int4 *>(a.xd_in) + (u - uq));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = base + j * kPhThreads + tid;
        if (u < uq) reinterpret_cast<int4 *>(xq_s)[u] = v[j];
        else if (u < nu) reinterpret_cast<int4 *>(xd_s)[u - uq] = v[j];
      }
    }
    __syncthreads();
  }
  if (one_bar && nr > 0 && !slice_ok) {
    ok = false;
    if (tid == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
  }
  const int C = a.nchunks;                 // 1, 2, 4 or 8
  const int c = warp & (C - 1);            // this warp's chunk
  const int G = kPhWarps / C;              // warps per chunk
  const int i0 = warp / C;
  const int u0 = c * a.chunk_blocks + lane;
  const bool direct = C == 1 && !a.any_yq;
  float *part_s = reinterpret_cast<float *>(smem + a.smem_part);
  XChunk xc;
  if (nr > 0) load_chunk<QT>(xc, xq_s, xd_s, nb, c * a.chunk_blocks, a.chunk_blocks, lane);
  // The input has landed: only now queue (non-static) weight copies and the
  // L2 hints (an SM serves its reads in order, so anything queued first
  // would delay the input).
  if (!a.early) issue_slice();
  if (a.npf > 0 && warp == kPhWarps - 1) {
    // this CTA's share of the ranges to hint into L2, 16 KB per lane step
    size_t total = 0;
    for (int i = 0; i < a.npf; ++i) total += a.pf_bytes[i];
    const size_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
    size_t off = 0;
    for (int i = 0; i < a.npf; ++i) {
      const size_t b0 = max(lo, off), b1 = min(hi, off + a.pf_bytes[i]);
      if (b1 > b0) {
        const uintptr_t base = reinterpret_cast<uintptr_t>(a.pf_ptr[i]);
        const uintptr_t s0 = (base + (b0 - off) + 15) & ~static_cast<uintptr_t>(15);
        const uintptr_t e0 = (base + (b1 - off)) & ~static_cast<uintptr_t>(15);
        for (uintptr_t q = s0 + static_cast<uintptr_t>(lane) * 16384; q < e0; q += 32 * 16384)
          bulk_prefetch_l2(reinterpret_cast<const void *>(q),
                           static_cast<uint32_t>(e0 - q < 16384 ? e0 - q : 16384));
      }
      off += a.pf_bytes[i];
    }
  }
  if (nr > 0 && ok) {
    int pw = 0;  // pieces [0, pw) have landed
    for (int r0 = i0; r0 < nr; r0 += 4 * G) {
      const int rlast = min(nr - 1, r0 + 3 * G);
      while (!one_bar && pw < np && pt.start[pw] <= rlast) {
        if (!mbar_wait_warp(smem_addr(&bars[pw]), 0, a.wait_ns)) {
          ok = false;
          if (lane == 0 && atomicExch(&abort_flag, 1) == 0) set_status(a.status, kStatusTimeout);
          break;
        }
        ++pw;
      }
      if (!ok) break;
      float acc[4];
      if (QT == 1) {
        rows4_q4(acc, wq_s, wd_s, rowq, nb, r0, G, nr, xc, u0);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = r0 + G * j;
          acc[j] = row < nr ? row_part<QT>(wq_s + static_cast<size_t>(row) * rowq,
                                           wd_s + static_cast<size_t>(row) * nb, xc, u0, lane)
                            : 0.0f;
        }
      }
      const float v = reduce4(acc[0], acc[1], acc[2], acc[3], lane);
      const int row = r0 + G * (lane >> 3);
      if ((lane & 7) == 0 && row < nr) {
        if (direct) {
          int lr;
          const int j = phase_product(a, ra + row, &lr);
          if (in_bounds(lr >= 0 && lr < a.prod[j].rows, a.status)) a.prod[j].y[lr] = v;
        } else if (in_bounds(row * C + c < part_cap, a.status)) {
          part_s[row * C + c] = v;
        }
      }
    }
  }
  if (!direct) {
    __syncthreads();
    // Each row's float value: the sum of its K-chunks in a fixed order.
    // Rows of a product with a quantised output are stored by the warp that
    // quantises their 32-row block (below); with one K-chunk the other rows
    // are stored in the same pass, so one CTA barrier suffices.
    for (int row = tid; row < nr; row += kPhThreads) {
      int lr;
      const int j = phase_product(a, ra + row, &lr);
      if (C == 1 && a.prod[j].yq != nullptr) continue;
      if (!in_bounds((row + 1) * C <= part_cap && lr >= 0 && lr < a.prod[j].rows, a.status)) continue;
      float v = part_s[row * C];
      for (int cc = 1; cc < C; ++cc) v += part_s[row * C + cc];
      a.prod[j].y[lr] = v;
      part_s[row * C] = v;
    }
    if (a.any_yq) {
      if (C > 1) __syncthreads();
      // quantise each whole 32-row block of a product that asks for it,
      // from exactly the float values stored in y; one warp per block
      int t = 0;
      int off = 0;
      for (int j = 0; j < a.nproducts; off += a.prod[j].rows, ++j) {
        const int lo = max(ra, off), hi = min(rb, off + a.prod[j].rows);
        if (a.prod[j].yq == nullptr || hi <= lo) continue;
        for (int g = lo; g < hi; g += kQK, ++t) {
          if ((t & (kPhWarps - 1)) != warp) continue;
          const bool ok = in_bounds((g - ra + lane + 1) * C <= part_cap && g - off + lane >= 0 &&
                                        g - off + lane < a.prod[j].rows, a.status);
          const float v = ok ? part_s[(g - ra + lane) * C] : 0.0f;
          if (C == 1 && ok) a.prod[j].y[g - off + lane] = v;
          uint32_t m = __float_as_uint(fabsf(v));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
          const float amax = __uint_as_float(m);
          const float dd = amax / 127.0f;
          const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
          if (ok) a.prod[j].yq[g - off + lane] = static_cast<int8_t>(quant_one(v, id));
          if (lane == 0 && ok) a.prod[j].yd[(g - off) / kQK] = dd;
        }
      }
    }
  }
  // Gave up a wait: our copies may still be landing, wait for them (bounded).
  // With one barrier every warp knows the outcome since the input barrier;
  // with pieces a warp may have given up alone, so the CTA syncs first.
  if (!one_bar) __syncthreads();
  if (tid == 0 && (one_bar ? !ok : abort_flag != 0)) {
    for (int p = 0; p < (one_bar ? 1 : np); ++p) mbar_wait_bounded(smem_addr(&bars[p]), 0, kDrainWaitNs);
  }
}

template <int QT, int NW>
static cudaError_t launch_phase_t(const LaunchCtx &ctx, const FusedArgs &args) {
  constexpr int kPhWarps = NW;
  PhaseArgs pa;
  pa.a = args;
  FusedArgs &a = pa.a;
  const int nb = a.nb;
  int C = 1;
  while (C * kPhChunk < nb) C *= 2;
  // 16-byte bulk copies of whole scale rows need nb % 4 == 0
  if (C > kPhWarps || a.total_rows <= 0 || nb % 4 != 0) return cudaErrorNotSupported;
  a.nchunks = C;
  a.chunk_blocks = (nb + C - 1) / C;
  int grid = ctx.num_sms < a.total_rows ? ctx.num_sms : a.total_rows;
  grid = grid < kPhMaxGrid ? grid : kPhMaxGrid;
  const int rows_max = plan_rows(a, a.total_rows, grid, pa.bounds);
  const size_t rowq = static_cast<size_t>(nb) * (QT == 1 ? 16 : 32);
  auto up128 = [](size_t v) { return (v + 127) / 128 * 128; };
  const size_t xs = up128(static_cast<size_t>(nb) * (kQK + 4));
  const bool direct = C == 1 && !a.any_yq;
  const size_t ps = direct ? 0 : up128(static_cast<size_t>(rows_max) * C * 4);
  a.smem_part = static_cast<unsigned>(xs);
  a.smem_w = static_cast<unsigned>(xs + ps);
  a.smem_wd = static_cast<unsigned>(xs + ps + rows_max * rowq);
  const size_t smem = a.smem_wd + static_cast<size_t>(rows_max) * nb * 4;
  if (smem > kPhBudget) return cudaErrorNotSupported;
  diag_note("phase: products=%d rows=%d K=%d rows/CTA<=%d chunks=%d slice=%zuB input=%s q8_out=%d early=%d",
            a.nproducts, a.total_rows, nb * kQK, rows_max, C, smem - a.smem_w, a.x != nullptr ? "f32" : "q8",
            a.any_yq, a.early);
  auto kern = phase_kernel<QT, NW>;
  prefer_max_shared(kern);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(NW * 32), smem, ctx, pa);
}

cudaError_t launch_phase(const LaunchCtx &ctx, int qtype, const FusedArgs &a) {
  static_assert(sizeof(PhaseArgs) <= 4096, "kernel parameters");
  // MLQ_PHASE_WARPS=16|8: CTA width (A/B timing).  16 warps (two CTAs per
  // SM) reduce a slice faster; 8 would let four phases share an SM, which
  // measured slower on the TinyLlama layer chain.
  static const int wide = [] {
    const char *e = std::getenv("MLQ_PHASE_WARPS");
    return !(e != nullptr && e[0] == '8');
  }();
  // MLQ_PHASE_KERNEL=ring: always the ring kernel (A/B timing, tests)
  static const bool ring_only = [] {
    const char *e = std::getenv("MLQ_PHASE_KERNEL");
    return e != nullptr && e[0] == 'r';
  }();
  if (!ring_only) {
    cudaError_t e;
    if (wide) e = qtype == 1 ? launch_phase_t<1, 16>(ctx, a) : launch_phase_t<0, 16>(ctx, a);
    else e = qtype == 1 ? launch_phase_t<1, 8>(ctx, a) : launch_phase_t<0, 8>(ctx, a);
    if (e != cudaErrorNotSupported) return e;
  }
  // the CTA slices do not fit in shared memory: stream them through a ring
  return launch_phase_ring(ctx, qtype, a);
}

}  // namespace mlq
