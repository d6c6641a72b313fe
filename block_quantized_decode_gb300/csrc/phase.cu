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
#include "mlq_device.cuh"
#include "mlq_launch.h"

#include <cstdlib>

namespace mlq {

constexpr int kPhPieces = 16;
constexpr int kPhChunk = 64;                 // blocks of K per warp chunk: two per lane
constexpr size_t kPhBudget = 120 * 1024;     // dynamic shared memory of one CTA

// int32 -> float32 through the exponent bias: for |s| < 2^22 the float whose
// bit pattern is 0x4B400000 + s equals 1.5 * 2^23 + s exactly, so one
// subtraction of 1.5 * 2^23 yields s exactly.  The bias is folded into the
// dp4a accumulator, so the conversion costs one float subtraction.
constexpr int kMagicBits = 0x4B400000;
constexpr float kMagic = 12582912.0f;

// unsigned bytes of a times signed bytes of b, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The launch arguments: the phase plus its row split, computed on the host
// (rows [bounds[b], bounds[b+1]) of the concatenated products go to CTA b).
constexpr int kPhMaxGrid = 160;
struct PhaseArgs {
  FusedArgs a;
  int bounds[kPhMaxGrid + 1];
};

__device__ __forceinline__ int phase_product(const FusedArgs &a, int g, int *local) {
  int j = 0, off = 0;
  while (j + 1 < a.nproducts && g >= off + a.prod[j].rows) {
    off += a.prod[j].rows;
    ++j;
  }
  *local = g - off;
  return j;
}

// Quantise float x (nb blocks) into shared memory, eight lanes per block,
// all loads of up to eight passes issued before any block is reduced.
// CTA 0 also writes the copy asked for in xq_out / xd_out.
template <int NW>
__device__ __forceinline__ void phase_quantize(const FusedArgs &a, int8_t *xq_s, float *xd_s,
                                               int tid) {
  const int nb = a.nb;
  const int part = tid & 7;
  const bool writer = blockIdx.x == 0 && a.xq_out != nullptr;
  constexpr int kPer = NW * 32 / 8;
  constexpr int kPass = 8;
  // every CTA reads all of x: start each at another block to spread the requests
  const int rot = static_cast<int>((static_cast<long long>(blockIdx.x) * 37) % nb);
  for (int base0 = 0; base0 < nb; base0 += kPer * kPass) {
    float4 v[kPass];
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int i = base0 + p * kPer + (tid >> 3);
      const int b = i + rot < nb ? i + rot : i + rot - nb;
      v[p] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nb) v[p] = __ldcg(reinterpret_cast<const float4 *>(a.x + static_cast<size_t>(b) * kQK + part * 4));
    }
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      if (base0 + p * kPer >= nb) break;  // uniform across the CTA
      const int i = base0 + p * kPer + (tid >> 3);
      const int b = i + rot < nb ? i + rot : i + rot - nb;
      uint32_t m = max(max(__float_as_uint(fabsf(v[p].x)), __float_as_uint(fabsf(v[p].y))),
                       max(__float_as_uint(fabsf(v[p].z)), __float_as_uint(fabsf(v[p].w))));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      const float amax = __uint_as_float(m);
      const float dd = amax / 127.0f;
      const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
      const int q0 = quant_one(v[p].x, id), q1 = quant_one(v[p].y, id), q2 = quant_one(v[p].z, id),
                q3 = quant_one(v[p].w, id);
      const uint32_t packed = (q0 & 0xff) | ((q1 & 0xff) << 8) | ((q2 & 0xff) << 16) |
                              (static_cast<uint32_t>(q3 & 0xff) << 24);
      if (i < nb) {
        *reinterpret_cast<uint32_t *>(xq_s + b * kQK + part * 4) = packed;
        if (part == 0) xd_s[b] = dd;
        if (writer) {
          *reinterpret_cast<uint32_t *>(a.xq_out + static_cast<size_t>(b) * kQK + part * 4) = packed;
          if (part == 0) a.xd_out[b] = dd;
        }
      }
    }
  }
}

// A warp's chunk of the quantised input: lane l holds blocks u0 and u0 + 32
// (u0 = chunk start + l).  Q8_0 weights: the lane reads the two 16-byte
// halves of a block in the order h, 1 - h with h = bit 2 of the lane (no
// shared-memory bank conflicts), so x is held in that order too.
struct XChunk {
  int4 x[2][2];
  float d[2];
  int adj[2];   // dp4a start value: bias (+ the -8 fold of Q4_0, -8 * sum q)
  bool v[2];
};

template <int QT>
__device__ __forceinline__ void load_chunk(XChunk &c, const int8_t *xq, const float *xd, int nb,
                                           int cbeg, int cblocks, int lane) {
  // Lanes read their two 16-byte halves in the order h, 1 - h (h = bit 2 of
  // the lane): the eight lanes of a quarter warp then hit distinct banks.
  const int h = (lane >> 2) & 1;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int off = lane + 32 * k;
    const int u = cbeg + off;
    c.v[k] = off < cblocks && u < nb;
    int4 first = make_int4(0, 0, 0, 0), second = first;
    float d = 0.0f;
    if (c.v[k]) {
      const int4 *src = reinterpret_cast<const int4 *>(xq + static_cast<size_t>(u) * kQK);
      first = src[h];
      second = src[h ^ 1];
      d = xd[u];
    }
    if (QT == 1) {  // Q4_0: x[k][0] = elements 0..15 (low nibbles), x[k][1] = 16..31
      c.x[k][0] = h ? second : first;
      c.x[k][1] = h ? first : second;
    } else {        // Q8_0: kept in the lane's read order, as the weights are read
      c.x[k][0] = first;
      c.x[k][1] = second;
    }
    c.d[k] = d;
    int adj = kMagicBits;
    if (QT == 1) {
      constexpr int kOnes = 0x01010101;
      int sx = __dp4a(first.x, kOnes, 0);
      sx = __dp4a(first.y, kOnes, sx);
      sx = __dp4a(first.z, kOnes, sx);
      sx = __dp4a(first.w, kOnes, sx);
      sx = __dp4a(second.x, kOnes, sx);
      sx = __dp4a(second.y, kOnes, sx);
      sx = __dp4a(second.z, kOnes, sx);
      sx = __dp4a(second.w, kOnes, sx);
      adj -= 8 * sx;
    }
    c.adj[k] = adj;
  }
}

// sum over this lane's (at most two) blocks of ((float)sumi * dw) * dx
template <int QT>
__device__ __forceinline__ float row_part(const uint8_t *wrow, const float *drow, const XChunk &c,
                                          int u0, int lane) {
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (!c.v[k]) continue;
    const int u = u0 + 32 * k;
    const float dw = drow[u];
    int s;
    if (QT == 1) {
      const uint4 w = *reinterpret_cast<const uint4 *>(wrow + u * 16);
      const int4 xa = c.x[k][0], xb = c.x[k][1];
      constexpr uint32_t kLo = 0x0F0F0F0Fu, kHi = 0xF0F0F0F0u;
      int lo = __dp4a(static_cast<int>(w.x & kLo), xa.x, c.adj[k]);
      lo = __dp4a(static_cast<int>(w.y & kLo), xa.y, lo);
      lo = __dp4a(static_cast<int>(w.z & kLo), xa.z, lo);
      lo = __dp4a(static_cast<int>(w.w & kLo), xa.w, lo);
      int hi = dp4a_us(w.x & kHi, xb.x, 0);  // 16 * (high nibble) per byte: exact multiple of 16
      hi = dp4a_us(w.y & kHi, xb.y, hi);
      hi = dp4a_us(w.z & kHi, xb.z, hi);
      hi = dp4a_us(w.w & kHi, xb.w, hi);
      s = lo + (hi >> 4);
    } else {
      const int h = (lane >> 2) & 1;
      const uint4 w0 = *reinterpret_cast<const uint4 *>(wrow + u * 32 + 16 * h);
      const uint4 w1 = *reinterpret_cast<const uint4 *>(wrow + u * 32 + 16 * (h ^ 1));
      const int4 xa = c.x[k][0], xb = c.x[k][1];
      s = __dp4a(static_cast<int>(w0.x), xa.x, c.adj[k]);
      s = __dp4a(static_cast<int>(w0.y), xa.y, s);
      s = __dp4a(static_cast<int>(w0.z), xa.z, s);
      s = __dp4a(static_cast<int>(w0.w), xa.w, s);
      s = __dp4a(static_cast<int>(w1.x), xb.x, s);
      s = __dp4a(static_cast<int>(w1.y), xb.y, s);
      s = __dp4a(static_cast<int>(w1.z), xb.z, s);
      s = __dp4a(static_cast<int>(w1.w), xb.w, s);
    }
    const float sumi = __fsub_rn(__int_as_float(s), kMagic);
    acc = __fmaf_rn(__fmul_rn(sumi, dw), c.d[k], acc);
  }
  return acc;
}

// Q4_0, four rows at once, one of the lane's two blocks at a time: the
// four rows' shared-memory loads of a block are issued before any of its
// arithmetic (independent work for the scheduler, within 64 registers).
// Rows past the slice end (row >= nr) read the last row and contribute 0.
__device__ __forceinline__ void rows4_q4(float acc[4], const uint8_t *wq_s, const float *wd_s,
                                         size_t rowq, int nb, int r0, int G, int nr,
                                         const XChunk &c, int u0) {
  const uint8_t *wr[4];
  const float *dr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = min(r0 + G * j, nr - 1);
    wr[j] = wq_s + static_cast<size_t>(row) * rowq;
    dr[j] = wd_s + static_cast<size_t>(row) * nb;
    acc[j] = 0.0f;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (!c.v[k]) continue;
    const int u = u0 + 32 * k;
    uint4 w[4];
    float dw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w[j] = *reinterpret_cast<const uint4 *>(wr[j] + u * 16);
      dw[j] = dr[j][u];
    }
    constexpr uint32_t kLo = 0x0F0F0F0Fu, kHi = 0xF0F0F0F0u;
    const int4 xa = c.x[k][0], xb = c.x[k][1];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = w[j];
      int lo = __dp4a(static_cast<int>(q.x & kLo), xa.x, c.adj[k]);
      int hi = dp4a_us(q.x & kHi, xb.x, 0);  // 16 * (high nibble) per byte: exact multiple of 16
      lo = __dp4a(static_cast<int>(q.y & kLo), xa.y, lo);
      hi = dp4a_us(q.y & kHi, xb.y, hi);
      lo = __dp4a(static_cast<int>(q.z & kLo), xa.z, lo);
      hi = dp4a_us(q.z & kHi, xb.z, hi);
      lo = __dp4a(static_cast<int>(q.w & kLo), xa.w, lo);
      hi = dp4a_us(q.w & kHi, xb.w, hi);
      const float sumi = __fsub_rn(__int_as_float(lo + (hi >> 4)), kMagic);
      acc[j] = __fmaf_rn(__fmul_rn(sumi, dw[j]), c.d[k], acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = r0 + G * j < nr ? acc[j] : 0.0f;
}

// Four per-lane partial sums -> four warp sums.  Lane l returns the sum of
// row (l >> 3) & 3; fixed order, so the result is deterministic.
__device__ __forceinline__ float reduce4(float a0, float a1, float a2, float a3, int lane) {
  const bool b4 = (lane & 16) != 0;
  float k0 = b4 ? a2 : a0, k1 = b4 ? a3 : a1;
  const float s0 = b4 ? a0 : a2, s1 = b4 ? a1 : a3;
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  const bool b3 = (lane & 8) != 0;
  float k = b3 ? k1 : k0;
  const float s = b3 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, s, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

struct PieceTable {
  int n;
  int start[kPhPieces];  // first slice row
  int cnt[kPhPieces];
  int prod[kPhPieces];
  int lrow[kPhPieces];   // first row inside the product
};

template <int QT, int NW>
__global__ void __launch_bounds__(NW * 32, 32 / NW) phase_kernel(const __grid_constant__ PhaseArgs pa) {
  // One code image for both input kinds: every phase of a chain then runs
  // the same instructions, which stay in the SM's instruction cache.
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

  if (tid == 0) {
    // pieces of at most ceil(nr / 8) rows, never spanning two products
    const int rpp = nr > 0 ? (nr + kPhPieces / 2 - 1) / (kPhPieces / 2) : 1;
    int np = 0, off = 0;
    for (int j = 0; j < a.nproducts; ++j) {
      const int lo = max(ra, off) - off, hi = min(rb, off + a.prod[j].rows) - off;
      for (int r = lo; r < hi; r += rpp) {
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
    if (lane < np) {
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
  griddep_wait();  // the input (and, without static weights, W) may come from the previous kernel

  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + static_cast<size_t>(nb) * kQK);
  bool ok = true;
  if (IN == 0) {
    if (nr > 0 || (blockIdx.x == 0 && a.xq_out != nullptr)) phase_quantize<NW>(a, xq_s, xd_s, tid);
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
          a.prod[j].y[lr] = v;
        } else {
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
          const float v = part_s[(g - ra + lane) * C];
          if (C == 1) a.prod[j].y[g - off + lane] = v;
          uint32_t m = __float_as_uint(fabsf(v));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
          const float amax = __uint_as_float(m);
          const float dd = amax / 127.0f;
          const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
          a.prod[j].yq[g - off + lane] = static_cast<int8_t>(quant_one(v, id));
          if (lane == 0) a.prod[j].yd[(g - off) / kQK] = dd;
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

// ---- row split --------------------------------------------------------------
// A CTA boundary may fall anywhere, except inside a product whose output is
// quantised: there only at whole 32-row blocks of that product.
static int cut_down(const FusedArgs &a, int g) {  // largest allowed cut <= g
  int off = 0;
  for (int j = 0; j < a.nproducts; ++j) {
    const int end = off + a.prod[j].rows;
    if (g > off && g < end && a.prod[j].yq != nullptr) return off + ((g - off) & ~31);
    off = end;
  }
  return g;
}
static int cut_up(const FusedArgs &a, int g) {  // smallest allowed cut >= g
  int off = 0;
  for (int j = 0; j < a.nproducts; ++j) {
    const int end = off + a.prod[j].rows;
    if (g > off && g < end && a.prod[j].yq != nullptr) return off + ((g - off + 31) & ~31);
    off = end;
  }
  return g;
}
// Split `total` rows into `grid` runs of at most L rows at allowed cuts.
// balanced: each CTA takes its share of what is left (capped at L), so the
// rows spread over all CTAs; otherwise each takes as much as it may
// (greedy: uses the fewest CTAs, which decides whether L is feasible).
static bool split_rows(const FusedArgs &a, int total, int grid, int L, bool balanced, int *bounds) {
  int pos = 0;
  bounds[0] = 0;
  for (int b = 0; b < grid; ++b) {
    const int rem = total - pos;
    int take = L;
    if (balanced) {
      const int share = (rem + (grid - b) - 1) / (grid - b);
      take = share < L ? share : L;
    }
    int end = cut_down(a, pos + take < total ? pos + take : total);
    if (end <= pos && pos < total) {
      end = cut_up(a, pos + 1);
      if (end - pos > L) return false;
    }
    bounds[b + 1] = end;
    pos = end;
  }
  return pos == total;
}
// The split with the smallest largest run (the slowest CTA sets the time).
static int plan_rows(const FusedArgs &a, int total, int grid, int *bounds) {
  int lo = 1, hi = total;
  while (lo < hi) {  // smallest L the greedy split achieves
    const int mid = lo + (hi - lo) / 2;
    if (split_rows(a, total, grid, mid, false, bounds)) hi = mid;
    else lo = mid + 1;
  }
  if (!split_rows(a, total, grid, lo, true, bounds)) split_rows(a, total, grid, lo, false, bounds);
  int mx = 0;
  for (int b = 0; b < grid; ++b) mx = bounds[b + 1] - bounds[b] > mx ? bounds[b + 1] - bounds[b] : mx;
  return mx;
}

template <int QT, int NW>
static cudaError_t launch_phase_t(const LaunchCtx &ctx, const FusedArgs &args) {
  const int IN = args.x == nullptr ? 1 : 0;
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
  if (wide) return qtype == 1 ? launch_phase_t<1, 16>(ctx, a) : launch_phase_t<0, 16>(ctx, a);
  return qtype == 1 ? launch_phase_t<1, 8>(ctx, a) : launch_phase_t<0, 8>(ctx, a);
}

}  // namespace mlq
