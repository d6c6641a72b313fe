// phase_common.cuh -- pieces shared by the two phase kernels (phase.cu:
// the CTA's weight slice held whole in shared memory; phase_ring.cu: the
// slice streamed through a ring of shared-memory stages): the quantised
// input held in registers per warp K-chunk, the exact int32 -> float block
// sums, the four-row reduction, the in-CTA quantisation of a float input,
// and the host-side row split.  Definitions: page "Legacy-ISA ML Inference
// Runtime -- Design Spec", Sec. 4 (Q4_0 / Q8_0 blocks, block dot), Sec. 5
// (quantize_q8 rounding, matvec).
#pragma once

#include "mlq_device.cuh"
#include "mlq_launch.h"

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
// With `writer`, the CTA also writes the quantisation to xq_out / xd_out.
template <int NW>
__device__ __forceinline__ void quantize_input(const float *x, int nb, int8_t *xq_out,
                                               float *xd_out, bool writer, int8_t *xq_s,
                                               float *xd_s, int tid) {
  const int part = tid & 7;
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
      if (i < nb) v[p] = __ldcg(reinterpret_cast<const float4 *>(x + static_cast<size_t>(b) * kQK + part * 4));
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
          *reinterpret_cast<uint32_t *>(xq_out + static_cast<size_t>(b) * kQK + part * 4) = packed;
          if (part == 0) xd_out[b] = dd;
        }
      }
    }
  }
}
// The quantised input, already in shared memory, to xq_out / xd_out (16-byte
// units; nb is a multiple of 4): for a CTA that quantised its input before
// the dependency wait, when it may only write once that wait has returned.
__device__ __forceinline__ void store_input_copy(const int8_t *xq_s, const float *xd_s, int nb, int8_t *xq_out,
                                                 float *xd_out, int tid, int nthreads) {
  const int uq = nb * 2, nu = nb * 2 + nb / 4;
  for (int u = tid; u < nu; u += nthreads) {
    if (u < uq) reinterpret_cast<int4 *>(xq_out)[u] = reinterpret_cast<const int4 *>(xq_s)[u];
    else reinterpret_cast<int4 *>(xd_out)[u - uq] = reinterpret_cast<const int4 *>(xd_s)[u - uq];
  }
}
template <int NW>
__device__ __forceinline__ void phase_quantize(const FusedArgs &a, int8_t *xq_s, float *xd_s,
                                               int tid) {
  quantize_input<NW>(a.x, a.nb, a.xq_out, a.xd_out, blockIdx.x == 0 && a.xq_out != nullptr, xq_s,
                     xd_s, tid);
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
// rows4_q4 for Q8_0 weights: the same block arithmetic as row_part<0>,
// with the shared-memory loads of the four rows issued before any dp4a.
__device__ __forceinline__ void rows4_q8(float acc[4], const uint8_t *wq_s, const float *wd_s,
                                         size_t rowq, int nb, int r0, int G, int nr,
                                         const XChunk &c, int u0, int lane) {
  const uint8_t *wr[4];
  const float *dr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = min(r0 + G * j, nr - 1);
    wr[j] = wq_s + static_cast<size_t>(row) * rowq;
    dr[j] = wd_s + static_cast<size_t>(row) * nb;
    acc[j] = 0.0f;
  }
  const int h = (lane >> 2) & 1;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (!c.v[k]) continue;
    const int u = u0 + 32 * k;
    uint4 w0[4], w1[4];
    float dw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w0[j] = *reinterpret_cast<const uint4 *>(wr[j] + u * 32 + 16 * h);
      w1[j] = *reinterpret_cast<const uint4 *>(wr[j] + u * 32 + 16 * (h ^ 1));
      dw[j] = dr[j][u];
    }
    const int4 xa = c.x[k][0], xb = c.x[k][1];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int s = __dp4a(static_cast<int>(w0[j].x), xa.x, c.adj[k]);
      s = __dp4a(static_cast<int>(w0[j].y), xa.y, s);
      s = __dp4a(static_cast<int>(w0[j].z), xa.z, s);
      s = __dp4a(static_cast<int>(w0[j].w), xa.w, s);
      s = __dp4a(static_cast<int>(w1[j].x), xb.x, s);
      s = __dp4a(static_cast<int>(w1[j].y), xb.y, s);
      s = __dp4a(static_cast<int>(w1[j].z), xb.z, s);
      s = __dp4a(static_cast<int>(w1[j].w), xb.w, s);
      const float sumi = __fsub_rn(__int_as_float(s), kMagic);
      acc[j] = __fmaf_rn(__fmul_rn(sumi, dw[j]), c.d[k], acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = r0 + G * j < nr ? acc[j] : 0.0f;
}

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


// ---- row split --------------------------------------------------------------
// A CTA boundary may fall anywhere, except inside a product whose output is
// quantised: there only at whole 32-row blocks of that product.
inline int cut_down(const FusedArgs &a, int g) {  // largest allowed cut <= g
  int off = 0;
  for (int j = 0; j < a.nproducts; ++j) {
    const int end = off + a.prod[j].rows;
    if (g > off && g < end && a.prod[j].yq != nullptr) return off + ((g - off) & ~31);
    off = end;
  }
  return g;
}
inline int cut_up(const FusedArgs &a, int g) {  // smallest allowed cut >= g
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
// front_heavy (balanced only): a share that falls between two allowed cuts
// is rounded up rather than down (within L), so the lower-numbered CTAs hold
// the larger shares.  CTAs of a launch start in index order as SMs free up
// (under programmatic dependent launch the last ones start several
// microseconds after the first), so the larger shares should go first.
inline bool split_rows(const FusedArgs &a, int total, int grid, int L, bool balanced, int *bounds,
                       bool front_heavy = false) {
  int pos = 0;
  bounds[0] = 0;
  for (int b = 0; b < grid; ++b) {
    const int rem = total - pos;
    int take = L;
    if (balanced) {
      const int share = (rem + (grid - b) - 1) / (grid - b);
      take = share < L ? share : L;
    }
    const int want = pos + take < total ? pos + take : total;
    int end = cut_down(a, want);
    if (front_heavy && end < want) {
      const int up = cut_up(a, want);
      if (up - pos <= L) end = up;
    }
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
inline int plan_rows(const FusedArgs &a, int total, int grid, int *bounds, bool front_heavy = false) {
  int lo = 1, hi = total;
  while (lo < hi) {  // smallest L the greedy split achieves
    const int mid = lo + (hi - lo) / 2;
    if (split_rows(a, total, grid, mid, false, bounds)) hi = mid;
    else lo = mid + 1;
  }
  if (!(front_heavy && split_rows(a, total, grid, lo, true, bounds, true)) &&
      !split_rows(a, total, grid, lo, true, bounds))
    split_rows(a, total, grid, lo, false, bounds);
  int mx = 0;
  for (int b = 0; b < grid; ++b) mx = bounds[b + 1] - bounds[b] > mx ? bounds[b + 1] - bounds[b] : mx;
  return mx;
}

}  // namespace mlq
