// layer.cu -- the floating-point steps of a decode layer around the
// products, each one launch, fused with the Q8_0 quantisation that follows
// it where the forward pass quantises the result.
//
// Definitions: page "Legacy-ISA ML Inference Runtime -- Design Spec",
// Sec. 5 (Kernel Interface: ml_k_rmsnorm, ml_k_softmax, ml_k_rope,
// ml_k_silu_mul, ml_k_add, ml_k_dot_f32, ml_k_axpy_f32; RoPE over the
// interleaved pairs (2i, 2i+1) with freq_i = theta^(-2i/head_dim) and cos/sin
// tables of [max_seq][head_dim/2]) and Sec. 6 (Forward pass per token:
// h = rmsnorm(x) -> quantize; rope(q, k, pos) and the KV cache row; per head
// s_t = dot(q_h, K_t) / sqrt(hd), softmax, o_h = sum_t p_t V_t; GQA: the KV
// head of query head h is h / (n_heads / n_kv_heads); g = silu(g) * u ->
// quantize; x += ...).  The readings (rmsnorm with eps inside the root, the
// KV cache row layout) are the oracle's.
//
// These steps move kilobytes, not megabytes: they are latency-bound, so each
// is one small launch, chained to its neighbours by programmatic dependent
// launch.  Reductions run in a fixed order (warp butterflies, then warps in
// index order), so results are deterministic; square roots and divisions
// are IEEE (no fast math), exp is CUDA's expf.
#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

constexpr int kNormThreads = 1024;
constexpr int kAttnThreads = 256;
constexpr int kMaxHeadDim = 256;  // MLQ_MAX_HEAD_DIM

// Sum over the CTA in a fixed order: butterflies inside each warp, then the
// warps' sums in index order by warp 0.  `red` holds one float per warp.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red may still be read from an earlier call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.0f;
  if (warp == 0) {
    s = lane < NT / 32 ? red[lane] : 0.0f;
    s = warp_sum(s);
  }
  if (threadIdx.x == 0) red[0] = s;
  __syncthreads();
  return red[0];
}
template <int NT>
__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float m = lane < NT / 32 ? red[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[0] = m;
  }
  __syncthreads();
  return red[0];
}

// Quantise the 32 values a warp holds (one per lane) as one Q8_0 block:
// the same element arithmetic as quantize.cu (Design Spec Sec. 5 rounding).
__device__ __forceinline__ void quant_block_warp(float v, int8_t *q, float *d, int lane) {
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float id = amax != 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
  q[lane] = static_cast<int8_t>(quant_one(v, id));
  if (lane == 0) *d = __fdiv_rn(amax, 127.0f);
}

// ---- rmsnorm (optionally after x += y), then optionally Q8_0 -------------
struct NormArgs {
  float *x;        // normalised input; with y, x += y first (written back)
  const float *y;  // or nullptr
  const float *w;
  float *h;        // fp32 output or nullptr
  int8_t *hq;      // Q8_0 output or nullptr (then hd too)
  float *hd;
  int n;
  float eps;
};

// Thread tid holds elements tid + 1024 j: the sum of squares and the
// per-block pass (block b = warp + 32 j, lane l -> element 32 b + l) use
// the same mapping, so x and w are loaded once, before the reduction.
constexpr int kNormRegs = 8;  // elements kept in registers per thread (n <= 8192)

__global__ void __launch_bounds__(kNormThreads, 1) rmsnorm_q8_kernel(const NormArgs a) {
  __shared__ float red[32];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  const bool regs = a.n <= kNormRegs * kNormThreads;
  float xv[kNormRegs], wv[kNormRegs];
  float ss = 0.0f;
  if (regs) {
#pragma unroll
    for (int j = 0; j < kNormRegs; ++j) {
      const int i = tid + j * kNormThreads;
      xv[j] = i < a.n ? a.x[i] : 0.0f;
      wv[j] = i < a.n ? a.w[i] : 0.0f;
      if (a.y != nullptr && i < a.n) xv[j] = __fadd_rn(xv[j], a.y[i]);
    }
#pragma unroll
    for (int j = 0; j < kNormRegs; ++j) {
      const int i = tid + j * kNormThreads;
      if (i < a.n) {
        if (a.y != nullptr) a.x[i] = xv[j];
        ss = __fmaf_rn(xv[j], xv[j], ss);
      }
    }
  } else {
    for (int i = tid; i < a.n; i += kNormThreads) {
      float v = a.x[i];
      if (a.y != nullptr) {
        v = __fadd_rn(v, a.y[i]);
        a.x[i] = v;
      }
      ss = __fmaf_rn(v, v, ss);
    }
  }
  ss = block_sum<kNormThreads>(ss, red);
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(a.n)), a.eps)));
  // h_j = w_j * (x_j * inv); one warp per 32-element block, so the block's
  // quantisation needs no shared memory
  const int lane = tid & 31, warp = tid >> 5;
  const int nblk = (a.n + 31) / 32;
  if (regs) {
#pragma unroll
    for (int j = 0; j < kNormRegs; ++j) {
      const int b = warp + j * (kNormThreads / 32);
      if (b < nblk) {  // warp-uniform
        const int i = tid + j * kNormThreads;
        const float hv = i < a.n ? __fmul_rn(wv[j], __fmul_rn(xv[j], inv)) : 0.0f;
        if (a.h != nullptr && i < a.n) a.h[i] = hv;
        if (a.hq != nullptr) quant_block_warp(hv, a.hq + b * 32, a.hd + b, lane);
      }
    }
  } else {
    for (int b = warp; b < nblk; b += kNormThreads / 32) {
      const int i = b * 32 + lane;
      float hv = 0.0f;
      if (i < a.n) {
        hv = __fmul_rn(a.w[i], __fmul_rn(a.x[i], inv));
        if (a.h != nullptr) a.h[i] = hv;
      }
      if (a.hq != nullptr) quant_block_warp(hv, a.hq + b * 32, a.hd + b, lane);
    }
  }
}

cudaError_t launch_rmsnorm_q8(const LaunchCtx &ctx, float *x, const float *y, const float *w,
                              float *h, int8_t *hq, float *hd, int n, float eps) {
  NormArgs a{x, y, w, h, hq, hd, n, eps};
  prefer_max_shared(rmsnorm_q8_kernel);
  return launch_kernel(rmsnorm_q8_kernel, dim3(1), dim3(kNormThreads), 0, ctx, a);
}

// ---- y += x -----------------------------------------------------------------
__global__ void add_kernel(float *y, const float *x, int n) {
  griddep_wait();
  griddep_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    y[i] = __fadd_rn(y[i], x[i]);
}

cudaError_t launch_add(const LaunchCtx &ctx, float *y, const float *x, int n) {
  const int blocks = (n + 255) / 256 < ctx.num_sms ? (n + 255) / 256 : ctx.num_sms;
  prefer_max_shared(add_kernel);
  return launch_kernel(add_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, ctx, y, x, n);
}

// ---- softmax of one vector (one CTA) -----------------------------------------
__global__ void __launch_bounds__(kNormThreads) softmax_kernel(float *x, int n) {
  __shared__ float red[32];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  float m = -INFINITY;
  for (int i = tid; i < n; i += kNormThreads) m = fmaxf(m, x[i]);
  m = block_max<kNormThreads>(m, red);
  float s = 0.0f;
  for (int i = tid; i < n; i += kNormThreads) s = __fadd_rn(s, expf(__fsub_rn(x[i], m)));
  s = block_sum<kNormThreads>(s, red);
  for (int i = tid; i < n; i += kNormThreads) x[i] = __fdiv_rn(expf(__fsub_rn(x[i], m)), s);
}

cudaError_t launch_softmax(const LaunchCtx &ctx, float *x, int n) {
  prefer_max_shared(softmax_kernel);
  return launch_kernel(softmax_kernel, dim3(1), dim3(kNormThreads), 0, ctx, x, n);
}

// ---- g = silu(g) * u, then optionally Q8_0 ------------------------------------
__global__ void silu_mul_q8_kernel(float *g, const float *u, int n, int8_t *gq, float *gd) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int nblk = (n + 31) / 32;
  for (int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblk; b += warps) {
    const int i = b * 32 + lane;
    float v = 0.0f;
    if (i < n) {
      const float a = g[i];
      v = __fmul_rn(__fdiv_rn(a, __fadd_rn(1.0f, expf(-a))), u[i]);
      g[i] = v;
    }
    if (gq != nullptr) quant_block_warp(v, gq + b * 32, gd + b, lane);
  }
}

cudaError_t launch_silu_mul_q8(const LaunchCtx &ctx, float *g, const float *u, int n, int8_t *gq,
                               float *gd) {
  const int nblk = (n + 31) / 32;
  int blocks = (nblk + 7) / 8;
  blocks = blocks < ctx.num_sms ? blocks : ctx.num_sms;
  prefer_max_shared(silu_mul_q8_kernel);
  return launch_kernel(silu_mul_q8_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, ctx, g, u, n, gq,
                       gd);
}

// ---- RoPE -------------------------------------------------------------------------
// Tables in double (an angle pos * freq in float would be off by ~1e-4 rad at
// pos ~ 2000), rounded once to float.
__global__ void rope_tables_kernel(float *cos_t, float *sin_t, int max_seq, int head_dim,
                                   float theta) {
  const int half = head_dim / 2;
  const long long total = static_cast<long long>(max_seq) * half;
  for (long long k = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; k < total;
       k += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(k / half), i = static_cast<int>(k % half);
    const double freq = pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(head_dim));
    const double ang = static_cast<double>(pos) * freq;
    cos_t[k] = static_cast<float>(cos(ang));
    sin_t[k] = static_cast<float>(sin(ang));
  }
}

cudaError_t launch_rope_tables(const LaunchCtx &ctx, float *cos_t, float *sin_t, int max_seq,
                               int head_dim, float theta) {
  const long long total = static_cast<long long>(max_seq) * (head_dim / 2);
  long long blocks = (total + 255) / 256;
  blocks = blocks < 4 * ctx.num_sms ? blocks : 4 * ctx.num_sms;
  rope_tables_kernel<<<static_cast<unsigned>(blocks > 0 ? blocks : 1), 256, 0, ctx.stream>>>(
      cos_t, sin_t, max_seq, head_dim, theta);
  return cudaGetLastError();
}

struct RopeArgs {
  float *q;            // n_heads x head_dim, rotated in place
  float *k;            // n_kv_heads x head_dim, rotated in place unless k_out
  float *k_out;        // or nullptr: the rotated k goes here (a KV cache row)
  const float *v;      // or nullptr: copied to v_out (the cache row)
  float *v_out;
  const float *cos_t;  // the table rows of the position, head_dim/2 each
  const float *sin_t;
  int head_dim, n_heads, n_kv_heads;
};

__global__ void rope_kernel(const RopeArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int half = a.head_dim / 2;
  const int nq = a.n_heads * half, nk = a.n_kv_heads * half;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < nq + nk; p += gridDim.x * blockDim.x) {
    const bool isq = p < nq;
    const int pp = isq ? p : p - nq;
    const int i = pp % half, e = 2 * pp;  // pair (2i, 2i+1) of its head, at element 2*pp
    const float *src = isq ? a.q : a.k;
    float *dst = isq ? a.q : (a.k_out != nullptr ? a.k_out : a.k);
    const float x0 = src[e], x1 = src[e + 1], c = a.cos_t[i], s = a.sin_t[i];
    dst[e] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    dst[e + 1] = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
  }
  if (a.v != nullptr)
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < a.n_kv_heads * a.head_dim;
         j += gridDim.x * blockDim.x)
      a.v_out[j] = a.v[j];
}

cudaError_t launch_rope(const LaunchCtx &ctx, const RopeArgs &a) {
  const int pairs = (a.n_heads + a.n_kv_heads) * (a.head_dim / 2);
  int blocks = (pairs + 255) / 256;
  blocks = blocks < ctx.num_sms ? blocks : ctx.num_sms;
  prefer_max_shared(rope_kernel);
  return launch_kernel(rope_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, ctx, a);
}

// ---- attention, then optionally Q8_0 --------------------------------------------
// Query head h's positions are cut into P slices (P <= 8), one per CTA of a
// thread-block cluster.  A CTA stages q_h in shared memory, computes the
// scores of its slice (one thread per position, the K row read with 16-byte
// loads), its slice's max m_p, the weights e_t = exp(s_t - m_p), their sum
// S_p and the unnormalised O_p = sum_t e_t V_t (each warp over part of the
// slice, whole rows, lanes across elements; warp partials added in order).
// After a cluster barrier CTA 0 combines the slices in rank order:
// M = max m_p, o = sum_p e^(m_p - M) O_p / sum_p e^(m_p - M) S_p, reading the
// others through distributed shared memory -- the softmax of all positions,
// deterministic -- and writes o (and its Q8_0 blocks).
struct AttnArgs {
  float *o;          // n_heads x head_dim
  int8_t *oq;        // Q8_0 of o, or nullptr (then od too)
  float *od;
  const float *q;    // n_heads x head_dim
  const float *kc;   // K cache: row t = n_kv_heads x head_dim
  const float *vc;   // V cache, same layout
  int n_pos, head_dim, n_heads, n_kv_heads;
  int P;             // CTAs (position slices) per head = cluster size
};

__device__ __forceinline__ int attn_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ void attn_cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float attn_ld_remote(const float *local, int rank) {
  uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(local)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__global__ void __launch_bounds__(kAttnThreads, 1) attention_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float red[32];
  griddep_wait();
  griddep_launch_dependents();
  const int p = attn_rank();
  const int h = blockIdx.x / a.P, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hd = a.head_dim, kv_dim = a.n_kv_heads * hd;
  const int g = h / (a.n_heads / a.n_kv_heads);
  const int t0 = static_cast<int>(static_cast<long long>(a.n_pos) * p / a.P);
  const int t1 = static_cast<int>(static_cast<long long>(a.n_pos) * (p + 1) / a.P);
  const int nt = t1 - t0;
  constexpr int kW = kAttnThreads / 32, kPer = kMaxHeadDim / 32;
  // shared memory: q | scores of the slice | warp partials | (m_p, S_p, O_p),
  // laid out for the largest slice in every CTA: CTA 0 reads the others'
  // (m_p, S_p, O_p) at its own offsets
  const int slice_max = (a.n_pos + a.P - 1) / a.P;
  float *qs = sm;
  float *s = sm + ((hd + 3) & ~3);
  float *part = s + ((slice_max + 3) & ~3);
  float *mine = part + kW * hd;  // [0] m_p, [1] S_p, [2..] O_p
  for (int i = tid; i < hd; i += kAttnThreads) qs[i] = a.q[static_cast<size_t>(h) * hd + i];
  __syncthreads();
  const float rs = __fsqrt_rn(static_cast<float>(hd));
  // four partial sums (one per float4 component, hd/4 terms each), added
  // pairwise: at most (hd/4 + 2) roundings on the way to each score
  const bool vec = (hd % 4 == 0) && (kv_dim % 4 == 0) && (reinterpret_cast<uintptr_t>(a.kc) & 15) == 0;
  for (int j = tid; j < nt; j += kAttnThreads) {
    const float *kt = a.kc + static_cast<size_t>(t0 + j) * kv_dim + static_cast<size_t>(g) * hd;
    float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f;
    if (vec) {
      const float4 *k4 = reinterpret_cast<const float4 *>(kt);
      const float4 *q4 = reinterpret_cast<const float4 *>(qs);
#pragma unroll 8
      for (int i = 0; i < hd / 4; ++i) {
        const float4 kv = __ldg(k4 + i), qv = q4[i];
        d0 = __fmaf_rn(qv.x, kv.x, d0);
        d1 = __fmaf_rn(qv.y, kv.y, d1);
        d2 = __fmaf_rn(qv.z, kv.z, d2);
        d3 = __fmaf_rn(qv.w, kv.w, d3);
      }
    } else {
      for (int i = 0; i < hd; i += 2) {
        d0 = __fmaf_rn(qs[i], __ldg(kt + i), d0);
        d1 = __fmaf_rn(qs[i + 1], __ldg(kt + i + 1), d1);
      }
    }
    s[j] = __fdiv_rn(__fadd_rn(__fadd_rn(d0, d1), __fadd_rn(d2, d3)), rs);
  }
  __syncthreads();
  float m = -INFINITY;
  for (int j = tid; j < nt; j += kAttnThreads) m = fmaxf(m, s[j]);
  m = block_max<kAttnThreads>(m, red);
  float sum = 0.0f;
  for (int j = tid; j < nt; j += kAttnThreads) {
    const float e = expf(__fsub_rn(s[j], m));
    s[j] = e;
    sum = __fadd_rn(sum, e);
  }
  sum = block_sum<kAttnThreads>(sum, red);  // ends with a barrier: every e_t is stored
  {
    // warp w sums slice positions [w nt / W, (w + 1) nt / W)
    const int j0 = static_cast<int>(static_cast<long long>(nt) * warp / kW);
    const int j1 = static_cast<int>(static_cast<long long>(nt) * (warp + 1) / kW);
    const float *vbase = a.vc + static_cast<size_t>(t0) * kv_dim + static_cast<size_t>(g) * hd + lane;
    float acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.0f;
#pragma unroll 4
    for (int j = j0; j < j1; ++j) {
      const float e = s[j];
      const float *vr = vbase + static_cast<size_t>(j) * kv_dim;
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (lane + 32 * k < hd) acc[k] = __fmaf_rn(e, __ldg(vr + 32 * k), acc[k]);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (lane + 32 * k < hd) part[warp * hd + lane + 32 * k] = acc[k];
  }
  __syncthreads();
  for (int i = tid; i < hd; i += kAttnThreads) {
    float v = 0.0f;
    for (int w = 0; w < kW; ++w) v = __fadd_rn(v, part[w * hd + i]);
    mine[2 + i] = v;
  }
  if (tid == 0) {
    mine[0] = m;
    mine[1] = sum;
  }
  attn_cluster_sync();
  if (p == 0) {
    // the slices' weights rescaled to the overall max, in rank order
    float M = -INFINITY;
    for (int r = 0; r < a.P; ++r) M = fmaxf(M, attn_ld_remote(mine, r));
    float S = 0.0f;
    for (int r = 0; r < a.P; ++r)
      S = __fmaf_rn(expf(__fsub_rn(attn_ld_remote(mine, r), M)), attn_ld_remote(mine + 1, r), S);
    float *oh = a.o + static_cast<size_t>(h) * hd;
    for (int i = tid; i < hd; i += kAttnThreads) {
      float v = 0.0f;
      for (int r = 0; r < a.P; ++r)
        v = __fmaf_rn(expf(__fsub_rn(attn_ld_remote(mine, r), M)), attn_ld_remote(mine + 2 + i, r), v);
      v = __fdiv_rn(v, S);
      oh[i] = v;
      part[i] = v;
    }
    if (a.oq != nullptr) {
      __syncthreads();
      for (int b = warp; b < hd / 32; b += kW) {
        const int blk = (h * hd) / 32 + b;
        quant_block_warp(part[b * 32 + lane], a.oq + blk * 32, a.od + blk, lane);
      }
    }
  }
  attn_cluster_sync();  // no CTA leaves while CTA 0 reads its shared memory
}

cudaError_t launch_attention(const LaunchCtx &ctx, AttnArgs a) {
  if (a.head_dim > kMaxHeadDim) return cudaErrorNotSupported;
  // slices of at least 32 positions, at most 8
  a.P = a.n_pos / 32;
  a.P = a.P < 1 ? 1 : (a.P > 8 ? 8 : a.P);
  const int slice = (a.n_pos + a.P - 1) / a.P;
  const size_t smem = (static_cast<size_t>((a.head_dim + 3) & ~3) + ((slice + 3) & ~3) +
                       static_cast<size_t>(kAttnThreads / 32) * a.head_dim + 2 + a.head_dim) * 4;
  if (smem > 200 * 1024) return cudaErrorNotSupported;
  auto kern = attention_kernel;
  prefer_max_shared(kern);
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(a.P);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_heads * a.P));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cfg.attrs = at;
  cfg.numAttrs = ctx.pdl ? 2 : 1;
  diag_launch_cfg(reinterpret_cast<const void *>(kern), cfg);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_rope_call(const LaunchCtx &ctx, float *q, float *k, float *k_out, const float *v,
                             float *v_out, const float *cos_t, const float *sin_t, int head_dim,
                             int n_heads, int n_kv_heads) {
  RopeArgs a{q, k, k_out, v, v_out, cos_t, sin_t, head_dim, n_heads, n_kv_heads};
  return launch_rope(ctx, a);
}

cudaError_t launch_attention_call(const LaunchCtx &ctx, float *o, int8_t *oq, float *od,
                                  const float *q, const float *kc, const float *vc, int n_pos,
                                  int head_dim, int n_heads, int n_kv_heads) {
  AttnArgs a{o, oq, od, q, kc, vc, n_pos, head_dim, n_heads, n_kv_heads, 1};
  return launch_attention(ctx, a);
}

}  // namespace mlq
