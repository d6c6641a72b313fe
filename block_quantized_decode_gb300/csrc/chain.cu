// chain.cu -- a whole decode step of block-quantized products in one
// persistent launch.
//
// A chain is a list of phases; phase p quantises one float32 vector x_p to
// Q8_0 and multiplies it with one or more weight matrices of the same width
// (e.g. Wq|Wk|Wv, or gate|up).  x_p may be the output of an earlier phase.
// Definitions as in quantize.cu / matvec.cu (page "Legacy-ISA ML Inference
// Runtime -- Design Spec", Sec. 4 and Sec. 5; the per-step data flow of a
// layer is its Sec. 6 "Forward pass").
//
// Why one launch: a decode step is a chain of dependent products whose
// weights do NOT depend on the activations.  Launched one kernel at a time,
// every boundary costs a ramp and a tail during which HBM idles.  Here one
// CTA per SM (cooperative launch, so all CTAs are resident) owns a balanced
// slice of every phase's rows; its producer warp streams the weight bytes of
// ALL phases, in order, through a ring of shared-memory stages with 1-D bulk
// copies, without ever waiting for activations -- it runs ahead across phase
// boundaries, bounded only by the ring's free slots.  The consumer warps
// (16 per CTA) step through the phases: wait at a grid-wide barrier until
// every CTA has written the previous phase's outputs, quantise x_p into
// shared memory themselves (same element arithmetic as quantize.cu, so the
// bytes are identical), then reduce each row of the phase's stages with
// dp4a (Q4_0: -8 folded through the per-block sum of qx; Q8_0: half blocks
// joined by one shuffle) and a warp-shuffle tree.
//
// Grid barrier: after a phase, each CTA's consumers sync, then one thread
// fences and adds 1 to that phase's counter in the caller's workspace; the
// next phase starts when the counter reaches gridDim.x (acquire loads,
// bounded wait).  The last CTA to finish resets every counter to 0, so the
// workspace is zero again for the next call.  Every wait is bounded: a
// give-up records MLQ_E_TIMEOUT, the CTA stops issuing copies, drains its
// own copies in flight (bounded) and still takes part in the final reset.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

constexpr int kChainConsumerWarps = 16;
constexpr int kChainThreads = (kChainConsumerWarps + 1) * 32;
constexpr int kChainMaxSlots = 8;

__device__ __forceinline__ void chain_mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kChainConsumerWarps * 32) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool chain_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
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

// Bytes of one weight row (quants then, separately, its scales).
template <int QT>
__device__ __forceinline__ int row_q_bytes(int nb) {
  return nb * (QT == 1 ? 16 : 32);
}

// Visit this CTA's chunks of phase p in order: f(product, first local row, rows).
template <typename F>
__device__ __forceinline__ void for_each_chunk(const ChainArgs &a, int p, int rpc, F &&f) {
  const ChainPhaseDev &ph = a.phase[p];
  long long total = 0;
  for (int j = ph.first; j < ph.first + ph.count; ++j) total += a.prod[j].rows;
  const long long lo = total * blockIdx.x / gridDim.x;
  const long long hi = total * (blockIdx.x + 1) / gridDim.x;
  long long off = 0;
  for (int j = ph.first; j < ph.first + ph.count; ++j) {
    const long long r0 = lo > off ? lo : off;
    const long long e = off + a.prod[j].rows;
    const long long r1 = hi < e ? hi : e;
    for (long long r = r0; r < r1; r += rpc) {
      const long long n = r1 - r < rpc ? r1 - r : rpc;
      f(j, static_cast<int>(r - off), static_cast<int>(n));
    }
    off = e;
  }
}

template <int QT>
__device__ __forceinline__ int rows_per_chunk(const ChainArgs &a, int nb) {
  const int rb = row_q_bytes<QT>(nb) + nb * 4;
  const int r = a.stage_bytes / rb;
  return r < 1 ? 1 : r;
}

// Q4_0 activation layout in shared memory: the 32 quants of block b at
// b*32, with the two 16-byte halves swapped when bit 2 of b is set, so the
// eight lanes of a quarter warp reading consecutive blocks hit distinct
// banks.
__device__ __forceinline__ int q4_half_offset(int b, int half) {
  return b * 32 + ((half ^ ((b >> 2) & 1)) << 4);
}

template <int QT>
__device__ __forceinline__ float row_dot(const uint8_t *wrow, const float *drow,
                                         const int8_t *xq_s, const float *xd_s, const int *sx_s,
                                         int nb, int lane) {
  float acc = 0.0f;
  if (QT == 1) {
#pragma unroll 2
    for (int u = lane; u < nb; u += 32) {
      const uint4 w = *reinterpret_cast<const uint4 *>(wrow + u * 16);
      const float dw = drow[u];
      const int4 xa = *reinterpret_cast<const int4 *>(xq_s + q4_half_offset(u, 0));
      const int4 xb = *reinterpret_cast<const int4 *>(xq_s + q4_half_offset(u, 1));
      constexpr uint32_t kLo = 0x0F0F0F0Fu;
      int s = __dp4a(static_cast<int>(w.x & kLo), xa.x, 0);
      s = __dp4a(static_cast<int>(w.y & kLo), xa.y, s);
      s = __dp4a(static_cast<int>(w.z & kLo), xa.z, s);
      s = __dp4a(static_cast<int>(w.w & kLo), xa.w, s);
      s = __dp4a(static_cast<int>((w.x >> 4) & kLo), xb.x, s);
      s = __dp4a(static_cast<int>((w.y >> 4) & kLo), xb.y, s);
      s = __dp4a(static_cast<int>((w.z >> 4) & kLo), xb.z, s);
      s = __dp4a(static_cast<int>((w.w >> 4) & kLo), xb.w, s);
      s -= 8 * sx_s[u];
      acc = __fmaf_rn(__fmul_rn(__int2float_rn(s), dw), xd_s[u], acc);
    }
  } else {
    const int upr = 2 * nb;
    const int iters = (upr + 31) >> 5;
#pragma unroll 2
    for (int k = 0; k < iters; ++k) {
      const int h = lane + 32 * k;
      const bool valid = h < upr;
      int s = 0;
      float dw = 0.0f;
      if (valid) {
        const uint4 w = *reinterpret_cast<const uint4 *>(wrow + h * 16);
        const int4 xa = *reinterpret_cast<const int4 *>(xq_s + h * 16);
        dw = drow[h >> 1];
        s = __dp4a(static_cast<int>(w.x), xa.x, 0);
        s = __dp4a(static_cast<int>(w.y), xa.y, s);
        s = __dp4a(static_cast<int>(w.z), xa.z, s);
        s = __dp4a(static_cast<int>(w.w), xa.w, s);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      if (valid && !(lane & 1)) acc = __fmaf_rn(__fmul_rn(__int2float_rn(s), dw), xd_s[h >> 1], acc);
    }
  }
  return warp_sum(acc);
}

// Quantise x (nb blocks of 32 floats, global) into shared memory; every
// consumer thread takes part.  Eight lanes per block, four elements each.
template <int QT>
__device__ __forceinline__ void quantize_phase_input(const ChainPhaseDev &ph, int8_t *xq_s,
                                                     float *xd_s, int *sx_s, int ctid) {
  const int nb = ph.nb;
  const int part = ctid & 7;
  const bool writer = blockIdx.x == 0 && ph.xq_out != nullptr;
  for (int base = 0; base < nb; base += kChainConsumerWarps * 4) {
    const int b = base + (ctid >> 3);
    const bool valid = b < nb;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    // x may have been written by other CTAs in this launch: read through L2.
    if (valid) v = __ldcg(reinterpret_cast<const float4 *>(ph.x + static_cast<size_t>(b) * kQK + part * 4));
    uint32_t m = max(max(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y))),
                     max(__float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w))));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const float amax = __uint_as_float(m);
    const float dd = amax / 127.0f;
    const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
    const int q0 = quant_one(v.x, id), q1 = quant_one(v.y, id), q2 = quant_one(v.z, id),
              q3 = quant_one(v.w, id);
    const uint32_t packed = (q0 & 0xff) | ((q1 & 0xff) << 8) | ((q2 & 0xff) << 16) |
                            (static_cast<uint32_t>(q3 & 0xff) << 24);
    int s4 = q0 + q1 + q2 + q3;
    s4 += __shfl_xor_sync(0xffffffffu, s4, 4);
    s4 += __shfl_xor_sync(0xffffffffu, s4, 2);
    s4 += __shfl_xor_sync(0xffffffffu, s4, 1);
    if (valid) {
      const int off = QT == 1 ? q4_half_offset(b, part >> 2) + (part & 3) * 4 : b * kQK + part * 4;
      *reinterpret_cast<uint32_t *>(xq_s + off) = packed;
      if (part == 0) {
        xd_s[b] = dd;
        sx_s[b] = s4;
      }
      if (writer) {
        *reinterpret_cast<uint32_t *>(ph.xq_out + static_cast<size_t>(b) * kQK + part * 4) = packed;
        if (part == 0) ph.xd_out[b] = dd;
      }
    }
  }
}

template <int QT>
__global__ void __launch_bounds__(kChainThreads, 1) decode_chain_kernel(const __grid_constant__ ChainArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kChainMaxSlots];
  __shared__ __align__(8) uint64_t empty_bar[kChainMaxSlots];
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int8_t *xq_s = reinterpret_cast<int8_t *>(smem);
  float *xd_s = reinterpret_cast<float *>(smem + a.kmax);
  int *sx_s = reinterpret_cast<int *>(smem + a.kmax + 4 * (a.kmax / kQK));
  uint8_t *ring = smem + a.xbuf_bytes;

  if (tid == 0) {
    for (int s = 0; s < a.ns; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kChainConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;  // producer lane only
  if (warp == kChainConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int use = 0;
      bool stop = false;
      for (int p = 0; p < a.nphases && !stop; ++p) {
        const int nb = a.phase[p].nb;
        const int rq = row_q_bytes<QT>(nb);
        for_each_chunk(a, p, rows_per_chunk<QT>(a, nb), [&](int j, int r, int n) {
          if (stop) return;
          const int slot = use % a.ns;
          if (use >= a.ns &&
              !chain_wait(smem_addr(&empty_bar[slot]), ((use / a.ns) - 1) & 1, abort_v, a.wait_ns)) {
            if (!*abort_v) set_status(a.status, kStatusTimeout);
            *abort_v = 1;
            stop = true;
            return;
          }
          const uint32_t qb = static_cast<uint32_t>(n) * rq;
          const uint32_t db = static_cast<uint32_t>(n) * nb * 4;
          uint8_t *dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
          const uint32_t fb = smem_addr(&full_bar[slot]);
          mbar_arrive_expect_tx(fb, qb + db);
          bulk_copy_g2s(smem_addr(dst), a.prod[j].wq + static_cast<size_t>(r) * rq, qb, fb);
          bulk_copy_g2s(smem_addr(dst + qb), a.prod[j].wd + static_cast<size_t>(r) * nb, db, fb);
          ++use;
          issued = use;
        });
      }
    }
  } else {
    // ------------------------------ consumers ------------------------------
    int use = 0;
    for (int p = 0; p < a.nphases; ++p) {
      if (p > 0) {
        if (tid == 0) {
          const unsigned target = gridDim.x;
          bool ok = a.wait_ns != 0;
          const uint64_t t0 = sm_cycles(), lim = limit_cycles(a.wait_ns);
          while (ok && ld_acquire_gpu(a.counters + (p - 1)) < target) {
            if (*abort_v || sm_cycles() - t0 > lim) ok = false;
          }
          if (!ok) {
            if (!*abort_v) set_status(a.status, kStatusTimeout);
            *abort_v = 1;
          }
        }
        consumers_sync();
        if (*abort_v) break;
      }
      const ChainPhaseDev &ph = a.phase[p];
      quantize_phase_input<QT>(ph, xq_s, xd_s, sx_s, tid);
      consumers_sync();
      const int nb = ph.nb;
      const int rq = row_q_bytes<QT>(nb);
      bool stop = false;
      for_each_chunk(a, p, rows_per_chunk<QT>(a, nb), [&](int j, int r, int n) {
        if (stop) return;
        const int slot = use % a.ns;
        if (!warp_wait([&] { return chain_wait(smem_addr(&full_bar[slot]), (use / a.ns) & 1, abort_v,
                                               a.wait_ns); })) {
          if (!*abort_v) set_status(a.status, kStatusTimeout);
          *abort_v = 1;
          stop = true;
          return;
        }
        const uint8_t *sq = ring + static_cast<size_t>(slot) * a.stage_bytes;
        const float *sd = reinterpret_cast<const float *>(sq + static_cast<size_t>(n) * rq);
        float *y = a.prod[j].y + r;
        for (int i = warp; i < n; i += kChainConsumerWarps) {
          const float v = row_dot<QT>(sq + static_cast<size_t>(i) * rq, sd + static_cast<size_t>(i) * nb,
                                      xq_s, xd_s, sx_s, nb, lane);
          if (lane == 0) y[i] = v;
        }
        __syncwarp();
        if (lane == 0) chain_mbar_arrive(smem_addr(&empty_bar[slot]));
        ++use;
      });
      consumers_sync();  // every row of this phase written, x_p no longer read
      if (*abort_v) break;
      if (tid == 0) {
        __threadfence();
        atomicAdd(a.counters + p, 1u);
      }
    }
  }

  __syncthreads();
  if (tid == kChainConsumerWarps * 32 && *abort_v) {
    // Copies this CTA issued may still be landing in its shared memory.
    for (int slot = 0; slot < a.ns && slot < issued; ++slot) {
      const int last = slot + ((issued - 1 - slot) / a.ns) * a.ns;
      mbar_wait_bounded(smem_addr(&full_bar[slot]), (last / a.ns) & 1, kDrainWaitNs);
    }
  }
  if (tid == 0) {
    __threadfence();
    const unsigned done = atomicAdd(a.counters + a.nphases, 1u);
    if (done == gridDim.x - 1) {  // last CTA out: leave the workspace zeroed
      for (int p = 0; p <= a.nphases; ++p) atomicExch(a.counters + p, 0u);
      __threadfence();
    }
  }
}

cudaError_t launch_decode_chain(const LaunchCtx &ctx, int qtype, const ChainArgs &args_in) {
  // The streaming kernel of stream.cu is the default; this one takes the
  // shapes it does not (K above 16384) and MLQ_CHAIN_KERNEL=legacy.
  const char *kind = std::getenv("MLQ_CHAIN_KERNEL");
  if (kind == nullptr || std::strcmp(kind, "legacy") != 0) {
    const cudaError_t e = launch_decode_stream(ctx, qtype, args_in);
    if (e != cudaErrorNotSupported) return e;
  }
  ChainArgs a = args_in;
  const size_t nbmax = static_cast<size_t>(a.kmax) / kQK;
  a.xbuf_bytes = static_cast<int>((static_cast<size_t>(a.kmax) + 8 * nbmax + 127) / 128 * 128);
  size_t rowmax = 0;
  for (int p = 0; p < a.nphases; ++p) {
    const size_t nb = static_cast<size_t>(a.phase[p].nb);
    const size_t rb = nb * (qtype == 1 ? 16 : 32) + nb * 4;
    if (rb > rowmax) rowmax = rb;
  }
  constexpr size_t kBudget = 220 * 1024;
  size_t stage = 48 * 1024;
  if (rowmax > stage) stage = (rowmax + 127) / 128 * 128;
  int ns = static_cast<int>((kBudget - a.xbuf_bytes) / stage);
  if (ns > kChainMaxSlots) ns = kChainMaxSlots;
  if (ns < 2) return cudaErrorNotSupported;
  a.ns = ns;
  a.stage_bytes = static_cast<int>(stage);
  a.status = ctx.status;
  a.wait_ns = ctx.wait_ns;
  const size_t smem = a.xbuf_bytes + static_cast<size_t>(ns) * stage;
  auto kern = qtype == 1 ? decode_chain_kernel<1> : decode_chain_kernel<0>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctx.num_sms));
  cfg.blockDim = dim3(kChainThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  diag_launch_cfg(reinterpret_cast<const void *>(kern), cfg);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// ---------------------------------------------------------------------------
// Variant without caller workspace, for callers that may not allocate device
// memory: the barrier counters live in a fixed device array of this file
// instead.  kStaticChainWords counters cover MLQ_CHAIN_MAX_PHASES + 1 words
// with room to spare (256 bytes in all).  Every device that loads the
// library holds this array until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned g_static_chain_counters[kStaticChainWords];

namespace {
std::mutex g_static_mu;
unsigned *g_static_addr[64] = {};
}  // namespace

cudaError_t static_chain_scratch(int device, unsigned **out) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_addr[device] == nullptr) {
    // The host-side name of a __device__ array is not a device address; ask
    // the runtime for it, with `device` current (the caller guarantees that).
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_chain_counters);
    if (e != cudaSuccess) return e;
    g_static_addr[device] = static_cast<unsigned *>(p);
  }
  *out = g_static_addr[device];
  return cudaSuccess;
}

cudaError_t launch_decode_chain_static(const LaunchCtx &ctx, int device, int qtype,
                                       const ChainArgs &args) {
  if (args.nphases + 1 > kStaticChainWords) return cudaErrorInvalidValue;
  unsigned *counters = nullptr;
  cudaError_t e = static_chain_scratch(device, &counters);
  if (e != cudaSuccess) return e;
  // The counters must start at zero.  A finished call leaves them zero, but
  // clear them anyway (no allocation involved) so that nothing depends on
  // how an earlier call ended.
  e = cudaMemsetAsync(counters, 0, static_cast<size_t>(args.nphases + 1) * sizeof(unsigned),
                      ctx.stream);
  if (e != cudaSuccess) return e;
  ChainArgs a = args;
  a.counters = counters;
  return launch_decode_chain(ctx, qtype, a);
}

}  // namespace mlq
