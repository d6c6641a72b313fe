// mlq_device.cuh -- sm_103a device helpers shared by the kernels of libmlq:
// inline-PTX wrappers for mbarriers, 1-D bulk (TMA) copies, L2 prefetch,
// streaming loads, programmatic-dependent-launch control, and the bounded
// wait that every kernel uses instead of an unbounded spin.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mlq {

constexpr int kQK = 32;                 // block size (Design Spec Sec. 4)
constexpr int kStatusTimeout = 7;       // == MLQ_E_TIMEOUT in mlq.h
constexpr int kStatusBounds = 8;        // == MLQ_E_BOUNDS in mlq.h
constexpr unsigned long long kDrainWaitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch -------------------------------------
// Block until every grid this one depends on has completed and its memory
// is visible.  A no-op when the kernel was launched without the attribute.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next kernel on the stream to be scheduled (it still waits in
// griddep_wait() for this grid to finish before touching our outputs).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier ------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// SM cycle counter: cheap to read, so polling it does not slow the wait
// loop.  Wait limits are given in nanoseconds and converted at 2 cycles per
// ns (about the 2.07 GHz maximum SM clock), so a limit is "about" that long.
__device__ __forceinline__ uint64_t sm_cycles() { return static_cast<uint64_t>(clock64()); }
__device__ __forceinline__ uint64_t limit_cycles(unsigned long long limit_ns) {
  return static_cast<uint64_t>(limit_ns) * 2u;
}
// Wait for phase `parity` of the mbarrier, giving up after about limit_ns
// nanoseconds.  limit_ns == 0 gives up at once (test hook: exercises the
// timeout path with no real hang).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = sm_cycles(), lim = limit_cycles(limit_ns);
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sm_cycles() - t0 > lim) return false;
  }
}

// The calling warp waits as one: lane 0 runs `wait` (a bounded wait), the
// other lanes wait at __syncwarp, which also orders the data the barrier
// guards for them after lane 0's acquire.  All 32 lanes must call it.  One
// poller per warp, not 32: every try_wait of every lane is an operation on
// the same barrier word, and measured on GB300 they queue -- with 512
// threads checking a few already-completed barriers, about 400 cycles each.
template <typename W>
__device__ __forceinline__ bool warp_wait(W &&wait) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait() ? 1 : 0;
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               unsigned long long limit_ns) {
  return warp_wait([&] { return mbar_wait_bounded(bar, parity, limit_ns); });
}

// ---- bulk asynchronous copies (TMA, non-tensor) -----------------------------
// Global -> shared, completion counted in bytes on `bar`.  dst, src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Hint: bring [src, src + bytes) into L2.  src 16-byte aligned, bytes a
// multiple of 16.  Never reads through L1, so it is safe before
// griddep_wait() even if the previous kernel writes the same bytes.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Prefetch the 16-byte-aligned interior of [p, p + bytes), at most `cap`
// bytes, in pieces the bulk engine accepts.
__device__ __forceinline__ void prefetch_range_l2(const void *p, size_t bytes, size_t cap) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uintptr_t e = a + (bytes < cap ? bytes : cap);
  a = (a + 15) & ~uintptr_t(15);
  e &= ~uintptr_t(15);
  constexpr uintptr_t kPiece = 1u << 16;
  while (a < e) {
    uintptr_t n = e - a < kPiece ? e - a : kPiece;
    bulk_prefetch_l2(reinterpret_cast<const void *>(a), static_cast<uint32_t>(n));
    a += n;
  }
}

// ---- streaming loads ------------------------------------------------------------
// L2 policy that marks lines for early eviction: weight bytes are used
// exactly once per call, so they should not push activations out of L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Read-only 128-bit load that does not allocate in L1 and carries the L2
// eviction policy `pol`.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t pol) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ float ld_stream_f32(const float *p, uint64_t pol) {
  float v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
  return v;
}

// ---- reductions -------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- Q8_0 quantisation of one element ---------------------------------------
// Design Spec Sec. 5 rounding: q = trunc(x*id + copysign(0.5, x)) with the
// multiply and the add each rounded to float32 (__fmul_rn / __fadd_rn are
// never contracted into an FMA), clamped to [-127, 127]; NaN (0 * inf when
// 127/amax overflows) stores 0.  Shared by every kernel that quantises, so
// their bytes are identical by construction.
__device__ __forceinline__ int quant_one(float x, float id) {
  float v = __fmul_rn(x, id);
  v = __fadd_rn(v, copysignf(0.5f, x));
  v = truncf(v);
  return v >= 127.0f ? 127 : (v <= -127.0f ? -127 : (v == v ? static_cast<int>(v) : 0));
}

// Record a device-side status (first writer wins).
__device__ __forceinline__ void set_status(int *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Index checks of the bounds-checking build (compiled with MLQ_CHECK_BOUNDS):
//   if (in_bounds(i < n, status)) buf[i] = v;
// records MLQ_E_BOUNDS and skips the access when the condition fails -- no
// trap and no early return (a return could strand the CTA's barriers).  In
// the normal build the check is the constant true and costs nothing.
#ifdef MLQ_CHECK_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, int *status) {
  if (!ok) set_status(status, kStatusBounds);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, int *) { return true; }
#endif

}  // namespace mlq
