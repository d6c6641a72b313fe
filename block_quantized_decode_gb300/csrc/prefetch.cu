// prefetch.cu -- bring byte ranges (typically the weights of the next
// products of a decode step) into L2 ahead of their use.
//
// Each CTA issues fire-and-forget bulk L2 prefetches
// (cp.async.bulk.prefetch.L2) for its share of every range and exits; the
// memory system keeps streaming after the kernel has finished, so HBM
// reads of later products overlap the computation of earlier ones.  A
// prefetch is only a hint and L2 is the device's point of coherence, so it
// can never make a later kernel read stale data; the kernel therefore does
// not wait for the previous kernel on the stream and lets the next one
// start at once.
#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

__global__ void __launch_bounds__(32) prefetch_l2_kernel(const PrefetchList list) {
  griddep_launch_dependents();
  // Split the concatenated ranges into gridDim.x equal 16-byte-aligned
  // slices; lane i of the CTA prefetches every 32nd 64 KiB piece of it.
  size_t total = 0;
  for (int r = 0; r < list.n; ++r) total += list.bytes[r];
  const size_t per = ((total + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
  const size_t lo = per * blockIdx.x;
  const size_t hi = lo + per < total ? lo + per : total;
  constexpr size_t kPiece = 64 * 1024;
  size_t base = 0;
  for (int r = 0; r < list.n; ++r) {
    const size_t rb = base, re = base + list.bytes[r];
    base = re;
    const size_t a = lo > rb ? lo : rb;
    const size_t e = hi < re ? hi : re;
    if (a >= e) continue;
    const uint8_t *p = static_cast<const uint8_t *>(list.ptr[r]) + (a - rb);
    const size_t len = e - a;
    for (size_t off = static_cast<size_t>(threadIdx.x) * kPiece; off < len; off += 32 * kPiece) {
      const size_t n = len - off < kPiece ? len - off : kPiece;
      prefetch_range_l2(p + off, n, kPiece);
    }
  }
}

cudaError_t launch_prefetch_l2(const LaunchCtx &ctx, const PrefetchList &list) {
  size_t total = 0;
  for (int r = 0; r < list.n; ++r) total += list.bytes[r];
  if (total == 0) return cudaSuccess;
  long long grid = static_cast<long long>((total + 64 * 1024 - 1) / (64 * 1024));
  if (grid > ctx.num_sms) grid = ctx.num_sms;
  return launch_kernel(prefetch_l2_kernel, dim3(static_cast<unsigned>(grid)), dim3(32), 0, ctx,
                       list);
}

}  // namespace mlq
