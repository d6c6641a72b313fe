// quantize.cu -- Q8_0 activation quantiser (page "Legacy-ISA ML Inference
// Runtime -- Design Spec", Sec. 4 "Q8 quantization" and Sec. 5 rounding
// rule).  Per block of 32 floats: amax = max|x|, d = amax/127,
// id = 127/amax (0 if amax = 0), q = trunc(x*id + copysign(0.5, x)) with the
// multiply and the add each rounded to float32 (__fmul_rn/__fadd_rn are
// never contracted into an FMA), clamped to [-127, 127]; NaN (0*inf when
// 127/amax overflows) stores 0.  IEEE division, denormals kept (this file is
// built without fast-math or flush-to-zero), so the bytes and scales are
// bit-identical to the definition.
//
// Layout: eight lanes per block, four consecutive floats per lane (one
// 128-bit load, one 32-bit store of four quants), so a warp covers four
// blocks = 512 B in, 128 B + 16 B out, fully coalesced.  The block maximum
// is reduced over the eight lanes on the float bit patterns (for
// non-negative floats the unsigned order is the numeric order).
#include "mlq_device.cuh"
#include "mlq_launch.h"

namespace mlq {

__global__ void __launch_bounds__(256) quantize_q8_kernel(const float *__restrict__ x,
                                                          int8_t *__restrict__ q,
                                                          float *__restrict__ d,
                                                          long long nblocks) {
  // Let the next kernel start its prologue now (it still waits for this
  // grid before reading our output); then wait for x, which may be the
  // output of the previous kernel on the stream.
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;   // which of the warp's four blocks
  const int part = lane & 7;   // which four elements of the block
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long g0 = warp0 * 4; g0 < nblocks; g0 += nwarps * 4) {
    const long long g = g0 + sub;
    const bool valid = g < nblocks;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) v = *reinterpret_cast<const float4 *>(x + g * kQK + part * 4);
    uint32_t m = max(max(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y))),
                     max(__float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w))));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const float amax = __uint_as_float(m);
    const float dd = amax / 127.0f;
    const float id = amax != 0.0f ? 127.0f / amax : 0.0f;
    if (valid) {
      const uint32_t packed = (quant_one(v.x, id) & 0xff) | ((quant_one(v.y, id) & 0xff) << 8) |
                              ((quant_one(v.z, id) & 0xff) << 16) |
                              (static_cast<uint32_t>(quant_one(v.w, id) & 0xff) << 24);
      *reinterpret_cast<uint32_t *>(q + g * kQK + part * 4) = packed;
      if (part == 0) d[g] = dd;
    }
  }
}

cudaError_t launch_quantize_q8(const LaunchCtx &ctx, const float *x, int8_t *q, float *d, int m,
                               int k) {
  const long long nblocks = static_cast<long long>(m) * (k / kQK);
  if (nblocks == 0) return cudaSuccess;
  const long long warps = (nblocks + 3) / 4;
  long long grid = (warps + 7) / 8;
  const long long cap = static_cast<long long>(ctx.num_sms) * 8;
  if (grid > cap) grid = cap;
  prefer_max_shared(quantize_q8_kernel);
  return launch_kernel(quantize_q8_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, ctx,
                       x, q, d, nblocks);
}

}  // namespace mlq
