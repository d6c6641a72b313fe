// mma_frag.cuh -- fp16 operand conversions and scaling helpers shared by
// the tensor-core small-M kernels (gemm_mma.cu, gemm_mma_cluster.cu).
//
// All conversions are exact: a nibble minus 8 and an int8 are small
// integers, which fp16 holds exactly, and an m16n8k16 block sum of them
// (at most 32 * 8 * 127 in magnitude) is an exact integer in the fp32
// accumulator.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace mlq {

__device__ __forceinline__ uint32_t nib_to_h2(uint32_t w) {
  // two nibbles already in bits 0..3 and 16..19 -> half2 (n0 - 8, n1 - 8)
  uint32_t v = (w & 0x000F000Fu) | 0x64006400u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&v), __half2half2(__ushort_as_half(0x6408)));
  return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t s8_to_h2(uint32_t biased, uint32_t sel) {
  // biased = int8 ^ 0x80 per byte; pick two bytes into the mantissa of 1024
  uint32_t v;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(v) : "r"(biased), "r"(0x64646464u), "r"(sel));
  const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&v), __half2half2(__ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

// acc(2) = (d(2) * s) * x(2) + acc(2), rounded per step as in the definition
__device__ __forceinline__ void scale_acc2(unsigned long long &acc, float d0, float d1, float s,
                                           unsigned long long x2) {
  unsigned long long t;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(pack2(d0, d1)), "l"(pack2(s, s)));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(t), "l"(x2));
}

}  // namespace mlq
