// Small inline-PTX helpers shared by the librx kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace rxk {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes == 0 fills the destination with 0.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (lo, hi) rounded to nearest bf16 and packed, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x on the special-function unit (PTX ex2.approx).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA and integer pipes instead of the special-function unit
// (Cody-Waite range reduction with a polynomial, the scheme FlashAttention-4
// uses to relieve the SFU in softmax): x = n + f with n the nearest integer
// (adding 1.5 * 2^23 leaves n in the low mantissa bits; subtracting it back
// is exact) and f in [-1/2, 1/2]; 2^f by a cubic whose coefficients minimise
// the maximum relative error on [-1/2, 1/2] (a Remez exchange, derived for
// this library: 7.5e-5, far below the 2^-9 of the bf16 rounding P gets);
// 2^n added to the exponent field.  x below -125 gives 0 (2^-125 would be
// the smallest result), as the SFU's flushed result does.
__device__ __forceinline__ float poly_exp2(float x) {
  const float xc = fmaxf(x, -125.0f);
  const float t = xc + 12582912.0f;  // 1.5 * 2^23
  const float f = xc - (t - 12582912.0f);
  const float p = fmaf(fmaf(fmaf(0.05517166905792616f, f, 0.2426111221932161f), f,
                            0.6932609854606553f),
                       f, 0.9999280735394012f);
  const float r = __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
  return x < -125.0f ? 0.0f : r;
}

// Programmatic dependent launch: wait until the kernels this grid depends on
// (the previous ones on its stream) have completed and their writes are
// visible; a no-op in a grid launched without that attribute.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
// Let the next kernel on the stream, if launched with programmatic stream
// serialization, start launching before this grid completes.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

}  // namespace rxk
