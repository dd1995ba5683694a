// Shared device helpers of the MoE kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

#define MOE_DEVINL __device__ __forceinline__

typedef __nv_bfloat16 bf16_t;

// Record the first device-side error in the caller's status word (0 = none).
MOE_DEVINL void moe_set_status(int32_t *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (a no-op for a plain launch).
MOE_DEVINL void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

MOE_DEVINL float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MOE_DEVINL float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

MOE_DEVINL uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 8 bf16 <-> 8 fp32 through one 16-byte word.
MOE_DEVINL void bf16x8_to_f32(const uint4 &u, float *f) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

MOE_DEVINL uint4 f32_to_bf16x8(const float *f) {
  uint4 u;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

MOE_DEVINL uint4 ld_nc_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

MOE_DEVINL void st_v4(void *p, const uint4 &v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// sigmoid(z) = 1 / (1 + e^-z) in fp32 with the hardware exponential and
// reciprocal (relative error ~1e-6, far below the bf16 rounding of the
// SwiGLU outputs it feeds).  e^-z overflowing to inf gives exactly 0.
// 1 / (1 + e^-z) with the approximate reciprocal (rcp.approx.ftz: within
// 1 ulp; 1 / +inf = 0), far inside the bf16 rounding of the epilogue outputs
MOE_DEVINL float sigmoid_f(float z) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + __expf(-z)));
  return r;
}
