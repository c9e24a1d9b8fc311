// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// Raise a device status flag (see mla_device_flag in mla.h).
__device__ __forceinline__ void raise_flag(unsigned int* flags, unsigned int bit) {
  if (flags) atomicOr(flags, bit);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Rotary angle pos * base^(-2j/d) and its cos/sin, taken in double: a float
// product pos*theta loses ~1e-3 rad at pos ~ 6.5e4, far above fp32 tolerance.
__device__ __forceinline__ void rope_cos_sin(int pos, int j, int d, double base, float* c,
                                             float* s) {
  double theta = pow(base, -2.0 * (double)j / (double)d);
  double sn, cs;
  sincos((double)pos * theta, &sn, &cs);
  *c = (float)cs;
  *s = (float)sn;
}

// Rotary frequencies as fixed-point fractions of a turn: turns = theta / (2 pi)
// in 0.64 fixed point.  Then pos * turns (mod 2^64) is the angle pos * theta
// modulo 2 pi, formed with one integer multiply: the reduction needs no
// floating point, and its error is the rounding of `turns` times pos (about
// 2^-39 turn at pos 2^17), far below the float sincos that follows.  (FP64,
// which the product would otherwise need, runs at a small fraction of the
// fp32 rate on this GPU.)
inline uint64_t rope_turns(double theta) {
  return (uint64_t)(theta * 0.15915494309189535 * 18446744073709551616.0);
}

// cos/sin of the rotary angle pos * theta, theta given as rope_turns(theta):
// the top 32 bits of the product, read as a signed fraction of a turn, give
// the angle reduced to [-pi, pi).
__device__ __forceinline__ void rope_cs_turns(int pos, uint64_t turns, float* c, float* s) {
  const uint64_t ph = (uint64_t)(uint32_t)pos * turns;
  const float ang = (float)(int32_t)(uint32_t)(ph >> 32) * 1.4629180792671596e-09f;  // 2 pi / 2^32
  sincosf(ang, s, c);
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel in the stream start its prologue.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialisation allowed (pdl == false: a plain launch).
template <typename Kern, typename Arg>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Arg& arg,
                       bool pdl = true) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, arg);
}

// %globaltimer in nanoseconds.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Float -> uint32 key whose unsigned order equals the float order; -0.0 is
// first turned into +0.0 so that the two compare equal.
__device__ __forceinline__ uint32_t ordered_key(float x) {
  x = x + 0.0f;
  uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// Two floats -> packed bf16x2 (round to nearest even).
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}

}  // namespace mla
