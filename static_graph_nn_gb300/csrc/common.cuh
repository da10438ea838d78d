// Shared device helpers for the training-step kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace mg {

typedef __nv_bfloat16 bf16;

// Element load/store in either storage type, arithmetic in fp32.
__device__ __forceinline__ float ld_elem(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const bf16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_elem(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elem(bf16* p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// GELU, tanh form: 0.5 z (1 + tanh(u)), u = sqrt(2/pi) (z + 0.044715 z^3).
__device__ __forceinline__ float gelu_tanh_f(float z) {
  const float k0 = 0.7978845608028654f, k1 = 0.044715f;
  float u = k0 * (z + k1 * z * z * z);
  return 0.5f * z * (1.0f + tanhf(u));
}

// d/dz of the tanh-form GELU: 0.5 (1 + t) + 0.5 z (1 - t^2) sqrt(2/pi) (1 + 3*0.044715 z^2).
__device__ __forceinline__ float gelu_tanh_grad_f(float z) {
  const float k0 = 0.7978845608028654f, k1 = 0.044715f;
  float z2 = z * z;
  float t = tanhf(k0 * (z + k1 * z2 * z));
  return 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * k0 * (1.0f + 3.0f * k1 * z2);
}

__device__ __forceinline__ float apply_act(int act, float z) {
  if (act == ACT_RELU) return z > 0.0f ? z : 0.0f;
  if (act == ACT_GELU) return gelu_tanh_f(z);
  return z;
}

// Derivative factor of the activation, from the saved tensor: ReLU reads the
// saved output h (h > 0 exactly when z > 0), GELU reads the saved input z.
__device__ __forceinline__ float act_grad_from_saved(int act, float saved) {
  if (act == ACT_RELU) return saved > 0.0f ? 1.0f : 0.0f;
  if (act == ACT_GELU) return gelu_tanh_grad_f(saved);
  return 1.0f;
}

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

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024); all threads get it.
__device__ __forceinline__ float block_sum(float v, float* red /* >= 32 floats */) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.0f;
  return warp_sum(t);
}

__device__ __forceinline__ float block_max(float v, float* red) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : -INFINITY;
  return warp_max(t);
}


// Running softmax partial over 32 accumulator values of a row at columns n0..
// (those below g.N), each taken as it will be stored (plus the bias, rounded
// to the output type), kept in base 2: pm = max of x log2(e), ps = sum of
// 2^(x log2(e) - pm).  For GEMM outputs with no activation, residual or saved
// value.
__device__ __forceinline__ void softmax_partial32(const GemmArgs& g, int n0, const float (&v)[32],
                                                  float& pm, float& ps) {
  constexpr float kLog2e = 1.4426950408889634f;
  float x[32];
  float cm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    float t = v[j] + (g.bias && n < g.N ? g.bias[n] : 0.0f);
    if (g.out_type == DT_BF16) t = __bfloat162float(__float2bfloat16_rn(t));
    x[j] = n < g.N ? t * kLog2e : -INFINITY;
    cm = fmaxf(cm, x[j]);
  }
  if (cm == -INFINITY) return;
  if (cm > pm) {
    ps = (pm == -INFINITY) ? 0.0f : ps * exp2f(pm - cm);
    pm = cm;
  }
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x[j] - pm));
    acc += e;
  }
  ps += acc;
}

}  // namespace mg
