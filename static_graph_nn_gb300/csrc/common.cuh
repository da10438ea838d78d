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

// 32 bytes in one store (a full L2 sector per lane): 16 floats as bf16, or 8
// floats; p 32-byte aligned.
__device__ __forceinline__ void st32b(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st16bf(bf16* p, const float* f) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  st32b(p, w);
}
__device__ __forceinline__ void st8f32(float* p, const float* f) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(f[i]);
  st32b(p, w);
}

// 16 bf16 values from one 32-byte load (p 32-byte aligned), widened.
__device__ __forceinline__ void ld16bf(const bf16* p, float* f) {
  uint32_t w[8];
  asm("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Column sums over a warp's 32 rows: lane l holds row l's 32 consecutive
// columns in x; returns the sum of column l over the 32 lanes.  A butterfly
// reduce-scatter: at each of five steps every lane keeps one half of its
// remaining columns (the upper half if its lane bit is set), sends the other
// half to the partner lane and adds what it receives, so the additions run
// in a fixed order (deterministic).  x is clobbered.
__device__ __forceinline__ float warp_colsum32(float (&x)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = up ? x[j] : x[j + w];
      const float keep = up ? x[j + w] : x[j];
      x[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return x[0];
}

// Bias-gradient partials of one epilogue chunk (GemmArgs::col_part): v holds
// this lane's row (row m of a 32-row group starting at a multiple of 32) at
// columns n0 .. n0+31 as computed before the final rounding; rows at or
// beyond M and columns at or beyond N count as zero.  All 32 lanes call it.
template <typename TO>
__device__ __forceinline__ void col_partial32(const GemmArgs& g, int m, int n0, int lane,
                                              float (&v)[32]) {
  const bool row_ok = m < g.M;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float r = sizeof(TO) == 2 ? __bfloat162float(__float2bfloat16_rn(v[j])) : v[j];
    v[j] = row_ok && n0 + j < g.N ? r : 0.0f;
  }
  const float t = warp_colsum32(v, lane);
  if (n0 + lane < g.N) g.col_part[(size_t)(m >> 5) * g.N + n0 + lane] = t;
}

// One Adam step of one parameter (t = step, 1-based; lr_bc1 = lr / (1 - b1^t),
// inv_sqrt_bc2 = 1 / sqrt(1 - b2^t)): m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2,
// p -= lr_bc1 m / (sqrt(v) inv_sqrt_bc2 + eps).  Shared by the optimizer
// kernel and the weight-gradient epilogue, so both give the same bits.
__device__ __forceinline__ void adam_one(float& p, float g, float& m, float& v, float lr_bc1,
                                         float inv_sqrt_bc2, float b1, float b2, float eps) {
  m = b1 * m + (1.0f - b1) * g;
  v = b2 * v + (1.0f - b2) * g * g;
  p -= lr_bc1 * m / (sqrtf(v) * inv_sqrt_bc2 + eps);
}

// Adam update fused into a weight-gradient epilogue (GemmArgs::upd_p set):
// gr holds the fp32 gradients of row m, columns n0 .. n0+31 (as stored in
// out); the parameters, moments and bf16 copy share out's layout.
__device__ __forceinline__ void adam_update32(const GemmArgs& g, bool vec, int m, int n0,
                                              const float (&gr)[32]) {
  const float lr_bc1 = g.upd_scal[0], inv = g.upd_scal[1];
  const float b1 = g.upd_b1, b2 = g.upd_b2, eps = g.upd_eps;
  const size_t base = (size_t)m * g.ldo + n0;
  if (vec && n0 + 32 <= g.N) {
    float4* p4 = reinterpret_cast<float4*>(g.upd_p + base);
    float4* m4 = reinterpret_cast<float4*>(g.upd_m + base);
    float4* v4 = reinterpret_cast<float4*>(g.upd_v + base);
    uint2* s4 = reinterpret_cast<uint2*>(static_cast<bf16*>(g.upd_shadow) + base);
#pragma unroll
    for (int h = 0; h < 2; ++h) {   // 16 columns at a time: their 12 loads in flight together
      float4 pp[4], mm[4], vv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        pp[q] = p4[4 * h + q];
        mm[q] = m4[4 * h + q];
        vv[q] = v4[4 * h + q];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float* gq = gr + 16 * h + 4 * q;
        adam_one(pp[q].x, gq[0], mm[q].x, vv[q].x, lr_bc1, inv, b1, b2, eps);
        adam_one(pp[q].y, gq[1], mm[q].y, vv[q].y, lr_bc1, inv, b1, b2, eps);
        adam_one(pp[q].z, gq[2], mm[q].z, vv[q].z, lr_bc1, inv, b1, b2, eps);
        adam_one(pp[q].w, gq[3], mm[q].w, vv[q].w, lr_bc1, inv, b1, b2, eps);
        p4[4 * h + q] = pp[q];
        m4[4 * h + q] = mm[q];
        v4[4 * h + q] = vv[q];
        __nv_bfloat162 lo = __floats2bfloat162_rn(pp[q].x, pp[q].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(pp[q].z, pp[q].w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        s4[4 * h + q] = u;
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (n0 + j >= g.N) continue;
    const size_t k = base + j;
    float pp = g.upd_p[k], mm = g.upd_m[k], vv = g.upd_v[k];
    adam_one(pp, gr[j], mm, vv, lr_bc1, inv, b1, b2, eps);
    g.upd_p[k] = pp;
    g.upd_m[k] = mm;
    g.upd_v[k] = vv;
    static_cast<bf16*>(g.upd_shadow)[k] = __float2bfloat16_rn(pp);
  }
}

}  // namespace mg
