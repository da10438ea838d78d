// Multi-tensor optimizer update over the flat parameter buffers (README
// Contents section: SGD and Adam; Adam moments exist only when requested).
//
// One launch updates every tensor: a chunk table lists runs of at most
// 2048 elements of one tensor, one block per chunk, float4 accesses.  The
// same pass writes the bf16 copy of each updated weight for the next forward.
//
// Adam (t = step, 1-based): m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2,
// p -= (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps).
// LaProp (the published algorithm of Ziyin, Wang & Ueda, 2020; the paper's
// checkpoint notes name it beside Adam): v = b2 v + (1-b2) g^2,
// m = b1 m + (1-b1) g / (sqrt(v) / sqrt(1 - b2^t) + eps),
// p -= (lr / (1 - b1^t)) m.
// SGD with heavy-ball momentum mu: b = mu b + g, p -= lr b.
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

__global__ void step_scalars_kernel(float* dst, float lr_bc1, float inv_sqrt_bc2) {
  dst[0] = lr_bc1;
  dst[1] = inv_sqrt_bc2;
}

__global__ void __launch_bounds__(256) adam_kernel(const Chunk* chunks, float* p, const float* g,
                                                   float* m, float* v, bf16* shadow, float lr_bc1,
                                                   float inv_sqrt_bc2, float b1, float b2,
                                                   float eps) {
  const Chunk c = chunks[blockIdx.x];
  const long long base = c.start;
  const int n4 = c.len >> 2;
  float4* p4 = reinterpret_cast<float4*>(p + base);
  const float4* g4 = reinterpret_cast<const float4*>(g + base);
  float4* m4 = reinterpret_cast<float4*>(m + base);
  float4* v4 = reinterpret_cast<float4*>(v + base);
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    float4 pp = p4[i], gg = g4[i], mm = m4[i], vv = v4[i];
    adam_one(pp.x, gg.x, mm.x, vv.x, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    adam_one(pp.y, gg.y, mm.y, vv.y, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    adam_one(pp.z, gg.z, mm.z, vv.z, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    adam_one(pp.w, gg.w, mm.w, vv.w, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    p4[i] = pp;
    m4[i] = mm;
    v4[i] = vv;
    if (shadow && c.shadow) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(pp.z, pp.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(shadow + base)[i] = packed;
    }
  }
  for (int i = (n4 << 2) + threadIdx.x; i < c.len; i += blockDim.x) {
    long long k = base + i;
    float pp = p[k], mm = m[k], vv = v[k];
    adam_one(pp, g[k], mm, vv, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    p[k] = pp;
    m[k] = mm;
    v[k] = vv;
    if (shadow && c.shadow) shadow[k] = __float2bfloat16_rn(pp);
  }
}

__device__ __forceinline__ void laprop_one(float& p, float g, float& m, float& v, float lr_bc1,
                                           float inv_sqrt_bc2, float b1, float b2, float eps) {
  v = b2 * v + (1.0f - b2) * g * g;
  m = b1 * m + (1.0f - b1) * g / (sqrtf(v) * inv_sqrt_bc2 + eps);
  p -= lr_bc1 * m;
}

__device__ __forceinline__ void shadow4(bf16* shadow, long long base, int i, const float4& pp) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(pp.z, pp.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(shadow + base)[i] = packed;
}

__global__ void __launch_bounds__(256) laprop_kernel(const Chunk* chunks, float* p, const float* g,
                                                     float* m, float* v, bf16* shadow, float lr_bc1,
                                                     float inv_sqrt_bc2, float b1, float b2,
                                                     float eps) {
  const Chunk c = chunks[blockIdx.x];
  const long long base = c.start;
  const int n4 = c.len >> 2;
  float4* p4 = reinterpret_cast<float4*>(p + base);
  const float4* g4 = reinterpret_cast<const float4*>(g + base);
  float4* m4 = reinterpret_cast<float4*>(m + base);
  float4* v4 = reinterpret_cast<float4*>(v + base);
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    float4 pp = p4[i], gg = g4[i], mm = m4[i], vv = v4[i];
    laprop_one(pp.x, gg.x, mm.x, vv.x, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    laprop_one(pp.y, gg.y, mm.y, vv.y, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    laprop_one(pp.z, gg.z, mm.z, vv.z, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    laprop_one(pp.w, gg.w, mm.w, vv.w, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    p4[i] = pp;
    m4[i] = mm;
    v4[i] = vv;
    if (shadow && c.shadow) shadow4(shadow, base, i, pp);
  }
  for (int i = (n4 << 2) + threadIdx.x; i < c.len; i += blockDim.x) {
    long long k = base + i;
    float pp = p[k], mm = m[k], vv = v[k];
    laprop_one(pp, g[k], mm, vv, lr_bc1, inv_sqrt_bc2, b1, b2, eps);
    p[k] = pp;
    m[k] = mm;
    v[k] = vv;
    if (shadow && c.shadow) shadow[k] = __float2bfloat16_rn(pp);
  }
}

__global__ void __launch_bounds__(256) momentum_kernel(const Chunk* chunks, float* p,
                                                       const float* g, float* b, bf16* shadow,
                                                       float lr, float mu) {
  const Chunk c = chunks[blockIdx.x];
  const long long base = c.start;
  const int n4 = c.len >> 2;
  float4* p4 = reinterpret_cast<float4*>(p + base);
  const float4* g4 = reinterpret_cast<const float4*>(g + base);
  float4* b4 = reinterpret_cast<float4*>(b + base);
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    float4 pp = p4[i], gg = g4[i], bb = b4[i];
    bb.x = mu * bb.x + gg.x; bb.y = mu * bb.y + gg.y; bb.z = mu * bb.z + gg.z; bb.w = mu * bb.w + gg.w;
    pp.x -= lr * bb.x; pp.y -= lr * bb.y; pp.z -= lr * bb.z; pp.w -= lr * bb.w;
    p4[i] = pp;
    b4[i] = bb;
    if (shadow && c.shadow) shadow4(shadow, base, i, pp);
  }
  for (int i = (n4 << 2) + threadIdx.x; i < c.len; i += blockDim.x) {
    long long k = base + i;
    const float bb = mu * b[k] + g[k];
    const float pp = p[k] - lr * bb;
    b[k] = bb;
    p[k] = pp;
    if (shadow && c.shadow) shadow[k] = __float2bfloat16_rn(pp);
  }
}

__global__ void __launch_bounds__(256) sgd_kernel(const Chunk* chunks, float* p, const float* g,
                                                  bf16* shadow, float lr) {
  const Chunk c = chunks[blockIdx.x];
  for (int i = threadIdx.x; i < c.len; i += blockDim.x) {
    long long k = c.start + i;
    float pp = p[k] - lr * g[k];
    p[k] = pp;
    if (shadow && c.shadow) shadow[k] = __float2bfloat16_rn(pp);
  }
}

__global__ void __launch_bounds__(256) cast_shadow_kernel(const Chunk* chunks, const float* p,
                                                          bf16* shadow) {
  const Chunk c = chunks[blockIdx.x];
  if (!c.shadow) return;
  for (int i = threadIdx.x; i < c.len; i += blockDim.x) {
    long long k = c.start + i;
    shadow[k] = __float2bfloat16_rn(p[k]);
  }
}

template <typename T>
__global__ void cast_f32_kernel(const T* src, float* dst, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = ld_elem(src, i);
}

__global__ void nonfinite_kernel(const float* d, size_t n, unsigned long long* first) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    if (!isfinite(d[i])) atomicMin(first, (unsigned long long)i);
}

}  // namespace

cudaError_t write_step_scalars(float* dst, float lr_bc1, float inv_sqrt_bc2, cudaStream_t s) {
  step_scalars_kernel<<<1, 1, 0, s>>>(dst, lr_bc1, inv_sqrt_bc2);
  return cudaGetLastError();
}

bool optimizer_kernel_info(const void* func, OptKernelInfo* info) {
  // argument lists of the update kernels above: pointers are 8 bytes, scalars 4
  static const int two_moment[11] = {8, 8, 8, 8, 8, 8, 4, 4, 4, 4, 4};
  static const int momentum[7] = {8, 8, 8, 8, 8, 4, 4};
  static const int sgd[5] = {8, 8, 8, 8, 4};
  static const int scalars[3] = {8, 4, 4};
  const int* sizes = nullptr;
  if (func == reinterpret_cast<const void*>(adam_kernel) ||
      func == reinterpret_cast<const void*>(laprop_kernel)) {
    sizes = two_moment;
    info->nargs = 11;
    info->i_lr_bc1 = 6;
    info->i_inv_sqrt_bc2 = 7;
    info->i_lr = -1;
  } else if (func == reinterpret_cast<const void*>(step_scalars_kernel)) {
    sizes = scalars;
    info->nargs = 3;
    info->i_lr_bc1 = 1;
    info->i_inv_sqrt_bc2 = 2;
    info->i_lr = -1;
  } else if (func == reinterpret_cast<const void*>(momentum_kernel)) {
    sizes = momentum;
    info->nargs = 7;
    info->i_lr_bc1 = info->i_inv_sqrt_bc2 = -1;
    info->i_lr = 5;
  } else if (func == reinterpret_cast<const void*>(sgd_kernel)) {
    sizes = sgd;
    info->nargs = 5;
    info->i_lr_bc1 = info->i_inv_sqrt_bc2 = -1;
    info->i_lr = 4;
  } else {
    return false;
  }
  for (int i = 0; i < info->nargs; ++i) info->size[i] = sizes[i];
  return true;
}

cudaError_t adam_update(const Chunk* chunks, int n_chunks, float* p, const float* g, float* m,
                        float* v, void* shadow, float lr_over_bc1, float inv_sqrt_bc2,
                        float beta1, float beta2, float eps, cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  adam_kernel<<<n_chunks, 256, 0, s>>>(chunks, p, g, m, v, (bf16*)shadow, lr_over_bc1,
                                       inv_sqrt_bc2, beta1, beta2, eps);
  return cudaGetLastError();
}

cudaError_t laprop_update(const Chunk* chunks, int n_chunks, float* p, const float* g, float* m,
                          float* v, void* shadow, float lr_over_bc1, float inv_sqrt_bc2,
                          float beta1, float beta2, float eps, cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  laprop_kernel<<<n_chunks, 256, 0, s>>>(chunks, p, g, m, v, (bf16*)shadow, lr_over_bc1,
                                         inv_sqrt_bc2, beta1, beta2, eps);
  return cudaGetLastError();
}

cudaError_t momentum_update(const Chunk* chunks, int n_chunks, float* p, const float* g, float* b,
                            void* shadow, float lr, float mu, cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  momentum_kernel<<<n_chunks, 256, 0, s>>>(chunks, p, g, b, (bf16*)shadow, lr, mu);
  return cudaGetLastError();
}

cudaError_t sgd_update(const Chunk* chunks, int n_chunks, float* p, const float* g, void* shadow,
                       float lr, cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  sgd_kernel<<<n_chunks, 256, 0, s>>>(chunks, p, g, (bf16*)shadow, lr);
  return cudaGetLastError();
}

cudaError_t cast_shadow(const Chunk* chunks, int n_chunks, const float* p, void* shadow,
                        cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  cast_shadow_kernel<<<n_chunks, 256, 0, s>>>(chunks, p, (bf16*)shadow);
  return cudaGetLastError();
}

cudaError_t cast_to_f32(DType t, const void* src, float* dst, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int grid = (int)((n + 255) / 256 < 152 * 8 ? (n + 255) / 256 : 152 * 8);
  if (t == DT_F32)
    cast_f32_kernel<float><<<grid, 256, 0, s>>>((const float*)src, dst, n);
  else
    cast_f32_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)src, dst, n);
  return cudaGetLastError();
}

cudaError_t find_nonfinite(const float* data, size_t n, unsigned long long* first_bad,
                           cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int grid = (int)((n + 255) / 256 < 152 * 8 ? (n + 255) / 256 : 152 * 8);
  nonfinite_kernel<<<grid, 256, 0, s>>>(data, n, first_bad);
  return cudaGetLastError();
}

}  // namespace mg
