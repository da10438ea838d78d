// Loss kernels: row softmax cross-entropy (+ its gradient) and mean squared
// error (+ its gradient), the reduction archetype of the Meganeura README
// (Example section: cross_entropy_loss(logits, labels) with a dense [B, C]
// label tensor; "Why Meganeura" section: the reduction kernel archetype).
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "../../include/mg.h"
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

// Deterministic sum of v[0..n) times scale, one block.
__global__ void __launch_bounds__(1024) reduce_sum_kernel(const float* v, int n, float scale,
                                                          float* out) {
  __shared__ float red[32];
  float s = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += v[i];
  s = block_sum(s, red);
  if (threadIdx.x == 0) *out = s * scale;
}

// One block per row.  Pass 1: running (max, sum of exp) per thread, merged
// across the block; pass 2: gradient.  Labels: dense fp32 [B, C] or int32 ids.
template <typename T, bool DENSE>
__global__ void __launch_bounds__(256) ce_kernel(const T* logits, int C, long long ld,
                                                 const void* labels, T* dlogits,
                                                 float* row_loss, float inv_b) {
  __shared__ float red[32];
  __shared__ float sh_m, sh_s;
  const int r = blockIdx.x;
  const T* z = logits + (size_t)r * ld;
  T* dz = dlogits + (size_t)r * ld;

  float m = -INFINITY, s = 0.0f;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    float x = ld_elem(z, c);
    if (x > m) {
      s = s * expf(m - x) + 1.0f;
      m = x;
    } else {
      s += expf(x - m);
    }
  }
  // merge (m, s) across the block
  float bm = block_max(m, red);
  float sc = (m == -INFINITY) ? 0.0f : s * expf(m - bm);
  float bs = block_sum(sc, red);
  if (threadIdx.x == 0) {
    sh_m = bm;
    sh_s = bs;
  }
  __syncthreads();
  const float lse = sh_m + logf(sh_s);

  float ysum = 1.0f, yz = 0.0f;
  if (DENSE) {
    const float* y = static_cast<const float*>(labels) + (size_t)r * C;
    float a = 0.0f, b = 0.0f;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
      float yc = y[c];
      a += yc;
      b += yc * ld_elem(z, c);
    }
    ysum = block_sum(a, red);
    yz = block_sum(b, red);
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
      float p = expf(ld_elem(z, c) - lse);
      st_elem(dz, c, (p * ysum - y[c]) * inv_b);
    }
    if (threadIdx.x == 0) row_loss[r] = lse * ysum - yz;
  } else {
    const int t = static_cast<const int*>(labels)[r];
    const bool ok = t >= 0 && t < C;      // an id outside [0, C) poisons the loss (NaN)
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
      float p = expf(ld_elem(z, c) - lse);
      st_elem(dz, c, (p - (c == t ? 1.0f : 0.0f)) * inv_b);
    }
    if (threadIdx.x == 0) row_loss[r] = ok ? lse - ld_elem(z, t) : __int_as_float(0x7fc00000);
  }
}

// The gradient pass of a bf16 row given its log-sum-exp: dense labels' sums,
// dlogits = (softmax * sum(y) - y) / B, the row's loss.
template <bool DENSE>
__device__ __forceinline__ void ce_vec_tail(const bf16* z, bf16* dz, int C, const void* labels,
                                            int r, float lse, float* red, float* row_loss,
                                            float inv_b) {
  const int nv = C >> 3;
  float ysum = 1.0f, yz = 0.0f;
  int t = -1;
  const float* y = DENSE ? static_cast<const float*>(labels) + (size_t)r * C : nullptr;
  if (DENSE) {
    float a = 0.0f, b = 0.0f;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float4 y0 = reinterpret_cast<const float4*>(y)[2 * v];
      float4 y1 = reinterpret_cast<const float4*>(y)[2 * v + 1];
      uint4 u = reinterpret_cast<const uint4*>(z)[v];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
      float2 t0 = __bfloat1622float2(h[0]), t1 = __bfloat1622float2(h[1]);
      float2 t2 = __bfloat1622float2(h[2]), t3 = __bfloat1622float2(h[3]);
      a += y0.x + y0.y + y0.z + y0.w + y1.x + y1.y + y1.z + y1.w;
      b += y0.x * t0.x + y0.y * t0.y + y0.z * t1.x + y0.w * t1.y + y1.x * t2.x + y1.y * t2.y +
           y1.z * t3.x + y1.w * t3.y;
    }
    ysum = block_sum(a, red);
    yz = block_sum(b, red);
  } else {
    t = static_cast<const int*>(labels)[r];
  }
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 u = reinterpret_cast<const uint4*>(z)[v];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
    float g[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 q = __bfloat1622float2(h[i]);
      g[2 * i] = expf(q.x - lse);
      g[2 * i + 1] = expf(q.y - lse);
    }
    if (DENSE) {
      float4 y0 = reinterpret_cast<const float4*>(y)[2 * v];
      float4 y1 = reinterpret_cast<const float4*>(y)[2 * v + 1];
      const float yy[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = (g[i] * ysum - yy[i]) * inv_b;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = (g[i] - (v * 8 + i == t ? 1.0f : 0.0f)) * inv_b;
    }
    uint4 o;
    uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 hh = __floats2bfloat162_rn(g[2 * i], g[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&hh);
    }
    reinterpret_cast<uint4*>(dz)[v] = o;
  }
  if (threadIdx.x == 0) {
    if (DENSE)
      row_loss[r] = lse * ysum - yz;
    else
      row_loss[r] = (t >= 0 && t < C) ? lse - __bfloat162float(z[t]) : __int_as_float(0x7fc00000);
  }
}

// bf16 logits whose rows are whole 16-byte vectors (C % 8 == 0): the same two
// passes with 8 columns per access.
template <bool DENSE>
__global__ void __launch_bounds__(256) ce_kernel_vec(const bf16* logits, int C, long long ld,
                                                     const void* labels, bf16* dlogits,
                                                     float* row_loss, float inv_b) {
  __shared__ float red[32];
  __shared__ float sh_m, sh_s;
  const int r = blockIdx.x;
  const bf16* z = logits + (size_t)r * ld;
  bf16* dz = dlogits + (size_t)r * ld;
  const int nv = C >> 3;
  float m = -INFINITY, s = 0.0f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 u = reinterpret_cast<const uint4*>(z)[v];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      x[2 * i] = t.x;
      x[2 * i + 1] = t.y;
    }
    float vm = x[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) vm = fmaxf(vm, x[i]);
    if (vm > m) {
      s = (m == -INFINITY) ? 0.0f : s * expf(m - vm);
      m = vm;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) s += expf(x[i] - m);
  }
  float bm = block_max(m, red);
  float sc = (m == -INFINITY) ? 0.0f : s * expf(m - bm);
  float bs = block_sum(sc, red);
  if (threadIdx.x == 0) {
    sh_m = bm;
    sh_s = bs;
  }
  __syncthreads();
  const float lse = sh_m + logf(sh_s);
  ce_vec_tail<DENSE>(z, dz, C, labels, r, lse, red, row_loss, inv_b);
}

// Same from per-row softmax partials written by the head GEMM's epilogue (in
// base 2: max of x log2 e and the sum of 2^(x log2 e - max), per 128-column
// chunk), combined into the log-sum-exp, then the gradient pass.
template <bool DENSE>
__global__ void __launch_bounds__(256) ce_kernel_part(const bf16* logits, int C, long long ld,
                                                      const float2* parts, int nparts,
                                                      const void* labels, bf16* dlogits,
                                                      float* row_loss, float inv_b) {
  __shared__ float red[32];
  __shared__ float sh_m, sh_s;
  const int r = blockIdx.x;
  // partials in base 2: (max of x log2 e, sum of 2^(x log2 e - max))
  const float2* pr = parts + (size_t)r * nparts;
  float m = -INFINITY;
  for (int k = threadIdx.x; k < nparts; k += blockDim.x) m = fmaxf(m, pr[k].x);
  const float bm = block_max(m, red);
  float s = 0.0f;
  for (int k = threadIdx.x; k < nparts; k += blockDim.x) {
    const float2 q = pr[k];
    if (q.x > -INFINITY) s += q.y * exp2f(q.x - bm);
  }
  const float bs = block_sum(s, red);
  if (threadIdx.x == 0) {
    sh_m = bm;
    sh_s = bs;
  }
  __syncthreads();
  const float lse = (sh_m + log2f(sh_s)) * 0.6931471805599453f;   // back to base e
  ce_vec_tail<DENSE>(logits + (size_t)r * ld, dlogits + (size_t)r * ld, C, labels, r, lse, red,
                     row_loss, inv_b);
}

template <typename T>
__global__ void __launch_bounds__(256) mse_kernel(const T* o, const T* t, size_t n, T* dout,
                                                  float* partials, float two_over_n) {
  __shared__ float red[32];
  float acc = 0.0f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float d = ld_elem(o, i) - ld_elem(t, i);
    acc += d * d;
    st_elem(dout, i, d * two_over_n);
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = acc;
}

}  // namespace

cudaError_t ce_loss(DType t, const void* logits, int B, int C, long long ld, int label_kind,
                    const void* labels, void* dlogits, float* row_loss, float* loss,
                    cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  float inv_b = 1.0f / (float)B;
  if (t == DT_F32) {
    if (label_kind == 0)
      ce_kernel<float, true><<<B, 256, 0, s>>>((const float*)logits, C, ld, labels,
                                               (float*)dlogits, row_loss, inv_b);
    else
      ce_kernel<float, false><<<B, 256, 0, s>>>((const float*)logits, C, ld, labels,
                                                (float*)dlogits, row_loss, inv_b);
  } else if (C % 8 == 0 && ld % 8 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0 &&
             (reinterpret_cast<uintptr_t>(dlogits) & 15) == 0 &&
             (label_kind == 1 || (reinterpret_cast<uintptr_t>(labels) & 15) == 0)) {
    if (label_kind == 0)
      ce_kernel_vec<true><<<B, 256, 0, s>>>((const bf16*)logits, C, ld, labels, (bf16*)dlogits,
                                            row_loss, inv_b);
    else
      ce_kernel_vec<false><<<B, 256, 0, s>>>((const bf16*)logits, C, ld, labels, (bf16*)dlogits,
                                             row_loss, inv_b);
  } else {
    if (label_kind == 0)
      ce_kernel<bf16, true><<<B, 256, 0, s>>>((const bf16*)logits, C, ld, labels,
                                              (bf16*)dlogits, row_loss, inv_b);
    else
      ce_kernel<bf16, false><<<B, 256, 0, s>>>((const bf16*)logits, C, ld, labels,
                                               (bf16*)dlogits, row_loss, inv_b);
  }
  reduce_sum_kernel<<<1, 1024, 0, s>>>(row_loss, B, inv_b, loss);
  return cudaGetLastError();
}

cudaError_t ce_loss_from_partials(const void* logits, int B, int C, long long ld,
                                  const float2* parts, int nparts, int label_kind,
                                  const void* labels, void* dlogits, float* row_loss,
                                  float* loss, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  if (C % 8 || ld % 8 || (reinterpret_cast<uintptr_t>(logits) & 15) ||
      (reinterpret_cast<uintptr_t>(dlogits) & 15) ||
      (label_kind == 0 && (reinterpret_cast<uintptr_t>(labels) & 15)) || nparts != (C + 127) / 128)
    return cudaErrorInvalidValue;
  const float inv_b = 1.0f / (float)B;
  if (label_kind == 0)
    ce_kernel_part<true><<<B, 256, 0, s>>>((const bf16*)logits, C, ld, parts, nparts, labels,
                                           (bf16*)dlogits, row_loss, inv_b);
  else
    ce_kernel_part<false><<<B, 256, 0, s>>>((const bf16*)logits, C, ld, parts, nparts, labels,
                                            (bf16*)dlogits, row_loss, inv_b);
  reduce_sum_kernel<<<1, 1024, 0, s>>>(row_loss, B, inv_b, loss);
  return cudaGetLastError();
}

// Same with 16-byte accesses: V elements of o, t and dout per step.
template <typename T>
__global__ void __launch_bounds__(256) mse_kernel_vec(const T* o, const T* t, size_t n, T* dout,
                                                      float* partials, float two_over_n) {
  constexpr int V = 16 / sizeof(T);
  __shared__ float red[32];
  float acc = 0.0f;
  const size_t nv = n / V;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 uo = reinterpret_cast<const uint4*>(o)[i];
    const uint4 ut = reinterpret_cast<const uint4*>(t)[i];
    uint4 ud;
    const T* eo = reinterpret_cast<const T*>(&uo);
    const T* et = reinterpret_cast<const T*>(&ut);
    T* ed = reinterpret_cast<T*>(&ud);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float d = ld_elem(eo, k) - ld_elem(et, k);
      acc += d * d;
      st_elem(ed, k, d * two_over_n);
    }
    reinterpret_cast<uint4*>(dout)[i] = ud;
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = acc;
}

cudaError_t mse_loss(DType t, const void* o, const void* target, size_t n, void* dout,
                     float* partials, int n_partials, float* loss, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  float two_over_n = (float)(2.0 / (double)n);
  const size_t V = (t == DT_F32) ? 4 : 8;
  const bool vec = n % V == 0 && ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(target) |
                                   reinterpret_cast<uintptr_t>(dout)) & 15) == 0;
  if (vec && t == DT_F32)
    mse_kernel_vec<float><<<n_partials, 256, 0, s>>>((const float*)o, (const float*)target, n,
                                                     (float*)dout, partials, two_over_n);
  else if (vec)
    mse_kernel_vec<bf16><<<n_partials, 256, 0, s>>>((const bf16*)o, (const bf16*)target, n,
                                                    (bf16*)dout, partials, two_over_n);
  else if (t == DT_F32)
    mse_kernel<float><<<n_partials, 256, 0, s>>>((const float*)o, (const float*)target, n,
                                                 (float*)dout, partials, two_over_n);
  else
    mse_kernel<bf16><<<n_partials, 256, 0, s>>>((const bf16*)o, (const bf16*)target, n,
                                                (bf16*)dout, partials, two_over_n);
  reduce_sum_kernel<<<1, 1024, 0, s>>>(partials, n_partials, (float)(1.0 / (double)n), loss);
  return cudaGetLastError();
}

}  // namespace mg

// ---------------------------------------------------------------------------
// Softmax cross-entropy without any device allocation.
//
// For callers that are not allowed to allocate device memory -- code running
// inside another framework's plugin or kernel-enqueue hook, or a process whose
// device memory is already reserved by its own caching allocator -- and so
// cannot create a plan (mg_step_plan_create allocates the plan's workspace).
// The per-row losses that the plan keeps in its workspace live here in a
// fixed file-scope device array instead.  Every GPU that loads the library
// holds this array (kNoAllocMaxRows floats, 256 KB) until the process exits.
namespace {

constexpr int kNoAllocMaxRows = 65536;
__device__ __align__(256) float g_noalloc_row_loss[kNoAllocMaxRows];

// The array's device address is looked up once per device context and kept
// with that context's id: a cudaDeviceReset (or any re-creation of the
// primary context) loads the module again, possibly at another address, and
// the new context has a new id, so the address is looked up again.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct ScratchSlot {
  unsigned long long ctx_id;
  float* ptr;
};

std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 256;
ScratchSlot g_noalloc_scratch[kMaxDevices] = {};   // per device: context id, device address

// Id of the calling thread's current context; false when there is none yet
// or the driver lacks the calls.
bool current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    looked_up = true;
  }
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" mg_status mg_softmax_ce_noalloc(int dtype, const void* logits, int rows, int cols,
                                           int label_kind, const void* labels, void* dlogits,
                                           float* loss, mg_stream_t stream) {
  using namespace mg;
  if (!logits || !labels || !dlogits || !loss) {
    set_global_error("mg_softmax_ce_noalloc: logits, labels, dlogits and loss must be non-NULL");
    return MG_ERR_INVALID_ARG;
  }
  if ((dtype != 0 && dtype != 1) || (label_kind != 0 && label_kind != 1)) {
    set_global_error("mg_softmax_ce_noalloc: dtype and label_kind must be 0 or 1");
    return MG_ERR_INVALID_ARG;
  }
  if (rows < 1 || rows > kNoAllocMaxRows || cols < 1) {
    set_global_error("mg_softmax_ce_noalloc: rows must be in [1, 65536] and cols >= 1");
    return MG_ERR_INVALID_ARG;
  }
  char msg[256];
  // An error left pending by earlier work on this thread is reported as such,
  // not as a failure of this call's launches (and nothing is launched).
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg,
             "mg_softmax_ce_noalloc: a CUDA error was already pending before the call (%s); "
             "nothing launched", cudaGetErrorString(e));
    set_global_error(msg);
    return MG_ERR_CUDA;
  }
  int dev = -1;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_global_error("mg_softmax_ce_noalloc: no usable current CUDA device");
    return MG_ERR_CUDA;
  }
  float* scratch = nullptr;
  {
    // Set-up on the first call in each device context: look up the array's
    // device address (host code cannot use the array's name as a device
    // pointer).
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    unsigned long long id = 0;
    const bool have_id = current_ctx_id(&id);
    ScratchSlot& slot = g_noalloc_scratch[dev];
    if (!have_id || !slot.ptr || slot.ctx_id != id) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_row_loss);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        snprintf(msg, sizeof msg, "mg_softmax_ce_noalloc: cudaGetSymbolAddress failed (%s)",
                 cudaGetErrorString(e));
        set_global_error(msg);
        return MG_ERR_CUDA;
      }
      // the lookup made the context current if it was not yet
      slot.ptr = static_cast<float*>(p);
      slot.ctx_id = current_ctx_id(&id) ? id : 0;
      if (!slot.ctx_id) slot.ptr = nullptr;   // no id to key it on: look it up every call
      scratch = static_cast<float*>(p);
    } else {
      scratch = slot.ptr;
    }
  }
  // Every row's slot is written before the reduction reads it, so the array
  // needs no clearing between calls.
  e = ce_loss(dtype == 1 ? DT_BF16 : DT_F32, logits, rows, cols, cols, label_kind, labels,
              dlogits, scratch, loss, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "mg_softmax_ce_noalloc: kernel launch failed (%s)",
             cudaGetErrorString(e));
    set_global_error(msg);
    return MG_ERR_CUDA;
  }
  return MG_OK;
}
