// RMSNorm forward/backward and column sums (bias and gamma gradients): the
// reduction archetype of the Meganeura README ("Why Meganeura" section).
//
// RMSNorm: r = 1/sqrt(mean(x^2) + eps), y = x r gamma.  Backward with g = dy
// gamma: dx = r (g - x r^2 mean(g x)), dgamma = sum_rows dy x r.
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

constexpr int NORM_THREADS = 256;
constexpr int NORM_MAX_PER_THREAD = 16;   // d <= 4096

template <typename T>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_fwd_kernel(const T* x, const float* gamma,
                                                                    T* y, float* rstd, int rows,
                                                                    int d, float eps) {
  __shared__ float red[32];
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* xr = x + (size_t)r * d;
    float v[NORM_MAX_PER_THREAD];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < NORM_MAX_PER_THREAD; ++i) {
      int c = threadIdx.x + i * NORM_THREADS;
      v[i] = c < d ? ld_elem(xr, c) : 0.0f;
      ss += v[i] * v[i];
    }
    ss = block_sum(ss, red);
    float rs = 1.0f / sqrtf(ss / (float)d + eps);
    if (threadIdx.x == 0) rstd[r] = rs;
    T* yr = y + (size_t)r * d;
#pragma unroll
    for (int i = 0; i < NORM_MAX_PER_THREAD; ++i) {
      int c = threadIdx.x + i * NORM_THREADS;
      if (c < d) st_elem(yr, c, v[i] * rs * gamma[c]);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_bwd_kernel(
    const T* dy, const T* x, const float* rstd, const float* gamma, const T* dadd, T* dx,
    float* dgamma_partials, int rows, int d) {
  __shared__ float red[32];
  float dg[NORM_MAX_PER_THREAD];
#pragma unroll
  for (int i = 0; i < NORM_MAX_PER_THREAD; ++i) dg[i] = 0.0f;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* dyr = dy + (size_t)r * d;
    const T* xr = x + (size_t)r * d;
    const float rs = rstd[r];
    float xv[NORM_MAX_PER_THREAD], gv[NORM_MAX_PER_THREAD];
    float gx = 0.0f;
#pragma unroll
    for (int i = 0; i < NORM_MAX_PER_THREAD; ++i) {
      int c = threadIdx.x + i * NORM_THREADS;
      float dyc = c < d ? ld_elem(dyr, c) : 0.0f;
      xv[i] = c < d ? ld_elem(xr, c) : 0.0f;
      gv[i] = c < d ? dyc * gamma[c] : 0.0f;
      dg[i] += dyc * xv[i] * rs;
      gx += gv[i] * xv[i];
    }
    if (dx) {
      gx = block_sum(gx, red) / (float)d;
      const float k = rs * rs * gx;
      T* dxr = dx + (size_t)r * d;
      const T* ar = dadd ? dadd + (size_t)r * d : nullptr;
#pragma unroll
      for (int i = 0; i < NORM_MAX_PER_THREAD; ++i) {
        int c = threadIdx.x + i * NORM_THREADS;
        if (c < d) {
          float val = rs * (gv[i] - xv[i] * k);
          if (ar) val += ld_elem(ar, c);
          st_elem(dxr, c, val);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NORM_MAX_PER_THREAD; ++i) {
    int c = threadIdx.x + i * NORM_THREADS;
    if (c < d) dgamma_partials[(size_t)blockIdx.x * d + c] = dg[i];
  }
}

// bf16 rows with d a multiple of 8: each thread owns 16-byte vectors (8
// columns) v = tid, tid + 256, ... of every row it visits.
constexpr int NV_MAX = 4;   // d <= 256 * 8 * 4 = 8192

__device__ __forceinline__ void ld8(const bf16* p, float* f) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void st8(bf16* p, const float* f) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = u;
}

// NV = vectors per thread (d <= 2048 NV for 256 threads); gamma stays in
// registers across the rows a block visits.
template <int NV>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_fwd_vec(const bf16* x, const float* gamma,
                                                                bf16* y, float* rstd, int rows,
                                                                int d, float eps) {
  __shared__ float red[32];
  const int nvec = d >> 3;
  float gm[NV][8];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vi = threadIdx.x + i * NORM_THREADS;
#pragma unroll
    for (int j = 0; j < 8; ++j) gm[i][j] = vi < nvec ? gamma[vi * 8 + j] : 0.0f;
  }
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const bf16* xr = x + (size_t)r * d;
    float v[NV][8];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      int vi = threadIdx.x + i * NORM_THREADS;
      if (vi < nvec) {
        ld8(xr + vi * 8, v[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += v[i][j] * v[i][j];
      }
    }
    ss = block_sum(ss, red);
    const float rs = 1.0f / sqrtf(ss / (float)d + eps);
    if (threadIdx.x == 0) rstd[r] = rs;
    bf16* yr = y + (size_t)r * d;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      int vi = threadIdx.x + i * NORM_THREADS;
      if (vi < nvec) {
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = v[i][j] * rs * gm[i][j];
        st8(yr + vi * 8, o);
      }
    }
  }
}

template <int NV>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_bwd_vec(const bf16* dy, const bf16* x,
                                                                const float* rstd,
                                                                const float* gamma,
                                                                const bf16* dadd, bf16* dx,
                                                                float* dgamma_partials, int rows,
                                                                int d) {
  __shared__ float red[32];
  const int nvec = d >> 3;
  float dg[NV][8], gm[NV][8];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vi = threadIdx.x + i * NORM_THREADS;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      dg[i][j] = 0.0f;
      gm[i][j] = vi < nvec ? gamma[vi * 8 + j] : 0.0f;
    }
  }
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const float rs = rstd[r];
    float xv[NV][8], gv[NV][8];
    float gx = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      int vi = threadIdx.x + i * NORM_THREADS;
      if (vi < nvec) {
        float dyv[8];
        ld8(dy + (size_t)r * d + vi * 8, dyv);
        ld8(x + (size_t)r * d + vi * 8, xv[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          gv[i][j] = dyv[j] * gm[i][j];
          dg[i][j] += dyv[j] * xv[i][j] * rs;
          gx += gv[i][j] * xv[i][j];
        }
      }
    }
    if (dx) {
      gx = block_sum(gx, red) / (float)d;
      const float k = rs * rs * gx;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        int vi = threadIdx.x + i * NORM_THREADS;
        if (vi < nvec) {
          float o[8], a[8];
          if (dadd) ld8(dadd + (size_t)r * d + vi * 8, a);
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] = rs * (gv[i][j] - xv[i][j] * k) + (dadd ? a[j] : 0.0f);
          st8(dx + (size_t)r * d + vi * 8, o);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    int vi = threadIdx.x + i * NORM_THREADS;
    if (vi < nvec) {
#pragma unroll
      for (int j = 0; j < 8; ++j) dgamma_partials[(size_t)blockIdx.x * d + vi * 8 + j] = dg[i][j];
    }
  }
}

// partials[chunk, c] = sum of src[r, c] over the rows of this chunk.
template <typename T>
__global__ void __launch_bounds__(256) colsum_pass1(const T* src, int rows, int cols, long long ld,
                                                    float* partials) {
  int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  int chunks = gridDim.y;
  int per = (rows + chunks - 1) / chunks;
  int r0 = blockIdx.y * per, r1 = min(rows, r0 + per);
  float s = 0.0f;
  for (int r = r0; r < r1; ++r) s += ld_elem(src, (size_t)r * ld + c);
  partials[(size_t)blockIdx.y * cols + c] = s;
}

// Same, each thread summing 16 bytes of columns (8 bf16 or 4 fp32) with
// 16-byte loads, four rows in flight.
template <typename T>
__global__ void __launch_bounds__(256) colsum_pass1_vec(const T* src, int rows, int cols,
                                                        long long ld, float* partials) {
  constexpr int V = 16 / sizeof(T);
  const int cg = blockIdx.x * blockDim.x + threadIdx.x;
  if (cg * V >= cols) return;
  const int chunks = gridDim.y;
  const int per = (rows + chunks - 1) / chunks;
  const int r0 = blockIdx.y * per, r1 = min(rows, r0 + per);
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  const T* base = src + (size_t)cg * V;
  int r = r0;
  for (; r + 4 <= r1; r += 4) {
    uint4 u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) u[q] = *reinterpret_cast<const uint4*>(base + (size_t)(r + q) * ld);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const T* e = reinterpret_cast<const T*>(&u[q]);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += ld_elem(e, i);
    }
  }
  for (; r < r1; ++r) {
    const uint4 u = *reinterpret_cast<const uint4*>(base + (size_t)r * ld);
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] += ld_elem(e, i);
  }
  float4* out = reinterpret_cast<float4*>(partials + (size_t)blockIdx.y * cols + (size_t)cg * V);
#pragma unroll
  for (int i = 0; i < V / 4; ++i) out[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
}

// out[c] = sum over chunks of partials[chunk, c]: a block takes 32 columns,
// its eight warps eight interleaved subsets of the chunks (coalesced 128-byte
// rows), combined through shared memory.
__global__ void __launch_bounds__(256) colsum_pass2_wide(const float* partials, int chunks,
                                                         int cols, float* out) {
  __shared__ float red[8][32];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float s = 0.0f;
  if (c < cols)
    for (int k = grp; k < chunks; k += 8) s += partials[(size_t)k * cols + c];
  red[grp][lane] = s;
  __syncthreads();
  if (grp == 0 && c < cols) {
    float t = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) t += red[q][lane];
    out[c] = t;
  }
}

}  // namespace

cudaError_t colsum(DType t, const void* src, int rows, int cols, long long ld, float* partials,
                   size_t partial_floats, float* out, cudaStream_t s) {
  if (cols <= 0) return cudaSuccess;
  if (rows <= 0 || partial_floats < (size_t)cols) return cudaErrorInvalidValue;
  const int V = (t == DT_F32) ? 4 : 8;
  const bool vec = cols % V == 0 && ld % V == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  // about two blocks per SM over columns x row chunks, within the partials buffer
  const int gx = vec ? (cols / V + 255) / 256 : (cols + 255) / 256;
  long long chunks = kColsumBlocks / gx;
  if (chunks < 1) chunks = 1;
  if (chunks > rows) chunks = rows;
  if (chunks > (long long)(partial_floats / cols)) chunks = (long long)(partial_floats / cols);
  dim3 g1(gx, (unsigned)chunks);
  if (vec) {
    if (t == DT_F32)
      colsum_pass1_vec<float><<<g1, 256, 0, s>>>((const float*)src, rows, cols, ld, partials);
    else
      colsum_pass1_vec<bf16><<<g1, 256, 0, s>>>((const bf16*)src, rows, cols, ld, partials);
  } else {
    if (t == DT_F32)
      colsum_pass1<float><<<g1, 256, 0, s>>>((const float*)src, rows, cols, ld, partials);
    else
      colsum_pass1<bf16><<<g1, 256, 0, s>>>((const bf16*)src, rows, cols, ld, partials);
  }
  colsum_pass2_wide<<<(cols + 31) / 32, 256, 0, s>>>(partials, (int)chunks, cols, out);
  return cudaGetLastError();
}

cudaError_t colsum_partials(const float* partials, int chunks, int cols, float* out,
                            cudaStream_t s) {
  if (cols <= 0) return cudaSuccess;
  if (chunks <= 0) return cudaErrorInvalidValue;
  colsum_pass2_wide<<<(cols + 31) / 32, 256, 0, s>>>(partials, chunks, cols, out);
  return cudaGetLastError();
}

cudaError_t rmsnorm_fwd(DType t, const void* x, const float* gamma, void* y, float* rstd, int rows,
                        int d, float eps, cudaStream_t s) {
  if (d > NORM_THREADS * NORM_MAX_PER_THREAD) return cudaErrorInvalidValue;
  int grid = rows < 152 * 16 ? rows : 152 * 16;
  if (t == DT_BF16 && d % 8 == 0 && d <= NORM_THREADS * 8 * NV_MAX &&
      (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
    const int nv = (d / 8 + NORM_THREADS - 1) / NORM_THREADS;
    if (nv == 1)
      rmsnorm_fwd_vec<1><<<grid, NORM_THREADS, 0, s>>>((const bf16*)x, gamma, (bf16*)y, rstd, rows, d, eps);
    else if (nv == 2)
      rmsnorm_fwd_vec<2><<<grid, NORM_THREADS, 0, s>>>((const bf16*)x, gamma, (bf16*)y, rstd, rows, d, eps);
    else
      rmsnorm_fwd_vec<NV_MAX><<<grid, NORM_THREADS, 0, s>>>((const bf16*)x, gamma, (bf16*)y, rstd, rows, d, eps);
    return cudaGetLastError();
  }
  if (t == DT_F32)
    rmsnorm_fwd_kernel<float><<<grid, NORM_THREADS, 0, s>>>((const float*)x, gamma, (float*)y,
                                                            rstd, rows, d, eps);
  else
    rmsnorm_fwd_kernel<bf16><<<grid, NORM_THREADS, 0, s>>>((const bf16*)x, gamma, (bf16*)y, rstd,
                                                           rows, d, eps);
  return cudaGetLastError();
}

cudaError_t rmsnorm_bwd(DType t, const void* dy, const void* x, const float* rstd,
                        const float* gamma, const void* dadd, void* dx, float* dgamma_partials,
                        int row_chunks, float* dgamma, int rows, int d, cudaStream_t s) {
  if (d > NORM_THREADS * NORM_MAX_PER_THREAD) return cudaErrorInvalidValue;
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (t == DT_BF16 && d % 8 == 0 && d <= NORM_THREADS * 8 * NV_MAX && al(dy) && al(x) &&
      al(dadd) && al(dx)) {
    const int nv = (d / 8 + NORM_THREADS - 1) / NORM_THREADS;
    auto kern = nv == 1 ? rmsnorm_bwd_vec<1> : nv == 2 ? rmsnorm_bwd_vec<2> : rmsnorm_bwd_vec<NV_MAX>;
    // one wave: as many blocks as can be resident at once (at most row_chunks)
    int occ = 0, dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NORM_THREADS, 0) == cudaSuccess &&
        occ > 0 && occ * sms < row_chunks)
      row_chunks = occ * sms;
    kern<<<row_chunks, NORM_THREADS, 0, s>>>((const bf16*)dy, (const bf16*)x, rstd, gamma,
                                             (const bf16*)dadd, (bf16*)dx, dgamma_partials, rows, d);
    colsum_pass2_wide<<<(d + 31) / 32, 256, 0, s>>>(dgamma_partials, row_chunks, d, dgamma);
    return cudaGetLastError();
  }
  if (t == DT_F32)
    rmsnorm_bwd_kernel<float><<<row_chunks, NORM_THREADS, 0, s>>>(
        (const float*)dy, (const float*)x, rstd, gamma, (const float*)dadd, (float*)dx,
        dgamma_partials, rows, d);
  else
    rmsnorm_bwd_kernel<bf16><<<row_chunks, NORM_THREADS, 0, s>>>(
        (const bf16*)dy, (const bf16*)x, rstd, gamma, (const bf16*)dadd, (bf16*)dx,
        dgamma_partials, rows, d);
  colsum_pass2_wide<<<(d + 31) / 32, 256, 0, s>>>(dgamma_partials, row_chunks, d, dgamma);
  return cudaGetLastError();
}

}  // namespace mg
