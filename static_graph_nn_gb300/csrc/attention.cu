// Causal self-attention forward and backward (bf16 storage, fp32 math), the
// attention archetype of the Meganeura README ("Why Meganeura" section;
// Environment variables section: a flash forward and a backward made of a
// separate dQ kernel and a fused dK/dV kernel).
//
// Per (batch b, head h): S = Q K^T / sqrt(Dh) with keys j > i masked,
// P = softmax(S), O = P V.  Blockwise with an online softmax: the forward
// saves LSE_i = log sum_j exp(S_ij) so the backward recomputes P without
// storing it.  Backward: D_i = sum_c dO_ic O_ic; dV = P^T dO; dP = dO V^T;
// dS = P (dP - D); dQ = dS K / sqrt(Dh); dK = dS^T Q / sqrt(Dh).
//
// Layout: qkv [nb*S, 3*H*Dh] = [Q | K | V], head h in columns h*Dh.. of each
// third; o and dO [nb*S, H*Dh]; lse and D [nb, H, S] fp32.
//
// CUDA-core version: two threads per row, each owning half of the head
// dimension; partial dot products are combined with one shuffle.
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

constexpr int DH = 64;
constexpr int HALF = DH / 2;
constexpr int ROWS = 64;            // rows (queries or keys) per block
constexpr int THREADS = 2 * ROWS;
constexpr int TILE = 32;            // keys (or queries) staged per step
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float half_dot(const float* a, const float* b) {
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < HALF; ++c) s = fmaf(a[c], b[c], s);
  return s + __shfl_xor_sync(0xffffffffu, s, 1);
}

__global__ void __launch_bounds__(THREADS) attn_fwd_kernel(const bf16* qkv, bf16* o, float* lse,
                                                           int S, int H) {
  __shared__ __align__(16) float kt[TILE][DH];
  __shared__ __align__(16) float vt[TILE][DH];
  const int b = blockIdx.z, h = blockIdx.y;
  const int row_l = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int i = blockIdx.x * ROWS + row_l;                 // query index in the sequence
  const int d = H * DH, ld = 3 * d;
  const float scale2 = LOG2E / sqrtf((float)DH);
  const bf16* base = qkv + (size_t)b * S * ld;

  float q[HALF], acc[HALF];
#pragma unroll
  for (int c = 0; c < HALF; ++c) {
    q[c] = __bfloat162float(base[(size_t)i * ld + h * DH + half * HALF + c]) * scale2;
    acc[c] = 0.0f;
  }
  float m = -INFINITY, l = 0.0f;
  const int kmax = blockIdx.x * ROWS + ROWS;               // keys < kmax can be visible
  for (int j0 = 0; j0 < kmax; j0 += TILE) {
    __syncthreads();
    for (int e = threadIdx.x; e < TILE * DH; e += THREADS) {
      int jj = e / DH, c = e % DH;
      size_t r = (size_t)(j0 + jj) * ld;
      kt[jj][c] = __bfloat162float(base[r + d + h * DH + c]);
      vt[jj][c] = __bfloat162float(base[r + 2 * d + h * DH + c]);
    }
    __syncthreads();
    float s[TILE];
    float tmax = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < TILE; ++jj) {
      float v = half_dot(q, &kt[jj][half * HALF]);
      s[jj] = (j0 + jj <= i) ? v : -INFINITY;
      tmax = fmaxf(tmax, s[jj]);
    }
    float mnew = fmaxf(m, tmax);
    if (mnew == -INFINITY) continue;                       // nothing visible yet
    float corr = exp2f(m - mnew);
    l *= corr;
#pragma unroll
    for (int c = 0; c < HALF; ++c) acc[c] *= corr;
#pragma unroll
    for (int jj = 0; jj < TILE; ++jj) {
      float p = exp2f(s[jj] - mnew);
      l += p;
#pragma unroll
      for (int c = 0; c < HALF; ++c) acc[c] = fmaf(p, vt[jj][half * HALF + c], acc[c]);
    }
    m = mnew;
  }
  const float inv = 1.0f / l;
  bf16* orow = o + ((size_t)b * S + i) * d + h * DH + half * HALF;
#pragma unroll
  for (int c = 0; c < HALF; ++c) orow[c] = __float2bfloat16_rn(acc[c] * inv);
  if (half == 0) lse[((size_t)b * H + h) * S + i] = (m + log2f(l)) / LOG2E;
}

// D_i = sum_c dO_ic O_ic, one thread per (row, head).
// D[b, h, i] = sum_c dO[i, h, c] O[i, h, c]: one warp per row (all heads),
// 16-byte loads; the eight lanes that hold a head's 64 values reduce it with
// shuffles.  Rows are H * 64 elements, so each lane's vectors start 16-byte
// aligned when the tensors do.
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const bf16* o, const bf16* dout,
                                                           float* dsum, int nb, int S, int H) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);   // b*S + i
  const int lane = threadIdx.x & 31;
  if (row >= nb * S) return;
  const int b = row / S, i = row % S;
  const uint4* orow = reinterpret_cast<const uint4*>(o + (size_t)row * H * DH);
  const uint4* drow = reinterpret_cast<const uint4*>(dout + (size_t)row * H * DH);
  const int nvec = H * DH / 8;
  for (int v0 = 0; v0 < nvec; v0 += 32) {
    const int v = v0 + lane;
    float s = 0.0f;
    if (v < nvec) {
      const uint4 a = orow[v], c = drow[v];
      const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* hc = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = __bfloat1622float2(ha[k]), y = __bfloat1622float2(hc[k]);
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
      }
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    if ((lane & 7) == 0 && v < nvec) dsum[((size_t)b * H + (v >> 3)) * S + i] = s;
  }
}

// dQ: one query row per thread pair, loop over visible keys.
__global__ void __launch_bounds__(THREADS) attn_bwd_dq_kernel(const bf16* qkv, const bf16* dout,
                                                              const float* lse, const float* dsum,
                                                              bf16* dqkv, int S, int H) {
  __shared__ __align__(16) float kt[TILE][DH];
  __shared__ __align__(16) float vt[TILE][DH];
  const int b = blockIdx.z, h = blockIdx.y;
  const int row_l = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int i = blockIdx.x * ROWS + row_l;
  const int d = H * DH, ld = 3 * d;
  const float scale = 1.0f / sqrtf((float)DH);
  const bf16* base = qkv + (size_t)b * S * ld;
  float q[HALF], g[HALF], dq[HALF];
#pragma unroll
  for (int c = 0; c < HALF; ++c) {
    q[c] = __bfloat162float(base[(size_t)i * ld + h * DH + half * HALF + c]) * scale;
    g[c] = __bfloat162float(dout[((size_t)b * S + i) * d + h * DH + half * HALF + c]);
    dq[c] = 0.0f;
  }
  const float L = lse[((size_t)b * H + h) * S + i];
  const float Di = dsum[((size_t)b * H + h) * S + i];
  const int kmax = blockIdx.x * ROWS + ROWS;
  for (int j0 = 0; j0 < kmax; j0 += TILE) {
    __syncthreads();
    for (int e = threadIdx.x; e < TILE * DH; e += THREADS) {
      int jj = e / DH, c = e % DH;
      size_t r = (size_t)(j0 + jj) * ld;
      kt[jj][c] = __bfloat162float(base[r + d + h * DH + c]);
      vt[jj][c] = __bfloat162float(base[r + 2 * d + h * DH + c]);
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < TILE; ++jj) {
      float sv = half_dot(q, &kt[jj][half * HALF]);
      float dp = half_dot(g, &vt[jj][half * HALF]);
      float p = (j0 + jj <= i) ? expf(sv - L) : 0.0f;
      float ds = p * (dp - Di);
#pragma unroll
      for (int c = 0; c < HALF; ++c) dq[c] = fmaf(ds, kt[jj][half * HALF + c], dq[c]);
    }
  }
  bf16* out = dqkv + ((size_t)b * S + i) * ld + h * DH + half * HALF;
#pragma unroll
  for (int c = 0; c < HALF; ++c) out[c] = __float2bfloat16_rn(dq[c] * scale);
}

// Fused dK/dV: one key row per thread pair, loop over the queries that see it.
__global__ void __launch_bounds__(THREADS) attn_bwd_dkdv_kernel(const bf16* qkv, const bf16* dout,
                                                                const float* lse, const float* dsum,
                                                                bf16* dqkv, int S, int H) {
  __shared__ __align__(16) float qt[TILE][DH];
  __shared__ __align__(16) float gt[TILE][DH];
  __shared__ float lt[TILE], dt[TILE];
  const int b = blockIdx.z, h = blockIdx.y;
  const int row_l = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int j = blockIdx.x * ROWS + row_l;
  const int d = H * DH, ld = 3 * d;
  const float scale = 1.0f / sqrtf((float)DH);
  const bf16* base = qkv + (size_t)b * S * ld;
  float k[HALF], v[HALF], dk[HALF], dv[HALF];
#pragma unroll
  for (int c = 0; c < HALF; ++c) {
    k[c] = __bfloat162float(base[(size_t)j * ld + d + h * DH + half * HALF + c]) * scale;
    v[c] = __bfloat162float(base[(size_t)j * ld + 2 * d + h * DH + half * HALF + c]);
    dk[c] = 0.0f;
    dv[c] = 0.0f;
  }
  const int i_first = blockIdx.x * ROWS;                   // queries < i_first see no key here
  for (int i0 = i_first; i0 < S; i0 += TILE) {
    __syncthreads();
    for (int e = threadIdx.x; e < TILE * DH; e += THREADS) {
      int ii = e / DH, c = e % DH;
      qt[ii][c] = __bfloat162float(base[(size_t)(i0 + ii) * ld + h * DH + c]);
      gt[ii][c] = __bfloat162float(dout[((size_t)b * S + i0 + ii) * d + h * DH + c]);
    }
    if (threadIdx.x < TILE) {
      lt[threadIdx.x] = lse[((size_t)b * H + h) * S + i0 + threadIdx.x];
      dt[threadIdx.x] = dsum[((size_t)b * H + h) * S + i0 + threadIdx.x];
    }
    __syncthreads();
#pragma unroll 4
    for (int ii = 0; ii < TILE; ++ii) {
      float sv = half_dot(k, &qt[ii][half * HALF]);
      float dp = half_dot(v, &gt[ii][half * HALF]);
      float p = (i0 + ii >= j) ? expf(sv - lt[ii]) : 0.0f;
      float ds = p * (dp - dt[ii]);
#pragma unroll
      for (int c = 0; c < HALF; ++c) {
        dv[c] = fmaf(p, gt[ii][half * HALF + c], dv[c]);
        dk[c] = fmaf(ds, qt[ii][half * HALF + c], dk[c]);
      }
    }
  }
  bf16* outk = dqkv + ((size_t)b * S + j) * ld + d + h * DH + half * HALF;
  bf16* outv = dqkv + ((size_t)b * S + j) * ld + 2 * d + h * DH + half * HALF;
#pragma unroll
  for (int c = 0; c < HALF; ++c) {
    outk[c] = __float2bfloat16_rn(dk[c] * scale);
    outv[c] = __float2bfloat16_rn(dv[c]);
  }
}

}  // namespace

int attn_bwd_launches() { return 3; }

cudaError_t attn_bwd_pre(const void* o, const void* dout, float* dsum, int nb, int S, int H,
                         cudaStream_t s) {
  if ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout)) & 15)
    return cudaErrorInvalidValue;
  const int rows = nb * S;
  attn_bwd_pre_kernel<<<(rows + 7) / 8, 256, 0, s>>>((const bf16*)o, (const bf16*)dout, dsum, nb,
                                                     S, H);
  return cudaGetLastError();
}

cudaError_t attn_fwd(const void* qkv, void* o, float* lse, int nb, int S, int H, int Dh,
                     cudaStream_t s) {
  if (Dh != DH || S % ROWS != 0) return cudaErrorInvalidValue;
  dim3 grid(S / ROWS, H, nb);
  attn_fwd_kernel<<<grid, THREADS, 0, s>>>((const bf16*)qkv, (bf16*)o, lse, S, H);
  return cudaGetLastError();
}

cudaError_t attn_bwd(const void* qkv, const void* o, const void* dout, const float* lse,
                     float* dsum, void* dqkv, int nb, int S, int H, int Dh, cudaStream_t s) {
  if (Dh != DH || S % ROWS != 0) return cudaErrorInvalidValue;
  cudaError_t e = attn_bwd_pre(o, dout, dsum, nb, S, H, s);
  if (e != cudaSuccess) return e;
  dim3 grid(S / ROWS, H, nb);
  attn_bwd_dq_kernel<<<grid, THREADS, 0, s>>>((const bf16*)qkv, (const bf16*)dout, lse, dsum,
                                               (bf16*)dqkv, S, H);
  attn_bwd_dkdv_kernel<<<grid, THREADS, 0, s>>>((const bf16*)qkv, (const bf16*)dout, lse, dsum,
                                                 (bf16*)dqkv, S, H);
  return cudaGetLastError();
}

}  // namespace mg
