// Register-blocked CUDA-core GEMM with a fused epilogue.
//
// This is the strict-f32 matmul of the library: fp32 operands, fp32 FFMA
// accumulation, no tensor cores and no TF32 (the pages' "portable scalar
// matmul" path, README Environment variables section, kept separate from the
// reduced-precision tiles as the abstract's strict f32 protocol requires).  It
// also serves bf16 GEMMs whose widths do not meet the tensor-memory-access
// alignment rule (a row that is not a multiple of 16 bytes, e.g. 10 classes).
//
// Tile 128x128x16, 256 threads, 8x8 outputs per thread split in two 4x4
// quadrants (rows ty*4 and 64+ty*4, cols tx*4 and 64+tx*4) so that shared-memory
// reads are float4 and conflict-free.  Operands are staged through registers
// one K-tile ahead of the compute (double-buffered shared memory).
//
// Compensated variant (strict forward GEMMs): every product and partial sum
// carries its exact rounding error -- TwoProduct by FMA and TwoSum (Ogita,
// Rump and Oishi, "Accurate sum and dot product", SIAM J. Sci. Comput. 2005,
// algorithm Dot2) -- so the result is as accurate as if computed in twice the
// working precision and then rounded to fp32.  The graph's stored values are
// then the correctly rounded ones, and a ReLU decides on the sign of the exact
// pre-activation except within ~1e-13 of the kink.  Still fp32 FFMA/FADD only.
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, PAD = 4, NT = 256;

template <typename T>
__device__ __forceinline__ float ldg_or0(const T* p, long long i, bool ok) {
  return ok ? ld_elem(p, (size_t)i) : 0.0f;
}

template <typename T, bool A_MN, bool B_K>
__device__ __forceinline__ void load_tiles(const GemmArgs& g, int m0, int n0, int k0, int tid,
                                           float ra[8], float rb[8]) {
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  if (A_MN) {  // A[k*lda + m]: 16 k-rows x 128 m, 8 consecutive m per thread
    int k = tid >> 4, mm = (tid & 15) * 8;
    int gk = k0 + k;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gm = m0 + mm + i;
      ra[i] = ldg_or0(A, (long long)gk * g.lda + gm, gk < g.K && gm < g.M);
    }
  } else {  // A[m*lda + k]: 128 m-rows x 16 k, 8 consecutive k per thread
    int m = tid >> 1, kk = (tid & 1) * 8;
    int gm = m0 + m;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gk = k0 + kk + i;
      ra[i] = ldg_or0(A, (long long)gm * g.lda + gk, gk < g.K && gm < g.M);
    }
  }
  if (!B_K) {  // B[k*ldb + n]
    int k = tid >> 4, nn = (tid & 15) * 8;
    int gk = k0 + k;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gn = n0 + nn + i;
      rb[i] = ldg_or0(B, (long long)gk * g.ldb + gn, gk < g.K && gn < g.N);
    }
  } else {  // B[n*ldb + k]
    int n = tid >> 1, kk = (tid & 1) * 8;
    int gn = n0 + n;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gk = k0 + kk + i;
      rb[i] = ldg_or0(B, (long long)gn * g.ldb + gk, gk < g.K && gn < g.N);
    }
  }
}

template <bool A_MN, bool B_K>
__device__ __forceinline__ void store_tiles(float (*As)[BM + PAD], float (*Bs)[BN + PAD], int tid,
                                            const float ra[8], const float rb[8]) {
  if (A_MN) {
    int k = tid >> 4, mm = (tid & 15) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) As[k][mm + i] = ra[i];
  } else {
    int m = tid >> 1, kk = (tid & 1) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) As[kk + i][m] = ra[i];
  }
  if (!B_K) {
    int k = tid >> 4, nn = (tid & 15) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) Bs[k][nn + i] = rb[i];
  } else {
    int n = tid >> 1, kk = (tid & 1) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) Bs[kk + i][n] = rb[i];
  }
}

// Epilogue, rounding at the boundaries of graph values (a no-op for fp32):
// forward  Z = round(acc + b); H = act(Z) or skip + Z; stored rounded;
// backward dH = round(acc) when an activation derivative follows, then
//          dZ = dH * act'(saved) (+ the skip's gradient), stored rounded.
template <typename TO>
__device__ __forceinline__ float round_value(float v) {
  return sizeof(TO) == 2 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

template <typename TO, typename TX>
__device__ __forceinline__ void epilogue_elem(const GemmArgs& g, const float* bias, int m, int n,
                                              float v) {
  if (bias) v += bias[n];
  if (g.act || g.resid || g.out_z) v = round_value<TO>(v);
  if (g.out_z) st_elem(static_cast<TX*>(g.out_z), (size_t)m * g.ldz + n, v);
  if (g.act) v = apply_act(g.act, v);
  if (g.dact) {
    v = round_value<TO>(v);
    v *= act_grad_from_saved(g.dact, ld_elem(static_cast<const TX*>(g.saved), (size_t)m * g.lds + n));
  }
  if (g.resid) v += ld_elem(static_cast<const TX*>(g.resid), (size_t)m * g.ldr + n);
  st_elem(static_cast<TO*>(g.out), (size_t)m * g.ldo + n, v);
}

// s + c += a*b with the rounding errors of the product and the sum kept in c.
__device__ __forceinline__ void dot2_step(float a, float b, float& s, float& c) {
  float p = __fmul_rn(a, b);
  float pe = __fmaf_rn(a, b, -p);            // a*b - p exactly
  float t = __fadd_rn(s, p);
  float z = __fsub_rn(t, s);
  float se = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(p, z));   // s + p - t exactly
  s = t;
  c = __fadd_rn(c, __fadd_rn(pe, se));
}

template <typename T, typename TO, typename TX, bool A_MN, bool B_K, bool COMP>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const GemmArgs g) {
  __shared__ __align__(16) float As[2][BK][BM + PAD];
  __shared__ __align__(16) float Bs[2][BK][BN + PAD];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

  float acc[8][8];
  float cmp[COMP ? 8 : 1][COMP ? 8 : 1];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  if (COMP) {
#pragma unroll
    for (int i = 0; i < (COMP ? 8 : 1); ++i)
#pragma unroll
      for (int j = 0; j < (COMP ? 8 : 1); ++j) cmp[i][j] = 0.0f;
    // the bias is the first term of the compensated sum: Z = round(b + x.w)
    if (g.bias) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
        float b = n < g.N ? g.bias[n] : 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i][j] = b;
      }
    }
  }
  const float* epi_bias = COMP ? nullptr : g.bias;

  float ra[8], rb[8];
  load_tiles<T, A_MN, B_K>(g, m0, n0, 0, tid, ra, rb);
  store_tiles<A_MN, B_K>(As[0], Bs[0], tid, ra, rb);
  __syncthreads();

  const int nk = (g.K + BK - 1) / BK;
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    const bool more = kt + 1 < nk;
    if (more) load_tiles<T, A_MN, B_K>(g, m0, n0, (kt + 1) * BK, tid, ra, rb);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[8];
      float4 a0 = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4]);
      float4 a1 = *reinterpret_cast<const float4*>(&As[cur][kk][64 + ty * 4]);
      float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4]);
      float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][kk][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
      if (COMP) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) dot2_step(a[i], b[j], acc[i][j], cmp[COMP ? i : 0][COMP ? j : 0]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
    }
    if (more) store_tiles<A_MN, B_K>(As[cur ^ 1], Bs[cur ^ 1], tid, ra, rb);
    __syncthreads();
  }

  if (COMP) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = __fadd_rn(acc[i][j], cmp[COMP ? i : 0][COMP ? j : 0]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (n < g.N) epilogue_elem<TO, TX>(g, epi_bias, m, n, acc[i][j]);
    }
  }
}

// Small or skinny GEMMs (few output tiles, e.g. 10 classes): one warp per
// output element, lanes split K; the compensated variant combines the lanes'
// (sum, error) pairs with TwoSum so the result stays correctly rounded.
template <typename T, typename TO, typename TX, bool COMP>
__global__ void __launch_bounds__(256) gemm_warp_kernel(const GemmArgs g) {
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)g.M * g.N) return;          // whole warps only
  const int m = (int)(wid / g.N), n = (int)(wid % g.N);
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  float s = 0.0f, c = 0.0f;
  if (COMP && lane == 0 && g.bias) s = g.bias[n];
  for (int k = lane; k < g.K; k += 32) {
    float a = ld_elem(A, g.a_mn ? (size_t)k * g.lda + m : (size_t)m * g.lda + k);
    float b = ld_elem(B, g.b_k ? (size_t)n * g.ldb + k : (size_t)k * g.ldb + n);
    if (COMP)
      dot2_step(a, b, s, c);
    else
      s = fmaf(a, b, s);
  }
  float v;
  if (COMP) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float so = __shfl_xor_sync(0xffffffffu, s, off);
      float co = __shfl_xor_sync(0xffffffffu, c, off);
      float t = __fadd_rn(s, so);
      float z = __fsub_rn(t, s);
      float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(so, z));
      s = t;
      c = __fadd_rn(__fadd_rn(c, co), e);
    }
    v = __fadd_rn(s, c);
  } else {
    v = warp_sum(s);
  }
  if (lane == 0) epilogue_elem<TO, TX>(g, COMP ? nullptr : g.bias, m, n, v);
}

template <typename T, typename TO, typename TX, bool COMP>
cudaError_t launch_warp(const GemmArgs& g, cudaStream_t s) {
  long long threads = (long long)g.M * g.N * 32;
  gemm_warp_kernel<T, TO, TX, COMP><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(g);
  return cudaGetLastError();
}

// Weight gradients with few output columns (dW = X^T dZ, A M-major, B
// N-major, N <= 32): lanes take 32 consecutive rows m (coalesced A reads), the
// 8 warps of a block split K, and the block adds its warps' partial sums.
template <typename T, typename TO, typename TX>
__global__ void __launch_bounds__(256) gemm_dw_narrow_kernel(const GemmArgs g) {
  __shared__ float red[8][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int m = blockIdx.x * 32 + lane, n = blockIdx.y;
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  const int per = (g.K + 7) / 8;
  const int k0 = w * per, k1 = min(g.K, k0 + per);
  float acc = 0.0f;
  if (m < g.M) {
#pragma unroll 8
    for (int k = k0; k < k1; ++k)
      acc = fmaf(ld_elem(A, (size_t)k * g.lda + m), ld_elem(B, (size_t)k * g.ldb + n), acc);
  }
  red[w][lane] = acc;
  __syncthreads();
  if (w == 0 && m < g.M) {
    float v = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) v += red[i][lane];
    epilogue_elem<TO, TX>(g, g.bias, m, n, v);
  }
}

template <typename T, typename TO, typename TX>
cudaError_t launch_dw_narrow(const GemmArgs& g, cudaStream_t s) {
  gemm_dw_narrow_kernel<T, TO, TX><<<dim3((g.M + 31) / 32, g.N), 256, 0, s>>>(g);
  return cudaGetLastError();
}

template <typename T, typename TO, typename TX, bool A_MN, bool B_K, bool COMP = false>
cudaError_t launch1(const GemmArgs& g, cudaStream_t s) {
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM);
  gemm_simt_kernel<T, TO, TX, A_MN, B_K, COMP><<<grid, NT, 0, s>>>(g);
  return cudaGetLastError();
}

}  // namespace

// Layouts used by the schedule: forward (A K-major, B N-major), dX (A K-major,
// B K-major), dW (A M-major, B N-major, fp32 output).
cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (g.a_mn && !g.b_k && g.N <= 32 && g.out_type == DT_F32 && !g.act && !g.dact && !g.resid &&
      !g.out_z) {   // narrow weight gradient
    if (g.in_type == DT_F32) return launch_dw_narrow<float, float, float>(g, s);
    return launch_dw_narrow<bf16, float, bf16>(g, s);
  }
  if ((long long)g.M * g.N <= 65536 && g.K >= 64) {   // too few tiles: warp per output
    if (g.in_type == DT_F32) {
      if (!g.a_mn && !g.b_k) return launch_warp<float, float, float, true>(g, s);
      return launch_warp<float, float, float, false>(g, s);
    }
    if (g.out_type == DT_F32) return launch_warp<bf16, float, bf16, false>(g, s);
    return launch_warp<bf16, bf16, bf16, false>(g, s);
  }
  if (g.in_type == DT_F32) {   // strict path: everything fp32
    if (!g.a_mn && !g.b_k) return launch1<float, float, float, false, false, true>(g, s);
    if (!g.a_mn && g.b_k) return launch1<float, float, float, false, true>(g, s);
    if (g.a_mn && !g.b_k) return launch1<float, float, float, true, false>(g, s);
    return cudaErrorNotSupported;
  }
  if (g.out_type == DT_F32) {
    if (g.a_mn && !g.b_k) return launch1<bf16, float, bf16, true, false>(g, s);
    return cudaErrorNotSupported;
  }
  if (!g.a_mn && !g.b_k) return launch1<bf16, bf16, bf16, false, false>(g, s);
  if (!g.a_mn && g.b_k) return launch1<bf16, bf16, bf16, false, true>(g, s);
  return cudaErrorNotSupported;
}

}  // namespace mg
