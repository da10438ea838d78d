// Register-blocked CUDA-core GEMM with a fused epilogue.
//
// This is the strict-f32 matmul of the library: fp32 operands, fp32 FFMA
// accumulation, no tensor cores and no TF32 (the scalar f32 matmul the
// README's Environment variables section describes, kept separate from the
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
// It has a kernel of its own (gemm_dot2_kernel, 64x64 tiles, 4x4 outputs per
// thread): its per-output state is twice the plain kernel's.
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, PAD = 4, NT = 256;

template <typename T>
__device__ __forceinline__ float ldg_or0(const T* p, long long i, bool ok) {
  return ok ? ld_elem(p, (size_t)i) : 0.0f;
}

// Eight consecutive fp32 elements as two 16-byte loads when they are in
// bounds and 16-byte aligned (false: load them element by element).
__device__ __forceinline__ bool load8_vec(const float* p, long long i, bool all_in, float r[8]) {
  const float* q = p + i;
  if (!all_in || (reinterpret_cast<uintptr_t>(q) & 15) != 0) return false;
  const float4 u = reinterpret_cast<const float4*>(q)[0];
  const float4 v = reinterpret_cast<const float4*>(q)[1];
  r[0] = u.x; r[1] = u.y; r[2] = u.z; r[3] = u.w;
  r[4] = v.x; r[5] = v.y; r[6] = v.z; r[7] = v.w;
  return true;
}
__device__ __forceinline__ bool load8_vec(const bf16*, long long, bool, float*) { return false; }

// The eight consecutive elements of A (or B) a thread stages per K tile.
template <typename T, bool A_MN>
__device__ __forceinline__ void load_a(const GemmArgs& g, int m0, int k0, int tid, float ra[8]) {
  const T* A = static_cast<const T*>(g.A);
  if (A_MN) {  // A[k*lda + m]: 16 k-rows x 128 m, 8 consecutive m per thread
    int k = tid >> 4, mm = (tid & 15) * 8;
    int gk = k0 + k;
    if (load8_vec(A, (long long)gk * g.lda + m0 + mm, gk < g.K && m0 + mm + 8 <= g.M, ra)) return;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gm = m0 + mm + i;
      ra[i] = ldg_or0(A, (long long)gk * g.lda + gm, gk < g.K && gm < g.M);
    }
  } else {  // A[m*lda + k]: 128 m-rows x 16 k, 8 consecutive k per thread
    int m = tid >> 1, kk = (tid & 1) * 8;
    int gm = m0 + m;
    if (load8_vec(A, (long long)gm * g.lda + k0 + kk, gm < g.M && k0 + kk + 8 <= g.K, ra)) return;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gk = k0 + kk + i;
      ra[i] = ldg_or0(A, (long long)gm * g.lda + gk, gk < g.K && gm < g.M);
    }
  }
}

template <typename T, bool B_K>
__device__ __forceinline__ void load_b(const GemmArgs& g, int n0, int k0, int tid, float rb[8]) {
  const T* B = static_cast<const T*>(g.B);
  if (!B_K) {  // B[k*ldb + n]
    int k = tid >> 4, nn = (tid & 15) * 8;
    int gk = k0 + k;
    if (load8_vec(B, (long long)gk * g.ldb + n0 + nn, gk < g.K && n0 + nn + 8 <= g.N, rb)) return;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gn = n0 + nn + i;
      rb[i] = ldg_or0(B, (long long)gk * g.ldb + gn, gk < g.K && gn < g.N);
    }
  } else {  // B[n*ldb + k]
    int n = tid >> 1, kk = (tid & 1) * 8;
    int gn = n0 + n;
    if (load8_vec(B, (long long)gn * g.ldb + k0 + kk, gn < g.N && k0 + kk + 8 <= g.K, rb)) return;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gk = k0 + kk + i;
      rb[i] = ldg_or0(B, (long long)gn * g.ldb + gk, gk < g.K && gn < g.N);
    }
  }
}

template <typename T, bool A_MN, bool B_K>
__device__ __forceinline__ void load_tiles(const GemmArgs& g, int m0, int n0, int k0, int tid,
                                           float ra[8], float rb[8]) {
  load_a<T, A_MN>(g, m0, k0, tid, ra);
  load_b<T, B_K>(g, n0, k0, tid, rb);
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

// Two CTAs per SM (128 registers, four warps per SM sub-partition to hide
// the FFMA latency chains).  A strict weight gradient split over K
// (blockIdx.z = split, k_per > 0) writes its partial tile to its slice of
// split_ws.
template <typename T, typename TO, typename TX, bool A_MN, bool B_K>
__global__ void __launch_bounds__(NT, 2) gemm_simt_kernel(const GemmArgs gin, int k_per) {
  GemmArgs g = gin;
  int k_lo = 0;
  if (k_per > 0) {
    k_lo = blockIdx.z * k_per;
    g.K = min(gin.K, k_lo + k_per);
    g.out = gin.split_ws + (size_t)blockIdx.z * gin.M * gin.N;
    g.ldo = gin.N;
  }
  __shared__ __align__(16) float As[2][BK][BM + PAD];
  __shared__ __align__(16) float Bs[2][BK][BN + PAD];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  float ra[8], rb[8];
  load_tiles<T, A_MN, B_K>(g, m0, n0, k_lo, tid, ra, rb);
  store_tiles<A_MN, B_K>(As[0], Bs[0], tid, ra, rb);
  __syncthreads();

  const int nk = (g.K - k_lo + BK - 1) / BK;
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    const bool more = kt + 1 < nk;
    if (more) load_tiles<T, A_MN, B_K>(g, m0, n0, k_lo + (kt + 1) * BK, tid, ra, rb);
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
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) store_tiles<A_MN, B_K>(As[cur ^ 1], Bs[cur ^ 1], tid, ra, rb);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (n < g.N) epilogue_elem<TO, TX>(g, g.bias, m, n, acc[i][j]);
    }
  }
}

// Compensated forward (fp32, A = X [M, K] K-major, B = W [K, N] N-major):
// 64x64 tiles, 256 threads with 4x4 outputs each, three CTAs per SM.  Every
// output's sum runs in the same order as in the plain kernel (the bias first,
// then k ascending), so the tiling does not change a bit of the result; the
// small per-thread tile keeps the 16 sums and 16 error terms in registers with
// room for the Dot2 temporaries of several outputs in flight (measured on
// GB300: 2.8x the rate of an 8x8-per-thread tiling at 255 registers).
constexpr int DBM = 64, DBN = 64, DPAD = 4;

__global__ void __launch_bounds__(NT, 3) gemm_dot2_kernel(const GemmArgs g) {
  __shared__ __align__(16) float As[2][BK][DBM + DPAD];
  __shared__ __align__(16) float Bs[2][BK][DBN];
  const float* A = static_cast<const float*>(g.A);
  const float* B = static_cast<const float*>(g.B);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * DBM, n0 = blockIdx.x * DBN;
  // staging: A row tid / 4, k (tid % 4) * 4 .. +3; B k row tid / 16, n (tid % 16) * 4 .. +3
  const int am = tid >> 2, ak = (tid & 3) * 4, bk = tid >> 4, bn = (tid & 15) * 4;
  const bool a_vec = (g.lda & 3) == 0 && (reinterpret_cast<uintptr_t>(A) & 15) == 0;
  const bool b_vec = (g.ldb & 3) == 0 && (reinterpret_cast<uintptr_t>(B) & 15) == 0;
  float ra[4], rb[4];
  auto load = [&](int k0) {
    const int gm = m0 + am, gk = k0 + ak;
    if (a_vec && gm < g.M && gk + 4 <= g.K) {
      const float4 u = *reinterpret_cast<const float4*>(A + (size_t)gm * g.lda + gk);
      ra[0] = u.x; ra[1] = u.y; ra[2] = u.z; ra[3] = u.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ra[i] = (gm < g.M && gk + i < g.K) ? A[(size_t)gm * g.lda + gk + i] : 0.0f;
    }
    const int gkb = k0 + bk, gn = n0 + bn;
    if (b_vec && gkb < g.K && gn + 4 <= g.N) {
      const float4 u = *reinterpret_cast<const float4*>(B + (size_t)gkb * g.ldb + gn);
      rb[0] = u.x; rb[1] = u.y; rb[2] = u.z; rb[3] = u.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        rb[i] = (gkb < g.K && gn + i < g.N) ? B[(size_t)gkb * g.ldb + gn + i] : 0.0f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 4; ++i) As[buf][ak + i][am] = ra[i];
    *reinterpret_cast<float4*>(&Bs[buf][bk][bn]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
  };

  float acc[4][4], cmp[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // the bias is the first term of the compensated sum: Z = round(b + x.w)
    const int n = n0 + tx * 4 + j;
    const float b = (g.bias && n < g.N) ? g.bias[n] : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i][j] = b;
      cmp[i][j] = 0.0f;
    }
  }
  load(0);
  store(0);
  __syncthreads();
  const int nk = (g.K + BK - 1) / BK;
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    const bool more = kt + 1 < nk;
    if (more) load((kt + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4]);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w}, b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) dot2_step(a[i], b[j], acc[i][j], cmp[i][j]);
    }
    if (more) store(cur ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < g.N) epilogue_elem<float, float>(g, nullptr, m, n, __fadd_rn(acc[i][j], cmp[i][j]));
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

// ---- bf16 GEMMs with one narrow side (a head of a few classes) ------------
// The narrow operand is held in shared memory as fp32; the wide one streams
// through once.  Same epilogue arithmetic as above.

int sm_count_simt() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

__device__ __forceinline__ void unpack8(const bf16* p, float (&f)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void pack8(bf16* p, const float (&f)[8]) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = u;
}

// epilogue_elem on eight consecutive outputs of row m (bf16 output and
// auxiliaries) with 16-byte loads and stores.
__device__ __forceinline__ void epilogue8_bf16(const GemmArgs& g, int m, int n0, float (&v)[8]) {
  float sv[8], rs[8], z[8];
  if (g.dact) unpack8(static_cast<const bf16*>(g.saved) + (size_t)m * g.lds + n0, sv);
  if (g.resid) unpack8(static_cast<const bf16*>(g.resid) + (size_t)m * g.ldr + n0, rs);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float x = v[j];
    if (g.bias) x += g.bias[n0 + j];
    if (g.act || g.resid || g.out_z) x = round_value<bf16>(x);
    z[j] = x;
    if (g.act) x = apply_act(g.act, x);
    if (g.dact) {
      x = round_value<bf16>(x);
      x *= act_grad_from_saved(g.dact, sv[j]);
    }
    if (g.resid) x += rs[j];
    v[j] = x;
  }
  if (g.out_z) pack8(static_cast<bf16*>(g.out_z) + (size_t)m * g.ldz + n0, z);
  pack8(static_cast<bf16*>(g.out) + (size_t)m * g.ldo + n0, v);
}

// Copies the bf16 matrix src (rows x cols, row stride ld) into shared memory
// through put(r, c, value) with many loads in flight: 16-byte loads of the
// flat array when the rows are contiguous and aligned, else eight scalar
// loads per thread per round.
template <typename F>
__device__ __forceinline__ void stage_bf16(const bf16* src, int rows, int cols, long long ld,
                                           F put) {
  const int total = rows * cols;
  if (ld == cols && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
    const int nv = total / 8;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int base = threadIdx.x; base < nv; base += 4 * blockDim.x) {
      uint4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = base + u * blockDim.x;
        t[u] = q < nv ? s4[q] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = base + u * blockDim.x;
        if (q >= nv) continue;
        const uint32_t w[4] = {t[u].x, t[u].y, t[u].z, t[u].w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[p]));
          const int e = 8 * q + 2 * p;
          const int r0 = e / cols, r1 = (e + 1) / cols;
          put(r0, e - r0 * cols, f.x);
          put(r1, e + 1 - r1 * cols, f.y);
        }
      }
    }
    for (int e = 8 * nv + threadIdx.x; e < total; e += blockDim.x) {
      const int r = e / cols;
      put(r, e - r * cols, __bfloat162float(src[e]));
    }
    return;
  }
  for (int base = threadIdx.x; base < total; base += 8 * blockDim.x) {
    float t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * blockDim.x;
      const int r = i / cols, c = i - r * cols;
      t[u] = i < total ? __bfloat162float(src[(size_t)r * ld + c]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * blockDim.x;
      if (i < total) {
        const int r = i / cols;
        put(r, i - r * cols, t[u]);
      }
    }
  }
}

// Forward, N <= NP: out[m][n] = sum_k A[m][k] B[k][n] (A K-major, B N-major).
// B is held transposed in shared memory ([NP][ks], zero padded to k2, a
// multiple of 256).  A warp owns R rows at a time; lane l takes the eight
// consecutive k at 8l + 256i of each row (one 16-byte load); the partial sums
// are reduced across the warp and lane n applies the epilogue to column n.
template <int NP, int R, typename TO>
__global__ void __launch_bounds__(256) skinny_fwd_kernel(const GemmArgs g, int k2, int vec8) {
  extern __shared__ __align__(16) float sbt[];
  const int ks = k2 + 4;   // row stride: 16-byte aligned, rows four banks apart
  for (int i = threadIdx.x; i < NP * ks; i += blockDim.x) sbt[i] = 0.0f;
  __syncthreads();
  stage_bf16(static_cast<const bf16*>(g.B), g.K, g.N, g.ldb,
             [&](int k, int n, float v) { sbt[n * ks + k] = v; });
  __syncthreads();
  const bf16* A = static_cast<const bf16*>(g.A);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int m0 = (blockIdx.x * warps + warp) * R; m0 < g.M; m0 += gridDim.x * warps * R) {
    float acc[R][NP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int n = 0; n < NP; ++n) acc[r][n] = 0.0f;
    for (int k = 8 * lane; k < k2; k += 256) {
      float a[R][8];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int m = m0 + r;
        const bf16* ap = A + (size_t)m * g.lda + k;
        if (vec8 && m < g.M && k + 8 <= g.K) {
          unpack8(ap, a[r]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) a[r][j] = (m < g.M && k + j < g.K) ? __bfloat162float(ap[j]) : 0.0f;
        }
      }
#pragma unroll
      for (int n = 0; n < NP; ++n) {
        const float4 b0 = *reinterpret_cast<const float4*>(&sbt[n * ks + k]);
        const float4 b1 = *reinterpret_cast<const float4*>(&sbt[n * ks + k + 4]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float t = acc[r][n];
          t = fmaf(a[r][0], b0.x, t); t = fmaf(a[r][1], b0.y, t);
          t = fmaf(a[r][2], b0.z, t); t = fmaf(a[r][3], b0.w, t);
          t = fmaf(a[r][4], b1.x, t); t = fmaf(a[r][5], b1.y, t);
          t = fmaf(a[r][6], b1.z, t); t = fmaf(a[r][7], b1.w, t);
          acc[r][n] = t;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int n = 0; n < NP; ++n) {
        const float v = warp_sum(acc[r][n]);
        if (lane == n && n < g.N && m0 + r < g.M) epilogue_elem<TO, bf16>(g, g.bias, m0 + r, n, v);
      }
  }
}

// Input gradient, K <= 32: out[m][n] = sum_k A[m][k] B[n][k] (A K-major, B
// K-major).  B is held in shared memory as [K][n8] (n8 = N rounded up to 8);
// a thread computes eight consecutive outputs of a row.
template <typename TO>
__global__ void __launch_bounds__(256) skinny_dx_kernel(const GemmArgs g, int n8, int vec) {
  extern __shared__ __align__(16) float sw[];
  for (int i = threadIdx.x; i < n8 * g.K; i += blockDim.x) sw[i] = 0.0f;
  __syncthreads();
  stage_bf16(static_cast<const bf16*>(g.B), g.N, g.K, g.ldb,
             [&](int n, int k, float v) { sw[k * n8 + n] = v; });
  __syncthreads();
  const bf16* A = static_cast<const bf16*>(g.A);
  const int nc = n8 / 8;
  const long long total = (long long)g.M * nc;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(idx / nc), n0 = 8 * (int)(idx - (long long)m * nc);
    const bf16* ap = A + (size_t)m * g.lda;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k = 0; k < g.K; ++k) {
      const float a = __bfloat162float(ap[k]);
      const float4 w0 = *reinterpret_cast<const float4*>(&sw[k * n8 + n0]);
      const float4 w1 = *reinterpret_cast<const float4*>(&sw[k * n8 + n0 + 4]);
      acc[0] = fmaf(a, w0.x, acc[0]); acc[1] = fmaf(a, w0.y, acc[1]);
      acc[2] = fmaf(a, w0.z, acc[2]); acc[3] = fmaf(a, w0.w, acc[3]);
      acc[4] = fmaf(a, w1.x, acc[4]); acc[5] = fmaf(a, w1.y, acc[5]);
      acc[6] = fmaf(a, w1.z, acc[6]); acc[7] = fmaf(a, w1.w, acc[7]);
    }
    if (vec && n0 + 8 <= g.N) {
      epilogue8_bf16(g, m, n0, acc);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (n0 + j < g.N) epilogue_elem<TO, bf16>(g, g.bias, m, n0 + j, acc[j]);
    }
  }
}

// Weight gradient, N <= NP, plain fp32 output: out[m][n] = sum_k A[k][m]
// B[k][n] (A M-major, B N-major).  A block owns 32*MV rows of the output (MV
// consecutive per lane) and kper rows of K, whose rows of B it holds in shared
// memory; its eight warps take interleaved k, U rows' loads in flight at a
// time, then add their partial sums in warp order (deterministic).  With
// several K ranges (gridDim.y > 1) the blocks add into a zeroed output with
// atomics.
template <int NP, int MV>
__global__ void __launch_bounds__(256) skinny_dw_kernel(const GemmArgs g, int kper, int vec) {
  constexpr int U = 8;
  extern __shared__ __align__(16) float sb[];   // [kper][NP]
  __shared__ float red[NP][MV][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mb = blockIdx.x * 32 * MV, m0 = mb + lane * MV;
  const int k0 = blockIdx.y * kper, kn = min(g.K, k0 + kper) - k0;
  const bf16* A = static_cast<const bf16*>(g.A);
  for (int i = threadIdx.x; i < kn * NP; i += blockDim.x) sb[i] = 0.0f;
  __syncthreads();
  stage_bf16(static_cast<const bf16*>(g.B) + (size_t)k0 * g.ldb, kn, g.N, g.ldb,
             [&](int r, int n, float v) { sb[r * NP + n] = v; });
  __syncthreads();
  float acc[MV][NP];
#pragma unroll
  for (int j = 0; j < MV; ++j)
#pragma unroll
    for (int n = 0; n < NP; ++n) acc[j][n] = 0.0f;
  for (int kk = warp; kk < kn; kk += 8 * U) {
    float a[U][MV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = kk + 8 * u;
      const bf16* ap = A + (size_t)(k0 + r) * g.lda + m0;
      if (r < kn && vec && m0 + MV <= g.M) {
        if constexpr (MV == 4) {
          const uint2 q = *reinterpret_cast<const uint2*>(ap);
          const float2 t0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
          const float2 t1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
          a[u][0] = t0.x; a[u][1] = t0.y; a[u][2] = t1.x; a[u][3] = t1.y;
        } else {
          static_assert(MV == 2, "two or four rows per lane");
          const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(ap));
          a[u][0] = t.x; a[u][1] = t.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < MV; ++j)
          a[u][j] = (r < kn && m0 + j < g.M) ? __bfloat162float(ap[j]) : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = kk + 8 * u;
      if (r >= kn) break;
#pragma unroll
      for (int n = 0; n < NP; n += 4) {
        const float4 b = *reinterpret_cast<const float4*>(&sb[r * NP + n]);
#pragma unroll
        for (int j = 0; j < MV; ++j) {
          acc[j][n] = fmaf(a[u][j], b.x, acc[j][n]);
          acc[j][n + 1] = fmaf(a[u][j], b.y, acc[j][n + 1]);
          acc[j][n + 2] = fmaf(a[u][j], b.z, acc[j][n + 2]);
          acc[j][n + 3] = fmaf(a[u][j], b.w, acc[j][n + 3]);
        }
      }
    }
  }
  for (int w = 0; w < 8; ++w) {
    if (warp == w) {
#pragma unroll
      for (int j = 0; j < MV; ++j)
#pragma unroll
        for (int n = 0; n < NP; ++n) red[n][j][lane] = (w ? red[n][j][lane] : 0.0f) + acc[j][n];
    }
    __syncthreads();
  }
  float* out = static_cast<float*>(g.out);
  for (int i = threadIdx.x; i < NP * MV * 32; i += blockDim.x) {
    const int n = i / (MV * 32), j = (i / 32) % MV, l = i % 32;
    const int m = mb + l * MV + j;
    if (m < g.M && n < g.N) {
      float* o = out + (size_t)m * g.ldo + n;
      if (gridDim.y > 1)
        atomicAdd(o, red[n][j][l]);
      else
        *o = red[n][j][l];
    }
  }
}

constexpr size_t kSkinnySmem = 96 * 1024;

size_t skinny_fwd_smem(const GemmArgs& g) {
  const int np = g.N <= 16 ? 16 : 32;
  return (size_t)np * (((g.K + 255) & ~255) + 4) * 4;
}

size_t skinny_dx_smem(const GemmArgs& g) { return (size_t)((g.N + 7) & ~7) * g.K * 4; }

template <typename K>
cudaError_t allow_smem(K kern, bool& done) {
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSkinnySmem);
  if (e == cudaSuccess) done = true;
  return e;
}

template <int NP, int R, typename TO>
cudaError_t launch_skinny_fwd(const GemmArgs& g, cudaStream_t s) {
  static bool attr = false;
  cudaError_t e = allow_smem(skinny_fwd_kernel<NP, R, TO>, attr);
  if (e != cudaSuccess) return e;
  const int k2 = (g.K + 255) & ~255;
  const int vec8 = (reinterpret_cast<uintptr_t>(g.A) & 15u) == 0 && (g.lda & 7) == 0;
  const int need = (g.M + 8 * R - 1) / (8 * R);
  const int grid = need < 2 * sm_count_simt() ? need : 2 * sm_count_simt();
  skinny_fwd_kernel<NP, R, TO><<<grid, 256, skinny_fwd_smem(g), s>>>(g, k2, vec8);
  return cudaGetLastError();
}

template <typename TO>
cudaError_t launch_skinny_dx(const GemmArgs& g, cudaStream_t s) {
  static bool attr = false;
  cudaError_t e = allow_smem(skinny_dx_kernel<TO>, attr);
  if (e != cudaSuccess) return e;
  const int n8 = (g.N + 7) & ~7;
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const int vec = sizeof(TO) == 2 && g.aux_type == DT_BF16 && al(g.out) && al(g.out_z) &&
                  al(g.saved) && al(g.resid) && ((g.ldo | g.ldz | g.lds | g.ldr) & 7) == 0;
  const long long items = (long long)g.M * (n8 / 8);
  const long long need = (items + 255) / 256;
  const int grid = (int)(need < 4LL * sm_count_simt() ? need : 4LL * sm_count_simt());
  skinny_dx_kernel<TO><<<grid, 256, skinny_dx_smem(g), s>>>(g, n8, vec);
  return cudaGetLastError();
}

template <int NP, int MV>
cudaError_t launch_skinny_dw(const GemmArgs& g, cudaStream_t s) {
  static bool attr = false;
  cudaError_t e = allow_smem(skinny_dw_kernel<NP, MV>, attr);
  if (e != cudaSuccess) return e;
  const int bx = (g.M + 32 * MV - 1) / (32 * MV);
  const int kcap = (int)(kSkinnySmem / (NP * 4)) & ~7;   // rows of B a block can hold
  int ks = (sm_count_simt() + bx - 1) / bx;              // about one block per SM
  const int kmax = (g.K + 63) / 64;                      // at least 64 rows of K per block
  if (ks > kmax) ks = kmax;
  if (ks < (g.K + kcap - 1) / kcap) ks = (g.K + kcap - 1) / kcap;
  if (ks < 1) ks = 1;
  int kper = (g.K + ks - 1) / ks;
  kper = (kper + 7) & ~7;                                // 16-byte aligned row ranges of B
  if (kper > kcap) kper = kcap;
  ks = (g.K + kper - 1) / kper;
  if (ks > 1) {
    e = g.ldo == g.N ? cudaMemsetAsync(g.out, 0, (size_t)g.M * g.N * 4, s)
                     : cudaMemset2DAsync(g.out, (size_t)g.ldo * 4, 0, (size_t)g.N * 4, g.M, s);
    if (e != cudaSuccess) return e;
  }
  const int vec = (reinterpret_cast<uintptr_t>(g.A) & (2u * MV - 1)) == 0 && (g.lda % MV) == 0;
  skinny_dw_kernel<NP, MV><<<dim3(bx, ks), 256, (size_t)kper * NP * 4, s>>>(g, kper, vec);
  return cudaGetLastError();
}

// Which narrow-side kernel runs g (0 forward, 1 input gradient, 2 weight
// gradient); false if none does.
bool skinny_kind(const GemmArgs& g, int* kind) {
  if (g.in_type != DT_BF16 || g.K <= 0) return false;
  const bool plain = !g.bias && !g.act && !g.out_z && !g.dact && !g.resid;
  if (!g.a_mn && !g.b_k && g.N <= 32 && skinny_fwd_smem(g) <= kSkinnySmem &&
      (g.aux_type == DT_BF16 || (!g.out_z && !g.dact && !g.resid))) {
    *kind = 0;   // forward
    return true;
  }
  if (!g.a_mn && g.b_k && g.K <= 32 && skinny_dx_smem(g) <= kSkinnySmem &&
      (g.aux_type == DT_BF16 || (!g.out_z && !g.dact && !g.resid))) {
    *kind = 1;   // input gradient
    return true;
  }
  if (g.a_mn && !g.b_k && g.N <= 32 && g.out_type == DT_F32 && plain) {
    *kind = 2;   // weight gradient
    return true;
  }
  return false;
}

cudaError_t gemm_skinny(const GemmArgs& g, int kind, cudaStream_t s) {
  const bool f32 = g.out_type == DT_F32;
  if (kind == 0) {
    if (g.N <= 16) return f32 ? launch_skinny_fwd<16, 4, float>(g, s) : launch_skinny_fwd<16, 4, bf16>(g, s);
    return f32 ? launch_skinny_fwd<32, 2, float>(g, s) : launch_skinny_fwd<32, 2, bf16>(g, s);
  }
  if (kind == 1) return f32 ? launch_skinny_dx<float>(g, s) : launch_skinny_dx<bf16>(g, s);
  if (g.N <= 16) return launch_skinny_dw<16, 4>(g, s);
  return launch_skinny_dw<32, 2>(g, s);
}

template <typename T, typename TO, typename TX, bool A_MN, bool B_K>
cudaError_t launch1(const GemmArgs& g, cudaStream_t s) {
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM);
  gemm_simt_kernel<T, TO, TX, A_MN, B_K><<<grid, NT, 0, s>>>(g, 0);
  return cudaGetLastError();
}

cudaError_t launch_dot2(const GemmArgs& g, cudaStream_t s) {
  dim3 grid((g.N + DBN - 1) / DBN, (g.M + DBM - 1) / DBM);
  gemm_dot2_kernel<<<grid, NT, 0, s>>>(g);
  return cudaGetLastError();
}

// Splits of a strict weight gradient (fp32 operands and output, no epilogue)
// whose 128x128 tiles leave SMs idle: enough splits to give about two CTAs
// per SM, at most 8, each at least 256 deep in K.
int strict_dw_splits(const GemmArgs& g) {
  if (!(g.in_type == DT_F32 && g.a_mn && !g.b_k && g.out_type == DT_F32 && !g.bias && !g.act &&
        !g.out_z && !g.dact && !g.resid))
    return 1;
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int tiles = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  int sp = (2 * sms + tiles - 1) / tiles;
  if (sp > 8) sp = 8;
  while (sp > 1 && g.K / sp < 256) --sp;
  return sp;
}

// out = sum over splits of the partial tiles, in split order.
__global__ void __launch_bounds__(256) split_sum_kernel(const float* ws, int splits, int M, int N,
                                                       float* out, long long ldo) {
  const size_t mn = (size_t)M * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < mn;
       i += (size_t)gridDim.x * blockDim.x) {
    float v = ws[i];
    for (int s = 1; s < splits; ++s) v += ws[(size_t)s * mn + i];
    out[(i / N) * ldo + (i % N)] = v;
  }
}

cudaError_t launch_strict_dw_split(const GemmArgs& g, int splits, cudaStream_t s) {
  const int k_per = ((g.K + splits - 1) / splits + BK - 1) / BK * BK;
  const int used = (g.K + k_per - 1) / k_per;
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, used);
  gemm_simt_kernel<float, float, float, true, false><<<grid, NT, 0, s>>>(g, k_per);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t mn = (size_t)g.M * g.N;
  int blocks = (int)((mn + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  split_sum_kernel<<<blocks, 256, 0, s>>>(g.split_ws, used, g.M, g.N, static_cast<float*>(g.out),
                                          g.ldo);
  return cudaGetLastError();
}

}  // namespace

size_t gemm_simt_split_floats(const GemmArgs& g) {
  int kind = 0;
  if (g.M <= 0 || g.N <= 0 || skinny_kind(g, &kind)) return 0;
  if (g.a_mn && !g.b_k && g.N <= 32) return 0;                 // narrow weight gradient
  if ((long long)g.M * g.N <= 65536 && g.K >= 64) return 0;    // warp per output
  const int sp = strict_dw_splits(g);
  return sp > 1 ? (size_t)sp * g.M * g.N : 0;
}

bool gemm_simt_skinny(const GemmArgs& g) {
  int kind = 0;
  return skinny_kind(g, &kind);
}

// Layouts used by the schedule: forward (A K-major, B N-major), dX (A K-major,
// B K-major), dW (A M-major, B N-major, fp32 output).
cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  int kind = 0;
  if (skinny_kind(g, &kind)) return gemm_skinny(g, kind, s);
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
    if (!g.a_mn && !g.b_k) return launch_dot2(g, s);   // forward: compensated
    if (!g.a_mn && g.b_k) return launch1<float, float, float, false, true>(g, s);
    if (g.a_mn && !g.b_k) {
      const int sp = strict_dw_splits(g);
      if (sp > 1 && g.split_ws && (size_t)sp * g.M * g.N <= g.split_ws_floats)
        return launch_strict_dw_split(g, sp, s);
      return launch1<float, float, float, true, false>(g, s);
    }
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
