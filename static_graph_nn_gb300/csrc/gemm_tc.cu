// bf16 GEMM on the 5th-generation tensor cores (tcgen05) with TMA-fed
// shared-memory stages, fp32 accumulators in tensor memory (TMEM) and the same
// fused epilogue as the CUDA-core GEMM.  This is the matmul archetype of the
// Meganeura README ("Why Meganeura" section) on its reduced-precision path
// (Environment variables section: validated f16/bf16 input tiles), and it
// serves the forward, input-gradient and weight-gradient GEMMs of every layer:
//   forward  Z  = X  W     A = X  [M,K] K-major,   B = W  [K,N] N-major
//   dX       dH = dZ W^T   A = dZ [M,K] K-major,   B = W  [N,K] K-major
//   dW       dW = X^T dZ   A = X  [K,M] M-major,   B = dZ [K,N] N-major
//
// One persistent CTA per SM, 320 threads in three roles:
//   warp 0      TMA producer: loads 128xBK tiles of A and BNxBK tiles of B into
//               a ring of shared-memory stages (128-byte swizzle);
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16) from
//               one elected lane; tcgen05.commit frees each stage and
//               publishes each finished accumulator;
//   warps 2-9   epilogue: tcgen05.ld of one accumulator row per thread (two
//               warps per TMEM lane quarter, each taking half the columns),
//               bias, activation, derivative mask, residual, store to global;
//               the accumulator is released once its last columns are in
//               registers.
// Two accumulators in TMEM (2 x BN columns) let the epilogue of tile i overlap
// the main loop of tile i+1.  Every mbarrier wait is bounded; on expiry the
// kernel records the failure in an error word and unwinds instead of hanging.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace mg {
namespace {

using namespace tc;

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;              // 64 bf16 = 128 bytes = one swizzle row
constexpr int TC_THREADS = 320;          // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
struct TcParams {
  GemmArgs g;
  int tiles_m, tiles_n, k_blocks;
  int splits, kb_per;                  // split-K: K blocks [s*kb_per, (s+1)*kb_per) per split
  int vec;                             // epilogue pointers/strides allow 16-byte vectors
  int vec32;                           // out, out_z, saved and resid rows allow 32-byte accesses
  int* err;                            // set to 1 on a timed-out wait
};

template <typename TO>
__device__ __forceinline__ float round_value_tc(float v) {
  return sizeof(TO) == 2 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

__device__ __forceinline__ void load8_bf16(const bf16* p, float* f) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void store8_bf16(bf16* p, const float* f) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = u;
}

// Epilogue of 32 consecutive columns of one row (same rounding points as the
// CUDA-core GEMM's epilogue).  Full, aligned chunks move in 16-byte vectors.
// On return v holds the values stored (before their rounding to TO) at the
// columns below N.
template <typename TO>
__device__ __forceinline__ void epilogue_row32(const GemmArgs& g, bool vec, bool vec32, int m,
                                               int n0, float (&v)[32]) {
  const bool full = vec && n0 + 32 <= g.N;
  if (full) {
    if (g.bias) {
      const float4* b4 = reinterpret_cast<const float4*>(g.bias + n0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 b = b4[q];
        v[4 * q] += b.x; v[4 * q + 1] += b.y; v[4 * q + 2] += b.z; v[4 * q + 3] += b.w;
      }
    }
    if (g.act || g.resid || g.out_z) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = round_value_tc<TO>(v[j]);
    }
    if (g.out_z) {
      bf16* z = static_cast<bf16*>(g.out_z) + (size_t)m * g.ldz + n0;
#pragma unroll
      if (vec32) {
        st16bf(z, v);
        st16bf(z + 16, v + 16);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) store8_bf16(z + 8 * q, v + 8 * q);
      }
    }
    if (g.act) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = apply_act(g.act, v[j]);
    }
    if (g.dact) {
      const bf16* sv = static_cast<const bf16*>(g.saved) + (size_t)m * g.lds + n0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float f[16];
        if (vec32) {
          ld16bf(sv + 16 * q, f);
        } else {
          load8_bf16(sv + 16 * q, f);
          load8_bf16(sv + 16 * q + 8, f + 8);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[16 * q + i] = round_value_tc<TO>(v[16 * q + i]) * act_grad_from_saved(g.dact, f[i]);
      }
    }
    if (g.resid) {
      const bf16* rv = static_cast<const bf16*>(g.resid) + (size_t)m * g.ldr + n0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float f[16];
        if (vec32) {
          ld16bf(rv + 16 * q, f);
        } else {
          load8_bf16(rv + 16 * q, f);
          load8_bf16(rv + 16 * q + 8, f + 8);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * q + i] += f[i];
      }
    }
    TO* out = static_cast<TO*>(g.out) + (size_t)m * g.ldo + n0;
    if (vec32) {
      if (sizeof(TO) == 2) {
        st16bf(reinterpret_cast<bf16*>(out), v);
        st16bf(reinterpret_cast<bf16*>(out) + 16, v + 16);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) st8f32(reinterpret_cast<float*>(out) + 8 * q, v + 8 * q);
      }
    } else if (sizeof(TO) == 2) {
#pragma unroll
      for (int q = 0; q < 4; ++q) store8_bf16(reinterpret_cast<bf16*>(out) + 8 * q, v + 8 * q);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(out)[q] =
            make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
    }
    return;
  }
  // ragged or unaligned chunk: element by element
  const size_t rz = (size_t)m * g.ldz, rs = (size_t)m * g.lds, rr = (size_t)m * g.ldr;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    if (n >= g.N) continue;
    float x = v[j];
    if (g.bias) x += g.bias[n];
    if (g.act || g.resid || g.out_z) x = round_value_tc<TO>(x);
    if (g.out_z) static_cast<bf16*>(g.out_z)[rz + n] = __float2bfloat16_rn(x);
    if (g.act) x = apply_act(g.act, x);
    if (g.dact) {
      x = round_value_tc<TO>(x);
      x *= act_grad_from_saved(g.dact, __bfloat162float(static_cast<const bf16*>(g.saved)[rs + n]));
    }
    if (g.resid) x += __bfloat162float(static_cast<const bf16*>(g.resid)[rr + n]);
    st_elem(static_cast<TO*>(g.out), (size_t)m * g.ldo + n, x);
    v[j] = x;
  }
}

// Split-K partial sum of 32 consecutive fp32 columns of one row, added into
// the (zeroed) output with vector atomics.  Used only for plain fp32 outputs
// (weight gradients: no bias, activation or residual in the epilogue).
__device__ __forceinline__ void split_add_row32(const GemmArgs& g, bool vec, int m, int n0,
                                                const float (&v)[32]) {
  float* out = static_cast<float*>(g.out) + (size_t)m * g.ldo + n0;
  if (vec && n0 + 32 <= g.N) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      atomicAdd(reinterpret_cast<float4*>(out) + q,
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (n0 + j < g.N) atomicAdd(out + j, v[j]);
}

template <int BN, int STAGES, typename TO, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams P) {
  constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;
  constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  constexpr uint32_t TMEM_COLS = 2 * BN;   // two accumulators
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned stage ring
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = P.tiles_m * P.tiles_n * P.splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x) {
        const int tile = item / P.splits, sp = item % P.splits;
        const int m0 = (tile / P.tiles_n) * TC_BM, n0 = (tile % P.tiles_n) * BN;
        const int kb0 = sp * P.kb_per, kb1 = min(P.k_blocks, kb0 + P.kb_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) { *abort_flag = 1; atomicExch(P.err, 1); break; }
          mbar_expect_tx(&full[stage], A_BYTES + B_BYTES);
          const int k0 = kb * TC_BK;
          uint8_t* a = sA + stage * A_BYTES;
          uint8_t* b = sB + stage * B_BYTES;
          if (A_MN) {   // [K rows][M]: boxes of 64 M x BK rows
#pragma unroll
            for (int i = 0; i < TC_BM / 64; ++i) tma_load_2d(a + i * 64 * TC_BK * 2, &tmA, &full[stage], m0 + i * 64, k0);
          } else {      // [M rows][K]: one box of 128 rows x 64 K
            tma_load_2d(a, &tmA, &full[stage], k0, m0);
          }
          if (B_MN) {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i) tma_load_2d(b + i * 64 * TC_BK * 2, &tmB, &full[stage], n0 + i * 64, k0);
          } else {
            tma_load_2d(b, &tmB, &full[stage], k0, n0);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(TC_BM, BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x, ++it) {
        const int sp = item % P.splits;
        const int kb0 = sp * P.kb_per, kb1 = min(P.k_blocks, kb0 + P.kb_per);
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&tempty[acc], use ^ 1)) { *abort_flag = 1; atomicExch(P.err, 1); break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + stage * A_BYTES);
          const uint32_t b = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k) {
            const uint64_t ad = A_MN ? smem_desc(a + k * 2048, 64 * TC_BK * 2, 1024)
                                     : smem_desc(a + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc(b + k * 2048, 64 * TC_BK * 2, 1024)
                                     : smem_desc(b + k * 32, 16, 1024);
            mma_bf16(d, ad, bd, idesc, (kb > kb0 || k) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);           // frees the stage when these MMAs finish
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; atomicExch(P.err, 1); break; }
        mma_commit(&tfull[acc]);               // accumulator ready for the epilogue
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;          // columns half*BN/2 .. (half+1)*BN/2-1
    const int row_in_tile = quarter * 32 + lane;
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const int tile = item / P.splits;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&tfull[acc], use)) { *abort_flag = 1; atomicExch(P.err, 1); break; }
      if (*abort_flag) break;
      tc_fence_after();
      const int m0 = (tile / P.tiles_n) * TC_BM, n0 = (tile % P.tiles_n) * BN;
      const int m = m0 + row_in_tile;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      static_assert(BN == 256, "softmax partials cover 128 columns per epilogue warp");
      float pm = -INFINITY, ps = 0.0f;             // softmax partial of this row's 128 columns
      auto chunk = [&](int c, uint32_t (&r)[32]) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if (m < P.g.M && n0 + c * 32 < P.g.N) {
          if (P.splits > 1) {
            split_add_row32(P.g, P.vec != 0, m, n0 + c * 32, v);
          } else {
            if (P.g.lse_part) softmax_partial32(P.g, n0 + c * 32, v, pm, ps);
            epilogue_row32<TO>(P.g, P.vec != 0, P.vec32 != 0, m, n0 + c * 32, v);
            if (sizeof(TO) == 4 && P.g.upd_p) adam_update32(P.g, P.vec != 0, m, n0 + c * 32, v);
          }
        }
        // warp-uniform: the warp's 32-row group starts below M, the chunk below N
        if (P.g.col_part && (m & ~31) < P.g.M && n0 + c * 32 < P.g.N)
          col_partial32<TO>(P.g, m, n0 + c * 32, lane, v);
      };
      // two pairs of 32-column chunks; the accumulator is released to the MMA
      // thread once the second pair is in registers, before its epilogue runs
#pragma unroll 1
      for (int cp = 0; cp < 2; ++cp) {
        const int c0 = half * (BN / 64) + 2 * cp;
        uint32_t r0[32], r1[32];
        tmem_ld32_async(taddr + c0 * 32, r0);
        tmem_ld32_async(taddr + (c0 + 1) * 32, r1);
        tmem_wait_regs(r0);
        reg_fence(r1);
        if (cp == 1) {
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
        }
        chunk(c0, r0);
        chunk(c0 + 1, r1);
      }
      if (P.g.lse_part && m < P.g.M && n0 + half * (BN / 2) < P.g.N)
        P.g.lse_part[(size_t)m * P.g.lse_ld + (n0 + half * (BN / 2)) / 128] = make_float2(pm, ps);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2D bf16 tensor [rows][cols] (cols contiguous, row stride ld elements), box
// box_cols x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, long long rows, long long cols, long long ld,
              int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int BN, int STAGES, typename TO, bool A_MN, bool B_MN>
cudaError_t launch_tc(const GemmArgs& g, int* err, cudaStream_t s) {
  CUtensorMap ma, mb;
  // A: logical [M, K].  K-major storage [M rows][K]; M-major storage [K rows][M].
  bool ok = A_MN ? make_map(&ma, g.A, g.K, g.M, g.lda, 64, TC_BK)
                 : make_map(&ma, g.A, g.M, g.K, g.lda, TC_BK, TC_BM);
  // B: logical [K, N].  N-major storage [K rows][N]; K-major storage [N rows][K].
  ok = ok && (B_MN ? make_map(&mb, g.B, g.K, g.N, g.ldb, 64, TC_BK)
                   : make_map(&mb, g.B, g.N, g.K, g.ldb, TC_BK, BN));
  if (!ok) return cudaErrorInvalidValue;
  TcParams P;
  P.g = g;
  P.tiles_m = (g.M + TC_BM - 1) / TC_BM;
  P.tiles_n = (g.N + BN - 1) / BN;
  P.k_blocks = (g.K + TC_BK - 1) / TC_BK;
  P.splits = 1;
  P.kb_per = P.k_blocks;
  P.err = err;
  {
    auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const long long lds = (g.ldz | g.lds | g.ldr | g.ldo);
    P.vec = al(g.bias) && al(g.out_z) && al(g.saved) && al(g.resid) && al(g.out) &&
            al(g.upd_p) && al(g.upd_m) && al(g.upd_v) && al(g.upd_shadow) && (lds & 7) == 0;
    auto al32 = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    const long long out_elems32 = g.out_type == DT_F32 ? 8 : 16;   // elements per 32 bytes
    P.vec32 = P.vec && al32(g.out) && al32(g.out_z) && al32(g.saved) && al32(g.resid) &&
              g.ldo % out_elems32 == 0 && (g.out_z == nullptr || g.ldz % 16 == 0) &&
              (g.saved == nullptr || g.lds % 16 == 0) && (g.resid == nullptr || g.ldr % 16 == 0);
  }
  const size_t smem = 1024 + (size_t)STAGES * (TC_BM + BN) * TC_BK * 2 + (2 * STAGES + 4) * 8 + 16;
  auto kern = gemm_tc_kernel<BN, STAGES, TO, A_MN, B_MN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int tiles = P.tiles_m * P.tiles_n;
  {
    double steps;
    P.splits = gemm_tc_splits(g, &steps);
    if (P.splits > 1) {
      P.kb_per = (P.k_blocks + P.splits - 1) / P.splits;
      P.splits = (P.k_blocks + P.kb_per - 1) / P.kb_per;
      cudaError_t e = g.ldo == g.N
                          ? cudaMemsetAsync(g.out, 0, (size_t)g.M * g.N * 4, s)
                          : cudaMemset2DAsync(g.out, (size_t)g.ldo * 4, 0, (size_t)g.N * 4, g.M, s);
      if (e != cudaSuccess) return e;
    }
  }
  const int items = tiles * P.splits;
  const int grid = items < num_sms() ? items : num_sms();
  kern<<<grid, TC_THREADS, smem, s>>>(ma, mb, P);
  return cudaGetLastError();
}

}  // namespace

bool gemm_tc_eligible(const GemmArgs& g) {
  if (g.in_type != DT_BF16 || g.K <= 0) return false;
  // TMA: 16-byte aligned bases and row strides
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al(g.A) || !al(g.B)) return false;
  if ((g.lda * 2) % 16 || (g.ldb * 2) % 16) return false;
  if (g.a_mn && g.b_k) return false;
  if (g.out_type == DT_F32 && !g.a_mn) return false;   // only dW writes fp32
  return encode_fn() != nullptr;
}

// Split-K for plain fp32 outputs (weight gradients) when the 128x256 tiles
// leave SMs idle: the split count that minimises rounds of work / splits, with
// at least 4 K blocks per split; the partial sums are added into a zeroed
// output.  *steps: the estimated duration in K-block steps of one SM at the
// SM-pair kernel's per-SM MMA rate; this kernel's steps take about 1.5x as
// long (one SM's shared memory feeds its 128x256 MMAs at about 2/3 of their
// rate).
int gemm_tc_splits(const GemmArgs& g, double* steps) {
  const int sms = num_sms();
  const int tiles = ((g.M + TC_BM - 1) / TC_BM) * ((g.N + 255) / 256);
  const int kb = (g.K + TC_BK - 1) / TC_BK;
  const bool plain = g.out_type == DT_F32 && !g.bias && !g.act && !g.out_z && !g.dact && !g.resid &&
                     !g.col_part && !g.upd_p;
  int splits = 1;
  double best = (double)((tiles + sms - 1) / sms);
  if (plain && tiles < sms) {
    best = 1.0;
    for (int sp = 2; sp <= 8 && kb / sp >= 4; ++sp) {
      const double cost = (double)((tiles * sp + sms - 1) / sms) / sp + 0.02 * sp;
      if (cost < best - 1e-9) {
        best = cost;
        splits = sp;
      }
    }
  }
  if (steps) *steps = 1.5 * best * kb;
  return splits;
}

cudaError_t gemm_tc(const GemmArgs& g, int* err, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (g.a_mn) return launch_tc<256, 4, float, true, true>(g, err, s);   // dW (fp32 out)
  if (g.b_k) return launch_tc<256, 4, bf16, false, false>(g, err, s);   // dX
  return launch_tc<256, 4, bf16, false, true>(g, err, s);                // forward
}

}  // namespace mg
