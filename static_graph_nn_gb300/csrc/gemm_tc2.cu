// bf16 GEMM on a CTA pair (tcgen05 cta_group::2): 256x256 output tiles
// computed by the tensor cores of two SMs, with the same fused epilogue as the
// single-SM kernel in gemm_tc.cu (see there for the three GEMM layouts).
//
// Why a pair: a 128x256x16 single-SM MMA reads 12 KB of operands from shared
// memory every 128 cycles while TMA writes the next 12 KB, about 1.5x what one
// SM's shared memory delivers.  With cta_group::2 each SM holds its 128 rows
// of A and only half (128 columns) of B; the pair's tensor cores exchange the
// B halves, so each SM moves 8 KB in and 8 KB out per 128 cycles.
//
// Cluster of 2 CTAs, one per SM, 320 threads each:
//   warp 0      (both CTAs) TMA producer for this CTA's A rows and B columns;
//               both CTAs' loads complete on the leader's full barrier
//               (cp.async.bulk.tensor .cta_group::2), whose expected byte
//               count the leader sets for the pair;
//   warp 1      leader CTA: allocates TMEM (2 x 256 columns, shared address in
//               both SMs), waits for both CTAs' stages and issues
//               tcgen05.mma.cta_group::2 (M=256, N=256, K=16); its commits are
//               multicast to both CTAs (stage free, accumulator full);
//   warps 2-9   (both CTAs) epilogue on this CTA's 128 accumulator rows, two
//               warps per TMEM lane quarter splitting the 256 columns; a
//               remote arrive on the leader's accumulator-free barrier once
//               the last TMEM loads are in registers, then the rest of the
//               epilogue (32-byte global accesses where rows allow them).
// Every wait is bounded; on expiry the error word is set and the pair unwinds.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace mg {
namespace {

using namespace tc;

constexpr int P_BM = 128;          // rows per CTA (256 per pair)
constexpr int P_BNH = 128;         // B columns per CTA (256 per pair)
constexpr int P_BN = 256;
constexpr int P_BK = 64;
constexpr int P_STAGES = 7;
constexpr int P_THREADS = 320;          // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t P_A_BYTES = P_BM * P_BK * 2;
constexpr uint32_t P_B_BYTES = P_BNH * P_BK * 2;

struct PairParams {
  GemmArgs g;
  int tiles_m, tiles_n, k_blocks;   // tiles_m counts 256-row pair tiles
  int splits, kb_per;               // split-K: K blocks [s*kb_per, (s+1)*kb_per) per split
  int vec;
  int vec32;                        // out, out_z, saved and resid rows allow 32-byte accesses
  int* err;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same object in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

// Arrive on a barrier of another CTA of the cluster.  Default semantics
// (release at CTA scope): it signals that this thread's TMEM reads are done
// (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync), and must not
// wait for the thread's global stores to reach cluster scope -- nothing the
// waiting MMA thread reads depends on them.  (With .release.cluster each
// epilogue warp stalled on a memory barrier per tile, holding the
// accumulator until its output stores were acknowledged.)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on the
// leader CTA's barrier (cluster address bar_cluster).
__device__ __forceinline__ void tma_load_2d_to_leader(void* dst, const CUtensorMap* map,
                                                      uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.aligned;\nbarrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive on the barrier at this offset in both CTAs once the pair's MMAs issued
// so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

template <typename TO>
__device__ __forceinline__ float rv(float v) {
  return sizeof(TO) == 2 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

__device__ __forceinline__ void ld8f(const bf16* p, float* f) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void st8f(bf16* p, const float* f) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = u;
}

// One split's partial sums of 32 columns of one row, added into the (zeroed)
// fp32 output; plain weight-gradient outputs only.
__device__ __forceinline__ void split_add32(const GemmArgs& g, bool vec, int m, int n0,
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

// Epilogue of 32 columns of one row; identical arithmetic to gemm_tc.cu.  On
// return v holds the values stored (before their rounding to TO) at the
// columns below N.
template <typename TO>
__device__ __forceinline__ void epi32(const GemmArgs& g, bool vec, bool vec32, int m, int n0,
                                      float (&v)[32]) {
  if (vec && n0 + 32 <= g.N) {
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
      for (int j = 0; j < 32; ++j) v[j] = rv<TO>(v[j]);
    }
    if (g.out_z) {
      bf16* z = static_cast<bf16*>(g.out_z) + (size_t)m * g.ldz + n0;
      if (vec32) {
        st16bf(z, v);
        st16bf(z + 16, v + 16);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) st8f(z + 8 * q, v + 8 * q);
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
          ld8f(sv + 16 * q, f);
          ld8f(sv + 16 * q + 8, f + 8);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[16 * q + i] = rv<TO>(v[16 * q + i]) * act_grad_from_saved(g.dact, f[i]);
      }
    }
    if (g.resid) {
      const bf16* rp = static_cast<const bf16*>(g.resid) + (size_t)m * g.ldr + n0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float f[16];
        if (vec32) {
          ld16bf(rp + 16 * q, f);
        } else {
          ld8f(rp + 16 * q, f);
          ld8f(rp + 16 * q + 8, f + 8);
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
      for (int q = 0; q < 4; ++q) st8f(reinterpret_cast<bf16*>(out) + 8 * q, v + 8 * q);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(out)[q] = make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
    }
    return;
  }
  const size_t rz = (size_t)m * g.ldz, rs = (size_t)m * g.lds, rr = (size_t)m * g.ldr;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    if (n >= g.N) continue;
    float x = v[j];
    if (g.bias) x += g.bias[n];
    if (g.act || g.resid || g.out_z) x = rv<TO>(x);
    if (g.out_z) static_cast<bf16*>(g.out_z)[rz + n] = __float2bfloat16_rn(x);
    if (g.act) x = apply_act(g.act, x);
    if (g.dact) {
      x = rv<TO>(x);
      x *= act_grad_from_saved(g.dact, __bfloat162float(static_cast<const bf16*>(g.saved)[rs + n]));
    }
    if (g.resid) x += __bfloat162float(static_cast<const bf16*>(g.resid)[rr + n]);
    st_elem(static_cast<TO*>(g.out), (size_t)m * g.ldo + n, x);
    v[j] = x;
  }
}

template <typename TO, bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const PairParams P) {
  constexpr uint32_t TMEM_COLS = 2 * P_BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + P_STAGES * P_A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + P_STAGES * P_B_BYTES);
  uint64_t* empty = full + P_STAGES;
  uint64_t* tfull = empty + P_STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int n_items = P.tiles_m * P.tiles_n * P.splits;   // (tile, K split) work items

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * 256);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();                      // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int item = pair; item < n_items && !*abort_flag; item += npairs) {
        const int tile = item / P.splits, sp = item % P.splits;
        const int m0 = (tile / P.tiles_n) * 2 * P_BM + rank * P_BM;
        const int n0 = (tile % P.tiles_n) * P_BN + rank * P_BNH;
        const int kb0 = sp * P.kb_per, kb1 = min(P.k_blocks, kb0 + P.kb_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1)) { *abort_flag = 1; atomicExch(P.err, 1); break; }
          // both CTAs' bytes complete on the leader's full barrier
          if (leader) mbar_expect_tx(&full[stage], 2 * (P_A_BYTES + P_B_BYTES));
          const uint32_t fb = map_to(&full[stage], 0);
          const int k0 = kb * P_BK;
          uint8_t* a = sA + stage * P_A_BYTES;
          uint8_t* b = sB + stage * P_B_BYTES;
          if (A_MN) {
            tma_load_2d_to_leader(a, &tmA, fb, m0, k0);
            tma_load_2d_to_leader(a + 64 * P_BK * 2, &tmA, fb, m0 + 64, k0);
          } else {
            tma_load_2d_to_leader(a, &tmA, fb, k0, m0);
          }
          if (B_MN) {
            tma_load_2d_to_leader(b, &tmB, fb, n0, k0);
            tma_load_2d_to_leader(b + 64 * P_BK * 2, &tmB, fb, n0 + 64, k0);
          } else {
            tma_load_2d_to_leader(b, &tmB, fb, k0, n0);
          }
          if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- leader: MMA issuer for the pair ----------------
      constexpr uint32_t idesc = instr_desc(2 * P_BM, P_BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int item = pair; item < n_items && !*abort_flag; item += npairs, ++it) {
        const int sp = item % P.splits;
        const int kb0 = sp * P.kb_per, kb1 = min(P.k_blocks, kb0 + P.kb_per);
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_cluster(&tempty[acc], use ^ 1)) { *abort_flag = 1; atomicExch(P.err, 1); break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * P_BN);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + stage * P_A_BYTES);
          const uint32_t b = smem_u32(sB + stage * P_B_BYTES);
#pragma unroll
          for (int k = 0; k < P_BK / 16; ++k) {
            const uint64_t ad = A_MN ? smem_desc(a + k * 2048, 64 * P_BK * 2, 1024)
                                     : smem_desc(a + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc(b + k * 2048, 64 * P_BK * 2, 1024)
                                     : smem_desc(b + k * 32, 16, 1024);
            mma_bf16_pair(d, ad, bd, idesc, (kb > kb0 || k) ? 1u : 0u);
          }
          mma_commit_pair(&empty[stage]);        // frees stage s in both CTAs
          if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; atomicExch(P.err, 1); break; }
        mma_commit_pair(&tfull[acc]);            // accumulators ready in both CTAs
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9, both CTAs) ----------------
    const int quarter = warp & 3;                // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;            // columns half*128 .. half*128+127
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t leader_tempty[2] = {map_to(&tempty[0], 0), map_to(&tempty[1], 0)};
    int it = 0;
    for (int item = pair; item < n_items; item += npairs, ++it) {
      const int tile = item / P.splits;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&tfull[acc], use)) { *abort_flag = 1; atomicExch(P.err, 1); break; }
      if (*abort_flag) break;
      tc_fence_after();
      const int m0 = (tile / P.tiles_n) * 2 * P_BM + rank * P_BM;
      const int n0 = (tile % P.tiles_n) * P_BN;
      const int m = m0 + row_in_tile;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * P_BN);
      float pm = -INFINITY, ps = 0.0f;             // softmax partial of this row's 128 columns
      auto chunk = [&](int c, uint32_t (&r)[32]) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if (m < P.g.M && n0 + c * 32 < P.g.N) {
          if (P.splits > 1) {
            split_add32(P.g, P.vec != 0, m, n0 + c * 32, v);
          } else {
            if (P.g.lse_part) softmax_partial32(P.g, n0 + c * 32, v, pm, ps);
            epi32<TO>(P.g, P.vec != 0, P.vec32 != 0, m, n0 + c * 32, v);
            if (sizeof(TO) == 4 && P.g.upd_p) adam_update32(P.g, P.vec != 0, m, n0 + c * 32, v);
          }
        }
        // warp-uniform: the warp's 32-row group starts below M, the chunk below N
        if (P.g.col_part && (m & ~31) < P.g.M && n0 + c * 32 < P.g.N)
          col_partial32<TO>(P.g, m, n0 + c * 32, lane, v);
      };
      // two pairs of 32-column chunks; the second pair's TMEM loads are this
      // warp's last reads of the accumulator, which is released to the MMA
      // thread before that pair's epilogue (loads, math, stores) runs
#pragma unroll 1
      for (int cp = 0; cp < 2; ++cp) {
        const int c0 = half * (P_BN / 64) + 2 * cp;
        uint32_t r0[32], r1[32];
        tmem_ld32_async(taddr + c0 * 32, r0);
        tmem_ld32_async(taddr + (c0 + 1) * 32, r1);
        tmem_wait_regs(r0);
        reg_fence(r1);
        if (cp == 1) {
          tc_fence_before();
          mbar_arrive_remote(leader_tempty[acc]);
        }
        chunk(c0, r0);
        chunk(c0 + 1, r1);
      }
      if (P.g.lse_part && m < P.g.M && n0 + half * (P_BN / 2) < P.g.N)
        P.g.lse_part[(size_t)m * P.g.lse_ld + (n0 + half * (P_BN / 2)) / 128] = make_float2(pm, ps);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();                      // no remote arrive or MMA still targets either CTA
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn2() {
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

bool make_map2(CUtensorMap* map, const void* base, long long rows, long long cols, long long ld,
               int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn2();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count2() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

constexpr size_t kPairSmem = 1024 + (size_t)P_STAGES * (P_A_BYTES + P_B_BYTES) + (2 * P_STAGES + 4) * 8 + 16;

// Clusters of two that can be resident at once (GPCs may not pair every SM);
// every instantiation of the kernel has the same shape of launch.
int pair_slots() {
  static int n = 0;
  if (!n) {
    auto kern = gemm_pair_kernel<float, true, true>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count2() / 2));
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = kPairSmem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c, kern, &cfg) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      c = sm_count2() / 2;
    }
    n = c;
  }
  return n;
}

// Split-K of the pair kernel, chosen as for the single-SM kernel (plain fp32
// outputs whose 256x256 tiles leave pairs idle, at least 4 K blocks per
// split), with a larger charge per split: a pair's partial tile is twice a
// single SM's, so each split adds twice the atomic traffic per slot.  *steps:
// estimated duration in K-block steps of one SM.
int pair_splits(const GemmArgs& g, double* steps) {
  const int slots = pair_slots();
  const int tiles = ((g.M + 2 * P_BM - 1) / (2 * P_BM)) * ((g.N + P_BN - 1) / P_BN);
  const int kb = (g.K + P_BK - 1) / P_BK;
  const bool plain = g.out_type == DT_F32 && !g.bias && !g.act && !g.out_z && !g.dact && !g.resid &&
                     !g.col_part && !g.upd_p;
  int splits = 1;
  double best = (double)((tiles + slots - 1) / slots);
  if (plain && tiles < slots) {
    best = 1.0;
    for (int sp = 2; sp <= 8 && kb / sp >= 4; ++sp) {
      const double cost = (double)((tiles * sp + slots - 1) / slots) / sp + 0.05 * sp;
      if (cost < best - 1e-9) {
        best = cost;
        splits = sp;
      }
    }
  }
  if (steps) *steps = best * kb;
  return splits;
}

template <typename TO, bool A_MN, bool B_MN>
cudaError_t launch_pair(const GemmArgs& g, int* err, cudaStream_t s) {
  CUtensorMap ma, mb;
  bool ok = A_MN ? make_map2(&ma, g.A, g.K, g.M, g.lda, 64, P_BK)
                 : make_map2(&ma, g.A, g.M, g.K, g.lda, P_BK, P_BM);
  ok = ok && (B_MN ? make_map2(&mb, g.B, g.K, g.N, g.ldb, 64, P_BK)
                   : make_map2(&mb, g.B, g.N, g.K, g.ldb, P_BK, P_BNH));
  if (!ok) return cudaErrorInvalidValue;
  PairParams P;
  P.g = g;
  P.tiles_m = (g.M + 2 * P_BM - 1) / (2 * P_BM);
  P.tiles_n = (g.N + P_BN - 1) / P_BN;
  P.k_blocks = (g.K + P_BK - 1) / P_BK;
  P.splits = pair_splits(g, nullptr);
  P.kb_per = P.k_blocks;
  if (P.splits > 1) {
    P.kb_per = (P.k_blocks + P.splits - 1) / P.splits;
    P.splits = (P.k_blocks + P.kb_per - 1) / P.kb_per;
  }
  P.err = err;
  {
    auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const long long lds = (g.ldz | g.lds | g.ldr | g.ldo);
    P.vec = al(g.bias) && al(g.out_z) && al(g.saved) && al(g.resid) && al(g.out) && al(g.upd_p) &&
            al(g.upd_m) && al(g.upd_v) && al(g.upd_shadow) && (lds & 7) == 0;
    auto al32 = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    const long long out_elems32 = g.out_type == DT_F32 ? 8 : 16;   // elements per 32 bytes
    P.vec32 = P.vec && al32(g.out) && al32(g.out_z) && al32(g.saved) && al32(g.resid) &&
              g.ldo % out_elems32 == 0 && (g.out_z == nullptr || g.ldz % 16 == 0) &&
              (g.saved == nullptr || g.lds % 16 == 0) && (g.resid == nullptr || g.ldr % 16 == 0);
  }
  const size_t smem = kPairSmem;
  auto kern = gemm_pair_kernel<TO, A_MN, B_MN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (P.splits > 1) {   // the splits' partial sums are added into a zeroed output
    cudaError_t e = g.ldo == g.N
                        ? cudaMemsetAsync(g.out, 0, (size_t)g.M * g.N * 4, s)
                        : cudaMemset2DAsync(g.out, (size_t)g.ldo * 4, 0, (size_t)g.N * 4, g.M, s);
    if (e != cudaSuccess) return e;
  }
  const int items = P.tiles_m * P.tiles_n * P.splits;
  int pairs = pair_slots();
  if (items < pairs) pairs = items;
  kern<<<2 * pairs, P_THREADS, smem, s>>>(ma, mb, P);
  return cudaGetLastError();
}

}  // namespace

bool gemm_pair_eligible(const GemmArgs& g) {
  // the estimated durations of the two kernels, waves of (split) tiles times
  // their K-block steps; below 128 rows or columns a pair is mostly padding
  if (g.M < 128 || g.N < 128 || g.K < 64) return false;
  double pair_steps = 0, single_steps = 0;
  pair_splits(g, &pair_steps);
  gemm_tc_splits(g, &single_steps);
  return pair_steps < single_steps;
}

int gemm_pair_split_count(const GemmArgs& g) { return pair_splits(g, nullptr); }

cudaError_t gemm_pair(const GemmArgs& g, int* err, cudaStream_t s) {
  if (g.a_mn) return launch_pair<float, true, true>(g, err, s);    // dW (fp32 out)
  if (g.b_k) return launch_pair<bf16, false, false>(g, err, s);    // dX
  return launch_pair<bf16, false, true>(g, err, s);                 // forward
}

}  // namespace mg
