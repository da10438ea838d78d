// Causal attention on the 5th-generation tensor cores (tcgen05), head_dim 64,
// the attention archetype of the Meganeura README ("Why Meganeura" section)
// with its kernel split (Environment variables section): a flash forward, and
// a backward made of a separate dQ kernel and a fused dK/dV kernel.
//
// Per (batch b, head h): S = Q K^T / sqrt(64), keys j > query i masked,
// P = softmax(S), O = P V; the forward saves LSE_i.  Backward with
// D_i = sum_c dO_ic O_ic:  P = exp(S - LSE), dP = dO V^T, dS = P (dP - D),
// dV = P^T dO, dK = dS^T Q / 8, dQ = dS K / 8.
//
// Every kernel: one CTA per (128-row block, head, sequence), 288 threads.
// Warp 0 lane 0 issues TMA loads and tcgen05.mma; warps 1-8 each own one TMEM
// lane quarter (32 rows of the 128-row block) and one half of the 128 columns,
// read S / dP with tcgen05.ld, do the softmax arithmetic in fp32 and write bf16
// P / dS tiles into shared memory in the 128-byte-swizzled K-major layout the
// next MMA reads.  The two warps that share a row exchange its maximum through
// shared memory (forward only).
//   forward: S = Q K_j^T (TMEM) -> P (smem) -> O_j = P V_j (TMEM, two slots);
//            O, the running max and sum stay in registers (online softmax).
//   dK/dV:   per key block, over the query blocks that see it:
//            S^T = K Q_i^T and dP^T = V dO_i^T (keys are the M dimension), so
//            P^T and dS^T are written row by row and feed dV += P^T dO_i and
//            dK += dS^T Q_i directly; dV, dK accumulate in TMEM.
//   dQ:      per query block, over the visible key blocks: S, dP, then
//            dQ += dS K_j accumulated in TMEM.
// All mbarrier waits are bounded; on expiry the error word is set and the CTA
// unwinds.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace mg {
namespace {

using namespace tc;

constexpr int AD = 64;                      // head dimension
constexpr int AB = 128;                     // rows (queries / keys) per block
constexpr uint32_t TILE = AB * AD * 2;      // one [128][64] bf16 tile: 16 KB
constexpr uint32_t PTILE = 2 * TILE;        // one [128][128] bf16 tile: 32 KB (two K atoms)
constexpr int NSW = 8;                      // softmax / elementwise warps (two per TMEM lane quarter)
constexpr int AT_THREADS = 32 * (1 + NSW);
constexpr int NSWT = 32 * NSW;              // their thread count
constexpr float LOG2E = 1.4426950408889634f;

struct AttnArgs {
  int S, H;
  bf16* o;          // forward output [nb*S, H*64]
  float* lse;       // [nb, H, S]
  const float* dsum;  // D [nb, H, S] (backward)
  bf16* dqkv;       // [nb*S, 3*H*64] (backward)
  int* err;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void fail_wait(int* err, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(err, 1);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// K-major descriptors: a [128 rows][64 cols] tile (SBO 1024); k-step of 16 = 32 bytes.
__device__ __forceinline__ uint64_t kdesc(const uint8_t* tile, int kstep) {
  return smem_desc(smem_u32(tile) + kstep * 32, 16, 1024);
}
// K-major descriptor into a [128 rows][128 cols] tile stored as two 64-col atoms.
__device__ __forceinline__ uint64_t kdesc_p(const uint8_t* ptile, int kstep) {
  return smem_desc(smem_u32(ptile) + (kstep >> 2) * TILE + (kstep & 3) * 32, 16, 1024);
}
// MN-major descriptor: the same [128 rows = K][64 cols = N] tile read with K
// along the rows; k-step of 16 rows = 2048 bytes.
__device__ __forceinline__ uint64_t mndesc(const uint8_t* tile, int kstep) {
  return smem_desc(smem_u32(tile) + kstep * 2048, 8192, 1024);
}

// 32 fp32 values times scale -> bf16, four 16-byte global stores.
__device__ __forceinline__ void store8_bf16_row(bf16* out, const float* v, float scale) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 hv = __floats2bfloat162_rn(v[q * 8 + 2 * i] * scale, v[q * 8 + 2 * i + 1] * scale);
      w[i] = *reinterpret_cast<uint32_t*>(&hv);
    }
    reinterpret_cast<uint4*>(out)[q] = u;
  }
}

// Barrier among the softmax / elementwise warps only (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

constexpr uint32_t IDESC_128x128_KK = instr_desc(128, 128, 0, 0);
constexpr uint32_t IDESC_128x64_KMN = instr_desc(128, 64, 0, 1);

// 32 fp32 values -> bf16, written as four 16-byte chunks of row r (column
// chunks cc0..cc0+3 of a two-atom [128][128] tile).
__device__ __forceinline__ void store_row_chunk(uint8_t* ptile, int r, int cc0, const float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int cc = cc0 + q;
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 hv = __floats2bfloat162_rn(v[q * 8 + 2 * i], v[q * 8 + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(ptile + (cc >> 3) * TILE + sw128(r, cc & 7)) = u;
  }
}

// Same, from fp32 values kept as raw bits (computed in place in the TMEM load registers).
__device__ __forceinline__ void store_row_chunk_bits(uint8_t* ptile, int r, int cc0, const uint32_t* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int cc = cc0 + q;
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(v[q * 8 + 2 * i]),
                                                __uint_as_float(v[q * 8 + 2 * i + 1]));
      w[i] = *reinterpret_cast<uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(ptile + (cc >> 3) * TILE + sw128(r, cc & 7)) = u;
  }
}

// ============================================================ forward
__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_fwd_tc(const __grid_constant__ CUtensorMap tm_qkv, const AttnArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + TILE;           // [2]
  uint8_t* sV = sK + 2 * TILE;       // [2]
  uint8_t* sP = sV + 2 * TILE;       // 32 KB
  uint64_t* bar = reinterpret_cast<uint64_t*>(sP + PTILE);
  uint64_t *q_full = bar, *kv_full = bar + 1, *kv_empty = bar + 3, *s_full = bar + 5,
           *s_free = bar + 6, *p_full = bar + 7, *o_full = bar + 8, *o_free = bar + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red_max = reinterpret_cast<float*>(bar + 16);    // [2 iterations][2 halves][128]
  float* red_l = red_max + 4 * AB;                        // [2 halves][128]

  const int nqb = A.S / AB;
  const int qb = nqb - 1 - blockIdx.x;             // longest rows of work first
  const int h = blockIdx.y, b = blockIdx.z;
  const int nkb = qb + 1;
  const int d = A.H * AD;
  const int row0 = b * A.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], NSWT);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, NSWT);
    mbar_init(p_full, NSWT);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = *tmem_slot;            // columns 0..127
  const uint32_t tO0 = tS + 128;             // two 64-column slots

  if (warp == 0) {
    if (lane == 0) {
      auto load_kv = [&](int j) {
        mbar_expect_tx(&kv_full[j & 1], 2 * TILE);
        tma_load_2d(sK + (j & 1) * TILE, &tm_qkv, &kv_full[j & 1], d + h * AD, row0 + j * AB);
        tma_load_2d(sV + (j & 1) * TILE, &tm_qkv, &kv_full[j & 1], 2 * d + h * AD, row0 + j * AB);
      };
      auto mma_pv = [&](int i) -> bool {
        if (!mbar_wait(p_full, i & 1)) return false;
        if (i >= 2 && !mbar_wait(&o_free[i & 1], ((i - 2) >> 1) & 1)) return false;
        tc_fence_after();
        const uint8_t* v = sV + (i & 1) * TILE;
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16(tO0 + (i & 1) * 64, kdesc_p(sP, kk), mndesc(v, kk), IDESC_128x64_KMN, kk > 0);
        mma_commit(&o_full[i & 1]);
        mma_commit(&kv_empty[i & 1]);
        return true;
      };
      bool ok = true;
      mbar_expect_tx(q_full, TILE);
      tma_load_2d(sQ, &tm_qkv, q_full, h * AD, row0 + qb * AB);
      load_kv(0);
      if (nkb > 1) load_kv(1);
      for (int j = 0; j < nkb && ok; ++j) {
        ok = mbar_wait(&kv_full[j & 1], (j >> 1) & 1) && (j > 0 || mbar_wait(q_full, 0)) &&
             (j == 0 || mbar_wait(s_free, (j - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint8_t* k = sK + (j & 1) * TILE;
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(tS, kdesc(sQ, kk), kdesc(k, kk), IDESC_128x128_KK, kk > 0);
        mma_commit(s_full);
        if (j > 0) ok = mma_pv(j - 1);
        if (ok && j + 1 < nkb && j + 1 >= 2) {
          ok = mbar_wait(&kv_empty[(j + 1) & 1], ((j - 1) >> 1) & 1);
          if (ok) load_kv(j + 1);
        }
      }
      if (ok) ok = mma_pv(nkb - 1);
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    const int quarter = warp & 3;
    const int half = (warp - 1) >> 2;            // columns half*64 .. half*64+63
    const int r = quarter * 32 + lane;
    const int qi = qb * AB + r;                  // query position in the sequence
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float scale2 = LOG2E * 0.125f;         // log2(e) / sqrt(64)
    float o[32];                                 // O columns half*32 .. half*32+31
#pragma unroll
    for (int c = 0; c < 32; ++c) o[c] = 0.0f;
    float m = -INFINITY, l = 0.0f, alpha_prev = 0.0f;
    bool ok = true;
    // Every thread passes the same named barriers, also after a failed wait,
    // so that a timeout never leaves the other warps blocked at a barrier.
    for (int j = 0; j < nkb; ++j) {
      ok = ok && mbar_wait(s_full, j & 1);
      const bool diag = (j == qb);
      uint32_t sr[2][32];
      float mx = -INFINITY;
      if (ok) {
        tc_fence_after();
        tmem_ld32_async(tS + lane_off + half * 64, sr[0]);
        tmem_ld32_async(tS + lane_off + half * 64 + 32, sr[1]);
        tmem_wait();
        tc_fence_before();
        mbar_arrive(s_free);                       // S is in registers: the next QK^T may start
        if (diag) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (half * 64 + c * 32 + t <= r) mx = fmaxf(mx, __uint_as_float(sr[c][t]));
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int t = 0; t < 32; ++t) mx = fmaxf(mx, __uint_as_float(sr[c][t]));
        }
      }
      float* rm = red_max + (j & 1) * 2 * AB;
      rm[half * AB + r] = mx;
      named_sync(1, NSWT);
      if (!ok) continue;
      mx = fmaxf(rm[r], rm[AB + r]);
      const float m_new = fmaxf(m, mx * scale2);
      const float alpha = exp2f(m - m_new);
      if (j > 0) {   // fold in O_{j-1}; its MMA has also finished reading P
        ok = mbar_wait(&o_full[(j - 1) & 1], ((j - 1) >> 1) & 1);
        if (!ok) continue;
        tc_fence_after();
        float v[32];
        tmem_ld32(tO0 + ((j - 1) & 1) * 64 + half * 32 + lane_off, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t] = o[t] * alpha_prev + v[t];
        tc_fence_before();
        mbar_arrive(&o_free[(j - 1) & 1]);
      }
      float lsum = 0.0f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          float e = exp2f(__uint_as_float(sr[c][t]) * scale2 - m_new);
          if (diag && half * 64 + c * 32 + t > r) e = 0.0f;
          sr[c][t] = __float_as_uint(e);
          lsum += e;
        }
        store_row_chunk_bits(sP, r, (half * 2 + c) * 4, sr[c]);
      }
      fence_proxy_async();
      mbar_arrive(p_full);
      l = l * alpha + lsum;
      m = m_new;
      alpha_prev = alpha;
    }
    ok = ok && mbar_wait(&o_full[(nkb - 1) & 1], ((nkb - 1) >> 1) & 1);
    if (ok) {
      tc_fence_after();
      float v[32];
      tmem_ld32(tO0 + ((nkb - 1) & 1) * 64 + half * 32 + lane_off, v);
#pragma unroll
      for (int t = 0; t < 32; ++t) o[t] = o[t] * alpha_prev + v[t];
    }
    red_l[half * AB + r] = l;
    named_sync(1, NSWT);
    if (ok) {
      const float lt = red_l[r] + red_l[AB + r];
      const float inv = 1.0f / lt;
      store8_bf16_row(A.o + (size_t)(row0 + qi) * d + h * AD + half * 32, o, inv);
      if (half == 0) A.lse[((size_t)b * A.H + h) * A.S + qi] = (m + log2f(lt)) / LOG2E;
    } else {
      fail_wait(A.err, abort_flag);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*tmem_slot, 256);
  }
}

// ============================================================ backward dK/dV
__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tm_qkv,
                     const __grid_constant__ CUtensorMap tm_do, const AttnArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sK = sm;
  uint8_t* sV = sK + TILE;
  uint8_t* sQ = sV + TILE;            // [2]
  uint8_t* sdO = sQ + 2 * TILE;       // [2]
  uint8_t* sPt = sdO + 2 * TILE;      // 32 KB
  uint8_t* sdSt = sPt + PTILE;        // 32 KB
  float* sL = reinterpret_cast<float*>(sdSt + PTILE);   // [2][128] LSE of the query block
  float* sD = sL + 2 * AB;                               // [2][128] D of the query block
  uint64_t* bar = reinterpret_cast<uint64_t*>(sD + 2 * AB);
  uint64_t *kv_full = bar, *in_full = bar + 1, *in_empty = bar + 3, *st_full = bar + 5,
           *st_free = bar + 6, *ds_full = bar + 7, *acc_done = bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int nqb = A.S / AB;
  const int jb = blockIdx.x;                       // key block; most work first
  const int h = blockIdx.y, b = blockIdx.z;
  const int n_it = nqb - jb;                       // query blocks jb .. nqb-1
  const int d = A.H * AD;
  const int row0 = b * A.S;
  const size_t lrow = ((size_t)b * A.H + h) * A.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 1);
    }
    mbar_init(st_full, 1);
    mbar_init(st_free, NSWT);
    mbar_init(ds_full, NSWT);
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tSt = *tmem_slot, tdPt = tSt + 128, tdV = tSt + 256, tdK = tSt + 320;

  if (warp == 0) {
    if (lane == 0) {
      auto load_in = [&](int t) {
        const int i = jb + t, bf = t & 1;
        mbar_expect_tx(&in_full[bf], 2 * TILE + 2 * AB * 4);
        tma_load_2d(sQ + bf * TILE, &tm_qkv, &in_full[bf], h * AD, row0 + i * AB);
        tma_load_2d(sdO + bf * TILE, &tm_do, &in_full[bf], h * AD, row0 + i * AB);
        bulk_load(sL + bf * AB, A.lse + lrow + i * AB, AB * 4, &in_full[bf]);
        bulk_load(sD + bf * AB, A.dsum + lrow + i * AB, AB * 4, &in_full[bf]);
      };
      auto mma_acc = [&](int t) -> bool {
        if (!mbar_wait(ds_full, t & 1)) return false;
        tc_fence_after();
        const int bf = t & 1;
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16(tdV, kdesc_p(sPt, kk), mndesc(sdO + bf * TILE, kk), IDESC_128x64_KMN, (t | kk) > 0);
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16(tdK, kdesc_p(sdSt, kk), mndesc(sQ + bf * TILE, kk), IDESC_128x64_KMN, (t | kk) > 0);
        mma_commit(acc_done);
        mma_commit(&in_empty[bf]);
        return true;
      };
      bool ok = true;
      mbar_expect_tx(kv_full, 2 * TILE);
      tma_load_2d(sK, &tm_qkv, kv_full, d + h * AD, row0 + jb * AB);
      tma_load_2d(sV, &tm_qkv, kv_full, 2 * d + h * AD, row0 + jb * AB);
      load_in(0);
      if (n_it > 1) load_in(1);
      for (int t = 0; t < n_it && ok; ++t) {
        ok = mbar_wait(&in_full[t & 1], (t >> 1) & 1) && (t > 0 || mbar_wait(kv_full, 0)) &&
             (t == 0 || mbar_wait(st_free, (t - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint8_t* q = sQ + (t & 1) * TILE;
        const uint8_t* g = sdO + (t & 1) * TILE;
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(tSt, kdesc(sK, kk), kdesc(q, kk), IDESC_128x128_KK, kk > 0);
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(tdPt, kdesc(sV, kk), kdesc(g, kk), IDESC_128x128_KK, kk > 0);
        mma_commit(st_full);
        if (t > 0) ok = mma_acc(t - 1);
        if (ok && t + 1 < n_it && t + 1 >= 2) {
          ok = mbar_wait(&in_empty[(t + 1) & 1], ((t - 1) >> 1) & 1);
          if (ok) load_in(t + 1);
        }
      }
      if (ok) ok = mma_acc(n_it - 1);
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    const int quarter = warp & 3;
    const int half = (warp - 1) >> 2;            // query columns half*64 .. +63
    const int r = quarter * 32 + lane;
    const int kj = jb * AB + r;                  // key position
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float scale2 = LOG2E * 0.125f;
    bool ok = true;
    for (int t = 0; t < n_it; ++t) {
      const int bf = t & 1;
      if (!mbar_wait(st_full, t & 1) || !mbar_wait(&in_full[bf], (t >> 1) & 1) ||
          (t > 0 && !mbar_wait(acc_done, (t - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool diag = (t == 0);                // query block jb holds the diagonal
      const float* L = sL + bf * AB;
      const float* Dv = sD + bf * AB;
#pragma unroll 1
      for (int c4 = 2 * half; c4 < 2 * half + 2; ++c4) {
        float s[32], dp[32];
        tmem_ld32(tSt + lane_off + c4 * 32, s);
        tmem_ld32(tdPt + lane_off + c4 * 32, dp);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = reinterpret_cast<const float4*>(L + c4 * 32)[e4];
          const float4 d4 = reinterpret_cast<const float4*>(Dv + c4 * 32)[e4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = e4 * 4 + u;
            float p = exp2f(s[e] * scale2 - lv[u] * LOG2E);
            if (diag && c4 * 32 + e < r) p = 0.0f;     // query < key
            s[e] = p;
            dp[e] = p * (dp[e] - dv[u]);
          }
        }
        store_row_chunk(sPt, r, c4 * 4, s);
        store_row_chunk(sdSt, r, c4 * 4, dp);
      }
      tc_fence_before();
      mbar_arrive(st_free);
      fence_proxy_async();
      mbar_arrive(ds_full);
    }
    if (ok && mbar_wait(acc_done, (n_it - 1) & 1)) {
      tc_fence_after();
      bf16* outk = A.dqkv + (size_t)(row0 + kj) * 3 * d + d + h * AD + half * 32;
      bf16* outv = A.dqkv + (size_t)(row0 + kj) * 3 * d + 2 * d + h * AD + half * 32;
      float v[32];
      tmem_ld32(tdV + lane_off + half * 32, v);
      store8_bf16_row(outv, v, 1.0f);
      tmem_ld32(tdK + lane_off + half * 32, v);
      store8_bf16_row(outk, v, 0.125f);
    } else {
      fail_wait(A.err, abort_flag);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*tmem_slot, 512);
  }
}

// ============================================================ backward dQ
__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tm_qkv,
                   const __grid_constant__ CUtensorMap tm_do, const AttnArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm;
  uint8_t* sdO = sQ + TILE;
  uint8_t* sK = sdO + TILE;           // [2]
  uint8_t* sV = sK + 2 * TILE;        // [2]
  uint8_t* sdS = sV + 2 * TILE;       // 32 KB
  uint64_t* bar = reinterpret_cast<uint64_t*>(sdS + PTILE);
  uint64_t *q_full = bar, *kv_full = bar + 1, *kv_empty = bar + 3, *s_full = bar + 5,
           *s_free = bar + 6, *ds_full = bar + 7, *acc_done = bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int nqb = A.S / AB;
  const int ib = nqb - 1 - blockIdx.x;             // most work first
  const int h = blockIdx.y, b = blockIdx.z;
  const int n_it = ib + 1;                         // key blocks 0 .. ib
  const int d = A.H * AD;
  const int row0 = b * A.S;
  const size_t lrow = ((size_t)b * A.H + h) * A.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, NSWT);
    mbar_init(ds_full, NSWT);
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = *tmem_slot, tdP = tS + 128, tdQ = tS + 256;

  if (warp == 0) {
    if (lane == 0) {
      auto load_kv = [&](int t) {
        const int bf = t & 1;
        mbar_expect_tx(&kv_full[bf], 2 * TILE);
        tma_load_2d(sK + bf * TILE, &tm_qkv, &kv_full[bf], d + h * AD, row0 + t * AB);
        tma_load_2d(sV + bf * TILE, &tm_qkv, &kv_full[bf], 2 * d + h * AD, row0 + t * AB);
      };
      auto mma_acc = [&](int t) -> bool {
        if (!mbar_wait(ds_full, t & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16(tdQ, kdesc_p(sdS, kk), mndesc(sK + (t & 1) * TILE, kk), IDESC_128x64_KMN,
                   (t | kk) > 0);
        mma_commit(acc_done);
        mma_commit(&kv_empty[t & 1]);
        return true;
      };
      bool ok = true;
      mbar_expect_tx(q_full, 2 * TILE);
      tma_load_2d(sQ, &tm_qkv, q_full, h * AD, row0 + ib * AB);
      tma_load_2d(sdO, &tm_do, q_full, h * AD, row0 + ib * AB);
      load_kv(0);
      if (n_it > 1) load_kv(1);
      for (int t = 0; t < n_it && ok; ++t) {
        ok = mbar_wait(&kv_full[t & 1], (t >> 1) & 1) && (t > 0 || mbar_wait(q_full, 0)) &&
             (t == 0 || mbar_wait(s_free, (t - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint8_t* k = sK + (t & 1) * TILE;
        const uint8_t* v = sV + (t & 1) * TILE;
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(tS, kdesc(sQ, kk), kdesc(k, kk), IDESC_128x128_KK, kk > 0);
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(tdP, kdesc(sdO, kk), kdesc(v, kk), IDESC_128x128_KK, kk > 0);
        mma_commit(s_full);
        if (t > 0) ok = mma_acc(t - 1);
        if (ok && t + 1 < n_it && t + 1 >= 2) {
          ok = mbar_wait(&kv_empty[(t + 1) & 1], ((t - 1) >> 1) & 1);
          if (ok) load_kv(t + 1);
        }
      }
      if (ok) ok = mma_acc(n_it - 1);
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    const int quarter = warp & 3;
    const int half = (warp - 1) >> 2;            // key columns half*64 .. +63
    const int r = quarter * 32 + lane;
    const int qi = ib * AB + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float scale2 = LOG2E * 0.125f;
    const float L2 = A.lse[lrow + qi] * LOG2E;
    const float Di = A.dsum[lrow + qi];
    bool ok = true;
    for (int t = 0; t < n_it; ++t) {
      if (!mbar_wait(s_full, t & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[2][32], dr[2][32];
      tmem_ld32_async(tS + lane_off + half * 64, sr[0]);
      tmem_ld32_async(tS + lane_off + half * 64 + 32, sr[1]);
      tmem_ld32_async(tdP + lane_off + half * 64, dr[0]);
      tmem_ld32_async(tdP + lane_off + half * 64 + 32, dr[1]);
      tmem_wait();
      tc_fence_before();
      mbar_arrive(s_free);                         // S, dP are in registers
      if (t > 0 && !mbar_wait(acc_done, (t - 1) & 1)) {   // dS tile free again
        ok = false;
        break;
      }
      const bool diag = (t == ib);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int c4 = half * 2 + c;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float p = exp2f(__uint_as_float(sr[c][e]) * scale2 - L2);
          if (diag && c4 * 32 + e > r) p = 0.0f;      // key > query
          dr[c][e] = __float_as_uint(p * (__uint_as_float(dr[c][e]) - Di));
        }
        store_row_chunk_bits(sdS, r, c4 * 4, dr[c]);
      }
      fence_proxy_async();
      mbar_arrive(ds_full);
    }
    if (ok && mbar_wait(acc_done, (n_it - 1) & 1)) {
      tc_fence_after();
      float v[32];
      tmem_ld32(tdQ + lane_off + half * 32, v);
      store8_bf16_row(A.dqkv + (size_t)(row0 + qi) * 3 * d + h * AD + half * 32, v, 0.125f);
    } else {
      fail_wait(A.err, abort_flag);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*tmem_slot, 512);
  }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode() {
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

// [rows][cols] bf16, row stride ld elements, box 64 x 128, 128-byte swizzle.
bool map_128x64(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld) {
  EncodeTiledFn fn = encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t SMEM_FWD = 1024 + TILE * 5 + PTILE + 128 + 6 * AB * 4;
constexpr size_t SMEM_DKDV = 1024 + TILE * 6 + 2 * PTILE + 4 * AB * 4 + 128;
constexpr size_t SMEM_DQ = 1024 + TILE * 6 + PTILE + 128;

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

bool attn_tc_eligible(int S, int H, int Dh, const void* qkv) {
  return Dh == AD && S % AB == 0 && S > 0 && ((reinterpret_cast<uintptr_t>(qkv) & 15) == 0) &&
         encode() != nullptr;
}

cudaError_t attn_fwd_tc_launch(const void* qkv, void* o, float* lse, int nb, int S, int H,
                               int* err, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_fwd_tc, SMEM_FWD);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap m;
  if (!map_128x64(&m, qkv, (long long)nb * S, 3LL * H * AD, 3LL * H * AD)) return cudaErrorInvalidValue;
  AttnArgs a{S, H, (bf16*)o, lse, nullptr, nullptr, err};
  attn_fwd_tc<<<dim3(S / AB, H, nb), AT_THREADS, SMEM_FWD, s>>>(m, a);
  return cudaGetLastError();
}

cudaError_t attn_bwd_tc_launch(const void* qkv, const void* dout, const float* lse,
                               const float* dsum, void* dqkv, int nb, int S, int H, int* err,
                               cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_bwd_dkdv_tc, SMEM_DKDV);
    if (e == cudaSuccess) e = set_smem(attn_bwd_dq_tc, SMEM_DQ);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mq, mo;
  if (!map_128x64(&mq, qkv, (long long)nb * S, 3LL * H * AD, 3LL * H * AD) ||
      !map_128x64(&mo, dout, (long long)nb * S, (long long)H * AD, (long long)H * AD))
    return cudaErrorInvalidValue;
  AttnArgs a{S, H, nullptr, const_cast<float*>(lse), dsum, (bf16*)dqkv, err};
  attn_bwd_dkdv_tc<<<dim3(S / AB, H, nb), AT_THREADS, SMEM_DKDV, s>>>(mq, mo, a);
  attn_bwd_dq_tc<<<dim3(S / AB, H, nb), AT_THREADS, SMEM_DQ, s>>>(mq, mo, a);
  return cudaGetLastError();
}

}  // namespace mg
