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

// 2^x on the special-function unit, subnormal results flushed to zero (the
// probabilities they stand for are far below bf16 resolution next to the
// row maximum's 1); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float2 u2f2(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a), __uint_as_float(b));
}

constexpr uint32_t IDESC_128x128_KK = instr_desc(128, 128, 0, 0);
constexpr uint32_t IDESC_128x64_KMN = instr_desc(128, 64, 0, 1);

// 32 fp32 values held as raw bits (computed in place in the TMEM load
// registers) -> bf16, written as four 16-byte chunks of row r (column chunks
// cc0..cc0+3 of a two-atom [128][128] tile).
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
// Persistent, one CTA per SM.  A work unit is a pair of consecutive query
// blocks (2p, 2p+1) of one (head, sequence).  Warps 0-3 own query block 2p
// (tile 0) and warps 4-7 block 2p+1 (tile 1), one query row per thread; warp 8
// is the TMA producer, warp 9 issues the MMAs.  Per key block j and tile w:
//   S_w = Q_w K_j^T          TMEM, fp32, 128 columns
//   P_w = 2^(S_w/8 log2e - m) TMEM, bf16 pairs, 64 columns
//   O_w += P_w V_j           TMEM, fp32, 64 columns (A operand read from TMEM)
// While one tile's softmax runs, the tensor core works on the other tile.
// m is the row's reference maximum (log2 units); it is raised, and O and l
// rescaled, only when a block's maximum exceeds it by more than 8, so that
// P <= 2^8.  Tile 0 skips key block 2p+1, which lies after all its queries.
// Units are dealt to the CTAs heaviest first in snake order.
constexpr int FWD_THREADS = 320;
constexpr int FWD_NST = 3;                            // K/V ring stages
constexpr uint32_t F_S = 0, F_P = 256, F_O = 384;     // TMEM columns of S, P, O (tile 0)
constexpr float RESCALE_T = 8.0f;

struct FwdUnit {
  int p, h, b, n0, n1;   // pair, head, sequence; key blocks of tile 0 / tile 1 (0: no tile 1)
};

__device__ __forceinline__ bool fwd_unit(int k, int n_units, int npair, int nqb, int H, FwdUnit& U) {
  const int G = gridDim.x;
  const int u = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  if (u >= n_units) return false;
  const int hb = n_units / npair;
  U.p = npair - 1 - u / hb;
  U.h = (u % hb) % H;
  U.b = (u % hb) / H;
  U.n0 = 2 * U.p + 1;
  U.n1 = (2 * U.p + 1 < nqb) ? 2 * U.p + 2 : 0;
  return true;
}

// 32 fp32 S values (raw bits) of row r at columns col0.. : keys after the
// query get -inf when the block is the diagonal one.
__device__ __forceinline__ void mask_diag(uint32_t (&v)[32], int col0, int r) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (col0 + e > r) v[e] = 0xff800000u;
}

__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_tc(const __grid_constant__ CUtensorMap tm_qkv, const AttnArgs A, int nb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm;                          // [2 slots][2 tiles]
  uint8_t* sK = sQ + 4 * TILE;               // [FWD_NST]
  uint8_t* sV = sK + FWD_NST * TILE;         // [FWD_NST]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sV + FWD_NST * TILE);
  uint64_t *q_full = bar, *q_empty = bar + 2, *kv_full = bar + 4, *kv_empty = kv_full + FWD_NST;
  uint64_t *s_full = kv_empty + FWD_NST, *p_full = s_full + 2, *o_done = s_full + 4,
           *o_free = s_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 24);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int nqb = A.S / AB;
  const int npair = (nqb + 1) / 2;
  const int n_units = npair * A.H * nb;
  const int d = A.H * AD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_free[i], 128);
    }
    for (int i = 0; i < FWD_NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 9) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      FwdUnit U;
      for (int k = 0; ok && fwd_unit(k, n_units, npair, nqb, A.H, U); ++k) {
        const int row0 = U.b * A.S, slot = k & 1;
        const int nmax = U.n1 ? U.n1 : U.n0;
        ok = mbar_wait(&q_empty[slot], ((k >> 1) & 1) ^ 1);
        if (!ok) break;
        mbar_expect_tx(&q_full[slot], (U.n1 ? 2 : 1) * TILE);
        tma_load_2d(sQ + (2 * slot) * TILE, &tm_qkv, &q_full[slot], U.h * AD, row0 + 2 * U.p * AB);
        if (U.n1)
          tma_load_2d(sQ + (2 * slot + 1) * TILE, &tm_qkv, &q_full[slot], U.h * AD,
                      row0 + (2 * U.p + 1) * AB);
        for (int j = 0; j < nmax; ++j, ++g) {
          const int st = g % FWD_NST;
          ok = mbar_wait(&kv_empty[st], ((g / FWD_NST) & 1) ^ 1);
          if (!ok) break;
          mbar_expect_tx(&kv_full[st], 2 * TILE);
          tma_load_2d(sK + st * TILE, &tm_qkv, &kv_full[st], d + U.h * AD, row0 + j * AB);
          tma_load_2d(sV + st * TILE, &tm_qkv, &kv_full[st], 2 * d + U.h * AD, row0 + j * AB);
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      int c[2] = {0, 0};     // S/P iterations issued per tile
      int uo[2] = {0, 0};    // units started per tile
      // the previous step, whose P V products are still to be issued
      int pv_st = -1, pv_act = 0, pv_first = 0;
      auto issue_pv = [&](int w) -> bool {
        // P_w of tile-iteration c[w]-1 is complete (this also frees S_w)
        if (!mbar_wait(&p_full[w], (c[w] - 1) & 1)) return false;
        if ((pv_first >> w) & 1) {
          if (uo[w] > 1 && !mbar_wait(&o_free[w], (uo[w] - 2) & 1)) return false;
        }
        tc_fence_after();
        const uint8_t* v = sV + pv_st * TILE;
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16_ts(tbase + F_O + 64 * w, tbase + F_P + 64 * w + kk * 8, mndesc(v, kk),
                      IDESC_128x64_KMN, !(((pv_first >> w) & 1) && kk == 0));
        mma_commit(&o_done[w]);
        return true;
      };
      FwdUnit U;
      for (int k = 0; ok && fwd_unit(k, n_units, npair, nqb, A.H, U); ++k) {
        const int slot = k & 1;
        const int nmax = U.n1 ? U.n1 : U.n0;
        ok = mbar_wait(&q_full[slot], (k >> 1) & 1);
        for (int j = 0; ok && j < nmax; ++j, ++g) {
          const int st = g % FWD_NST;
          const int act = (j < U.n0 ? 1 : 0) | (j < U.n1 ? 2 : 0);
          ok = mbar_wait(&kv_full[st], (g / FWD_NST) & 1);
          if (!ok) break;
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            if ((pv_act >> w) & 1) {
              ok = issue_pv(w);
              if (!ok) break;
            }
            if ((act >> w) & 1) {
              tc_fence_after();
              const uint8_t* q = sQ + (2 * slot + w) * TILE;
              const uint8_t* kt = sK + st * TILE;
#pragma unroll
              for (int kk = 0; kk < AD / 16; ++kk)
                mma_bf16(tbase + F_S + 128 * w, kdesc(q, kk), kdesc(kt, kk), IDESC_128x128_KK, kk > 0);
              mma_commit(&s_full[w]);
              ++c[w];
            }
          }
          if (!ok) break;
          if (pv_act) mma_commit(&kv_empty[pv_st]);
          if (j == nmax - 1) mma_commit(&q_empty[slot]);
          if (j == 0) {   // counted after the previous unit's last P V products
            if (U.n0) ++uo[0];
            if (U.n1) ++uo[1];
          }
          pv_st = st;
          pv_act = act;
          pv_first = (j == 0) ? act : 0;
        }
      }
      if (ok && pv_act) {
        for (int w = 0; w < 2 && ok; ++w)
          if ((pv_act >> w) & 1) ok = issue_pv(w);
        if (ok) mma_commit(&kv_empty[pv_st]);
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    // ---------------- softmax: warps 0-3 tile 0, warps 4-7 tile 1 ----------------
    const int w = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tSw = tbase + F_S + 128 * w + lane_off;
    const uint32_t tPw = tbase + F_P + 64 * w + lane_off;
    const uint32_t tOw = tbase + F_O + 64 * w + lane_off;
    const float scale2 = LOG2E * 0.125f;      // log2(e) / sqrt(64)
    bool ok = true;
    int c = 0;
    FwdUnit U;
    for (int k = 0; ok && fwd_unit(k, n_units, npair, nqb, A.H, U); ++k) {
      const int nw = w ? U.n1 : U.n0;
      if (nw == 0) continue;
      const int qb = 2 * U.p + w;
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nw; ++j, ++c) {
        if (!mbar_wait(&s_full[w], c & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool diag = (j == qb);
        uint32_t buf[2][32];
        // pass 1: the row maximum (four 32-column chunks, next load in flight)
        float pm[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pm[e] = -INFINITY;
        tmem_ld32_async(tSw, buf[0]);
        tmem_wait_regs(buf[0]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t(&cur)[32] = buf[ch & 1];
          if (ch < 3) tmem_ld32_async(tSw + 32 * (ch + 1), buf[(ch + 1) & 1]);
          if (diag) mask_diag(cur, ch * 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) pm[e & 7] = fmaxf(pm[e & 7], __uint_as_float(cur[e]));
          if (ch < 3) tmem_wait_regs(buf[(ch + 1) & 1]);
        }
        const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                               fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * scale2;
        const bool need = mx > m + RESCALE_T;
        const float m_new = need ? mx : m;
        const float alpha = need ? exp2f(m - m_new) : 1.0f;
        // P_w and O_w are free once the previous P V product is done
        if (c > 0 && !mbar_wait(&o_done[w], (c - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // pass 2: P = 2^(s scale2 - m_new) as bf16 pairs into TMEM; row sum
        const float2 sc2 = make_float2(scale2, scale2), nm2 = make_float2(-m_new, -m_new);
        float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        tmem_ld32_async(tSw, buf[0]);
        tmem_wait_regs(buf[0]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t(&cur)[32] = buf[ch & 1];
          if (ch < 3) tmem_ld32_async(tSw + 32 * (ch + 1), buf[(ch + 1) & 1]);
          if (diag) mask_diag(cur, ch * 32, r);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 y = __ffma2_rn(u2f2(cur[e], cur[e + 1]), sc2, nm2);
            const float2 pe = make_float2(ex2(y.x), ex2(y.y));
            ls[(e >> 1) & 3] = __fadd2_rn(ls[(e >> 1) & 3], pe);
            __nv_bfloat162 hv = __floats2bfloat162_rn(pe.x, pe.y);
            pk[e >> 1] = *reinterpret_cast<uint32_t*>(&hv);
          }
          tmem_st16(tPw + 16 * ch, pk);
          if (ch < 3) tmem_wait_regs(buf[(ch + 1) & 1]);
        }
        const float2 lsp = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
        // O = O * alpha for the rows whose reference maximum moved
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t ov[32];
            tmem_ld32_async(tOw + 32 * hh, ov);
            tmem_wait_regs(ov);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 sc = __fmul2_rn(u2f2(ov[e], ov[e + 1]), a2);
              ov[e] = __float_as_uint(sc.x);
              ov[e + 1] = __float_as_uint(sc.y);
            }
            tmem_st16(tOw + 32 * hh, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
            tmem_st16(tOw + 32 * hh + 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[16]));
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[w]);
        l = l * alpha + (lsp.x + lsp.y);
        m = m_new;
      }
      if (!ok) break;
      // unit end: O_w / l -> bf16 output; LSE
      if (!mbar_wait(&o_done[w], (c - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int qi = qb * AB + r;
      const int row0 = U.b * A.S;
      bf16* out = A.o + (size_t)(row0 + qi) * d + U.h * AD;
      const float inv = 1.0f / l;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float ov[32];
        tmem_ld32(tOw + 32 * hh, ov);
        store8_bf16_row(out + 32 * hh, ov, inv);
      }
      A.lse[((size_t)U.b * A.H + U.h) * A.S + qi] = (m + log2f(l)) / LOG2E;
      tc_fence_before();
      mbar_arrive(&o_free[w]);
    }
    if (!ok) fail_wait(A.err, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
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
      const float2 sc2 = make_float2(scale2, scale2), nlog2 = make_float2(-LOG2E, -LOG2E);
#pragma unroll 1
      for (int c4 = 2 * half; c4 < 2 * half + 2; ++c4) {
        uint32_t s[32], dp[32];
        tmem_ld32_async(tSt + lane_off + c4 * 32, s);
        tmem_ld32_async(tdPt + lane_off + c4 * 32, dp);
        tmem_wait();
        if (diag) {   // queries before the key get -inf, so their 2^x is 0
          const int lim = r - c4 * 32;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < lim) s[e] = 0xff800000u;
        }
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = reinterpret_cast<const float4*>(L + c4 * 32)[e4];
          const float4 d4 = reinterpret_cast<const float4*>(Dv + c4 * 32)[e4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int e = e4 * 4 + u;
            const float2 l2 = u ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
            const float2 d2 = u ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
            // p = 2^(s * log2(e) / 8 - LSE * log2(e)), dS = p (dP - D)
            const float2 y = __ffma2_rn(u2f2(s[e], s[e + 1]), sc2, __fmul2_rn(l2, nlog2));
            const float2 pp = make_float2(ex2(y.x), ex2(y.y));
            const float2 ds = __fmul2_rn(pp, __fadd2_rn(u2f2(dp[e], dp[e + 1]), d2));
            s[e] = __float_as_uint(pp.x);
            s[e + 1] = __float_as_uint(pp.y);
            dp[e] = __float_as_uint(ds.x);
            dp[e + 1] = __float_as_uint(ds.y);
          }
        }
        store_row_chunk_bits(sPt, r, c4 * 4, s);
        store_row_chunk_bits(sdSt, r, c4 * 4, dp);
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
      if (t == ib) {   // keys after the query get -inf, so their 2^x is 0
        const int lim = r - half * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e > lim) sr[c][e] = 0xff800000u;
      }
      // p = 2^(s * log2(e) / 8 - LSE * log2(e)), dS = p (dP - D), two lanes at a time
      const float2 sc2 = make_float2(scale2, scale2), nl2 = make_float2(-L2, -L2),
                   nd2 = make_float2(-Di, -Di);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 y = __ffma2_rn(u2f2(sr[c][e], sr[c][e + 1]), sc2, nl2);
          const float2 pp = make_float2(ex2(y.x), ex2(y.y));
          const float2 ds = __fmul2_rn(pp, __fadd2_rn(u2f2(dr[c][e], dr[c][e + 1]), nd2));
          dr[c][e] = __float_as_uint(ds.x);
          dr[c][e + 1] = __float_as_uint(ds.y);
        }
        store_row_chunk_bits(sdS, r, (half * 2 + c) * 4, dr[c]);
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

constexpr size_t SMEM_FWD = 1024 + TILE * (4 + 2 * FWD_NST) + 256;
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
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int units = ((S / AB + 1) / 2) * H * nb;
  attn_fwd_tc<<<units < sms ? units : sms, FWD_THREADS, SMEM_FWD, s>>>(m, a, nb);
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
