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
// Forward: persistent, one CTA per SM over (pair of query blocks, head,
// sequence) units; S, P and O live in tensor memory (P is the A operand of
// P V, read from TMEM); each of two softmax groups owns one query tile of the
// pair, and each group's products have an MMA-issuing thread of their own
// (see below).
// Backward: the same persistent plan for the dK/dV kernel (per key block,
// over the query blocks that see it: S^T and dP^T with the keys as the M
// dimension, P^T and dS^T into TMEM, dV += P^T dO_i and dK += dS^T Q_i) and
// for the dQ kernel (per query block, over the visible key blocks: S, dP,
// dS into TMEM, dQ += dS K_j).
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
constexpr int NSW = 8;                      // softmax / elementwise warps (two per TMEM lane quarter)
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

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&hv);
}


// 32 fp32 S values (raw bits) of row r at columns col0.. : keys after the
// query get -inf when the block is the diagonal one.
__device__ __forceinline__ void mask_diag(uint32_t (&v)[32], int col0, int r) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (col0 + e > r) v[e] = 0xff800000u;
}

constexpr uint32_t IDESC_128x128_KK = instr_desc(128, 128, 0, 0);
constexpr uint32_t IDESC_128x64_KMN = instr_desc(128, 64, 0, 1);

// ============================================================ forward
// Persistent, one CTA per SM.  A work unit is one (sequence b, head h, pair of
// adjacent 128-row query blocks 2p, 2p+1), dealt to the CTAs heaviest first
// in snake order; the two query tiles share every K/V tile the CTA loads.
// Softmax group g (warps 4g .. 4g+3, one query row per thread) owns one of
// the two tiles -- the groups take the higher block of the pair in turn, so
// their work over a run balances -- with its own buffers
//   S[g] = Q_g K_j^T           TMEM, fp32, 128 columns
//   P[g] = 2^(S/8 log2e - m)   TMEM, bf16 pairs, 64 columns
//   O[g] += P[g] V_j           TMEM, fp32, 64 columns (A operand read from TMEM)
// and its own running maximum m and sum l per row; a group finishes its tile
// alone (no merge).  m is a reference maximum in log2 units, raised (and
// O[g], l rescaled) only when a block's maximum exceeds it by more than 8, so
// that P <= 2^8.
// Warp 8 is the TMA producer; warps 9 and 10 issue the MMAs of group 0 and
// group 1.  One issuing thread per group: a tcgen05.mma takes about 60 cycles
// to issue from one thread, and the products here are small (N = 128 for S,
// N = 64 for P V), so one thread issuing for both groups would leave the
// tensor pipe idle; two threads on two SM sub-partitions issue concurrently
// (measured on GB300: 45 -> 33 us on B8 S1024 H16).  Warp 11 is spare, so
// that each issuing warp has an SM sub-partition of its own.
constexpr int FWD_THREADS = 384;
constexpr int FWD_NST = 4;                                  // K/V ring stages
constexpr uint32_t F_S = 0, F_P = 256, F_O = 384;           // TMEM columns of S[0], P[0], O[0]
constexpr float RESCALE_T = 8.0f;

struct FwdUnit {
  int h, b;
  int qlo, qhi;        // query blocks 2p and 2p + 1; qhi < 0: the pair has one block
};

__device__ __forceinline__ bool fwd_unit(int k, int n_units, int npair, int nqb, int H,
                                         FwdUnit& U) {
  const int G = gridDim.x;
  const int u = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  if (u >= n_units) return false;
  const int hb = n_units / npair;
  const int p = npair - 1 - u / hb;
  U.h = (u % hb) % H;
  U.b = (u % hb) / H;
  U.qlo = 2 * p;
  U.qhi = 2 * p + 1 < nqb ? 2 * p + 1 : -1;
  return true;
}
// query block of group g in the CTA's k-th unit (-1: none) and its tile index
// in the unit's Q slot
__device__ __forceinline__ int fwd_grp_q(const FwdUnit& U, int k, int g) {
  return ((g ^ (k & 1)) == 0) ? U.qlo : U.qhi;
}
__device__ __forceinline__ int fwd_grp_t(int k, int g) { return g ^ (k & 1); }
// K/V blocks a unit loads
__device__ __forceinline__ int fwd_nkv(const FwdUnit& U) { return (U.qhi >= 0 ? U.qhi : U.qlo) + 1; }

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
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
  uint64_t *s_full = kv_empty + FWD_NST, *s_free = s_full + 2, *p_full = s_full + 4,
           *o_done = s_full + 6, *o_free = s_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int nqb = A.S / AB;
  const int npair = (nqb + 1) / 2;
  const int n_units = npair * A.H * nb;
  const int d = A.H * AD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 2);            // both groups' last S of the unit
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], NSWT / 2);      // one group
      mbar_init(&p_full[i], NSWT / 2);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_free[i], NSWT / 2);
    }
    for (int i = 0; i < FWD_NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 2);           // both groups' last P V of the block
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
      int gkv = 0;
      FwdUnit U;
      for (int k = 0; ok && fwd_unit(k, n_units, npair, nqb, A.H, U); ++k) {
        const int row0 = U.b * A.S, slot = k & 1;
        ok = mbar_wait(&q_empty[slot], ((k >> 1) & 1) ^ 1);
        if (!ok) break;
        mbar_expect_tx(&q_full[slot], (U.qhi >= 0 ? 2 : 1) * TILE);
        tma_load_2d(sQ + (2 * slot) * TILE, &tm_qkv, &q_full[slot], U.h * AD, row0 + U.qlo * AB);
        if (U.qhi >= 0)
          tma_load_2d(sQ + (2 * slot + 1) * TILE, &tm_qkv, &q_full[slot], U.h * AD,
                      row0 + U.qhi * AB);
        const int nkv = fwd_nkv(U);
        for (int j = 0; j < nkv; ++j, ++gkv) {
          const int st = gkv % FWD_NST;
          ok = mbar_wait(&kv_empty[st], ((gkv / FWD_NST) & 1) ^ 1);
          if (!ok) break;
          mbar_expect_tx(&kv_full[st], 2 * TILE);
          tma_load_2d(sK + st * TILE, &tm_qkv, &kv_full[st], d + U.h * AD, row0 + j * AB);
          tma_load_2d(sV + st * TILE, &tm_qkv, &kv_full[st], 2 * d + U.h * AD, row0 + j * AB);
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp == 9 || warp == 10) {
    // ---------------- MMA issuer of group g ----------------
    if (lane == 0) {
      const int g = warp - 9;
      constexpr uint64_t TSTEP = TILE >> 4;
      const uint64_t dq0 = kdesc(sQ, 0), dk0 = kdesc(sK, 0), dv0 = mndesc(sV, 0);
      // A cursor walks this group's items (unit k, key block j) in order:
      // base is the ring index of the unit's first K/V block, c the group's
      // item count, e its count of units with work.
      struct Cur {
        int k, j, n, base, c, e;
        FwdUnit U;
        bool valid;
      };
      auto enter = [&](Cur& c) {   // the group's next unit with work
        while ((c.valid = fwd_unit(c.k, n_units, npair, nqb, A.H, c.U))) {
          const int q = fwd_grp_q(c.U, c.k, g);
          if (q >= 0) {
            c.n = q + 1;
            return;
          }
          c.base += fwd_nkv(c.U);
          ++c.k;
        }
      };
      auto next = [&](Cur& c) {
        ++c.c;
        if (++c.j >= c.n) {
          c.base += fwd_nkv(c.U);
          c.j = 0;
          ++c.k;
          ++c.e;
          enter(c);
        }
      };
      Cur cs, cp;
      cs.k = cs.j = cs.base = cs.c = cs.e = 0;
      enter(cs);
      cp = cs;
      // The group's products come in a fixed order -- S of item c + 1 (once
      // the softmax has read S of item c) before P V of item c (once it has
      // written P of item c) -- so the issuer waits for each in turn.
      auto issue_s = [&]() -> bool {
        const int gkv = cs.base + cs.j, st = gkv % FWD_NST, slot = cs.k & 1;
        if (cs.j == 0 && !mbar_wait(&q_full[slot], (cs.k >> 1) & 1)) return false;
        if (!mbar_wait(&kv_full[st], (gkv / FWD_NST) & 1)) return false;
        if (cs.c > 0 && !mbar_wait(&s_free[g], (cs.c - 1) & 1)) return false;
        tc_fence_after();
        const uint64_t aq = dq0 + (uint64_t)(2 * slot + fwd_grp_t(cs.k, g)) * TSTEP;
        const uint64_t bk = dk0 + (uint64_t)st * TSTEP;
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(tbase + F_S + 128 * g, aq + kk * 2, bk + kk * 2, IDESC_128x128_KK, kk > 0);
        mma_commit(&s_full[g]);
        if (cs.j == cs.n - 1) {
          mma_commit(&q_empty[slot]);
          if (cs.U.qhi < 0) mma_commit(&q_empty[slot]);   // the other group had no block
        }
        next(cs);
        return true;
      };
      auto issue_pv = [&]() -> bool {
        if (!mbar_wait(&p_full[g], cp.c & 1)) return false;
        // a unit's first P V overwrites O[g]: the previous unit's O is read out
        if (cp.j == 0 && cp.e > 0 && !mbar_wait(&o_free[g], (cp.e - 1) & 1)) return false;
        tc_fence_after();
        const int st = (cp.base + cp.j) % FWD_NST;
        const uint64_t bv = dv0 + (uint64_t)st * TSTEP;
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16_ts(tbase + F_O + 64 * g, tbase + F_P + 64 * g + kk * 8, bv + kk * 128,
                      IDESC_128x64_KMN, kk > 0 || cp.j > 0);
        mma_commit(&o_done[g]);
        mma_commit(&kv_empty[st]);
        // the other group does not use this key block: its arrival too
        const int qo = fwd_grp_q(cp.U, cp.k, g ^ 1);
        if (qo < 0 || cp.j > qo) mma_commit(&kv_empty[st]);
        next(cp);
        return true;
      };
      bool ok = true;
      if (cs.valid) ok = issue_s();
      while (ok && cp.valid) {
        if (cs.valid) ok = issue_s();
        if (ok) ok = issue_pv();
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp < 8) {
    // ---------------- softmax: group g = warps 4g .. 4g+3, one row per thread ----------------
    const int quarter = warp & 3;
    const int g = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + F_S + 128 * g + lane_off;
    const uint32_t tP = tbase + F_P + 64 * g + lane_off;
    const uint32_t tO = tbase + F_O + 64 * g + lane_off;
    const float scale2 = LOG2E * 0.125f;
    bool ok = true;
    int c = 0;   // this group's item count
    FwdUnit U;
    for (int k = 0; ok && fwd_unit(k, n_units, npair, nqb, A.H, U); ++k) {
      const int q = fwd_grp_q(U, k, g);
      if (q < 0) continue;
      const int n = q + 1;
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < n; ++j, ++c) {
        if (!mbar_wait(&s_full[g], c & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the whole 128-column row of S in registers, then S[g] is released
        uint32_t sv[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32_async(tS + 32 * ch, sv[ch]);
        tmem_wait_regs(sv[0]);
        reg_fence(sv[1]);
        reg_fence(sv[2]);
        reg_fence(sv[3]);
        tc_fence_before();
        mbar_arrive(&s_free[g]);
        // the diagonal block: 32-key chunk `quarter` holds this warp's
        // diagonal (keys after the row masked), later chunks are masked whole
        const bool diag = (j == n - 1);
        const int lim = diag ? quarter : 3;   // last chunk with an unmasked key
        if (diag) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            if (ch == quarter) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (e > lane) sv[ch][e] = 0xff800000u;
            }
        }
        float pm[4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          pm[ch] = -INFINITY;
          if (ch <= lim) {
            // tree of three-input maxima: 32 -> 11 -> 4 -> 1
            float t1[11];
#pragma unroll
            for (int i = 0; i < 10; ++i)
              t1[i] = max3f(__uint_as_float(sv[ch][3 * i]), __uint_as_float(sv[ch][3 * i + 1]),
                            __uint_as_float(sv[ch][3 * i + 2]));
            t1[10] = fmaxf(__uint_as_float(sv[ch][30]), __uint_as_float(sv[ch][31]));
            const float t2a = max3f(t1[0], t1[1], t1[2]), t2b = max3f(t1[3], t1[4], t1[5]),
                        t2c = max3f(t1[6], t1[7], t1[8]), t2d = fmaxf(t1[9], t1[10]);
            pm[ch] = fmaxf(max3f(t2a, t2b, t2c), t2d);
          }
        }
        const float mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])) * scale2;
        const bool need = mx > m + RESCALE_T;
        const float m_new = need ? mx : m;
        const float alpha = need ? exp2f(m - m_new) : 1.0f;
        const float2 sc2 = make_float2(scale2, scale2), nm2 = make_float2(-m_new, -m_new);
        float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        // chunks 0-1 while the previous P V may still read P[g]; then wait for
        // it, store them and go on with chunks 2-3; masked chunks store zeros
        uint32_t pk[2][16];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          if (ch <= lim) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 y = __ffma2_rn(u2f2(sv[ch][e], sv[ch][e + 1]), sc2, nm2);
              const float2 pe = make_float2(ex2(y.x), ex2(y.y));
              ls[(e >> 1) & 1] = __fadd2_rn(ls[(e >> 1) & 1], pe);
              pk[ch][e >> 1] = pack_bf16(pe.x, pe.y);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[ch][e] = 0u;
          }
        }
        // P[g] and O[g] are free once this group's previous P V is done
        if (c >= 1 && !mbar_wait(&o_done[g], (c - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tP, pk[0]);
        tmem_st16(tP + 16, pk[1]);
#pragma unroll
        for (int ch = 2; ch < 4; ++ch) {
          uint32_t pq[16];
          if (ch <= lim) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 y = __ffma2_rn(u2f2(sv[ch][e], sv[ch][e + 1]), sc2, nm2);
              const float2 pe = make_float2(ex2(y.x), ex2(y.y));
              ls[(e >> 1) & 1] = __fadd2_rn(ls[(e >> 1) & 1], pe);
              pq[e >> 1] = pack_bf16(pe.x, pe.y);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) pq[e] = 0u;
          }
          tmem_st16(tP + 16 * ch, pq);
        }
        // O[g] = O[g] * alpha for the rows whose reference maximum moved
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t ov[32];
            tmem_ld32_async(tO + 32 * hh, ov);
            tmem_wait_regs(ov);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 sc = __fmul2_rn(u2f2(ov[e], ov[e + 1]), a2);
              ov[e] = __float_as_uint(sc.x);
              ov[e + 1] = __float_as_uint(sc.y);
            }
            tmem_st16(tO + 32 * hh, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
            tmem_st16(tO + 32 * hh + 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[16]));
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[g]);
        const float2 lsp = __fadd2_rn(ls[0], ls[1]);
        l = l * alpha + (lsp.x + lsp.y);
        m = m_new;
      }
      if (!ok) break;
      // unit end: O of this group's tile once its last P V is done
      if (!mbar_wait(&o_done[g], (c - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int qi = q * AB + r;
      bf16* orow = A.o + (size_t)(U.b * A.S + qi) * d + U.h * AD;
      const float inv_l = 1.0f / l;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float ov[32];
        tmem_ld32(tO + 32 * hh, ov);
        if (hh == 1) {
          tc_fence_before();
          mbar_arrive(&o_free[g]);            // O[g] is read: the next unit may overwrite it
        }
        store8_bf16_row(orow + 32 * hh, ov, inv_l);
      }
      A.lse[((size_t)U.b * A.H + U.h) * A.S + qi] = (m + log2f(l)) / LOG2E;
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

// ============================================================ backward
// Both backward kernels follow the forward's plan: persistent CTAs over
// (128-row block, head, sequence) units dealt heaviest first in snake order,
// warps 0-15 the elementwise work (warp w: TMEM lane quarter w & 3, columns
// 32 (w >> 2) .. +31), warp 16 the TMA producer, warps 17 and 18 the MMA
// issuers; S and dP are read from TMEM once and released, and the bf16
// products P / dS are written back into TMEM as the A operand of the
// accumulating MMAs.
constexpr int BWD_NST = 3;   // ring stages of the streamed operand pair

__device__ __forceinline__ bool bwd_unit(int k, int n_units, int hb, int H, int& major, int& h,
                                         int& b) {
  const int G = gridDim.x;
  const int u = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  if (u >= n_units) return false;
  major = u / hb;
  h = (u % hb) % H;
  b = (u % hb) / H;
  return true;
}

// 32 fp32 S^T values (raw bits) of key row r at query columns col0.. : queries
// before the key get -inf when the block is the diagonal one.
__device__ __forceinline__ void mask_diag_t(uint32_t (&v)[32], int col0, int r) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (col0 + e < r) v[e] = 0xff800000u;
}



// ------------------------------------------------------------ dK / dV
// Unit: key block jb; over the query blocks i = jb .. nqb-1 (keys are the M
// dimension, so every product is a row-major one for this CTA's key rows):
//   S^T = K Q_i^T, dP^T = V dO_i^T                      TMEM, fp32
//   P^T = 2^(S^T/8 log2e - LSE_i log2e), dS^T = P^T (dP^T - D_i)  -> TMEM bf16
//   dV += P^T dO_i, dK += dS^T Q_i                      TMEM, fp32
// dK is scaled by 1/8 when it is written out.
// Warps 0-15 do the elementwise work, four per TMEM lane quarter: warp w
// takes key rows 32 (w & 3) .. +31 and query columns 32 (w >> 2) .. +31, so
// that each SM sub-partition has four elementwise warps to hide the latency
// of the per-element chain (TMEM load, exp2, products, bf16 packing, TMEM
// store).  Warp 16 is the TMA producer; warps 17 and 18 issue the MMAs.
constexpr uint32_t DKV_S = 0, DKV_DP = 128, DKV_P = 256, DKV_DS = 320, DKV_DV = 384, DKV_DK = 448;
constexpr int DKV_THREADS = 608;
constexpr int DKV_EW = 512;                 // elementwise threads

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 fp32 values times scale -> bf16, two 16-byte global stores.
__device__ __forceinline__ void store16_bf16(bf16* out, const float* v, float scale) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint4 u;
    u.x = pack_bf16(v[q * 8 + 0] * scale, v[q * 8 + 1] * scale);
    u.y = pack_bf16(v[q * 8 + 2] * scale, v[q * 8 + 3] * scale);
    u.z = pack_bf16(v[q * 8 + 4] * scale, v[q * 8 + 5] * scale);
    u.w = pack_bf16(v[q * 8 + 6] * scale, v[q * 8 + 7] * scale);
    reinterpret_cast<uint4*>(out)[q] = u;
  }
}

__global__ void __launch_bounds__(DKV_THREADS, 1)
    attn_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tm_qkv,
                     const __grid_constant__ CUtensorMap tm_do, const AttnArgs A, int nb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sK = sm;                          // [2 slots]
  uint8_t* sV = sK + 2 * TILE;               // [2 slots]
  uint8_t* sQ = sV + 2 * TILE;               // [BWD_NST]
  uint8_t* sdO = sQ + BWD_NST * TILE;        // [BWD_NST]
  float* sL = reinterpret_cast<float*>(sdO + BWD_NST * TILE);   // [BWD_NST][128] LSE
  float* sD = sL + BWD_NST * AB;                                 // [BWD_NST][128] D
  uint64_t* bar = reinterpret_cast<uint64_t*>(sD + BWD_NST * AB);
  uint64_t *kv_full = bar, *kv_empty = bar + 2, *in_full = bar + 4, *in_empty = in_full + BWD_NST;
  uint64_t *st_full = in_empty + BWD_NST, *st_free = st_full + 1, *ds_full = st_full + 2,
           *acc_done = st_full + 3, *o_free = st_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int nqb = A.S / AB;
  const int hb = A.H * nb;
  const int n_units = nqb * hb;
  const int d = A.H * AD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // barriers the MMAs complete take one commit from each of the two issuers
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 2);
    }
    for (int i = 0; i < BWD_NST; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 2);
    }
    mbar_init(st_full, 2);
    mbar_init(st_free, DKV_EW);
    mbar_init(ds_full, DKV_EW);
    mbar_init(acc_done, 2);
    mbar_init(o_free, DKV_EW);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 16) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 16) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      int g = 0, jb, h, b;
      for (int k = 0; ok && bwd_unit(k, n_units, hb, A.H, jb, h, b); ++k) {
        const int row0 = b * A.S, slot = k & 1, n = nqb - jb;
        const size_t lrow = ((size_t)b * A.H + h) * A.S;
        ok = mbar_wait(&kv_empty[slot], ((k >> 1) & 1) ^ 1);
        if (!ok) break;
        mbar_expect_tx(&kv_full[slot], 2 * TILE);
        tma_load_2d(sK + slot * TILE, &tm_qkv, &kv_full[slot], d + h * AD, row0 + jb * AB);
        tma_load_2d(sV + slot * TILE, &tm_qkv, &kv_full[slot], 2 * d + h * AD, row0 + jb * AB);
        for (int j = 0; j < n; ++j, ++g) {
          const int i = jb + j, st = g % BWD_NST;
          ok = mbar_wait(&in_empty[st], ((g / BWD_NST) & 1) ^ 1);
          if (!ok) break;
          mbar_expect_tx(&in_full[st], 2 * TILE + 2 * AB * 4);
          tma_load_2d(sQ + st * TILE, &tm_qkv, &in_full[st], h * AD, row0 + i * AB);
          tma_load_2d(sdO + st * TILE, &tm_do, &in_full[st], h * AD, row0 + i * AB);
          bulk_load(sL + st * AB, A.lse + lrow + i * AB, AB * 4, &in_full[st]);
          bulk_load(sD + st * AB, A.dsum + lrow + i * AB, AB * 4, &in_full[st]);
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp == 17 || warp == 18) {
    // ---------------- MMA issuers ----------------
    // Issuer 0 (warp 17): S^T = K Q_i^T, then dV += P^T dO_i; issuer 1 (warp
    // 18): dP^T = V dO_i^T, then dK += dS^T Q_i.  Twelve MMAs each per block;
    // two issuing threads on two SM sub-partitions keep the tensor pipe fed
    // where one thread issuing all 24 small MMAs could not.  Each issues, in
    // order, its S-type product of block c + 1 (once the elementwise warps have
    // read block c's S^T and dP^T) before its accumulating product of block c
    // (once they have written P^T and dS^T of block c).
    if (lane == 0) {
      const int who = warp - 17;
      constexpr uint64_t TSTEP = TILE >> 4;
      const uint64_t da0 = who == 0 ? kdesc(sK, 0) : kdesc(sV, 0);        // K or V
      const uint64_t db0 = who == 0 ? kdesc(sQ, 0) : kdesc(sdO, 0);       // Q_i or dO_i
      const uint64_t dm0 = who == 0 ? mndesc(sdO, 0) : mndesc(sQ, 0);     // dO_i or Q_i
      const uint32_t t_st = tbase + (who == 0 ? DKV_S : DKV_DP);
      const uint32_t t_a = tbase + (who == 0 ? DKV_P : DKV_DS);
      const uint32_t t_acc = tbase + (who == 0 ? DKV_DV : DKV_DK);
      struct Cursor {
        int k, j, g, jb, h, b;
        bool valid;
      };
      auto advance = [&](Cursor& c) {
        ++c.g;
        if (++c.j >= nqb - c.jb) {
          c.j = 0;
          ++c.k;
          c.valid = bwd_unit(c.k, n_units, hb, A.H, c.jb, c.h, c.b);
        }
      };
      Cursor ca;
      ca.k = ca.j = ca.g = 0;
      ca.valid = bwd_unit(0, n_units, hb, A.H, ca.jb, ca.h, ca.b);
      Cursor cb = ca;
      auto issue_st = [&]() -> bool {
        const int st = ca.g % BWD_NST, slot = ca.k & 1;
        if (ca.j == 0 && !mbar_wait(&kv_full[slot], (ca.k >> 1) & 1)) return false;
        if (!mbar_wait(&in_full[st], (ca.g / BWD_NST) & 1)) return false;
        if (ca.g > 0 && !mbar_wait(st_free, (ca.g - 1) & 1)) return false;
        tc_fence_after();
        const uint64_t a = da0 + (uint64_t)slot * TSTEP, bq = db0 + (uint64_t)st * TSTEP;
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(t_st, a + kk * 2, bq + kk * 2, IDESC_128x128_KK, kk > 0);
        mma_commit(st_full);
        if (ca.j == nqb - ca.jb - 1) mma_commit(&kv_empty[slot]);
        advance(ca);
        return true;
      };
      auto issue_acc = [&]() -> bool {
        if (!mbar_wait(ds_full, cb.g & 1)) return false;
        // a unit's first block overwrites the accumulator: the previous
        // unit's dV / dK is read out
        if (cb.j == 0 && cb.k > 0 && !mbar_wait(o_free, (cb.k - 1) & 1)) return false;
        tc_fence_after();
        const int st = cb.g % BWD_NST;
        const uint64_t bm = dm0 + (uint64_t)st * TSTEP;
#pragma unroll
        for (int kk = 0; kk < AB / 16; ++kk)
          mma_bf16_ts(t_acc, t_a + kk * 8, bm + kk * 128, IDESC_128x64_KMN, kk > 0 || cb.j > 0);
        mma_commit(acc_done);
        mma_commit(&in_empty[st]);
        advance(cb);
        return true;
      };
      bool ok = true;
      if (ca.valid) ok = issue_st();
      while (ok && cb.valid) {
        if (ca.valid) ok = issue_st();
        if (ok) ok = issue_acc();
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp < 16) {
    // ---------------- elementwise: warps 0-15 ----------------
    const int quarter = warp & 3;
    const int part = warp >> 2;                    // query columns 32 part .. +31
    const int r = quarter * 32 + lane;             // key row within the block
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + DKV_S + 32 * part + lane_off;
    const uint32_t tDP = tbase + DKV_DP + 32 * part + lane_off;
    const uint32_t tP = tbase + DKV_P + 16 * part + lane_off;
    const uint32_t tDS = tbase + DKV_DS + 16 * part + lane_off;
    const float scale2 = LOG2E * 0.125f;
    const float2 sc2 = make_float2(scale2, scale2);
    bool ok = true;
    int g = 0, jb, h, b;
    for (int k = 0; ok && bwd_unit(k, n_units, hb, A.H, jb, h, b); ++k) {
      const int n = nqb - jb;
      for (int j = 0; j < n; ++j, ++g) {
        const int st = g % BWD_NST;
        if (!mbar_wait(st_full, g & 1) || !mbar_wait(&in_full[st], (g / BWD_NST) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[32], dv[32];
        tmem_ld32_async(tS, sv);
        tmem_ld32_async(tDP, dv);
        tmem_wait_regs(sv);
        reg_fence(dv);
        tc_fence_before();
        mbar_arrive(st_free);                      // S^T, dP^T may be overwritten
        if (j == 0) mask_diag_t(sv, 32 * part, r);
        const float* L = sL + st * AB + 32 * part;
        const float* Dv = sD + st * AB + 32 * part;
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = reinterpret_cast<const float4*>(L)[e4];
          const float4 d4 = reinterpret_cast<const float4*>(Dv)[e4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int e = e4 * 4 + u;
            const float2 nl = u ? make_float2(-l4.z * LOG2E, -l4.w * LOG2E)
                                : make_float2(-l4.x * LOG2E, -l4.y * LOG2E);
            const float2 nd = u ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
            const float2 y = __ffma2_rn(u2f2(sv[e], sv[e + 1]), sc2, nl);
            const float2 p = make_float2(ex2(y.x), ex2(y.y));
            const float2 ds = __fmul2_rn(p, __fadd2_rn(u2f2(dv[e], dv[e + 1]), nd));
            pp[e >> 1] = pack_bf16(p.x, p.y);
            pd[e >> 1] = pack_bf16(ds.x, ds.y);
          }
        }
        // P^T and dS^T are free once the previous block's dV, dK products are done
        if (g > 0 && !mbar_wait(acc_done, (g - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tP, pp);
        tmem_st16(tDS, pd);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (!ok) break;
      // unit end: dV and dK (x 1/8) of this CTA's key rows, 16 head columns per warp
      if (!mbar_wait(acc_done, (g - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const size_t row = (size_t)(b * A.S + jb * AB + r) * 3 * d;
      float v[16], w[16];
      tmem_ld16(tbase + DKV_DV + 16 * part + lane_off, v);
      tmem_ld16(tbase + DKV_DK + 16 * part + lane_off, w);
      tc_fence_before();
      mbar_arrive(o_free);
      store16_bf16(A.dqkv + row + 2 * d + h * AD + 16 * part, v, 1.0f);
      store16_bf16(A.dqkv + row + d + h * AD + 16 * part, w, 0.125f);
    }
    if (!ok) fail_wait(A.err, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 16) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ------------------------------------------------------------ dQ
// Unit: query block ib; over the key blocks j = 0 .. ib:
//   S = Q K_j^T, dP = dO V_j^T                          TMEM, fp32
//   dS = 2^(S/8 log2e - LSE log2e) (dP - D)             -> TMEM bf16, two buffers
//   dQ += dS K_j                                        TMEM, fp32
// dQ is scaled by 1/8 when it is written out.  Warps 0-15 elementwise (four
// per TMEM lane quarter, 32 key columns each, as in the dK/dV kernel), warp 16
// TMA, warps 17 and 18 MMA issuers.  dQ is accumulated as two halves over the
// block's keys (keys 0-63 and 64-127, one per issuer, summed when read out):
// two independent chains of four MMAs instead of one chain of eight.
constexpr uint32_t DQ_S = 0, DQ_DP = 128, DQ_DS = 256, DQ_DQ = 384, DQ_DQ2 = 448;
constexpr int DQ_THREADS = 608;
constexpr int DQ_EW = 512;

__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tm_qkv,
                   const __grid_constant__ CUtensorMap tm_do, const AttnArgs A, int nb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm;                          // [2 slots]
  uint8_t* sdO = sQ + 2 * TILE;              // [2 slots]
  uint8_t* sK = sdO + 2 * TILE;              // [BWD_NST]
  uint8_t* sV = sK + BWD_NST * TILE;         // [BWD_NST]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sV + BWD_NST * TILE);
  uint64_t *qd_full = bar, *qd_empty = bar + 2, *kv_full = bar + 4, *kv_empty = kv_full + BWD_NST;
  uint64_t *s_full = kv_empty + BWD_NST, *s_free = s_full + 1, *ds_full = s_full + 2,
           *dq_done = s_full + 4, *o_free = s_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int nqb = A.S / AB;
  const int hb = A.H * nb;
  const int n_units = nqb * hb;
  const int d = A.H * AD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // barriers that both issuers' MMAs complete take one commit from each
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 2);
      mbar_init(&ds_full[i], DQ_EW);
      mbar_init(&dq_done[i], 2);
    }
    for (int i = 0; i < BWD_NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 2);
    }
    mbar_init(s_full, 2);
    mbar_init(s_free, DQ_EW);
    mbar_init(o_free, DQ_EW);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 16) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 16) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      int g = 0, mj, h, b;
      for (int k = 0; ok && bwd_unit(k, n_units, hb, A.H, mj, h, b); ++k) {
        const int ib = nqb - 1 - mj, row0 = b * A.S, slot = k & 1;
        ok = mbar_wait(&qd_empty[slot], ((k >> 1) & 1) ^ 1);
        if (!ok) break;
        mbar_expect_tx(&qd_full[slot], 2 * TILE);
        tma_load_2d(sQ + slot * TILE, &tm_qkv, &qd_full[slot], h * AD, row0 + ib * AB);
        tma_load_2d(sdO + slot * TILE, &tm_do, &qd_full[slot], h * AD, row0 + ib * AB);
        for (int j = 0; j <= ib; ++j, ++g) {
          const int st = g % BWD_NST;
          ok = mbar_wait(&kv_empty[st], ((g / BWD_NST) & 1) ^ 1);
          if (!ok) break;
          mbar_expect_tx(&kv_full[st], 2 * TILE);
          tma_load_2d(sK + st * TILE, &tm_qkv, &kv_full[st], d + h * AD, row0 + j * AB);
          tma_load_2d(sV + st * TILE, &tm_qkv, &kv_full[st], 2 * d + h * AD, row0 + j * AB);
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp == 17 || warp == 18) {
    // ---------------- MMA issuers ----------------
    // Issuer 0 (warp 17): S = Q K_j^T, then dQ_lo += dS[:, 0:64] K_j[0:64];
    // issuer 1 (warp 18): dP = dO V_j^T, then dQ_hi += dS[:, 64:128]
    // K_j[64:128].  Each issues its S-type product of block c + 1 (once the
    // elementwise warps have read block c's S and dP) before its dQ half of
    // block c (once they have written dS of block c).
    if (lane == 0) {
      const int who = warp - 17;
      constexpr uint64_t TSTEP = TILE >> 4;
      const uint64_t da0 = who == 0 ? kdesc(sQ, 0) : kdesc(sdO, 0);   // Q or dO
      const uint64_t db0 = who == 0 ? kdesc(sK, 0) : kdesc(sV, 0);    // K_j or V_j
      const uint64_t mk0 = mndesc(sK, 0);
      const uint32_t t_st = tbase + (who == 0 ? DQ_S : DQ_DP);
      struct Cursor {
        int k, j, g, ib, h, b;
        bool valid;
      };
      auto load_unit = [&](Cursor& c) {
        int mj;
        c.valid = bwd_unit(c.k, n_units, hb, A.H, mj, c.h, c.b);
        c.ib = nqb - 1 - mj;
      };
      auto advance = [&](Cursor& c) {
        ++c.g;
        if (++c.j > c.ib) {
          c.j = 0;
          ++c.k;
          load_unit(c);
        }
      };
      Cursor ca;
      ca.k = ca.j = ca.g = 0;
      load_unit(ca);
      Cursor cb = ca;
      auto issue_st = [&]() -> bool {
        const int st = ca.g % BWD_NST, slot = ca.k & 1;
        if (ca.j == 0 && !mbar_wait(&qd_full[slot], (ca.k >> 1) & 1)) return false;
        if (!mbar_wait(&kv_full[st], (ca.g / BWD_NST) & 1)) return false;
        if (ca.g > 0 && !mbar_wait(s_free, (ca.g - 1) & 1)) return false;
        tc_fence_after();
        const uint64_t a = da0 + (uint64_t)slot * TSTEP, bk = db0 + (uint64_t)st * TSTEP;
#pragma unroll
        for (int kk = 0; kk < AD / 16; ++kk)
          mma_bf16(t_st, a + kk * 2, bk + kk * 2, IDESC_128x128_KK, kk > 0);
        mma_commit(s_full);
        if (ca.j == ca.ib) mma_commit(&qd_empty[slot]);
        advance(ca);
        return true;
      };
      auto issue_dq = [&]() -> bool {
        const int pb = cb.g & 1;
        if (!mbar_wait(&ds_full[pb], (cb.g >> 1) & 1)) return false;
        // dQ is overwritten at a unit's first block: the previous unit's dQ is read out
        if (cb.j == 0 && cb.k > 0 && !mbar_wait(o_free, (cb.k - 1) & 1)) return false;
        tc_fence_after();
        const int st = cb.g % BWD_NST;
        const uint64_t bk = mk0 + (uint64_t)st * TSTEP;
        const int k0 = 4 * who;                    // this issuer's half of the keys
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts(tbase + (who == 0 ? DQ_DQ : DQ_DQ2), tbase + DQ_DS + 64 * pb + (k0 + kk) * 8,
                      bk + (k0 + kk) * 128, IDESC_128x64_KMN, kk > 0 || cb.j > 0);
        mma_commit(&dq_done[pb]);
        mma_commit(&kv_empty[st]);                 // this issuer's use of K_j / V_j is done
        advance(cb);
        return true;
      };
      bool ok = true;
      if (ca.valid) ok = issue_st();
      while (ok && cb.valid) {
        if (ca.valid) ok = issue_st();
        if (ok) ok = issue_dq();
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else if (warp < 16) {
    // ---------------- elementwise: warps 0-15 ----------------
    const int quarter = warp & 3;
    const int part = warp >> 2;                    // key columns 32 part .. +31
    const int r = quarter * 32 + lane;             // query row within the block
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + DQ_S + 32 * part + lane_off;
    const uint32_t tDP = tbase + DQ_DP + 32 * part + lane_off;
    const uint32_t tDS = tbase + DQ_DS + 16 * part + lane_off;
    const float scale2 = LOG2E * 0.125f;
    const float2 sc2 = make_float2(scale2, scale2);
    bool ok = true;
    int g = 0, mj, h, b;
    for (int k = 0; ok && bwd_unit(k, n_units, hb, A.H, mj, h, b); ++k) {
      const int ib = nqb - 1 - mj;
      const size_t lrow = ((size_t)b * A.H + h) * A.S + ib * AB + r;
      const float L2 = A.lse[lrow] * LOG2E, Di = A.dsum[lrow];
      const float2 nl2 = make_float2(-L2, -L2), nd2 = make_float2(-Di, -Di);
      for (int j = 0; j <= ib; ++j, ++g) {
        if (!mbar_wait(s_full, g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[32], dv[32];
        tmem_ld32_async(tS, sv);
        tmem_ld32_async(tDP, dv);
        tmem_wait_regs(sv);
        reg_fence(dv);
        tc_fence_before();
        mbar_arrive(s_free);                       // S, dP may be overwritten
        if (j == ib) mask_diag(sv, 32 * part, r);
        uint32_t pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 y = __ffma2_rn(u2f2(sv[e], sv[e + 1]), sc2, nl2);
          const float2 p = make_float2(ex2(y.x), ex2(y.y));
          const float2 ds = __fmul2_rn(p, __fadd2_rn(u2f2(dv[e], dv[e + 1]), nd2));
          pd[e >> 1] = pack_bf16(ds.x, ds.y);
        }
        // dS[g & 1] was read by the dQ product of block g-2
        const int pb = g & 1;
        if (g >= 2 && !mbar_wait(&dq_done[pb], ((g - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tDS + 64 * pb, pd);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full[pb]);
      }
      if (!ok) break;
      // unit end: dQ x 1/8 of this CTA's query rows, 16 head columns per warp
      const int gl = g - 1;
      if (!mbar_wait(&dq_done[gl & 1], (gl >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[16], w[16];
      tmem_ld16(tbase + DQ_DQ + 16 * part + lane_off, v);
      tmem_ld16(tbase + DQ_DQ2 + 16 * part + lane_off, w);
      tc_fence_before();
      mbar_arrive(o_free);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += w[i];
      store16_bf16(A.dqkv + (size_t)(b * A.S + ib * AB + r) * 3 * d + h * AD + 16 * part, v,
                   0.125f);
    }
    if (!ok) fail_wait(A.err, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 16) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
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
constexpr size_t SMEM_DKDV = 1024 + TILE * (4 + 2 * BWD_NST) + 2 * BWD_NST * AB * 4 + 256;
constexpr size_t SMEM_DQ = 1024 + TILE * (4 + 2 * BWD_NST) + 256;

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
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int units = (S / AB) * H * nb;
  const int grid = units < sms ? units : sms;
  attn_bwd_dkdv_tc<<<grid, DKV_THREADS, SMEM_DKDV, s>>>(mq, mo, a, nb);
  attn_bwd_dq_tc<<<grid, DQ_THREADS, SMEM_DQ, s>>>(mq, mo, a, nb);
  return cudaGetLastError();
}

}  // namespace mg
