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
// Forward: persistent, one CTA per SM over (query block, head, sequence)
// units; S, P and O live in tensor memory (P is the A operand of P V, read from
// TMEM) and two softmax groups take alternate key blocks with their own
// running maximum and sum, merged at the end of the unit (see below).
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

// 2^x for two lanes on the FMA and integer pipes, which the special-function
// unit's ex2 leaves idle: 2^x = 2^j 2^f with j = round(x) (adding 1.5 * 2^23
// rounds to an integer and leaves j in the low mantissa bits), f = x - j in
// [-1/2, 1/2], 2^f from a cubic fitted for least maximum relative error by
// Lawson's iteratively reweighted least squares (8.4e-5, below bf16 rounding),
// and j added into the exponent field.  x is clamped below at -125, so keys
// masked with -inf give ~2^-125 instead of 0: nothing at bf16 resolution.
__device__ __forceinline__ float2 ex2_poly2(float2 x) {
  constexpr float RND = 12582912.0f;
  constexpr float C0 = 0.999919593334198f, C1 = 0.6932621598243713f,
                  C2 = 0.24271413683891296f, C3 = 0.055212993174791336f;
  x.x = fmaxf(x.x, -125.0f);
  x.y = fmaxf(x.y, -125.0f);
  const float2 t = __fadd2_rn(x, make_float2(RND, RND));
  const float2 j = __fadd2_rn(t, make_float2(-RND, -RND));
  const float2 f = __ffma2_rn(j, make_float2(-1.0f, -1.0f), x);
  float2 p = __ffma2_rn(make_float2(C3, C3), f, make_float2(C2, C2));
  p = __ffma2_rn(p, f, make_float2(C1, C1));
  p = __ffma2_rn(p, f, make_float2(C0, C0));
  return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(t.x) << 23)),
                     __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(t.y) << 23)));
}

constexpr uint32_t IDESC_128x128_KK = instr_desc(128, 128, 0, 0);
constexpr uint32_t IDESC_128x64_KMN = instr_desc(128, 64, 0, 1);

// ============================================================ forward
// Persistent, one CTA per SM; a work unit is one 128-row query block of one
// (head, sequence), dealt to the CTAs heaviest first in snake order.  Warp 8
// is the TMA producer, warp 9 issues the MMAs, warps 0-7 do the softmax in
// two groups: group p (warps 4p .. 4p+3, one query row per thread) takes the
// key blocks whose running index g has parity p, with its own buffers
//   S[p] = Q K_g^T            TMEM, fp32, 128 columns
//   P[p] = 2^(S/8 log2e - m)  TMEM, bf16 pairs, 64 columns
//   O[p] += P[p] V_g          TMEM, fp32, 64 columns (A operand read from TMEM)
// and its own running maximum m and sum l, so the two groups never wait for
// each other inside a unit (their warps share the SM sub-partitions and fill
// each other's latencies).  At the end of a unit the two partial results are
// merged: M = max(m0, m1), O = (O0 2^(m0-M) + O1 2^(m1-M)) / (l0 2^(m0-M) +
// l1 2^(m1-M)).  m is a reference maximum in log2 units; it is raised, and
// O[p] and l rescaled, only when a block's maximum exceeds it by more than 8,
// so that P <= 2^8.
constexpr int FWD_THREADS = 320;
constexpr int FWD_NST = 3;                                  // K/V ring stages
constexpr uint32_t F_S = 0, F_P = 256, F_O = 384;           // TMEM columns of S[0], P[0], O[0]
constexpr float RESCALE_T = 8.0f;

struct FwdUnit {
  int qb, h, b;   // query block, head, sequence; key blocks 0 .. qb
};

__device__ __forceinline__ bool fwd_unit(int k, int n_units, int nqb, int H, FwdUnit& U) {
  const int G = gridDim.x;
  const int u = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  if (u >= n_units) return false;
  const int hb = n_units / nqb;
  U.qb = nqb - 1 - u / hb;
  U.h = (u % hb) % H;
  U.b = (u % hb) / H;
  return true;
}

// 32 fp32 S values (raw bits) of row r at columns col0.. : keys after the
// query get -inf when the block is the diagonal one.
__device__ __forceinline__ void mask_diag(uint32_t (&v)[32], int col0, int r) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (col0 + e > r) v[e] = 0xff800000u;
}

// Barrier between the two warps that share a TMEM lane quarter (ids 1-4).
__device__ __forceinline__ void pair_sync(int quarter) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
}

__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_tc(const __grid_constant__ CUtensorMap tm_qkv, const AttnArgs A, int nb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm;                          // [2 slots]
  uint8_t* sK = sQ + 2 * TILE;               // [FWD_NST]
  uint8_t* sV = sK + FWD_NST * TILE;         // [FWD_NST]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sV + FWD_NST * TILE);
  uint64_t *q_full = bar, *q_empty = bar + 2, *kv_full = bar + 4, *kv_empty = kv_full + FWD_NST;
  uint64_t *s_full = kv_empty + FWD_NST, *s_free = s_full + 2, *p_full = s_full + 4,
           *o_done = s_full + 6, *o_free = s_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 24);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(bar + 32);    // [m, l][2 groups][128]: unit-end merge
  const int nqb = A.S / AB;
  const int n_units = nqb * A.H * nb;
  const int d = A.H * AD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], NSWT / 2);     // one softmax group
      mbar_init(&p_full[i], NSWT / 2);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(o_free, NSWT);                // both groups
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
      for (int k = 0; ok && fwd_unit(k, n_units, nqb, A.H, U); ++k) {
        const int row0 = U.b * A.S, slot = k & 1;
        ok = mbar_wait(&q_empty[slot], ((k >> 1) & 1) ^ 1);
        if (!ok) break;
        mbar_expect_tx(&q_full[slot], TILE);
        tma_load_2d(sQ + slot * TILE, &tm_qkv, &q_full[slot], U.h * AD, row0 + U.qb * AB);
        for (int j = 0; j <= U.qb; ++j, ++g) {
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
      // descriptors of the first tile of each buffer; a tile further is
      // TILE >> 4 further, a K step 32 bytes (K-major) or 16 rows (V, MN-major)
      constexpr uint64_t TSTEP = TILE >> 4;
      const uint64_t dq0 = kdesc(sQ, 0), dk0 = kdesc(sK, 0), dv0 = mndesc(sV, 0);
      // Two cursors walk the same sequence of (unit, key block): one issues
      // S = Q K^T as soon as the block's K/V and S buffer are ready, the
      // other P V as soon as the block's P is; neither waits on the other's
      // barriers, so the tensor core gets whichever product is ready first.
      struct Cursor {
        int k, j, g;
        FwdUnit U;
        bool valid;
      };
      auto advance = [&](Cursor& c) {
        ++c.g;
        if (++c.j > c.U.qb) {
          c.j = 0;
          ++c.k;
          c.valid = fwd_unit(c.k, n_units, nqb, A.H, c.U);
        }
      };
      Cursor cq, cp;
      cq.k = cq.j = cq.g = 0;
      cq.valid = fwd_unit(0, n_units, nqb, A.H, cq.U);
      cp = cq;
      bool ok = true;
      uint32_t idle = 0;
      while (cp.valid) {
        bool did = false;
        if (cq.valid) {
          const int st = cq.g % FWD_NST, sb = cq.g & 1, slot = cq.k & 1;
          // S[sb] was last read by its group two blocks ago
          if ((cq.j > 0 || mbar_test(&q_full[slot], (cq.k >> 1) & 1)) &&
              mbar_test(&kv_full[st], (cq.g / FWD_NST) & 1) &&
              (cq.g < 2 || mbar_test(&s_free[sb], ((cq.g - 2) >> 1) & 1))) {
            tc_fence_after();
            const uint64_t aq = dq0 + (uint64_t)slot * TSTEP;
            const uint64_t bk = dk0 + (uint64_t)st * TSTEP;
#pragma unroll
            for (int kk = 0; kk < AD / 16; ++kk)
              mma_bf16(tbase + F_S + 128 * sb, aq + kk * 2, bk + kk * 2, IDESC_128x128_KK, kk > 0);
            mma_commit(&s_full[sb]);
            if (cq.j == cq.U.qb) mma_commit(&q_empty[slot]);
            advance(cq);
            did = true;
          }
        }
        if (cp.g < cq.g) {
          const int pb = cp.g & 1;
          // a unit's first product overwrites O: the previous unit's O is read out
          if (mbar_test(&p_full[pb], (cp.g >> 1) & 1) &&
              (cp.j != 0 || cp.k == 0 || mbar_test(o_free, (cp.k - 1) & 1))) {
            tc_fence_after();
            const int st = cp.g % FWD_NST;
            const uint64_t bv = dv0 + (uint64_t)st * TSTEP;
#pragma unroll
            for (int kk = 0; kk < AB / 16; ++kk)
              mma_bf16_ts(tbase + F_O + 64 * pb, tbase + F_P + 64 * pb + kk * 8, bv + kk * 128,
                          IDESC_128x64_KMN, kk > 0 || cp.j >= 2);
            mma_commit(&o_done[pb]);
            mma_commit(&kv_empty[st]);
            advance(cp);
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (++idle > kWaitLimit) {
          ok = false;
          break;
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    // ---------------- softmax: two groups of four warps ----------------
    const int quarter = warp & 3;
    const int grp = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + F_S + 128 * grp + lane_off;
    const uint32_t tP = tbase + F_P + 64 * grp + lane_off;
    const uint32_t tO = tbase + F_O + 64 * grp + lane_off;
    const float scale2 = LOG2E * 0.125f;      // log2(e) / sqrt(64)
    bool ok = true;
    int g0 = 0;                               // running index of the unit's first block
    FwdUnit U;
    // Both groups pass the unit-end barrier, also after a failed wait, so
    // that a timeout never leaves the partner warp blocked there.
    for (int k = 0; fwd_unit(k, n_units, nqb, A.H, U); ++k) {
      const int n = U.qb + 1;
      float m = -INFINITY, l = 0.0f;
      int last = -1;                          // running index of this group's last block
      for (int j = (grp - g0) & 1; ok && j < n; j += 2) {
        const int gi = g0 + j;
        if (!mbar_wait(&s_full[grp], (gi >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the whole 128-column row of S in registers, then S[grp] is released
        uint32_t sv[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32_async(tS + 32 * ch, sv[ch]);
        tmem_wait_regs(sv[0]);
        reg_fence(sv[1]);
        reg_fence(sv[2]);
        reg_fence(sv[3]);
        tc_fence_before();
        mbar_arrive(&s_free[grp]);
        if (j == U.qb) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) mask_diag(sv[ch], 32 * ch, r);
        }
        float pm[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pm[e] = __uint_as_float(sv[0][e]);
#pragma unroll
        for (int e = 8; e < 128; ++e) pm[e & 7] = fmaxf(pm[e & 7], __uint_as_float(sv[e >> 5][e & 31]));
        const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                               fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * scale2;
        const bool need = mx > m + RESCALE_T;
        const float m_new = need ? mx : m;
        const float alpha = need ? exp2f(m - m_new) : 1.0f;
        // P[grp] and O[grp] are free once this group's previous P V is done
        if (gi >= 2 && !mbar_wait(&o_done[grp], ((gi - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float2 sc2 = make_float2(scale2, scale2), nm2 = make_float2(-m_new, -m_new);
        float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 y = __ffma2_rn(u2f2(sv[ch][e], sv[ch][e + 1]), sc2, nm2);
            // one pair in four on the FMA pipe, the rest on the SFU
            const float2 pe = ((e >> 1) & 3) == 3 ? ex2_poly2(y) : make_float2(ex2(y.x), ex2(y.y));
            ls[(e >> 1) & 1] = __fadd2_rn(ls[(e >> 1) & 1], pe);
            __nv_bfloat162 hv = __floats2bfloat162_rn(pe.x, pe.y);
            pk[e >> 1] = *reinterpret_cast<uint32_t*>(&hv);
          }
          tmem_st16(tP + 16 * ch, pk);
        }
        // O[grp] = O[grp] * alpha for the rows whose reference maximum moved
        if (last >= 0 && __any_sync(0xffffffffu, need)) {
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
        mbar_arrive(&p_full[grp]);
        const float2 lsp = __fadd2_rn(ls[0], ls[1]);
        l = l * alpha + (lsp.x + lsp.y);
        m = m_new;
        last = gi;
      }
      // unit end: this group's O is complete once its last P V is done
      if (ok && last >= 0) ok = mbar_wait(&o_done[grp], (last >> 1) & 1);
      xch[grp * AB + r] = m;
      xch[(2 + grp) * AB + r] = l;
      tc_fence_before();
      pair_sync(quarter);
      if (ok) {
        tc_fence_after();
        // group p had blocks in this unit unless the unit's only block went to the other
        const bool has0 = n >= 2 || (g0 & 1) == 0, has1 = n >= 2 || (g0 & 1) == 1;
        const float m0 = xch[r], m1 = xch[AB + r];
        const float M = fmaxf(has0 ? m0 : -INFINITY, has1 ? m1 : -INFINITY);
        const float w0 = has0 ? exp2f(m0 - M) : 0.0f, w1 = has1 ? exp2f(m1 - M) : 0.0f;
        const float L = (has0 ? xch[2 * AB + r] * w0 : 0.0f) + (has1 ? xch[3 * AB + r] * w1 : 0.0f);
        // this thread writes head dimensions 32 grp .. +31 of its row
        float o[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.0f;
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          if (!(p2 ? has1 : has0)) continue;
          float ov[32];
          tmem_ld32(tbase + F_O + 64 * p2 + 32 * grp + lane_off, ov);
          const float wp = p2 ? w1 : w0;
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = fmaf(ov[e], wp, o[e]);
        }
        const int qi = U.qb * AB + r;
        store8_bf16_row(A.o + (size_t)(U.b * A.S + qi) * d + U.h * AD + 32 * grp, o, 1.0f / L);
        if (grp == 0) A.lse[((size_t)U.b * A.H + U.h) * A.S + qi] = (M + log2f(L)) / LOG2E;
        tc_fence_before();
      }
      // xch is rewritten at the next unit's end only after both warps passed
      // this point (the next pair_sync orders it)
      pair_sync(quarter);
      mbar_arrive(o_free);
      g0 += n;
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
// warp 8 the TMA producer, warp 9 an event-driven MMA issuer, warps 0-7 the
// elementwise work (warp w: TMEM lane quarter w & 3, columns 64 (w >> 2) ..
// +63), S and dP read from TMEM once and released, and the bf16 products P /
// dS written back into TMEM as the A operand of the accumulating MMAs.
constexpr int BWD_THREADS = 320;
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

// Four 32-column TMEM loads of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld4x32(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3,
                                            uint32_t (&a)[32], uint32_t (&b)[32],
                                            uint32_t (&c)[32], uint32_t (&e)[32]) {
  tmem_ld32_async(t0, a);
  tmem_ld32_async(t1, b);
  tmem_ld32_async(t2, c);
  tmem_ld32_async(t3, e);
  tmem_wait_regs(a);
  reg_fence(b);
  reg_fence(c);
  reg_fence(e);
}

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&hv);
}

// ------------------------------------------------------------ dK / dV
// Unit: key block jb; over the query blocks i = jb .. nqb-1 (keys are the M
// dimension, so every product is a row-major one for this CTA's key rows):
//   S^T = K Q_i^T, dP^T = V dO_i^T                      TMEM, fp32
//   P^T = 2^(S^T/8 log2e - LSE_i log2e), dS^T = P^T (dP^T - D_i)  -> TMEM bf16
//   dV += P^T dO_i, dK += dS^T Q_i                      TMEM, fp32
// dK is scaled by 1/8 when it is written out.
constexpr uint32_t DKV_S = 0, DKV_DP = 128, DKV_P = 256, DKV_DS = 320, DKV_DV = 384, DKV_DK = 448;

__global__ void __launch_bounds__(BWD_THREADS, 1)
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < BWD_NST; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 1);
    }
    mbar_init(st_full, 1);
    mbar_init(st_free, NSWT);
    mbar_init(ds_full, NSWT);
    mbar_init(acc_done, 1);
    mbar_init(o_free, NSWT);
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
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint64_t TSTEP = TILE >> 4;
      const uint64_t dk0 = kdesc(sK, 0), dv0 = kdesc(sV, 0), dq0 = kdesc(sQ, 0),
                     ddo0 = kdesc(sdO, 0), mq0 = mndesc(sQ, 0), mdo0 = mndesc(sdO, 0);
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
      bool ok = true;
      uint32_t idle = 0;
      while (cb.valid) {
        bool did = false;
        if (ca.valid) {
          const int st = ca.g % BWD_NST, slot = ca.k & 1;
          if ((ca.j > 0 || mbar_test(&kv_full[slot], (ca.k >> 1) & 1)) &&
              mbar_test(&in_full[st], (ca.g / BWD_NST) & 1) &&
              (ca.g == 0 || mbar_test(st_free, (ca.g - 1) & 1))) {
            tc_fence_after();
            const uint64_t ak = dk0 + (uint64_t)slot * TSTEP, av = dv0 + (uint64_t)slot * TSTEP;
            const uint64_t bq = dq0 + (uint64_t)st * TSTEP, bo = ddo0 + (uint64_t)st * TSTEP;
#pragma unroll
            for (int kk = 0; kk < AD / 16; ++kk)
              mma_bf16(tbase + DKV_S, ak + kk * 2, bq + kk * 2, IDESC_128x128_KK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < AD / 16; ++kk)
              mma_bf16(tbase + DKV_DP, av + kk * 2, bo + kk * 2, IDESC_128x128_KK, kk > 0);
            mma_commit(st_full);
            if (ca.j == nqb - ca.jb - 1) mma_commit(&kv_empty[slot]);
            advance(ca);
            did = true;
          }
        }
        if (cb.g < ca.g) {
          // dV and dK overwrite their accumulators at a unit's first block:
          // the previous unit's results are read out
          if (mbar_test(ds_full, cb.g & 1) &&
              (cb.j != 0 || cb.k == 0 || mbar_test(o_free, (cb.k - 1) & 1))) {
            tc_fence_after();
            const int st = cb.g % BWD_NST;
            const uint64_t bo = mdo0 + (uint64_t)st * TSTEP, bq = mq0 + (uint64_t)st * TSTEP;
#pragma unroll
            for (int kk = 0; kk < AB / 16; ++kk)
              mma_bf16_ts(tbase + DKV_DV, tbase + DKV_P + kk * 8, bo + kk * 128, IDESC_128x64_KMN,
                          kk > 0 || cb.j > 0);
#pragma unroll
            for (int kk = 0; kk < AB / 16; ++kk)
              mma_bf16_ts(tbase + DKV_DK, tbase + DKV_DS + kk * 8, bq + kk * 128, IDESC_128x64_KMN,
                          kk > 0 || cb.j > 0);
            mma_commit(acc_done);
            mma_commit(&in_empty[st]);
            advance(cb);
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (++idle > kWaitLimit) {
          ok = false;
          break;
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    // ---------------- elementwise: warps 0-7 ----------------
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int r = quarter * 32 + lane;             // key row within the block
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + DKV_S + 64 * half + lane_off;
    const uint32_t tDP = tbase + DKV_DP + 64 * half + lane_off;
    const uint32_t tP = tbase + DKV_P + 32 * half + lane_off;
    const uint32_t tDS = tbase + DKV_DS + 32 * half + lane_off;
    const float scale2 = LOG2E * 0.125f;
    const float2 sc2 = make_float2(scale2, scale2), nlog2 = make_float2(-LOG2E, -LOG2E);
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
        uint32_t sv[2][32], dv[2][32];
        tmem_ld4x32(tS, tS + 32, tDP, tDP + 32, sv[0], sv[1], dv[0], dv[1]);
        tc_fence_before();
        mbar_arrive(st_free);                      // S^T, dP^T may be overwritten
        if (j == 0) {
          mask_diag_t(sv[0], 64 * half, r);
          mask_diag_t(sv[1], 64 * half + 32, r);
        }
        const float* L = sL + st * AB + 64 * half;
        const float* Dv = sD + st * AB + 64 * half;
        uint32_t pp[2][16], pd[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 l4 = reinterpret_cast<const float4*>(L + 32 * c)[e4];
            const float4 d4 = reinterpret_cast<const float4*>(Dv + 32 * c)[e4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              const int e = e4 * 4 + u;
              const float2 l2 = u ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
              const float2 d2 = u ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
              const float2 y = __ffma2_rn(u2f2(sv[c][e], sv[c][e + 1]), sc2, __fmul2_rn(l2, nlog2));
              const float2 p = ((e >> 1) & 3) == 3 ? ex2_poly2(y) : make_float2(ex2(y.x), ex2(y.y));
              const float2 ds = __fmul2_rn(p, __fadd2_rn(u2f2(dv[c][e], dv[c][e + 1]), d2));
              pp[c][e >> 1] = pack_bf16(p.x, p.y);
              pd[c][e >> 1] = pack_bf16(ds.x, ds.y);
            }
          }
        }
        // P^T and dS^T are free once the previous block's dV, dK products are done
        if (g > 0 && !mbar_wait(acc_done, (g - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tP, pp[0]);
        tmem_st16(tP + 16, pp[1]);
        tmem_st16(tDS, pd[0]);
        tmem_st16(tDS + 16, pd[1]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (!ok) break;
      // unit end: dV and dK (x 1/8) of this CTA's key rows
      if (!mbar_wait(acc_done, (g - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const size_t row = (size_t)(b * A.S + jb * AB + r) * 3 * d;
      float v[32];
      tmem_ld32(tbase + DKV_DV + 32 * half + lane_off, v);
      store8_bf16_row(A.dqkv + row + 2 * d + h * AD + 32 * half, v, 1.0f);
      tmem_ld32(tbase + DKV_DK + 32 * half + lane_off, v);
      store8_bf16_row(A.dqkv + row + d + h * AD + 32 * half, v, 0.125f);
      tc_fence_before();
      mbar_arrive(o_free);
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

// ------------------------------------------------------------ dQ
// Unit: query block ib; over the key blocks j = 0 .. ib:
//   S = Q K_j^T, dP = dO V_j^T                          TMEM, fp32
//   dS = 2^(S/8 log2e - LSE log2e) (dP - D)             -> TMEM bf16, two buffers
//   dQ += dS K_j                                        TMEM, fp32
// dQ is scaled by 1/8 when it is written out.
constexpr uint32_t DQ_S = 0, DQ_DP = 128, DQ_DS = 256, DQ_DQ = 384;

__global__ void __launch_bounds__(BWD_THREADS, 1)
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
      mbar_init(&ds_full[i], NSWT);
      mbar_init(&dq_done[i], 1);
    }
    for (int i = 0; i < BWD_NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, NSWT);
    mbar_init(o_free, NSWT);
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
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint64_t TSTEP = TILE >> 4;
      const uint64_t dq0 = kdesc(sQ, 0), ddo0 = kdesc(sdO, 0), dk0 = kdesc(sK, 0),
                     dv0 = kdesc(sV, 0), mk0 = mndesc(sK, 0);
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
      bool ok = true;
      uint32_t idle = 0;
      while (cb.valid) {
        bool did = false;
        if (ca.valid) {
          const int st = ca.g % BWD_NST, slot = ca.k & 1;
          if ((ca.j > 0 || mbar_test(&qd_full[slot], (ca.k >> 1) & 1)) &&
              mbar_test(&kv_full[st], (ca.g / BWD_NST) & 1) &&
              (ca.g == 0 || mbar_test(s_free, (ca.g - 1) & 1))) {
            tc_fence_after();
            const uint64_t aq = dq0 + (uint64_t)slot * TSTEP, ao = ddo0 + (uint64_t)slot * TSTEP;
            const uint64_t bk = dk0 + (uint64_t)st * TSTEP, bv = dv0 + (uint64_t)st * TSTEP;
#pragma unroll
            for (int kk = 0; kk < AD / 16; ++kk)
              mma_bf16(tbase + DQ_S, aq + kk * 2, bk + kk * 2, IDESC_128x128_KK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < AD / 16; ++kk)
              mma_bf16(tbase + DQ_DP, ao + kk * 2, bv + kk * 2, IDESC_128x128_KK, kk > 0);
            mma_commit(s_full);
            if (ca.j == ca.ib) mma_commit(&qd_empty[slot]);
            advance(ca);
            did = true;
          }
        }
        if (cb.g < ca.g) {
          const int pb = cb.g & 1;
          // dQ is overwritten at a unit's first block: the previous unit's dQ is read out
          if (mbar_test(&ds_full[pb], (cb.g >> 1) & 1) &&
              (cb.j != 0 || cb.k == 0 || mbar_test(o_free, (cb.k - 1) & 1))) {
            tc_fence_after();
            const int st = cb.g % BWD_NST;
            const uint64_t bk = mk0 + (uint64_t)st * TSTEP;
#pragma unroll
            for (int kk = 0; kk < AB / 16; ++kk)
              mma_bf16_ts(tbase + DQ_DQ, tbase + DQ_DS + 64 * pb + kk * 8, bk + kk * 128,
                          IDESC_128x64_KMN, kk > 0 || cb.j > 0);
            mma_commit(&dq_done[pb]);
            mma_commit(&kv_empty[st]);
            advance(cb);
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (++idle > kWaitLimit) {
          ok = false;
          break;
        }
      }
      if (!ok) fail_wait(A.err, abort_flag);
    }
  } else {
    // ---------------- elementwise: warps 0-7 ----------------
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int r = quarter * 32 + lane;             // query row within the block
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + DQ_S + 64 * half + lane_off;
    const uint32_t tDP = tbase + DQ_DP + 64 * half + lane_off;
    const uint32_t tDS = tbase + DQ_DS + 32 * half + lane_off;
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
        uint32_t sv[2][32], dv[2][32];
        tmem_ld4x32(tS, tS + 32, tDP, tDP + 32, sv[0], sv[1], dv[0], dv[1]);
        tc_fence_before();
        mbar_arrive(s_free);                       // S, dP may be overwritten
        if (j == ib) {
          mask_diag(sv[0], 64 * half, r);
          mask_diag(sv[1], 64 * half + 32, r);
        }
        uint32_t pd[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 y = __ffma2_rn(u2f2(sv[c][e], sv[c][e + 1]), sc2, nl2);
            const float2 p = ((e >> 1) & 3) == 3 ? ex2_poly2(y) : make_float2(ex2(y.x), ex2(y.y));
            const float2 ds = __fmul2_rn(p, __fadd2_rn(u2f2(dv[c][e], dv[c][e + 1]), nd2));
            pd[c][e >> 1] = pack_bf16(ds.x, ds.y);
          }
        }
        // dS[g & 1] was read by the dQ product of block g-2
        const int pb = g & 1;
        if (g >= 2 && !mbar_wait(&dq_done[pb], ((g - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tDS + 64 * pb, pd[0]);
        tmem_st16(tDS + 64 * pb + 16, pd[1]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full[pb]);
      }
      if (!ok) break;
      // unit end: dQ x 1/8 of this CTA's query rows
      const int gl = g - 1;
      if (!mbar_wait(&dq_done[gl & 1], (gl >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[32];
      tmem_ld32(tbase + DQ_DQ + 32 * half + lane_off, v);
      store8_bf16_row(A.dqkv + (size_t)(b * A.S + ib * AB + r) * 3 * d + h * AD + 32 * half, v,
                      0.125f);
      tc_fence_before();
      mbar_arrive(o_free);
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

constexpr size_t SMEM_FWD = 1024 + TILE * (2 + 2 * FWD_NST) + 256 + 4 * AB * 4;
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
  const int units = (S / AB) * H * nb;
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
  attn_bwd_dkdv_tc<<<grid, BWD_THREADS, SMEM_DKDV, s>>>(mq, mo, a, nb);
  attn_bwd_dq_tc<<<grid, BWD_THREADS, SMEM_DQ, s>>>(mq, mo, a, nb);
  return cudaGetLastError();
}

}  // namespace mg
