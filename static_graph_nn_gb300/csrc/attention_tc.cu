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
// Backward: one CTA per (128-row block, head, sequence), 288 threads.  Warp 0
// lane 0 issues TMA loads and tcgen05.mma; warps 1-8 each own one TMEM lane
// quarter (32 rows of the 128-row block) and one half of the 128 columns, read
// S / dP with tcgen05.ld, do the arithmetic in fp32 and write bf16 P / dS
// tiles into shared memory in the 128-byte-swizzled K-major layout the next
// MMA reads.
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

constexpr size_t SMEM_FWD = 1024 + TILE * (2 + 2 * FWD_NST) + 256 + 4 * AB * 4;
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
  attn_bwd_dkdv_tc<<<dim3(S / AB, H, nb), AT_THREADS, SMEM_DKDV, s>>>(mq, mo, a);
  attn_bwd_dq_tc<<<dim3(S / AB, H, nb), AT_THREADS, SMEM_DQ, s>>>(mq, mo, a);
  return cudaGetLastError();
}

}  // namespace mg
