// predict_max.cu — max-pooled block scores of the low-rank predictor.
//
// DSV page [nl], "Technische samenvatting" 2A (low-rank predictors W^Q_lr,
// W^K_lr whose logits approximate Q K^T) and 2B (one proxy per query group).
// The pages leave open how a (group, key block) tile of logits is reduced to
// one score; predict.cu takes the mean, this file the largest logit:
//   S[g, j] = max over i in group g, l in key block j of (Q_i W^Q) . (K_l W^K).
// A maximum does not commute with pooling, so every token is projected and
// every tile of logits is formed: an [N, N] x r contraction per (b, h), run
// on the tensor cores.
//
// Kernel 1 projects one 128-token tile of Q (or K) of one (b, h) per CTA to
// rank r in fp32 (the head's W staged in shared memory) and splits each value
// into two bf16 parts, v = hi + lo with |v - hi - lo| <= 2^-18 |v|.  Then
//   q . k = hi_q.hi_k + hi_q.lo_k + lo_q.hi_k   (each term off by ~2^-16 of |q_c k_c|)
// is ONE bf16 contraction over K = 3r: query rows are stored as [hi | hi | lo]
// and key rows as [hi | lo | hi], zero-padded to a multiple of 16, in the
// tensor core's K-major layout without swizzle (8-row x 8-element core
// matrices of 128 contiguous bytes), one 128-token tile after another.
//
// Kernel 2: persistent CTAs; a CTA takes four (for r > 48: two) 128-token
// query tiles of a (b, h) at a time against a run of key tiles.  Warp 0
// copies the query tiles and the key tiles through a ring (plain bulk copies:
// the workspace already holds the MMA layout), warp 1 issues one M=128, N=128, K=3r product (tcgen05,
// fp32 accumulation) per (query tile, key tile) into one of four TMEM
// accumulators, and warps 2-9, two groups of four taking alternate products,
// read each accumulator back (one warp per TMEM lane quarter), take the
// maximum of every block x block sub-tile and write the scores.  The three-input max.f32 used drops a NaN
// logit, as fmaxf does.
#include <cuda_bf16.h>
#include <limits.h>

#include "dsv_launch.h"

namespace dsv {
namespace {

constexpr int kTile = 128;               // tokens per MMA tile (M = N = 128)

// Workspace layout of one tensor's split rows.
template <int R>
struct MaxLayout {
  static constexpr int KP = (3 * R + 15) / 16 * 16;   // contraction length, padded to the MMA's K = 16
  static constexpr int KSTEPS = KP / 16;
  static constexpr int LBO = 128;                     // bytes between core matrices along K
  static constexpr int SBO = KP * 16;                 // bytes between 8-row groups
  static constexpr int TILE_BYTES = kTile * KP * 2;
  // byte offset of (row i of a tile, element e of the row)
  __host__ __device__ static constexpr int offset(int i, int e) {
    return (i >> 3) * SBO + (e >> 3) * 128 + (i & 7) * 16 + (e & 7) * 2;
  }
};

// grid (B*H*NT, 2), 128 threads: one 128-token tile per CTA, one token row per
// thread.  blockIdx.y = 0 projects Q with W^Q and writes [hi | hi | lo], 1
// projects K with W^K and writes [hi | lo | hi].  The head's W sits in shared
// memory as pairs (W[2m][c], W[2m+1][c]), so that a thread's row (in
// registers, bf16 pairs) meets it with packed two-lane FMAs; the two lanes of
// each sum are added at the end.  Rows past N (the last tile when
// N % 128 == 64) are written as zeros.
template <int D, int R>
__global__ void __launch_bounds__(kTile) lowrank_split_kernel(const __nv_bfloat16* __restrict__ Q,
                                                              const __nv_bfloat16* __restrict__ K,
                                                              const float* __restrict__ Wq,
                                                              const float* __restrict__ Wk, int H, int N, int NT,
                                                              uint8_t* __restrict__ qt, uint8_t* __restrict__ kt) {
  using L = MaxLayout<R>;
  extern __shared__ float4 sm4[];
  float2* w2 = reinterpret_cast<float2*>(sm4);  // [D/2][R]: (W[2m][c], W[2m+1][c])
  const int t = threadIdx.x;
  const int which = blockIdx.y;
  const long long tile = blockIdx.x;            // (b*H + h) * NT + tile index
  const long long bh = tile / NT;
  const int n = (int)(tile - bh * NT) * kTile + t;
  const float* W = (which ? Wk : Wq) + (bh % H) * (long long)D * R;
  for (int i = t; i < D * R / 2; i += kTile) {
    const int m = i / R, c = i - m * R;
    w2[i] = make_float2(__ldg(W + (2 * m) * R + c), __ldg(W + (2 * m + 1) * R + c));
  }
  __syncthreads();
  uint8_t* out = (which ? kt : qt) + tile * (long long)L::TILE_BYTES;
  // outputs per pass (bounds the accumulator registers); divides R, so that a
  // pass never reads W or writes pieces past column R
  constexpr int RH = R % 16 == 0 ? 16 : 8;
  static_assert(R % RH == 0 && RH % 8 == 0, "pass width must divide R");
  if (n < N) {
    // the whole row first (16 loads in flight), then the products, RH outputs at a time
    const uint4* X = reinterpret_cast<const uint4*>((which ? K : Q) + (bh * N + n) * D);
    uint32_t xw[D / 2];
#pragma unroll
    for (int q = 0; q < D / 8; ++q) {
      const uint4 v = __ldg(X + q);
      xw[4 * q] = v.x;
      xw[4 * q + 1] = v.y;
      xw[4 * q + 2] = v.z;
      xw[4 * q + 3] = v.w;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < R; c0 += RH) {
      uint64_t acc[RH];
#pragma unroll
      for (int c = 0; c < RH; ++c) acc[c] = 0ull;
#pragma unroll
      for (int m = 0; m < D / 2; ++m) {
        const uint64_t xp = f2_pack(__uint_as_float(xw[m] << 16), __uint_as_float(xw[m] & 0xFFFF0000u));
        const float4* wr = reinterpret_cast<const float4*>(w2 + m * R + c0);
#pragma unroll
        for (int c = 0; c < RH; c += 2) {
          const float4 ww = wr[c / 2];
          acc[c] = fma2(xp, f2_pack(ww.x, ww.y), acc[c]);
          acc[c + 1] = fma2(xp, f2_pack(ww.z, ww.w), acc[c + 1]);
        }
      }
      float v[RH], vl[RH];                        // the values and their low bf16 parts
#pragma unroll
      for (int c = 0; c < RH; ++c) {
        float lo, hi;
        f2_unpack(acc[c], lo, hi);
        v[c] = lo + hi;
        vl[c] = v[c] - __bfloat162float(__float2bfloat16_rn(v[c]));
      }
      // 16-byte pieces of the three parts: Q rows [hi | hi | lo], K rows [hi | lo | hi]
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const float* src = (which ? (part == 1) : (part == 2)) ? vl : v;
#pragma unroll
        for (int pc = 0; pc < RH; pc += 8) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) w4[e] = pack_bf16x2(src[pc + 2 * e], src[pc + 2 * e + 1]);
          *reinterpret_cast<uint4*>(out + L::offset(t, part * R + c0 + pc)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    }
#pragma unroll
    for (int e0 = 3 * R; e0 < L::KP; e0 += 8)
      *reinterpret_cast<uint4*>(out + L::offset(t, e0)) = make_uint4(0u, 0u, 0u, 0u);
  } else {
#pragma unroll
    for (int e0 = 0; e0 < L::KP; e0 += 8)
      *reinterpret_cast<uint4*>(out + L::offset(t, e0)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int R>
struct MaxTraits {
  using L = MaxLayout<R>;
  static constexpr int TB = L::TILE_BYTES;
  // key tiles per product: two (N = 256) for r <= 32 (at most six MMAs a
  // product), so that the hand-over around each product (barrier round trips,
  // the accumulator read-back) is paid once per 256 keys
  static constexpr int KT = L::KSTEPS <= 6 ? 2 : 1;
  static constexpr int NACC = 4 / KT;                            // TMEM accumulators of 128 * KT columns
  static constexpr int CG = 2 * KT;                              // 64-column groups of a product
  static constexpr int SB = KT * TB;                             // bytes of one key step (KT tiles)
  static constexpr int ZC = 8;                                   // key steps per cross-warp combine
  static constexpr int MISC = 8192;                              // barriers, partial maxima, slots
  // query tiles per CTA: 4 where they and a two-stage key ring fit (each key
  // step copied to shared memory then serves 4 products), else 2
  static constexpr int NQ = 4 * TB + 2 * SB + 1024 + MISC <= 227 * 1024 ? 4 : 2;
  static constexpr int RING_ROOM = 227 * 1024 - 1024 - NQ * TB - MISC;
  static constexpr int NSTAGE = RING_ROOM / SB >= 4 ? 4 : RING_ROOM / SB;
  static constexpr int SMEM_USED = 1024 + NQ * TB + NSTAGE * SB + MISC;
  // at least 120 KB, so that one CTA holds an SM (and its whole TMEM)
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static_assert(NSTAGE >= 2, "tile too large for a two-stage ring");
  static_assert(2 * ZC * NQ * 4 * CG * 4 + (1 + 2 * NSTAGE + 2 * NACC + 1) * 8 + 16 <= MISC, "misc area");
  static_assert(ZC * NQ * 4 * KT <= 256, "one combined score per reduction thread");
};

constexpr int kMaxThreads = 320;         // producer, MMA, two groups of 4 reduction warps

enum : unsigned int { MW_A = 1, MW_BFULL, MW_BEMPTY, MW_TFULL, MW_TEMPTY, MW_DRAIN };

// Order-preserving map of a non-NaN float to a signed integer (and back):
// negative values have their magnitude bits flipped.
__device__ __forceinline__ int float_key(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : b ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float key_float(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF); }

// Work is a sequence of steps w = ((b*H + h) * NG + tg) * NS + c: query-tile
// group tg (NQ query tiles from tg*NQ) of head (b, h) against key step c (key
// tiles KT*c .. KT*c + KT - 1; the workspace holds NTP = NS * KT tiles per
// head, the ones past N zero).  Persistent CTAs, one per SM, each take one
// contiguous range of steps of equal length (so no wave is left partly
// empty), reloading the query tiles when the range crosses into the next
// group.
struct MaxStep {
  long long bh;
  int tq0, nq, c;
  long long item;
};
template <int NQ>
__device__ __forceinline__ MaxStep max_step(long long w, int NT, int NS) {
  const int NG = (NT + NQ - 1) / NQ;
  MaxStep st;
  st.item = w / NS;
  st.c = (int)(w - st.item * NS);
  st.bh = st.item / NG;
  st.tq0 = (int)(st.item - st.bh * NG) * NQ;
  st.nq = NT - st.tq0 < NQ ? NT - st.tq0 : NQ;
  return st;
}

template <int BLOCK, int R>
__global__ void __launch_bounds__(kMaxThreads, 1)
    tile_max_mma_kernel(const uint8_t* __restrict__ qt, const uint8_t* __restrict__ kt, int NT, int NS, int G,
                        long long steps, float* __restrict__ S, Ctl ctl) {
  using T = MaxTraits<R>;
  using L = typename T::L;
  constexpr int TB = T::TB, SB = T::SB, KT = T::KT, NACC = T::NACC, CG = T::CG;
  constexpr int NSTAGE = T::NSTAGE, NQ = T::NQ;
  constexpr int NTP_PER_STEP = KT;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sA = smem_align1024(smem_raw);        // NQ query tiles
  uint8_t* sB = sA + NQ * TB;                     // NSTAGE key steps
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + NSTAGE * SB);
  uint64_t* a_full = bars;
  uint64_t* a_free = bars + 1;                    // the products on the current query tiles are done
  uint64_t* b_full = bars + 2;
  uint64_t* b_empty = b_full + NSTAGE;
  uint64_t* t_full = b_empty + NSTAGE;            // [NACC]
  uint64_t* t_empty = t_full + NACC;              // [NACC]
  uint64_t* drain = t_empty + NACC;
  int* part = reinterpret_cast<int*>(drain + 1);  // [2][ZC][NQ][4 quarters][CG], ordered keys
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(part + 2 * T::ZC * NQ * 4 * CG);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long w0 = steps * blockIdx.x / gridDim.x, w1 = steps * (blockIdx.x + 1) / gridDim.x;
  const long long NTP = (long long)NS * NTP_PER_STEP;   // tiles per head in the workspace
  const unsigned int kid = (unsigned int)KID_MAXPOOL << 8;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_free, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&t_full[a], 1);
      mbar_init(&t_empty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- copies ----------------
      long long cur = -1;
      int a_loads = 0;
      long long issued = 0;
      for (long long w = w0; w < w1; ++w) {
        const long long k = w - w0;
        const MaxStep st = max_step<NQ>(w, NT, NS);
        if (st.item != cur) {
          // the query tiles are overwritten once every product reading them is done
          if (a_loads > 0 &&
              !mbar_wait(a_free, (uint32_t)(a_loads - 1) & 1u, abort_flag, ctl, kid | MW_A))
            break;
          mbar_arrive_expect_tx(a_full, (uint32_t)(st.nq * TB));
          for (int rt = 0; rt < st.nq; ++rt)
            bulk_load(sA + rt * TB, qt + (st.bh * NTP + st.tq0 + rt) * (long long)TB, TB, a_full);
          ++a_loads;
          cur = st.item;
        }
        const int s = (int)(k % NSTAGE);
        if (!mbar_wait(&b_empty[s], ((uint32_t)(k / NSTAGE) & 1u) ^ 1u, abort_flag, ctl, kid | MW_BEMPTY)) break;
        mbar_arrive_expect_tx(&b_full[s], SB);
        bulk_load(sB + s * SB, kt + (st.bh * NTP + (long long)st.c * KT) * (long long)TB, SB, &b_full[s]);
        issued = k + 1;
      }
      // every copy started must land before the CTA exits
      if (a_loads > 0) mbar_wait(a_full, (uint32_t)(a_loads - 1) & 1u, nullptr, ctl, kid | MW_DRAIN);
      for (long long k = (issued > NSTAGE ? issued - NSTAGE : 0); k < issued; ++k)
        mbar_wait(&b_full[k % NSTAGE], (uint32_t)(k / NSTAGE) & 1u, nullptr, ctl, kid | MW_DRAIN);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The next key step's barrier and the next product's accumulator are
    // tested one step early; a wait whose test found the phase complete is
    // free.
    constexpr uint32_t ID = idesc_bf16_f32(kTile, kTile * KT, false, false);
    const uint64_t a0 = sdesc_noswz(smem_u32(sA), L::LBO, L::SBO);
    const uint64_t b0 = sdesc_noswz(smem_u32(sB), L::LBO, L::SBO);
    long long cur = -1;
    int a_uses = 0;
    long long p = 0;                                // product number: accumulator p % NACC, its use p / NACC
    bool ok = true;
    uint32_t tb = 0u, te = 1u;                      // product 0's accumulator is free
    for (long long w = w0; ok && w < w1; ++w) {
      const long long k = w - w0;
      const MaxStep st = max_step<NQ>(w, NT, NS);
      if (st.item != cur) {
        if (a_uses > 0) mma_commit_w(a_free);
        if (!mbar_wait_warp(a_full, (uint32_t)a_uses & 1u, abort_flag, ctl, kid | MW_A)) break;
        ++a_uses;
        cur = st.item;
      }
      const int s = (int)(k % NSTAGE);
      if (!mbar_wait_warp_tested(&b_full[s], (uint32_t)(k / NSTAGE) & 1u, tb, abort_flag, ctl, kid | MW_BFULL))
        break;
      tb = w + 1 < w1 ? mbar_test(&b_full[(k + 1) % NSTAGE], (uint32_t)((k + 1) / NSTAGE) & 1u) : 0u;
      for (int rt = 0; rt < st.nq; ++rt, ++p) {
        const int buf = (int)(p % NACC);
        if (!mbar_wait_warp_tested(&t_empty[buf], ((uint32_t)(p / NACC) & 1u) ^ 1u, te, abort_flag, ctl,
                                   kid | MW_TEMPTY)) {
          ok = false;
          break;
        }
        te = mbar_test(&t_empty[(p + 1) % NACC], ((uint32_t)((p + 1) / NACC) & 1u) ^ 1u);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < L::KSTEPS; ++kk)
          mma_ss_w(tmem + (uint32_t)(buf * kTile * KT), desc_off(a0, (uint32_t)(rt * TB + kk * 2 * L::LBO)),
                   desc_off(b0, (uint32_t)(s * SB + kk * 2 * L::LBO)), ID, kk > 0 ? 1u : 0u);
        mma_commit_w(&t_full[buf]);
      }
      if (ok) mma_commit_w(&b_empty[s]);
    }
    mma_commit_w(drain);
    mbar_wait_warp(drain, 0, nullptr, ctl, kid | MW_DRAIN);
  } else {
    // ------------- reduction warps: group grp takes the products p with p % 2 == grp; -------------
    // ------------- warp qd of a group reads TMEM lane quarter qd (tile rows 32*qd .. +31) -----------
    // Per product: the row maxima over each 64-column group of the product's
    // 128 * KT key columns, then the warp's maxima (redux on order-preserving
    // integer keys), kept in shared memory.  Two groups work on alternate
    // products, so that the latency of one product's waits, loads and
    // reductions overlaps the other's.  Every ZC steps all eight warps meet at
    // a named barrier and combine the quarters into scores.  Every warp runs
    // every step and barrier, also after a wait has given up (then without
    // waits or TMEM reads), so that no warp is left at the barrier.
    const int qd = warp & 3, grp = (warp - 2) >> 2;
    const int tid = threadIdx.x - 64;               // 0 .. 255
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    bool ok = true;
    long long p = 0;
    for (long long w = w0; w < w1; ++w) {
      const long long k = w - w0;
      const int z = (int)(k % T::ZC), zb = (int)(k / T::ZC) & 1;
      const int nq = max_step<NQ>(w, NT, NS).nq;
      for (int rt = 0; rt < nq; ++rt, ++p) {
        if ((int)(p & 1) != grp) continue;
        const int buf = (int)(p % NACC);
        if (ok) ok = mbar_wait_warp(&t_full[buf], (uint32_t)(p / NACC) & 1u, abort_flag, ctl, kid | MW_TFULL);
        int key[CG];
#pragma unroll
        for (int cg = 0; cg < CG; ++cg) key[cg] = INT_MIN;
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < KT; ++kc) {
            uint32_t v[128];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tmem_ld32(tmem + lane_off + (uint32_t)(buf * kTile * KT + kc * kTile + 32 * q), v + 32 * q);
            tmem_ld_wait();
            if (kc == KT - 1) {
              tc_fence_before();
              mbar_arrive(&t_empty[buf]);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t* x = v + 64 * hh;
              float a0 = __uint_as_float(x[0]), a1 = __uint_as_float(x[1]), a2 = __uint_as_float(x[2]),
                    a3 = __uint_as_float(x[3]);
#pragma unroll
              for (int i = 4; i < 60; i += 8) {     // columns 4 .. 59
                a0 = max3f(a0, __uint_as_float(x[i]), __uint_as_float(x[i + 1]));
                a1 = max3f(a1, __uint_as_float(x[i + 2]), __uint_as_float(x[i + 3]));
                a2 = max3f(a2, __uint_as_float(x[i + 4]), __uint_as_float(x[i + 5]));
                a3 = max3f(a3, __uint_as_float(x[i + 6]), __uint_as_float(x[i + 7]));
              }
              a0 = max3f(a0, __uint_as_float(x[60]), __uint_as_float(x[61]));
              a1 = max3f(a1, __uint_as_float(x[62]), __uint_as_float(x[63]));
              float m = fmaxf(max3f(a0, a1, a2), a3);   // NaN only if all 64 logits are NaN
              if (m != m) m = -INFINITY;
              key[2 * kc + hh] = __reduce_max_sync(0xffffffffu, float_key(m));
            }
          }
        }
        if (lane == 0) {
          int* pp = part + (((zb * T::ZC + z) * NQ + rt) * 4 + qd) * CG;
#pragma unroll
          for (int cg = 0; cg < CG; ++cg) pp[cg] = key[cg];
        }
      }
      if (z == T::ZC - 1 || w == w1 - 1) {
        asm volatile("bar.sync 1, 256;" ::: "memory");
        // one score per thread: (step k - z + zz, query tile rt, [query half ga,] key block jb)
        constexpr int PER = BLOCK == 128 ? KT : 4 * KT;
        const int item = tid / PER, sub = tid % PER;
        const int zz = item / NQ, rt = item % NQ;
        if (ok && zz <= z) {
          const MaxStep st = max_step<NQ>(w - z + zz, NT, NS);
          if (rt < st.nq) {
            const int* pb = part + (((zb * T::ZC + zz) * NQ + rt) * 4) * CG;   // [quarter][column group]
            const int tq = st.tq0 + rt;
            if (BLOCK == 128) {
              // key block jb: column groups 2 jb, 2 jb + 1 of all four quarters
              const int jb = sub, j = st.c * KT + jb;
              int m = INT_MIN;
#pragma unroll
              for (int q = 0; q < 4; ++q) m = max(m, max(pb[q * CG + 2 * jb], pb[q * CG + 2 * jb + 1]));
              if (j < G) S[(st.bh * G + tq) * (long long)G + j] = key_float(m);
            } else {
              // rows 0..63 (quarters 0, 1) are group 2*tq, rows 64..127 group 2*tq + 1;
              // column group jb is key block 2*KT*c + jb
              const int ga = sub / (2 * KT), jb = sub % (2 * KT);
              const int g = 2 * tq + ga, j = 2 * KT * st.c + jb;
              if (g < G && j < G)
                S[(st.bh * G + g) * (long long)G + j] = key_float(max(pb[(2 * ga) * CG + jb], pb[(2 * ga + 1) * CG + jb]));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int R>
cudaError_t launch_tile_max(const uint8_t* qt, const uint8_t* kt, const dsv_shape& s, int NT, int NS, float* scores,
                            const Ctl& ctl, cudaStream_t st) {
  const int G = s.N / s.block;
  auto kern = s.block == 128 ? tile_max_mma_kernel<128, R> : tile_max_mma_kernel<64, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MaxTraits<R>::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  constexpr int NQ = MaxTraits<R>::NQ;
  const long long steps = (long long)s.B * s.H * ((NT + NQ - 1) / NQ) * NS;
  const unsigned grid = (unsigned)(steps < nsm ? steps : nsm);
  kern<<<grid, kMaxThreads, MaxTraits<R>::SMEM, st>>>(qt, kt, NT, NS, G, steps, scores, ctl);
  return cudaGetLastError();
}

template <int D, int R>
cudaError_t launch_split(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s, int NTP,
                         uint8_t* qt, uint8_t* kt, cudaStream_t st) {
  const int smem = D * R * (int)sizeof(float);
  cudaError_t e =
      cudaFuncSetAttribute(lowrank_split_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((long long)s.B * s.H * NTP), 2);
  lowrank_split_kernel<D, R><<<grid, kTile, smem, st>>>(static_cast<const __nv_bfloat16*>(Q),
                                                        static_cast<const __nv_bfloat16*>(K), Wq, Wk, s.H, s.N, NTP,
                                                        qt, kt);
  return cudaGetLastError();
}

// 128-token tiles per head in the workspace: ceil(N / 128), rounded up to a
// whole number of key steps
template <int R>
int tiles_per_head(const dsv_shape& s) {
  constexpr int KT = MaxTraits<R>::KT;
  const int NT = (s.N + kTile - 1) / kTile;
  return (NT + KT - 1) / KT * KT;
}

template <int R>
size_t tiles_bytes(const dsv_shape& s) {
  return align256((size_t)s.B * s.H * (size_t)tiles_per_head<R>(s) * (size_t)MaxLayout<R>::TILE_BYTES);
}

template <int R>
cudaError_t launch_predict_max_r(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                                 float* scores, void* ws, const Ctl& ctl, cudaStream_t st) {
  const int NT = (s.N + kTile - 1) / kTile;
  const int NTP = tiles_per_head<R>(s);
  uint8_t* qt = static_cast<uint8_t*>(ws);
  uint8_t* kt = qt + tiles_bytes<R>(s);
  cudaError_t e = s.d == 128 ? launch_split<128, R>(Q, K, Wq, Wk, s, NTP, qt, kt, st)
                             : launch_split<64, R>(Q, K, Wq, Wk, s, NTP, qt, kt, st);
  if (e != cudaSuccess) return e;
  return launch_tile_max<R>(qt, kt, s, NT, NTP / MaxTraits<R>::KT, scores, ctl, st);
}

template <int R>
size_t ws_bytes_r(const dsv_shape& s) {
  return 2 * tiles_bytes<R>(s);
}

}  // namespace

size_t predict_max_ws_bytes(const dsv_shape& s) {
  switch (s.r) {
    case 8: return ws_bytes_r<8>(s);
    case 16: return ws_bytes_r<16>(s);
    case 24: return ws_bytes_r<24>(s);
    case 32: return ws_bytes_r<32>(s);
    case 40: return ws_bytes_r<40>(s);
    case 48: return ws_bytes_r<48>(s);
    case 56: return ws_bytes_r<56>(s);
    default: return ws_bytes_r<64>(s);
  }
}

cudaError_t launch_predict_max(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                               float* scores, void* ws, const Ctl& ctl, cudaStream_t st) {
  switch (s.r) {
    case 8: return launch_predict_max_r<8>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    case 16: return launch_predict_max_r<16>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    case 24: return launch_predict_max_r<24>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    case 32: return launch_predict_max_r<32>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    case 40: return launch_predict_max_r<40>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    case 48: return launch_predict_max_r<48>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    case 56: return launch_predict_max_r<56>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
    default: return launch_predict_max_r<64>(Q, K, Wq, Wk, s, scores, ws, ctl, st);
  }
}

}  // namespace dsv
