// attn_bwd.cu — gradient of the block-sparse attention, without atomics.
//
// DSV page [nl], "Technische samenvatting" 2A: stage 2 trains with sparse
// attention over the critical KV only, so the backward pass runs over the same
// (group, block) pairs as the forward.  With P_ij = exp(s_ij - lse_i):
//   D_i  = sum_c dO_ic O_ic                       (pre-pass, HBM-bound)
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i      (per key block)
//   dQ_i = scale sum_j dS_ij k_j                                  (per group)
//   dS_ij = P_ij (dO_i . v_j - D_i)
//
// Every output tile has exactly one owner CTA, so no atomics are needed:
//   kv kernel  one CTA per key block (b, h, j), looping over the ascending
//              transposed list of groups g that selected j:
//                S^T = K_j Q_g^T, dP^T = V_j dO_g^T       (tcgen05, smem x smem)
//                P^T, dS^T -> TMEM (bf16) by the compute warpgroup
//                dV += P^T dO_g, dK += dS^T Q_g           (tcgen05, TMEM x smem)
//   q kernel   one CTA per group (b, h, g), looping over its forward list:
//                S = Q_g K_j^T, dP = dO_g V_j^T; dS -> TMEM; dQ += dS K_j
// The price of no atomics is recomputing S and dP in both kernels (7 MMAs
// per pair instead of 5).  Warp roles and TMEM use mirror the forward kernel:
// warp 0 TMA, warp 1 MMA issue, warps 2..5 one tile row per thread.
#include <math.h>

#include "dsv_launch.h"

namespace dsv {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// D_i = sum_c dO_ic * O_ic
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         float* __restrict__ Dw, long long rows) {
  constexpr int TPR = D / 8;             // threads per row, 16 bytes each
  constexpr int RPC = 256 / TPR;         // rows per CTA
  const long long row = (long long)blockIdx.x * RPC + threadIdx.x / TPR;
  const int c = threadIdx.x % TPR;
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(O + row * D) + c);
    const uint4 b = __ldcs(reinterpret_cast<const uint4*>(dO + row * D) + c);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wb[i] << 16), acc);
      acc = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wb[i] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (row < rows && c == 0) Dw[row] = acc;
}

enum : unsigned int { W_KV = 1, W_GFULL, W_GEMPTY, W_S, W_P, W_ACC, W_DRAIN, W_KFULL, W_VFULL, W_KVEMPTY };

// ---------------------------------------------------------------------------
// dK, dV: one CTA per key block
// ---------------------------------------------------------------------------
template <int BETA, int D>
struct KVTraits {
  static constexpr int BM = 128;                   // MMA M: key rows incl. padding
  static constexpr int NCH = D / 64;
  static constexpr int A_CHUNK = BM * 128;         // K_j / V_j as A operands (padded rows)
  static constexpr int A_BYTES = NCH * A_CHUNK;
  static constexpr int B_CHUNK = BETA * 128;       // Q_g / dO_g tiles
  static constexpr int B_BYTES = NCH * B_CHUNK;
  static constexpr int NST = 2;
  static constexpr int VEC_BYTES = BETA * 4;       // lse_g or D_g
  static constexpr int STAGE_BYTES = (2 * B_BYTES + 2 * VEC_BYTES + 1023) / 1024 * 1024;  // keeps tiles 1024-aligned
  static constexpr int NBAR = 1 + 2 * NST + 3;
  static constexpr int SMEM_USED = 1024 + 2 * A_BYTES + NST * STAGE_BYTES + NBAR * 8 + 16;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t ST_COL = 0, DPT_COL = 128, DV_COL = 256, DK_COL = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
};

template <int BETA, int D>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const float* __restrict__ lse, const float* __restrict__ Dw,
                       const int32_t* __restrict__ bwd_ptr, const int32_t* __restrict__ bwd_col, int N, int G,
                       float scale, __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, Ctl ctl) {
  using T = KVTraits<BETA, D>;
  constexpr int NST = T::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = align_up_ptr<uint8_t>(smem_raw, 1024);
  uint8_t* sK = sbase;
  uint8_t* sV = sK + T::A_BYTES;
  uint8_t* sStage = sV + T::A_BYTES;              // NST x [Q_g | dO_g | lse | D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + NST * T::STAGE_BYTES);
  uint64_t* kv_full = bars;
  uint64_t* g_full = bars + 1;
  uint64_t* g_empty = g_full + NST;
  uint64_t* s_full = g_empty + NST;
  uint64_t* p_full = s_full + 1;
  uint64_t* acc_done = p_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x;               // (b*H + h)*nb + j
  const int nb = G;
  const long long bh = row / nb;
  const int j = (int)(row - bh * nb);
  const int start = bwd_ptr[row];
  const int cnt = bwd_ptr[row + 1] - start;
  const unsigned int kid = (unsigned int)KID_BWD_KV << 8;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&g_full[s], 1);
      mbar_init(&g_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (BETA < T::BM) {
    for (int t = 0; t < 2; ++t)
      for (int c = 0; c < T::NCH; ++c) {
        uint4* z = reinterpret_cast<uint4*>(sK + t * T::A_BYTES + c * T::A_CHUNK + BETA * 128);
        for (int i = threadIdx.x; i < (T::BM - BETA) * 128 / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
      }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, T::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long krow0 = bh * N + (long long)j * BETA;

  if (cnt <= 0) {
    if (cnt < 0 && threadIdx.x == 0) set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
    for (int i = threadIdx.x; i < BETA * D / 8; i += blockDim.x) {
      reinterpret_cast<uint4*>(dK + krow0 * D)[i] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(dV + krow0 * D)[i] = make_uint4(0, 0, 0, 0);
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(kv_full, 2 * BETA * D * 2);
      for (int c = 0; c < T::NCH; ++c) {
        tma_load_2d(sK + c * T::A_CHUNK, &tmK, kv_full, c * 64, (int)krow0);
        tma_load_2d(sV + c * T::A_CHUNK, &tmV, kv_full, c * 64, (int)krow0);
      }
      int issued = 0;
      for (int n = 0; n < cnt; ++n) {
        const int s = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        int g = bwd_col[start + n];
        if (!mbar_wait(&g_empty[s], ph ^ 1u, abort_flag, ctl, kid | W_GEMPTY)) break;
        if ((unsigned)g >= (unsigned)G) {
          set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
          g = 0;
        }
        const long long qrow = bh * N + (long long)g * BETA;
        uint8_t* st = sStage + s * T::STAGE_BYTES;
        mbar_arrive_expect_tx(&g_full[s], 2 * BETA * D * 2 + 2 * T::VEC_BYTES);
        for (int c = 0; c < T::NCH; ++c) {
          tma_load_2d(st + c * T::B_CHUNK, &tmQ, &g_full[s], c * 64, (int)qrow);
          tma_load_2d(st + T::B_BYTES + c * T::B_CHUNK, &tmdO, &g_full[s], c * 64, (int)qrow);
        }
        bulk_load(st + 2 * T::B_BYTES, lse + qrow, T::VEC_BYTES, &g_full[s]);
        bulk_load(st + 2 * T::B_BYTES + T::VEC_BYTES, Dw + qrow, T::VEC_BYTES, &g_full[s]);
        issued = n + 1;
      }
      mbar_wait(kv_full, 0, nullptr, ctl, kid | W_DRAIN);
      for (int n = (issued > NST ? issued - NST : 0); n < issued; ++n)
        mbar_wait(&g_full[n % NST], (uint32_t)(n / NST) & 1u, nullptr, ctl, kid | W_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t ID_S = idesc_bf16_f32(T::BM, BETA, false, false);   // S^T, dP^T: N = queries
      constexpr uint32_t ID_G = idesc_bf16_f32(T::BM, D, false, true);       // dV, dK: B MN-major
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aS = smem_u32(sStage);
      bool ok = mbar_wait(kv_full, 0, abort_flag, ctl, kid | W_KV);
      for (int n = 0; ok && n < cnt; ++n) {
        const int s = n % NST;
        if (!mbar_wait(&g_full[s], (uint32_t)(n / NST) & 1u, abort_flag, ctl, kid | W_GFULL)) break;
        tc_fence_after();
        const uint32_t aQg = aS + s * T::STAGE_BYTES, adOg = aQg + T::B_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * T::B_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + T::ST_COL, sdesc_sw128(aK + ao, 16, 1024), sdesc_sw128(aQg + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * T::B_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + T::DPT_COL, sdesc_sw128(aV + ao, 16, 1024), sdesc_sw128(adOg + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (!mbar_wait(p_full, (uint32_t)n & 1u, abort_flag, ctl, kid | W_P)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BETA / 16; ++kk) {
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + T::DV_COL, tmem + T::ST_COL + kk * 8,
                 sdesc_sw128(adOg + kk * 16 * 128, T::B_CHUNK, 1024), ID_G, acc);
          mma_ts(tmem + T::DK_COL, tmem + T::DPT_COL + kk * 8,
                 sdesc_sw128(aQg + kk * 16 * 128, T::B_CHUNK, 1024), ID_G, acc);
        }
        mma_commit(&g_empty[s]);
      }
      mma_commit(acc_done);
      mbar_wait(acc_done, 0, nullptr, ctl, kid | W_DRAIN);
    }
  } else {
    // ---------------- compute warpgroup: one key row per thread ----------------
    const int sp = warp & 3;
    const int kr = sp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    const float scale_log2 = scale * kLog2e;
    bool ok = true;
    for (int n = 0; n < cnt; ++n) {
      const int s = n % NST;
      if (!mbar_wait_warp(&g_full[s], (uint32_t)(n / NST) & 1u, abort_flag, ctl, kid | W_GFULL) ||
          !mbar_wait_warp(s_full, (uint32_t)n & 1u, abort_flag, ctl, kid | W_S)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* lse_s = reinterpret_cast<const float*>(sStage + s * T::STAGE_BYTES + 2 * T::B_BYTES);
      const float* dd_s = lse_s + BETA;
#pragma unroll
      for (int c = 0; c < BETA / 32; ++c) {
        uint32_t xs[32], xp[32];
        tmem_ld32(tmem + lane_off + T::ST_COL + c * 32, xs);
        tmem_ld32(tmem + lane_off + T::DPT_COL + c * 32, xp);
        tmem_ld_wait();
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int q0 = c * 32 + 2 * i;
          const float p0 = ex2(fmaf(__uint_as_float(xs[2 * i]), scale_log2, -lse_s[q0] * kLog2e));
          const float p1 = ex2(fmaf(__uint_as_float(xs[2 * i + 1]), scale_log2, -lse_s[q0 + 1] * kLog2e));
          const float d0 = p0 * (__uint_as_float(xp[2 * i]) - dd_s[q0]);
          const float d1 = p1 * (__uint_as_float(xp[2 * i + 1]) - dd_s[q0 + 1]);
          pw[i] = pack_bf16x2(p0, p1);
          dw[i] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tmem + lane_off + T::ST_COL + c * 16, pw);
        tmem_st16(tmem + lane_off + T::DPT_COL + c * 16, dw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait_warp(acc_done, 0, abort_flag, ctl, kid | W_ACC);
    if (ok) {
      tc_fence_after();
      const long long orow = krow0 + kr;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t col = t == 0 ? T::DV_COL : T::DK_COL;
        const float mul = t == 0 ? 1.0f : scale;
        __nv_bfloat16* outp = t == 0 ? dV : dK;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + col + c * 32, o);
          tmem_ld_wait();
          if (kr < BETA) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
            uint4* dst = reinterpret_cast<uint4*>(outp + orow * D + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, T::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// dQ: one CTA per query group
// ---------------------------------------------------------------------------
template <int BETA, int D>
struct QTraits {
  static constexpr int BM = 128;
  static constexpr int NCH = D / 64;
  static constexpr int A_CHUNK = BM * 128;         // Q_g / dO_g as A operands (padded rows)
  static constexpr int A_BYTES = NCH * A_CHUNK;
  static constexpr int KV_CHUNK = BETA * 128;
  static constexpr int KV_BYTES = NCH * KV_CHUNK;
  static constexpr int NST = (2 * A_BYTES + 6 * KV_BYTES + 2048 <= 227 * 1024) ? 3 : 2;
  static constexpr int NBAR = 1 + 3 * NST + 3;
  static constexpr int SMEM_USED = 1024 + 2 * A_BYTES + 2 * NST * KV_BYTES + NBAR * 8 + 16;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TX_BYTES = BETA * D * 2;
};

template <int BETA, int D>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                      const float* __restrict__ lse, const float* __restrict__ Dw,
                      const int32_t* __restrict__ fwd_ptr, const int32_t* __restrict__ fwd_col, int N, int G,
                      float scale, __nv_bfloat16* __restrict__ dQ, Ctl ctl) {
  using T = QTraits<BETA, D>;
  constexpr int NST = T::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = align_up_ptr<uint8_t>(smem_raw, 1024);
  uint8_t* sQ = sbase;
  uint8_t* sdO = sQ + T::A_BYTES;
  uint8_t* sK = sdO + T::A_BYTES;
  uint8_t* sV = sK + NST * T::KV_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NST * T::KV_BYTES);
  uint64_t* qd_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* kv_empty = v_full + NST;
  uint64_t* s_full = kv_empty + NST;
  uint64_t* p_full = s_full + 1;
  uint64_t* acc_done = p_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x;               // (b*H + h)*G + g
  const long long bh = row / G;
  const int g = (int)(row - bh * G);
  const int nb = G;
  const int start = fwd_ptr[row];
  const int cnt = fwd_ptr[row + 1] - start;
  const unsigned int kid = (unsigned int)KID_BWD_Q << 8;
  const long long qrow0 = bh * N + (long long)g * BETA;

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (BETA < T::BM) {
    for (int t = 0; t < 2; ++t)
      for (int c = 0; c < T::NCH; ++c) {
        uint4* z = reinterpret_cast<uint4*>(sQ + t * T::A_BYTES + c * T::A_CHUNK + BETA * 128);
        for (int i = threadIdx.x; i < (T::BM - BETA) * 128 / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
      }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, T::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (cnt <= 0) {
    if (cnt < 0 && threadIdx.x == 0) set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
    for (int i = threadIdx.x; i < BETA * D / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(dQ + qrow0 * D)[i] = make_uint4(0, 0, 0, 0);
  } else if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(qd_full, 2 * T::TX_BYTES);
      for (int c = 0; c < T::NCH; ++c) {
        tma_load_2d(sQ + c * T::A_CHUNK, &tmQ, qd_full, c * 64, (int)qrow0);
        tma_load_2d(sdO + c * T::A_CHUNK, &tmdO, qd_full, c * 64, (int)qrow0);
      }
      int issued = 0;
      int jn = fwd_col[start];
      for (int n = 0; n < cnt; ++n) {
        const int s = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        int j = jn;
        if (n + 1 < cnt) jn = fwd_col[start + n + 1];
        if (!mbar_wait(&kv_empty[s], ph ^ 1u, abort_flag, ctl, kid | W_KVEMPTY)) break;
        if ((unsigned)j >= (unsigned)nb) {
          set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
          j = 0;
        }
        const int krow = (int)(bh * N + (long long)j * BETA);
        mbar_arrive_expect_tx(&k_full[s], T::TX_BYTES);
        for (int c = 0; c < T::NCH; ++c)
          tma_load_2d(sK + s * T::KV_BYTES + c * T::KV_CHUNK, &tmK, &k_full[s], c * 64, krow);
        mbar_arrive_expect_tx(&v_full[s], T::TX_BYTES);
        for (int c = 0; c < T::NCH; ++c)
          tma_load_2d(sV + s * T::KV_BYTES + c * T::KV_CHUNK, &tmV, &v_full[s], c * 64, krow);
        issued = n + 1;
      }
      mbar_wait(qd_full, 0, nullptr, ctl, kid | W_DRAIN);
      for (int n = (issued > NST ? issued - NST : 0); n < issued; ++n) {
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        mbar_wait(&k_full[n % NST], ph, nullptr, ctl, kid | W_DRAIN);
        mbar_wait(&v_full[n % NST], ph, nullptr, ctl, kid | W_DRAIN);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16_f32(T::BM, BETA, false, false);
      constexpr uint32_t ID_Q = idesc_bf16_f32(T::BM, D, false, true);
      const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO), aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(qd_full, 0, abort_flag, ctl, kid | W_KV);
      for (int n = 0; ok && n < cnt; ++n) {
        const int s = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        if (!mbar_wait(&k_full[s], ph, abort_flag, ctl, kid | W_KFULL)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          const uint32_t bo = s * T::KV_BYTES + (kk >> 2) * T::KV_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + T::S_COL, sdesc_sw128(aQ + ao, 16, 1024), sdesc_sw128(aK + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
        if (!mbar_wait(&v_full[s], ph, abort_flag, ctl, kid | W_VFULL)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          const uint32_t bo = s * T::KV_BYTES + (kk >> 2) * T::KV_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + T::DP_COL, sdesc_sw128(adO + ao, 16, 1024), sdesc_sw128(aV + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (!mbar_wait(p_full, (uint32_t)n & 1u, abort_flag, ctl, kid | W_P)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BETA / 16; ++kk) {
          mma_ts(tmem + T::DQ_COL, tmem + T::S_COL + kk * 8,
                 sdesc_sw128(aK + s * T::KV_BYTES + kk * 16 * 128, T::KV_CHUNK, 1024), ID_Q,
                 (n > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&kv_empty[s]);
      }
      mma_commit(acc_done);
      mbar_wait(acc_done, 0, nullptr, ctl, kid | W_DRAIN);
    }
  } else {
    // ---------------- compute warpgroup: one query row per thread ----------------
    const int sp = warp & 3;
    const int r = sp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    const float scale_log2 = scale * kLog2e;
    const float lse2 = (r < BETA) ? lse[qrow0 + r] * kLog2e : 0.f;
    const float dd = (r < BETA) ? Dw[qrow0 + r] : 0.f;
    bool ok = true;
    for (int n = 0; n < cnt; ++n) {
      if (!mbar_wait_warp(s_full, (uint32_t)n & 1u, abort_flag, ctl, kid | W_S)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < BETA / 32; ++c) {
        uint32_t xs[32], xp[32];
        tmem_ld32(tmem + lane_off + T::S_COL + c * 32, xs);
        tmem_ld32(tmem + lane_off + T::DP_COL + c * 32, xp);
        tmem_ld_wait();
        uint32_t dw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(__uint_as_float(xs[2 * i]), scale_log2, -lse2));
          const float p1 = ex2(fmaf(__uint_as_float(xs[2 * i + 1]), scale_log2, -lse2));
          dw[i] = pack_bf16x2(p0 * (__uint_as_float(xp[2 * i]) - dd), p1 * (__uint_as_float(xp[2 * i + 1]) - dd));
        }
        tmem_st16(tmem + lane_off + T::S_COL + c * 16, dw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait_warp(acc_done, 0, abort_flag, ctl, kid | W_ACC);
    if (ok) {
      tc_fence_after();
      const long long orow = qrow0 + r;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + T::DQ_COL + c * 32, o);
        tmem_ld_wait();
        if (r < BETA) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * scale, __uint_as_float(o[2 * i + 1]) * scale);
          uint4* dst = reinterpret_cast<uint4*>(dQ + orow * D + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, T::TMEM_COLS);
}

template <int BETA, int D>
cudaError_t launch_bwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         const CUtensorMap& tmdO, const void* O, const void* dO, const float* lse, const dsv_shape& s,
                         const int32_t* fwd_ptr, const int32_t* fwd_col, const int32_t* bwd_ptr,
                         const int32_t* bwd_col, float scale, void* dQ, void* dK, void* dV, void* ws, const Ctl& ctl,
                         cudaStream_t st) {
  const int G = s.N / s.block;
  const long long rows = (long long)s.B * s.H * s.N;
  const long long groups = (long long)s.B * s.H * G;
  float* Dw = static_cast<float*>(ws);
  constexpr int RPC = 256 / (D / 8);
  bwd_rowdot_kernel<D><<<(unsigned)((rows + RPC - 1) / RPC), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), Dw, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kv = attn_bwd_kv_kernel<BETA, D>;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, KVTraits<BETA, D>::SMEM)) !=
      cudaSuccess)
    return e;
  kv<<<(unsigned)groups, 192, KVTraits<BETA, D>::SMEM, st>>>(tmQ, tmK, tmV, tmdO, lse, Dw, bwd_ptr, bwd_col, s.N, G,
                                                              scale, static_cast<__nv_bfloat16*>(dK),
                                                              static_cast<__nv_bfloat16*>(dV), ctl);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto qk = attn_bwd_q_kernel<BETA, D>;
  if ((e = cudaFuncSetAttribute(qk, cudaFuncAttributeMaxDynamicSharedMemorySize, QTraits<BETA, D>::SMEM)) !=
      cudaSuccess)
    return e;
  qk<<<(unsigned)groups, 192, QTraits<BETA, D>::SMEM, st>>>(tmQ, tmK, tmV, tmdO, lse, Dw, fwd_ptr, fwd_col, s.N, G,
                                                            scale, static_cast<__nv_bfloat16*>(dQ), ctl);
  return cudaGetLastError();
}

}  // namespace

size_t attn_bwd_ws_bytes(const dsv_shape& s) { return align256((size_t)s.B * s.H * s.N * sizeof(float)); }

cudaError_t launch_attn_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmdO, const void* O, const void* dO, const float* lse,
                            const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col,
                            const int32_t* bwd_ptr, const int32_t* bwd_col, float scale, void* dQ, void* dK,
                            void* dV, void* ws, const Ctl& ctl, cudaStream_t st) {
#define DSV_BWD(BE, DD)                                                                                        \
  return launch_bwd_t<BE, DD>(tmQ, tmK, tmV, tmdO, O, dO, lse, s, fwd_ptr, fwd_col, bwd_ptr, bwd_col, scale, dQ, \
                              dK, dV, ws, ctl, st)
  if (s.block == 128 && s.d == 128) DSV_BWD(128, 128);
  if (s.block == 128 && s.d == 64) DSV_BWD(128, 64);
  if (s.block == 64 && s.d == 128) DSV_BWD(64, 128);
  DSV_BWD(64, 64);
#undef DSV_BWD
}

}  // namespace dsv
