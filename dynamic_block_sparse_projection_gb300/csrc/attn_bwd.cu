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
//                P^T, dS^T -> TMEM (bf16) by the compute warps
//                dV += P^T dO_g, dK += dS^T Q_g           (tcgen05, TMEM x smem)
//              with the products of consecutive pairs interleaved so that
//              the tensor core runs one while the compute warps convert the
//              other's output.
//   q kernel   persistent CTAs (one per SM) working through the groups
//              (b, h, g), each looping over its forward list:
//                S = Q_g K_j^T, dP = dO_g V_j^T; dS -> TMEM; dQ += dS K_j
//              The rings and barrier phases run on across groups, so the
//              next group's tiles load while the current one finishes.  The
//              kv kernel keeps one CTA per block: persistent versions of it
//              (a static split of its uneven lists, and a shared work counter
//              with a shared-memory item queue) measured 11-22% slower.
// The price of no atomics is recomputing S and dP in both kernels (7 MMAs
// per pair instead of 5).
//
// Warp roles: warp 0 TMA producer (one lane), warp 1 TMEM allocator and MMA
// issuer (the whole warp; one elected lane issues), warps 2..9 compute; the q
// kernel adds warp 10 as the producer of its V ring.  A TMEM lane (tile row)
// belongs to the sub-partition warp % 4, so two compute warps share each row
// quarter and split its columns: two warps per SM sub-partition hide the
// latency of the TMEM loads and the exponentials.
#include <math.h>

#include "dsv_launch.h"

namespace dsv {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 320;          // 2 control warps + 8 compute warps
constexpr int kQVWarp = 10;            // q kernel: V producer warp
constexpr int kQThreads = 352;         // q kernel: 3 control warps + 8 compute warps
constexpr int kComputeThreads = 256;

// ---------------------------------------------------------------------------
// Pre-pass: D_i = sum_c dO_ic O_ic and -lse_i * log2(e) for the main kernels.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ Dw,
                                                         float* __restrict__ L2w, long long rows) {
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
  if (row < rows && c == 0) {
    Dw[row] = acc;
    L2w[row] = -lse[row] * kLog2e;
  }
}

enum : unsigned int {
  W_KV = 1, W_GFULL, W_GEMPTY, W_S, W_P, W_ACC, W_DRAIN, W_KFULL, W_VFULL, W_KVEMPTY, W_LD, W_SPFREE, W_DSFULL,
  W_DSEMPTY
};

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
  static constexpr int VEC_BYTES = BETA * 4;       // -lse2_g or D_g
  static constexpr int STAGE_BYTES = (2 * B_BYTES + 2 * VEC_BYTES + 1023) / 1024 * 1024;  // keeps tiles 1024-aligned
  static constexpr int NBAR = 1 + 2 * NST + 7;
  static constexpr int SMEM_USED = 1024 + 2 * A_BYTES + NST * STAGE_BYTES + NBAR * 8 + 16;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  // TMEM: S^T (fp32, BETA columns) at 0, dP^T at 128, dV at 256, dK at 256+D.
  // S^T and dP^T are whole-group products (N = BETA): an M=128, N=128
  // smem x smem product reads 8 KB in its 64 clocks, the shared-memory port's
  // rate, where a half-group (N = 64) product would need 6 KB in 32.  The
  // compute warps write P^T and dS^T (bf16 pairs) over the columns they read:
  // warp half hf owns queries [hf*W, hf*W + W) and packs them into its first
  // W/2 columns.
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int W = BETA / 2;               // columns per compute warp
  __host__ __device__ static constexpr uint32_t packed_col(int q) { return (uint32_t)((q / W) * W + (q % W) / 2); }
  // The compute warps hand P^T and dS^T over in two chunks (the first and the
  // second half of each warp's columns, one barrier each), so the tensor core
  // starts dV and dK on the first while they convert the second.
  __host__ __device__ static constexpr int chunk_of(int q) { return (q % W) / (W / 2); }
};

template <int BETA, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const float* __restrict__ L2w, const float* __restrict__ Dw,
                       const int32_t* __restrict__ bwd_ptr, const int32_t* __restrict__ bwd_col,
                       const int32_t* __restrict__ order, int N, int G, float scale,
                       __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, Ctl ctl) {
  using T = KVTraits<BETA, D>;
  constexpr int NST = T::NST;
  constexpr int W = T::W;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sbase = smem_align1024(smem_raw);
  uint8_t* sK = sbase;
  uint8_t* sV = sK + T::A_BYTES;
  uint8_t* sStage = sV + T::A_BYTES;              // NST x [Q_g | dO_g | lse2 | D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + NST * T::STAGE_BYTES);
  uint64_t* kv_full = bars;
  uint64_t* g_full = bars + 1;
  uint64_t* g_empty = g_full + NST;
  uint64_t* s_full = g_empty + NST;               // S^T in TMEM
  uint64_t* dp_full = s_full + 1;                 // dP^T in TMEM
  uint64_t* p_full = dp_full + 1;                 // [2] P^T chunk written back (bf16)
  uint64_t* ds_full = p_full + 2;                 // [2] dS^T chunk written back (bf16)
  uint64_t* acc_done = ds_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = order[blockIdx.x];        // (b*H + h)*nb + j, longest transposed lists first
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
    mbar_init(dp_full, 1);
    for (int c = 0; c < 2; ++c) {
      mbar_init(&p_full[c], kComputeThreads);
      mbar_init(&ds_full[c], kComputeThreads);
    }
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
  // Every CTA owns its SM's whole TMEM (512 columns), so the allocation starts
  // at lane 0, column 0: with that constant every TMEM address is known at
  // compile time and the MMA warp spends no instructions moving them into
  // uniform registers.  A different address is reported and nothing is run.
  const uint32_t tmem_base = *tmem_slot;
  constexpr uint32_t tmem = 0;
  const long long krow0 = bh * N + (long long)j * BETA;

  if (tmem_base != tmem) {
    if (threadIdx.x == 0) set_error(ctl, DSV_ERR_INTERNAL, (unsigned int)(row & 0x7fffffff));
  } else if (cnt <= 0) {
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
      int gn = bwd_col[start];
      for (int n = 0; n < cnt; ++n) {
        const int s = n % NST;
        const uint32_t ph = (uint32_t)(n / NST) & 1u;
        int g = gn;
        if (n + 1 < cnt) gn = bwd_col[start + n + 1];
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
        bulk_load(st + 2 * T::B_BYTES, L2w + qrow, T::VEC_BYTES, &g_full[s]);
        bulk_load(st + 2 * T::B_BYTES + T::VEC_BYTES, Dw + qrow, T::VEC_BYTES, &g_full[s]);
        issued = n + 1;
      }
      mbar_wait(kv_full, 0, nullptr, ctl, kid | W_DRAIN);
      for (int n = (issued > NST ? issued - NST : 0); n < issued; ++n)
        mbar_wait(&g_full[n % NST], (uint32_t)(n / NST) & 1u, nullptr, ctl, kid | W_DRAIN);
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
      // Order: S^T(0), dP^T(0), then per pair n
      //   dV(n) [P^T(n) written], S^T(n+1), dK(n) [dS^T(n) written], dP^T(n+1).
      // The tensor core runs S^T(n+1) while the compute warps turn dP^T(n)
      // into dS^T(n), and dK(n), dP^T(n+1) while they turn S^T(n+1) into
      // P^T(n+1).  A product that overwrites a TMEM buffer is issued after
      // the products that read it, and the tensor core runs them in order.
      // Each barrier is tested half-way through the products issued before
      // its wait: the MMA queue holds only a few products, so a wait that
      // sleeps, or pays the test's round trip, lets the tensor core drain.
      constexpr uint32_t ID_S = idesc_bf16_f32(T::BM, BETA, false, false);  // S^T, dP^T: N = BETA queries
      constexpr uint32_t ID_G = idesc_bf16_f32(T::BM, D, false, true);      // dV, dK: B MN-major
      const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dS0 = sdesc_sw128(smem_u32(sStage), 16, 1024);           // K-major view of a stage
      const uint64_t dSmn0 = sdesc_sw128(smem_u32(sStage), T::B_CHUNK, 1024);  // MN-major view
      // S^T = K_j Q_g^T (t = 0) or dP^T = V_j dO_g^T (t = 1); returns the test of `probe`
      auto issue_sdp = [&](int n, int t, uint64_t* probe, uint32_t probe_par) -> uint32_t {
        const uint64_t a0 = t ? dV0 : dK0;
        const uint64_t b0 = desc_off(dS0, (uint32_t)((n % NST) * T::STAGE_BYTES + t * T::B_BYTES));
        uint32_t r = 0u;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * T::B_CHUNK + (kk & 3) * 32;
          mma_ss_w(tmem + (t ? T::DP_COL : T::S_COL), desc_off(a0, ao), desc_off(b0, bo), ID_S, kk > 0 ? 1u : 0u);
          if (kk == D / 32 - 1 && probe != nullptr) r = mbar_test(probe, probe_par);
        }
        mma_commit_w(t ? dp_full : s_full);
        return r;
      };
      // chunk c of dV += P^T dO_g (t = 0) or dK += dS^T Q_g (t = 1); returns the test of `probe`
      auto issue_grad = [&](int n, int t, int c, uint64_t* probe, uint32_t probe_par) -> uint32_t {
        const uint64_t b0 = desc_off(dSmn0, (uint32_t)((n % NST) * T::STAGE_BYTES + (t ? 0 : T::B_BYTES)));
        uint32_t r = 0u;
        int m = 0;
#pragma unroll
        for (int kk = 0; kk < BETA / 16; ++kk) {
          if (T::chunk_of(kk * 16) != c) continue;
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          mma_ts_w(tmem + (t ? T::DK_COL : T::DV_COL), tmem + (t ? T::DP_COL : T::S_COL) + T::packed_col(kk * 16),
                   desc_off(b0, kk * 16 * 128), ID_G, acc);
          if (++m == BETA / 64 && probe != nullptr) r = mbar_test(probe, probe_par);
        }
        return r;
      };
      bool ok = mbar_wait_warp(kv_full, 0, abort_flag, ctl, kid | W_KV) &&
                mbar_wait_warp(&g_full[0], 0, abort_flag, ctl, kid | W_GFULL);
      uint32_t tp0 = 0u;
      if (ok) {
        tc_fence_after();
        issue_sdp(0, 0, nullptr, 0u);
        tp0 = issue_sdp(0, 1, &p_full[0], 0u);
      }
      for (int n = 0; ok && n < cnt; ++n) {
        const bool more = n + 1 < cnt;
        const uint32_t par = (uint32_t)n & 1u;
        const uint32_t tg = more ? mbar_test(&g_full[(n + 1) % NST], (uint32_t)((n + 1) / NST) & 1u) : 0u;
        if (!mbar_wait_warp_tested(&p_full[0], par, tp0, abort_flag, ctl, kid | W_P)) break;
        tc_fence_after();
        const uint32_t tp1 = issue_grad(n, 0, 0, &p_full[1], par);
        if (!mbar_wait_warp_tested(&p_full[1], par, tp1, abort_flag, ctl, kid | W_P)) break;
        tc_fence_after();
        issue_grad(n, 0, 1, nullptr, 0u);
        uint32_t td0 = 0u;
        if (more) {
          if (!mbar_wait_warp_tested(&g_full[(n + 1) % NST], (uint32_t)((n + 1) / NST) & 1u, tg, abort_flag, ctl,
                                     kid | W_GFULL))
            break;
          tc_fence_after();
          td0 = issue_sdp(n + 1, 0, &ds_full[0], par);
        }
        if (!mbar_wait_warp_tested(&ds_full[0], par, td0, abort_flag, ctl, kid | W_DSFULL)) break;
        tc_fence_after();
        const uint32_t td1 = issue_grad(n, 1, 0, &ds_full[1], par);
        if (!mbar_wait_warp_tested(&ds_full[1], par, td1, abort_flag, ctl, kid | W_DSFULL)) break;
        tc_fence_after();
        issue_grad(n, 1, 1, nullptr, 0u);
        mma_commit_w(&g_empty[n % NST]);
        if (more) tp0 = issue_sdp(n + 1, 1, &p_full[0], par ^ 1u);
      }
      mma_commit_w(acc_done);
      mbar_wait_warp(acc_done, 0, nullptr, ctl, kid | W_DRAIN);
    }
  } else {
    // ------------- compute warps: key row kr, W queries of the group -------------
    const int sp = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int kr = sp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    const float scale_log2 = scale * kLog2e;
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    const uint32_t cs = tmem + lane_off + T::S_COL + hf * W;
    const uint32_t cp = tmem + lane_off + T::DP_COL + hf * W;
    const int q0 = hf * W;                         // first query of this warp's columns
    bool ok = true;
    for (int n = 0; ok && n < cnt; ++n) {
      const int s = n % NST;
      if (!mbar_wait_warp(&g_full[s], (uint32_t)(n / NST) & 1u, abort_flag, ctl, kid | W_GFULL) ||
          !mbar_wait_warp(s_full, (uint32_t)n & 1u, abort_flag, ctl, kid | W_S)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* l4 = reinterpret_cast<const float4*>(sStage + s * T::STAGE_BYTES + 2 * T::B_BYTES) + q0 / 4;
      const float4* d4 = l4 + BETA / 4;
      uint32_t x[W];
      uint64_t p2[W / 2];                          // P^T of this row's W queries, fp32 pairs
      tmem_ld_w<W>(cs, x);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pw[W / 4];
#pragma unroll
        for (int q = c * (W / 8); q < (c + 1) * (W / 8); ++q) {
          const float4 L = l4[q];                  // -lse*log2(e) of four queries
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i0 = 4 * q + 2 * e;
            float x0, x1;
            f2_unpack(fma2(f2_pack(__uint_as_float(x[i0]), __uint_as_float(x[i0 + 1])), c2,
                           e ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y)), x0, x1);
            const float a = ex2(x0), b = ex2(x1);
            p2[2 * q + e] = f2_pack(a, b);
            pw[2 * q + e - c * (W / 4)] = pack_bf16x2(a, b);
          }
        }
        // each warp overwrites only the TMEM lanes and columns it has read
        tmem_st_w<W / 4>(cs + c * (W / 4), pw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[c]);
      }
      if (!mbar_wait_warp(dp_full, (uint32_t)n & 1u, abort_flag, ctl, kid | W_S)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld_w<W>(cp, x);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dw[W / 4];
#pragma unroll
        for (int q = c * (W / 8); q < (c + 1) * (W / 8); ++q) {
          const float4 Dd = d4[q];                 // D of four queries
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i0 = 4 * q + 2 * e;
            const uint64_t t = sub2(f2_pack(__uint_as_float(x[i0]), __uint_as_float(x[i0 + 1])),
                                    e ? f2_pack(Dd.z, Dd.w) : f2_pack(Dd.x, Dd.y));
            float d0, d1;
            f2_unpack(mul2(p2[2 * q + e], t), d0, d1);
            dw[2 * q + e - c * (W / 4)] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st_w<W / 4>(cp + c * (W / 4), dw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full[c]);
      }
    }
    if (ok) ok = mbar_wait_warp(acc_done, 0, abort_flag, ctl, kid | W_ACC);
    if (ok) {
      tc_fence_after();
      const long long orow = krow0 + kr;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t col = (t == 0 ? T::DV_COL : T::DK_COL) + hf * (D / 2);
        const float mul = t == 0 ? 1.0f : scale;
        __nv_bfloat16* outp = (t == 0 ? dV : dK) + orow * D + hf * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + col + c * 32, o);
          tmem_ld_wait();
          if (kr < BETA) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
            uint4* dst = reinterpret_cast<uint4*>(outp + c * 32);
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
  if (warp == 1) tmem_dealloc(tmem_base, T::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// dQ: persistent CTAs over the query groups
// ---------------------------------------------------------------------------
template <int BETA, int D>
struct QTraits {
  static constexpr int BM = 128;
  static constexpr int NCH = D / 64;
  static constexpr int A_CHUNK = BM * 128;         // Q_g and dO_g as the A operands of S and dP (padded rows)
  static constexpr int A_BYTES = NCH * A_CHUNK;
  static constexpr int KV_CHUNK = BETA * 128;
  static constexpr int KV_BYTES = NCH * KV_CHUNK;
  // K_j is read by S (early) and by dQ (late); V_j only by dP: separate rings,
  // each slot released as soon as its last product is done.
  static constexpr int NK = 3;
  static constexpr int NV = (2 * A_BYTES + 6 * KV_BYTES + 2048 <= 227 * 1024) ? 3 : 2;
  static constexpr int NBAR = 2 + 2 * NK + 2 * NV + 2 + 2 + 3;
  static constexpr int SMEM_USED = 1024 + 2 * A_BYTES + (NK + NV) * KV_BYTES + NBAR * 8 + 16;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  // TMEM: S and dP (fp32), dQ (fp32), dS (bf16 pairs, BETA/2 columns).  S and
  // dP take both operands from shared memory (an M=128, N=128 product reads 8 KB
  // in its 64 clocks, the port's 128 B/clock); dQ takes dS from TMEM.
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256, DS_COL = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TX_BYTES = BETA * D * 2;
  static constexpr int HALF = BETA / 2;
};

template <int BETA, int D>
__global__ void __launch_bounds__(kQThreads, 1)
    attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                      const float* __restrict__ L2w, const float* __restrict__ Dw,
                      const int32_t* __restrict__ fwd_ptr, const int32_t* __restrict__ fwd_col, long long items,
                      int N, int G, float scale, __nv_bfloat16* __restrict__ dQ, Ctl ctl) {
  using T = QTraits<BETA, D>;
  constexpr int NK = T::NK, NV = T::NV;
  constexpr int HALF = T::HALF;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sbase = smem_align1024(smem_raw);
  uint8_t* sdO = sbase;
  uint8_t* sQ = sdO + T::A_BYTES;
  uint8_t* sK = sQ + T::A_BYTES;
  uint8_t* sV = sK + NK * T::KV_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NV * T::KV_BYTES);
  uint64_t* qd_full = bars;                       // Q_g and dO_g landed in smem
  uint64_t* q_spare = bars + 1;                   // (unused)
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
  uint64_t* sp_free = s_full + 1;                 // compute threads have read S, dP
  uint64_t* ds_full = sp_free + 1;
  uint64_t* ds_empty = ds_full + 1;
  uint64_t* acc_done = ds_empty + 1;              // dQ of the current group is complete
  uint64_t* mma_drain = acc_done + 1;
  uint64_t* qd_free = mma_drain + 1;              // the current group's last dP product is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qd_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = G;
  const unsigned int kid = (unsigned int)KID_BWD_Q << 8;

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    mbar_init(q_spare, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(sp_free, kComputeThreads);
    mbar_init(ds_full, kComputeThreads);
    mbar_init(ds_empty, 1);
    mbar_init(acc_done, 1);
    mbar_init(mma_drain, 1);
    mbar_init(qd_free, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (BETA < T::BM) {
    for (int c = 0; c < T::NCH; ++c) {
      for (int t = 0; t < 2; ++t) {
        uint4* z = reinterpret_cast<uint4*>(sdO + t * T::A_BYTES + c * T::A_CHUNK + BETA * 128);
        for (int i = threadIdx.x; i < (T::BM - BETA) * 128 / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
      }
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
  // Every CTA owns its SM's whole TMEM (512 columns), so the allocation starts
  // at lane 0, column 0: with that constant every TMEM address is known at
  // compile time and the MMA warp spends no instructions moving them into
  // uniform registers.  A different address is reported and nothing is run.
  const uint32_t tmem_base = *tmem_slot;
  constexpr uint32_t tmem = 0;

  // The CTA works through groups blockIdx.x, blockIdx.x + gridDim.x, ...
  // Every role counts the pairs of the groups before the current one (gq: the
  // global pair index of ring slots and barrier phases) and the non-empty
  // groups (ne: the phase of qd_full, qd_free and acc_done), so the next group's
  // dO, K and V tiles load while the compute warps finish the current group.
  if (tmem_base != tmem) {
    if (threadIdx.x == 0) set_error(ctl, DSV_ERR_INTERNAL, blockIdx.x);
  } else if (warp == 0 || warp == kQVWarp) {
    // TMA producers, one per warp: warp 0 loads dO_g and the K ring,
    // warp 10 the V ring
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      const int nst = is_k ? NK : NV;
      uint8_t* ring = is_k ? sK : sV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      tma_prefetch_desc(map);
      if (is_k) {
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmQ);
      }
      uint32_t gq = 0;                            // tiles issued so far
      int qd_issued = 0;
      bool ok = true;
      ItemCursor cur(fwd_ptr, nullptr, items, false);
      long long row;
      int start, cnt;
      while (ok && cur.next(row, start, cnt)) {
        if (cnt <= 0) continue;
        const long long bh = row / G;
        const int g = (int)(row - bh * G);
        if (is_k) {
          // Q_g and dO_g are the A operands of every S and dP product: the
          // previous group's last ones must be done.  qd_free (one phase per
          // group) is at most one phase behind here; the per-pair s_full could
          // be two behind, and its parity would then alias.
          if (qd_issued > 0 && !mbar_wait(qd_free, (uint32_t)(qd_issued - 1) & 1u, abort_flag, ctl, kid | W_KVEMPTY))
            break;
          mbar_arrive_expect_tx(qd_full, 2 * T::TX_BYTES);
          const int qrow = (int)(bh * N + (long long)g * BETA);
          for (int c = 0; c < T::NCH; ++c) {
            tma_load_2d(sdO + c * T::A_CHUNK, &tmdO, qd_full, c * 64, qrow);
            tma_load_2d(sQ + c * T::A_CHUNK, &tmQ, qd_full, c * 64, qrow);
          }
          ++qd_issued;
        }
        int jn = fwd_col[start];
        for (int n = 0; n < cnt; ++n) {
          const int s = (int)(gq % (uint32_t)nst);
          const uint32_t ph = (gq / (uint32_t)nst) & 1u;
          int j = jn;
          if (n + 1 < cnt) jn = fwd_col[start + n + 1];
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, ctl, kid | W_KVEMPTY)) {
            ok = false;
            break;
          }
          if ((unsigned)j >= (unsigned)nb) {
            if (is_k) set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
            j = 0;
          }
          const int krow = (int)(bh * N + (long long)j * BETA);
          mbar_arrive_expect_tx(&full[s], T::TX_BYTES);
          for (int c = 0; c < T::NCH; ++c)
            tma_load_2d(ring + s * T::KV_BYTES + c * T::KV_CHUNK, map, &full[s], c * 64, krow);
          ++gq;
        }
      }
      // every copy this thread started must land before the CTA exits
      if (is_k && qd_issued > 0) mbar_wait(qd_full, (uint32_t)(qd_issued - 1) & 1u, nullptr, ctl, kid | W_DRAIN);
      for (uint32_t n = (gq > (uint32_t)nst ? gq - (uint32_t)nst : 0u); n < gq; ++n)
        mbar_wait(&full[n % (uint32_t)nst], (n / (uint32_t)nst) & 1u, nullptr, ctl, kid | W_DRAIN);
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
      constexpr uint32_t ID_S = idesc_bf16_f32(T::BM, BETA, false, false);
      constexpr uint32_t ID_Q = idesc_bf16_f32(T::BM, D, false, true);
      const uint64_t ddO0 = sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dKmn0 = sdesc_sw128(smem_u32(sK), T::KV_CHUNK, 1024);
      // tk / tv: early tests of K_n / V_n (see mbar_test); td: of dS of block n-1
      auto issue_sdp = [&](uint32_t gn, uint32_t tk, uint32_t tv, uint32_t* td) -> bool {
        const int sk = (int)(gn % NK), sv = (int)(gn % NV);
        if (!mbar_wait_warp_tested(&k_full[sk], (gn / NK) & 1u, tk, abort_flag, ctl, kid | W_KFULL)) return false;
        tc_fence_after();
        const uint64_t kb = desc_off(dK0, (uint32_t)sk * T::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t bo = (kk >> 2) * T::KV_CHUNK + (kk & 3) * 32;
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          mma_ss_w(tmem + T::S_COL, desc_off(dQ0, ao), desc_off(kb, bo), ID_S, kk > 0 ? 1u : 0u);
        }
        if (td != nullptr) *td = mbar_test(ds_full, (gn - 1) & 1u);
        if (!mbar_wait_warp_tested(&v_full[sv], (gn / NV) & 1u, tv, abort_flag, ctl, kid | W_VFULL)) return false;
        tc_fence_after();
        const uint64_t vb = desc_off(dV0, (uint32_t)sv * T::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * T::A_CHUNK + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * T::KV_CHUNK + (kk & 3) * 32;
          mma_ss_w(tmem + T::DP_COL, desc_off(ddO0, ao), desc_off(vb, bo), ID_S, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(s_full);
        mma_commit_w(&v_empty[sv]);   // V_j is only needed by dP
        return true;
      };
      uint32_t gq = 0;
      int ne = 0;
      bool ok = true;
      ItemCursor cur(fwd_ptr, nullptr, items, false);
      long long row;
      int start, cnt;
      while (ok && cur.next(row, start, cnt)) {
        if (cnt <= 0) continue;
        // S and dP are single-buffered: the previous group's last ones must
        // have been read by the compute warps (sp_free of its last pair)
        ok = mbar_wait_warp(qd_full, (uint32_t)ne & 1u, abort_flag, ctl, kid | W_KV) &&
             (gq == 0 || mbar_wait_warp(sp_free, (gq - 1) & 1u, abort_flag, ctl, kid | W_SPFREE));
        if (ok) ok = issue_sdp(gq, 0u, 0u, nullptr);
        if (ok && cnt == 1) mma_commit_w(qd_free);    // the group's last read of dO_g
        for (int n = 0; ok && n < cnt; ++n) {
          const uint32_t gn = gq + (uint32_t)n;
          uint32_t td = 0u;
          if (n + 1 < cnt) {
            const uint32_t tk = mbar_test(&k_full[(gn + 1) % NK], ((gn + 1) / NK) & 1u);
            const uint32_t tv = mbar_test(&v_full[(gn + 1) % NV], ((gn + 1) / NV) & 1u);
            // S and dP are single-buffered: overwrite them once the compute warps hold block n
            if (!mbar_wait_warp(sp_free, gn & 1u, abort_flag, ctl, kid | W_SPFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (!issue_sdp(gn + 1, tk, tv, &td)) {
              ok = false;
              break;
            }
            if (n + 2 == cnt) mma_commit_w(qd_free);    // the group's last read of dO_g
          }
          // ds_full of a group's first pair also means the compute warps have
          // read the previous group's dQ
          if (!mbar_wait_warp_tested(ds_full, gn & 1u, td, abort_flag, ctl, kid | W_DSFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int s = (int)(gn % NK);
          const uint64_t kmn = desc_off(dKmn0, (uint32_t)s * T::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < BETA / 16; ++kk) {
            mma_ts_w(tmem + T::DQ_COL, tmem + T::DS_COL + kk * 8, desc_off(kmn, kk * 16 * 128), ID_Q,
                     (n > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_w(&k_empty[s]);
          mma_commit_w(ds_empty);
        }
        if (!ok) break;
        mma_commit_w(acc_done);
        gq += (uint32_t)cnt;
        ++ne;
      }
      // TMEM is freed after the closing CTA-wide sync only once every MMA is done
      mma_commit_w(mma_drain);
      mbar_wait_warp(mma_drain, 0, nullptr, ctl, kid | W_DRAIN);
    }
  } else if (warp < kQVWarp) {
    // ------------- compute warps: query row r, key half hf -------------
    const int sp = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = sp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    const float scale_log2 = scale * kLog2e;
    bool ok = true;
    uint32_t gq = 0;
    int ne = 0;
    ItemCursor cur(fwd_ptr, nullptr, items, false);
    long long row;
    int start, cnt;
    while (ok && cur.next(row, start, cnt)) {
      const long long bh = row / G;
      const int g = (int)(row - bh * G);
      const long long qrow0 = bh * N + (long long)g * BETA;
      const long long orow = qrow0 + r;
      if (cnt <= 0) {
        // empty (or malformed) list: dQ = 0
        if (cnt < 0 && r == 0 && hf == 0) set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
        if (r < BETA) {
          uint4* dst = reinterpret_cast<uint4*>(dQ + orow * D + hf * (D / 2));
#pragma unroll
          for (int q = 0; q < D / 16; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const float nlse2 = (r < BETA) ? L2w[orow] : 0.f;   // -lse*log2(e)
      const float dd = (r < BETA) ? Dw[orow] : 0.f;

      uint32_t s_tested = 0u;
      for (int n = 0; n < cnt; ++n) {
        const uint32_t gn = gq + (uint32_t)n;
        if (!mbar_wait_warp_tested(s_full, gn & 1u, s_tested, abort_flag, ctl, kid | W_S)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t xs[HALF], xp[HALF];
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) {
          tmem_ld32(tmem + lane_off + T::S_COL + hf * HALF + c * 32, xs + c * 32);
          tmem_ld32(tmem + lane_off + T::DP_COL + hf * HALF + c * 32, xp + c * 32);
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(sp_free);
        const uint32_t e_tested = mbar_test(ds_empty, (gn & 1u) ^ 1u);
        // exponent, dP - D and dS on packed fp32 pairs
        uint32_t dw[HALF / 2];
        const uint64_t c2 = f2_pack(scale_log2, scale_log2), nl2 = f2_pack(nlse2, nlse2), dd2 = f2_pack(dd, dd);
#pragma unroll
        for (int i = 0; i < HALF / 2; ++i) {
          float x0, x1, d0, d1;
          f2_unpack(fma2(f2_pack(__uint_as_float(xs[2 * i]), __uint_as_float(xs[2 * i + 1])), c2, nl2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          const uint64_t t = sub2(f2_pack(__uint_as_float(xp[2 * i]), __uint_as_float(xp[2 * i + 1])), dd2);
          f2_unpack(mul2(f2_pack(p0, p1), t), d0, d1);
          dw[i] = pack_bf16x2(d0, d1);
        }
        // the single dS buffer is free once dQ of the previous block is done
        if (n + 1 < cnt) s_tested = mbar_test(s_full, (gn + 1) & 1u);
        if (!mbar_wait_warp_tested(ds_empty, (gn & 1u) ^ 1u, e_tested, abort_flag, ctl, kid | W_DSEMPTY)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c)
          tmem_st16(tmem + lane_off + T::DS_COL + hf * (HALF / 2) + c * 16, dw + c * 16);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (ok) ok = mbar_wait_warp(acc_done, (uint32_t)ne & 1u, abort_flag, ctl, kid | W_ACC);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + T::DQ_COL + hf * (D / 2) + c * 32, o);
        tmem_ld_wait();
        if (r < BETA) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * scale, __uint_as_float(o[2 * i + 1]) * scale);
          uint4* dst = reinterpret_cast<uint4*>(dQ + orow * D + hf * (D / 2) + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      gq += (uint32_t)cnt;
      ++ne;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, T::TMEM_COLS);
}

// The order in which the dK/dV kernel takes its key blocks, per chunk of
// consecutive (b, h) slices (one CTA per chunk; chunks keep their order and
// hold as many heads as leave their Q and dO in a part of L2).  Inside a
// chunk the few blocks whose transposed list is far longer than the chunk's
// mean (more than kLongFactor times it: the blocks nearly every group picks)
// go first, longest first, so that none of them starts in the grid's last
// wave; every other block follows in its natural order.  Blocks that run
// together are then neighbours in the latent, chosen by largely the same
// query groups, so the Q and dO tiles they load are shared in L2: on a
// 518k-token head (266 MB of Q and dO) ordering all blocks by list length
// instead spread the CTAs running together over the whole head and re-read
// its Q and dO from HBM ~44 times per launch.  Ties among long blocks in any
// order: a block's result does not depend on when it runs.
constexpr int kOrderThreads = 256;
constexpr int kMaxOrderLen = kMaxBlocksPerRow;   // a list holds at most G groups
constexpr int kLongFactor = 4;
__global__ void __launch_bounds__(kOrderThreads) kv_order_kernel(const int32_t* __restrict__ bwd_ptr,
                                                                 long long rows, int chunk, int maxlen,
                                                                 int32_t* __restrict__ order) {
  __shared__ int32_t cnt[kMaxOrderLen + 1];
  __shared__ int32_t wtot[kOrderThreads / 32];
  __shared__ int32_t s_nlong;
  const long long base = (long long)blockIdx.x * chunk;
  const int nb = (int)(rows - base < chunk ? rows - base : chunk);   // rows of this chunk
  const int32_t* P = bwd_ptr + base;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  // long: more than kLongFactor times the chunk's mean list length (and at least 64 groups)
  const long long total = (long long)P[nb] - P[0];
  const int thr = (int)max(64LL, kLongFactor * ((total + nb - 1) / nb));
  for (int i = t; i <= maxlen; i += kOrderThreads) cnt[i] = 0;
  if (t == 0) s_nlong = 0;
  __syncthreads();
  for (int r = t; r < nb; r += kOrderThreads) {
    const int len = min(maxlen, max(0, P[r + 1] - P[r]));
    if (len > thr) {
      atomicAdd(&cnt[len], 1);
      atomicAdd(&s_nlong, 1);
    }
  }
  __syncthreads();
  // long blocks: exclusive scan of their counts from the longest length down
  const int per = (maxlen + 1 + kOrderThreads - 1) / kOrderThreads;
  const int b0 = t * per;            // this thread's lengths, counted from the top: maxlen - b0 ...
  int loc = 0;
  for (int q = b0; q < min(maxlen + 1, b0 + per); ++q) loc += cnt[maxlen - q];
  int inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wtot[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = lane < kOrderThreads / 32 ? wtot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += v;
    }
    if (lane < kOrderThreads / 32) wtot[lane] = x;
  }
  __syncthreads();
  int run = (w > 0 ? wtot[w - 1] : 0) + inc - loc;
  for (int q = b0; q < min(maxlen + 1, b0 + per); ++q) {
    const int c = cnt[maxlen - q];
    cnt[maxlen - q] = run;
    run += c;
  }
  __syncthreads();
  for (int r = t; r < nb; r += kOrderThreads) {
    const int len = min(maxlen, max(0, P[r + 1] - P[r]));
    if (len > thr) order[base + atomicAdd(&cnt[len], 1)] = (int32_t)(base + r);
  }
  // the other blocks in natural order after them: exclusive scan of "short" over consecutive runs of rows
  const int nlong = s_nlong;
  const int span = (nb + kOrderThreads - 1) / kOrderThreads;
  const int r0 = t * span, r1 = min(nb, r0 + span);
  int mine = 0;
  for (int r = r0; r < r1; ++r) mine += (min(maxlen, max(0, P[r + 1] - P[r])) > thr) ? 0 : 1;
  __syncthreads();                   // wtot is reused
  int sinc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, sinc, o);
    if (lane >= o) sinc += v;
  }
  if (lane == 31) wtot[w] = sinc;
  __syncthreads();
  if (w == 0) {
    int x = lane < kOrderThreads / 32 ? wtot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += v;
    }
    if (lane < kOrderThreads / 32) wtot[lane] = x;
  }
  __syncthreads();
  int pos = nlong + (w > 0 ? wtot[w - 1] : 0) + sinc - mine;
  for (int r = r0; r < r1; ++r)
    if (min(maxlen, max(0, P[r + 1] - P[r])) <= thr) order[base + pos++] = (int32_t)(base + r);
}

template <int BETA, int D>
cudaError_t launch_kv_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const CUtensorMap& tmdO, const dsv_shape& s, const int32_t* bwd_ptr, const int32_t* bwd_col,
                        float scale, void* dK, void* dV, const float* Dw, const float* L2w, int32_t* order,
                        const Ctl& ctl, cudaStream_t st) {
  const int G = s.N / s.block;
  const long long groups = (long long)s.B * s.H * G;
  // heads per chunk: their Q and dO within ~48 MB of L2
  const long long head_bytes = 2LL * s.N * s.d * 2;
  const long long heads = (long long)s.B * s.H;
  long long hpc = (48LL << 20) / (head_bytes > 0 ? head_bytes : 1);
  hpc = hpc < 1 ? 1 : (hpc > heads ? heads : hpc);
  const long long chunk = hpc * G;
  kv_order_kernel<<<(unsigned)((groups + chunk - 1) / chunk), kOrderThreads, 0, st>>>(
      bwd_ptr, groups, (int)chunk, G < kMaxOrderLen ? G : kMaxOrderLen, order);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kv = attn_bwd_kv_kernel<BETA, D>;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, KVTraits<BETA, D>::SMEM)) !=
      cudaSuccess)
    return e;
  kv<<<(unsigned)groups, kThreads, KVTraits<BETA, D>::SMEM, st>>>(tmQ, tmK, tmV, tmdO, L2w, Dw, bwd_ptr, bwd_col,
                                                                   order, s.N, G, scale,
                                                                   static_cast<__nv_bfloat16*>(dK),
                                                                   static_cast<__nv_bfloat16*>(dV), ctl);
  return cudaGetLastError();
}

template <int BETA, int D>
cudaError_t launch_q_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmdO,
                       const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col, float scale, void* dQ,
                       const float* Dw, const float* L2w, const Ctl& ctl, cudaStream_t st) {
  const int G = s.N / s.block;
  const long long groups = (long long)s.B * s.H * G;
  auto qk = attn_bwd_q_kernel<BETA, D>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(qk, cudaFuncAttributeMaxDynamicSharedMemorySize, QTraits<BETA, D>::SMEM)) !=
      cudaSuccess)
    return e;
  // persistent: one CTA per SM (the CTA holds the SM's whole TMEM)
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)(groups < nsm ? groups : nsm);
  qk<<<grid, kQThreads, QTraits<BETA, D>::SMEM, st>>>(tmQ, tmK, tmV, tmdO, L2w, Dw, fwd_ptr, fwd_col, groups, s.N,
                                                      G, scale, static_cast<__nv_bfloat16*>(dQ), ctl);
  return cudaGetLastError();
}

// workspace: D_i, then -lse_i * log2(e), each B*H*N floats, then the dK/dV
// kernel's block order (B*H*nb ints), each part 256-byte aligned
const float* ws_D(const void* ws) { return static_cast<const float*>(ws); }
const float* ws_L2(const void* ws, const dsv_shape& s) {
  return reinterpret_cast<const float*>(static_cast<const char*>(ws) +
                                        align256((size_t)s.B * s.H * s.N * sizeof(float)));
}
int32_t* ws_order(const void* ws, const dsv_shape& s) {
  return reinterpret_cast<int32_t*>(const_cast<char*>(static_cast<const char*>(ws)) +
                                    2 * align256((size_t)s.B * s.H * s.N * sizeof(float)));
}

}  // namespace

size_t attn_bwd_ws_bytes(const dsv_shape& s) {
  return 2 * align256((size_t)s.B * s.H * s.N * sizeof(float)) +   // D and -lse*log2(e)
         align256((size_t)s.B * s.H * (s.N / s.block) * sizeof(int32_t));   // dK/dV block order
}

cudaError_t launch_attn_bwd_pre(const void* O, const void* dO, const float* lse, const dsv_shape& s, void* ws,
                                cudaStream_t st) {
  const long long rows = (long long)s.B * s.H * s.N;
  float* Dw = static_cast<float*>(ws);
  float* L2w = const_cast<float*>(ws_L2(ws, s));
  const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(O);
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(dO);
  if (s.d == 128) {
    constexpr int RPC = 256 / (128 / 8);
    bwd_rowdot_kernel<128><<<(unsigned)((rows + RPC - 1) / RPC), 256, 0, st>>>(o, g, lse, Dw, L2w, rows);
  } else {
    constexpr int RPC = 256 / (64 / 8);
    bwd_rowdot_kernel<64><<<(unsigned)((rows + RPC - 1) / RPC), 256, 0, st>>>(o, g, lse, Dw, L2w, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_kv(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const CUtensorMap& tmdO, const dsv_shape& s, const int32_t* bwd_ptr,
                               const int32_t* bwd_col, float scale, void* dK, void* dV, void* ws,
                               const Ctl& ctl, cudaStream_t st) {
#define DSV_KV(BE, DD) \
  return launch_kv_t<BE, DD>(tmQ, tmK, tmV, tmdO, s, bwd_ptr, bwd_col, scale, dK, dV, ws_D(ws), ws_L2(ws, s), \
                             ws_order(ws, s), ctl, st)
  if (s.block == 128 && s.d == 128) DSV_KV(128, 128);
  if (s.block == 128 && s.d == 64) DSV_KV(128, 64);
  if (s.block == 64 && s.d == 128) DSV_KV(64, 128);
  DSV_KV(64, 64);
#undef DSV_KV
}

cudaError_t launch_attn_bwd_q(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmdO,
                              const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col, float scale,
                              void* dQ, const void* ws, const Ctl& ctl, cudaStream_t st) {
#define DSV_Q(BE, DD) \
  return launch_q_t<BE, DD>(tmQ, tmK, tmV, tmdO, s, fwd_ptr, fwd_col, scale, dQ, ws_D(ws), ws_L2(ws, s), ctl, st)
  if (s.block == 128 && s.d == 128) DSV_Q(128, 128);
  if (s.block == 128 && s.d == 64) DSV_Q(128, 64);
  if (s.block == 64 && s.d == 128) DSV_Q(64, 128);
  DSV_Q(64, 64);
#undef DSV_Q
}

cudaError_t launch_attn_bwd(const void* Q, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmdO, const void* O, const void* dO, const float* lse,
                            const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col,
                            const int32_t* bwd_ptr, const int32_t* bwd_col, float scale, void* dQ, void* dK,
                            void* dV, void* ws, const Ctl& ctl, cudaStream_t st) {
  cudaError_t e = launch_attn_bwd_pre(O, dO, lse, s, ws, st);
  if (e != cudaSuccess) return e;
  if ((e = launch_attn_bwd_kv(tmQ, tmK, tmV, tmdO, s, bwd_ptr, bwd_col, scale, dK, dV, ws, ctl, st)) != cudaSuccess)
    return e;
  (void)Q;
  return launch_attn_bwd_q(tmQ, tmK, tmV, tmdO, s, fwd_ptr, fwd_col, scale, dQ, ws, ctl, st);
}

}  // namespace dsv
