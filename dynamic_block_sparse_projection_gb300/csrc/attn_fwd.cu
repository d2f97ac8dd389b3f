// attn_fwd.cu — block-sparse softmax attention forward on tcgen05 tensor cores.
//
// DSV page [nl], "Technische samenvatting" 2A (stage 2: only the critical
// subset of KV pairs is computed) and 2B (a query group shares its critical
// KV indices); [hi] 2B (grouping maximises coalescing and tensor-core use).
//
// Persistent CTAs, one per SM, each working through query groups (b, h, g)
// blockIdx.x, blockIdx.x + gridDim.x, ...: the group's `block` query rows form
// the M = 128 rows of every MMA (for block = 64 the upper 64 rows are zero
// padding).  For each key block j in the group's list:
//   S = Q K_j^T            tcgen05.mma, A = Q (smem), B = K_j (smem), D in TMEM
//   P = exp2(S*c - m)      softmax warpgroup, P written back to TMEM as bf16
//   O += P V_j             tcgen05.mma, A = P (TMEM), B = V_j (smem, MN-major)
// with an online softmax whose reference m is the first block's row maximum:
// a later block keeps it unless one of its values of P would exceed 2^64 (its
// block sum tells), and only then are the block's maximum taken, O rescaled
// and the block redone, so the common path computes no row maximum.
//
// Warp roles (224 threads):
//   warp 0      TMA producer of Q and the K_j ring (one lane).
//   warp 1      TMEM allocator and MMA issuer (the whole warp, one elected
//               lane issues each MMA and commit).
//   warps 2..5  softmax / epilogue; warp w owns TMEM lanes 32*(w%4)..+31,
//               i.e. one query row per thread.
//   warp 6      TMA producer of the V_j ring (one lane).
// TMEM columns: three S/P buffers at [0,128), [128,256), [256,384) and O at
// [384,384+d).  With three buffers the MMA warp queues S of block n+2 before
// it waits for P of block n, so the tensor core always has the next S
// products queued while the softmax runs, and the softmax of block n+1 can
// start as soon as that of block n is done.
//
// The rings, S/P buffers and barrier phases run on across groups, so the next
// group's Q and first K/V tiles load, and its first S products run, while the
// softmax warps finish the current group; the next group's first PV product
// waits for its P(0), which the softmax warps write only after they have read
// the current group's O.
//
// Ring slots are released without extra barriers: K slot n%3 is free once
// S(n) is done (s_full), V slot n%3 once O += P(n) V_n is done (o_done); the
// producer of tile n+3 waits for exactly that phase, which cannot be
// overtaken because S(n+3) / PV(n+3) need the very tile it is about to load.
#include <math.h>

#include "dsv_launch.h"

namespace dsv {

namespace {

template <int BETA, int D>
struct FwdTraits {
  static constexpr int BM = 128;                 // MMA M (query rows incl. padding)
  static constexpr int NCH = D / 64;             // 64-column (128-byte) chunks along d
  static constexpr int Q_CHUNK = BM * 128;       // bytes of one Q chunk
  static constexpr int KV_CHUNK = BETA * 128;    // bytes of one K or V chunk
  static constexpr int Q_BYTES = NCH * Q_CHUNK;
  static constexpr int KV_BYTES = NCH * KV_CHUNK;
  static constexpr int NST = 3;                  // K and V ring slots = S/P buffers
  static constexpr int NBAR = 1 + 2 * NST + 3 * NST + 2;
  static constexpr int SMEM_USED = 1024 + Q_BYTES + 2 * NST * KV_BYTES + NBAR * 8 + 16;
  static_assert(SMEM_USED <= 227 * 1024, "forward tiles exceed shared memory");
  // at least 120 KB so that one CTA owns an SM (and its 512 TMEM columns)
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t S_COL = 128;         // column stride of the S/P buffers
  static constexpr uint32_t O_COL = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TX_BYTES = BETA * D * 2;   // one K or V tile (and the Q tile)
};

constexpr int kVWarp = 6;                // V producer warp
constexpr int kFwdThreads = 224;         // 7 warps

enum : unsigned int { W_Q = 1, W_KEMPTY, W_K, W_P, W_V, W_S, W_O, W_OFINAL, W_DRAIN, W_QEMPTY };

template <int BETA, int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const int32_t* __restrict__ fwd_ptr,
                    const int32_t* __restrict__ fwd_col, long long rows, int N, int G, int nb, float scale_log2,
                    __nv_bfloat16* __restrict__ O, float* __restrict__ LSE, Ctl ctl) {
  using T = FwdTraits<BETA, D>;
  constexpr int NST = T::NST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sbase = smem_align1024(smem_raw);
  uint8_t* sQ = sbase;
  uint8_t* sK = sQ + T::Q_BYTES;
  uint8_t* sV = sK + NST * T::KV_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NST * T::KV_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* s_full = v_full + NST;    // [3] S(n) in buffer n%3; also frees K slot n%3
  uint64_t* p_full = s_full + NST;    // [3] P(n) written over S(n)
  uint64_t* o_done = p_full + NST;    // [3] O += P(n) V_n done; also frees V slot n%3
  uint64_t* o_final = o_done + NST;   // all PV products of the current row are done
  uint64_t* mma_drain = o_final + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned int kid = (unsigned int)KID_FWD << 8;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
      mbar_init(&o_done[s], 1);
    }
    mbar_init(o_final, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (BETA < T::BM) {
    // rows BETA..127 of every Q chunk are never loaded: make them zero
    for (int c = 0; c < T::NCH; ++c) {
      uint4* z = reinterpret_cast<uint4*>(sQ + c * T::Q_CHUNK + BETA * 128);
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

  // The CTA works through rows blockIdx.x, blockIdx.x + gridDim.x, ... (rows
  // with an empty list only get their zero output).  Every role counts the
  // key blocks of the rows before the current one (gq, the global index of
  // ring slots, S/P buffers and their barrier phases) and the non-empty rows
  // (ne, the phase of q_full and o_final), so the next row's Q and first K/V
  // tiles load, and its first S products run, while the softmax warps finish
  // the current row.
  if (tmem_base != tmem) {
    if (threadIdx.x == 0) set_error(ctl, DSV_ERR_INTERNAL, blockIdx.x);
  } else if (warp == 0 || warp == kVWarp) {
    // ---------------- TMA producers: warp 0 loads Q and the K ring, warp 6 the V ring ----------------
    // One producer per warp: lanes of one warp spinning on different barriers
    // would serialise each other.
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      uint8_t* ring = is_k ? sK : sV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* freed = is_k ? s_full : o_done;   // phase n of slot n%3: its last reader is done
      tma_prefetch_desc(map);
      if (is_k) tma_prefetch_desc(&tmQ);
      uint32_t gq = 0;                            // tiles issued so far
      int q_issued = 0;
      bool ok = true;
      ItemCursor cur(fwd_ptr, nullptr, rows, false);
      long long row;
      int start, cnt;
      while (ok && cur.next(row, start, cnt)) {
        if (cnt <= 0) continue;
        const long long bh = row / G;
        const int g = (int)(row - bh * G);
        if (is_k) {
          // Q is the A operand of every S product: the previous row's last one must be done
          if (q_issued > 0 &&
              !mbar_wait(&s_full[(gq - 1) % NST], (uint32_t)((gq - 1) / NST) & 1u, abort_flag, ctl, kid | W_QEMPTY))
            break;
          const int qrow = (int)(bh * N + (long long)g * BETA);
          mbar_arrive_expect_tx(q_full, T::TX_BYTES);
          for (int c = 0; c < T::NCH; ++c) tma_load_2d(sQ + c * T::Q_CHUNK, &tmQ, q_full, c * 64, qrow);
          ++q_issued;
        }
        int jn = fwd_col[start];
        for (int n = 0; n < cnt; ++n) {
          const int s = (int)(gq % NST);
          int j = jn;
          if (n + 1 < cnt) jn = fwd_col[start + n + 1];
          if (gq >= NST &&
              !mbar_wait(&freed[s], (uint32_t)((gq - NST) / NST) & 1u, abort_flag, ctl, kid | W_KEMPTY)) {
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
      if (is_k && q_issued > 0) mbar_wait(q_full, (uint32_t)(q_issued - 1) & 1u, nullptr, ctl, kid | W_DRAIN);
      for (uint32_t n = (gq > NST ? gq - NST : 0u); n < gq; ++n)
        mbar_wait(&full[n % NST], (uint32_t)(n / NST) & 1u, nullptr, ctl, kid | W_DRAIN);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t IDS = idesc_bf16_f32(T::BM, BETA, false, false);
    constexpr uint32_t IDO = idesc_bf16_f32(T::BM, D, false, true);
    // base descriptors; every MMA adds a compile-time offset
    const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_u32(sV), T::KV_CHUNK, 1024);
    // S(n) = Q K_n^T into buffer n%3
    auto issue_S = [&](uint32_t gn, int n) -> bool {
      const int s = (int)(gn % NST);
      if (!mbar_wait_warp(&k_full[s], (uint32_t)(gn / NST) & 1u, abort_flag, ctl, kid | W_K)) return false;
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)s * T::S_COL;
      const uint64_t kb = desc_off(dK0, (uint32_t)s * T::KV_BYTES);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        mma_ss_w(d_tmem, desc_off(dQ0, (kk >> 2) * T::Q_CHUNK + (kk & 3) * 32),
                 desc_off(kb, (kk >> 2) * T::KV_CHUNK + (kk & 3) * 32), IDS, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(&s_full[s]);
      return true;
    };
    uint32_t gq = 0;
    int ne = 0;
    bool ok = true;
    ItemCursor cur(fwd_ptr, nullptr, rows, false);
    long long row;
    int start, cnt;
    while (ok && cur.next(row, start, cnt)) {
      if (cnt <= 0) continue;
      ok = mbar_wait_warp(q_full, (uint32_t)ne & 1u, abort_flag, ctl, kid | W_Q);
      if (ok) ok = issue_S(gq, 0);
      if (ok && cnt > 1) ok = issue_S(gq + 1, 1);
      for (int n = 0; ok && n < cnt; ++n) {
        // S(n+2) reuses the buffer of P(n-1), whose PV product is already queued
        const uint32_t gn = gq + (uint32_t)n;
        const int s = (int)(gn % NST);
        const uint32_t ph = (gn / NST) & 1u;
        const uint32_t v_tested = mbar_test(&v_full[s], ph);   // V_n normally landed long ago
        if (n + 2 < cnt && !issue_S(gn + 2, n + 2)) {
          ok = false;
          break;
        }
        // P(0) of a row also means the softmax warps have read the previous row's O
        if (!mbar_wait_warp(&p_full[s], ph, abort_flag, ctl, kid | W_P)) {
          ok = false;
          break;
        }
        if (!mbar_wait_warp_tested(&v_full[s], ph, v_tested, abort_flag, ctl, kid | W_V)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t p_tmem = tmem + (uint32_t)s * T::S_COL;
        const uint64_t vb = desc_off(dV0, (uint32_t)s * T::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < BETA / 16; ++kk) {
          mma_ts_w(tmem + T::O_COL, p_tmem + kk * 8, desc_off(vb, kk * 16 * 128), IDO, (n > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit_w(&o_done[s]);
      }
      if (!ok) break;
      mma_commit_w(o_final);
      gq += (uint32_t)cnt;
      ++ne;
    }
    // TMEM is freed after the closing CTA-wide sync only once every MMA is done
    mma_commit_w(mma_drain);
    mbar_wait_warp(mma_drain, 0, nullptr, ctl, kid | W_DRAIN);
  } else if (warp < kVWarp) {
    // ---------------- softmax warpgroup (warps 2..5) ----------------
    const int sp = warp & 3;
    const int r = sp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    uint32_t gq = 0;
    int ne = 0;
    bool ok = true;
    ItemCursor cur(fwd_ptr, nullptr, rows, false);
    long long row;
    int start, cnt;
    while (ok && cur.next(row, start, cnt)) {
      const long long bh = row / G;
      const int g = (int)(row - bh * G);
      const long long orow = bh * N + (long long)g * BETA + r;
      if (cnt <= 0) {
        // empty (or malformed) list: O = 0, lse = -inf
        if (cnt < 0 && r == 0) set_error(ctl, DSV_ERR_BAD_INDEX, (unsigned int)(row & 0x7fffffff));
        if (r < BETA) {
          uint4* dst = reinterpret_cast<uint4*>(O + orow * D);
#pragma unroll
          for (int q = 0; q < D / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
          LSE[orow] = -INFINITY;
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      uint32_t s_tested = 0u;   // S(n) already known complete (tested during block n-1)
      for (int n = 0; n < cnt; ++n) {
        const uint32_t gn = gq + (uint32_t)n;
        const int s = (int)(gn % NST);
        if (!mbar_wait_warp_tested(&s_full[s], (gn / NST) & 1u, s_tested, abort_flag, ctl, kid | W_S)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sb = tmem + lane_off + (uint32_t)s * T::S_COL;
        uint32_t xr[BETA];
#pragma unroll
        for (int c = 0; c < BETA / 32; ++c) tmem_ld32(sb + c * 32, xr + c * 32);
        s_tested = (n + 1 < cnt) ? mbar_test(&s_full[(gn + 1) % NST], ((gn + 1) / NST) & 1u) : 0u;
        tmem_ld_wait();
        // row max as 8 independent partial maxima (short dependency chains),
        // two new values per three-input max
        auto row_max = [&]() -> float {
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = __uint_as_float(xr[i]);
#pragma unroll
          for (int j = 8; j < BETA; j += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              mx8[i] = j + 8 < BETA ? max3f(mx8[i], __uint_as_float(xr[j + i]), __uint_as_float(xr[j + 8 + i]))
                                    : fmaxf(mx8[i], __uint_as_float(xr[j + i]));
          return fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        };
        // P = exp2(S c - m): exponent and row sum on packed fp32 pairs
        uint32_t pk[BETA / 2];
        auto exponentiate = [&](float mref) -> float {
          const uint64_t c2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-mref, -mref);
          uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int j = 0; j < BETA / 2; ++j) {
            float x0, x1;
            f2_unpack(fma2(f2_pack(__uint_as_float(xr[2 * j]), __uint_as_float(xr[2 * j + 1])), c2, nm2), x0, x1);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            rs2[j & 3] = add2(rs2[j & 3], f2_pack(p0, p1));
            pk[j] = pack_bf16x2(p0, p1);
          }
          float a0, a1;
          f2_unpack(add2(add2(rs2[0], rs2[1]), add2(rs2[2], rs2[3])), a0, a1);
          return a0 + a1;
        };
        // The running maximum is the first block's; a later block keeps it
        // unless one of its values would exceed 2^kLazyLog2 (its block sum
        // tells: every value is at most the sum), in which case the block's
        // true maximum is taken, O rescaled and the block redone.  l and O stay
        // far inside the fp32 range (at most 2^kLazyLog2 per value, 4096
        // blocks of 128), so no row maximum is computed on the common path.
        constexpr float kLazyLog2 = 64.0f;
        float bsum;
        if (n == 0) {
          m = row_max() * scale_log2;
          bsum = exponentiate(m);
        } else {
          bsum = exponentiate(m);
          if (__any_sync(0xffffffffu, !(bsum <= 18446744073709551616.0f))) {   // 2^64
            const float m_new = fmaxf(m, row_max() * scale_log2);
            // rescale this warp's O rows once the previous PV product has landed
            const uint32_t gp = gn - 1;
            if (!mbar_wait_warp(&o_done[gp % NST], (gp / NST) & 1u, abort_flag, ctl, kid | W_O)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = ex2(m - m_new);
            l *= alpha;
            m = m_new;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tmem + lane_off + T::O_COL + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tmem_st32(tmem + lane_off + T::O_COL + c * 32, o);
            }
            tmem_st_wait();
            bsum = exponentiate(m);
          }
        }
        l += bsum;
#pragma unroll
        for (int c = 0; c < BETA / 32; ++c) tmem_st16(sb + c * 16, pk + c * 16);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[s]);
      }
      if (ok) ok = mbar_wait_warp(o_final, (uint32_t)ne & 1u, abort_flag, ctl, kid | W_OFINAL);
      if (!ok) break;
      tc_fence_after();
      const float inv = 1.0f / l;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + T::O_COL + c * 32, o);
        tmem_ld_wait();
        if (r < BETA) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(O + orow * D + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      if (r < BETA) LSE[orow] = (m + log2f(l)) * 0.69314718055994530942f;
      gq += (uint32_t)cnt;
      ++ne;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, T::TMEM_COLS);
}

template <int BETA, int D>
cudaError_t launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const dsv_shape& s,
                         const int32_t* fwd_ptr, const int32_t* fwd_col, float scale, void* O, float* lse,
                         const Ctl& ctl, cudaStream_t st) {
  using T = FwdTraits<BETA, D>;
  auto kern = attn_fwd_kernel<BETA, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  if (e != cudaSuccess) return e;
  const int G = s.N / s.block;
  const long long rows = (long long)s.B * s.H * G;
  const float scale_log2 = scale * 1.4426950408889634f;
  // persistent: one CTA per SM (the CTA holds the SM's whole TMEM)
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)(rows < nsm ? rows : nsm);
  kern<<<grid, kFwdThreads, T::SMEM, st>>>(tmQ, tmK, tmV, fwd_ptr, fwd_col, rows, s.N, G, G, scale_log2,
                                           static_cast<__nv_bfloat16*>(O), lse, ctl);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col, float scale,
                            void* O, float* lse, const Ctl& ctl, cudaStream_t st) {
  if (s.block == 128 && s.d == 128)
    return launch_fwd_t<128, 128>(tmQ, tmK, tmV, s, fwd_ptr, fwd_col, scale, O, lse, ctl, st);
  if (s.block == 128 && s.d == 64)
    return launch_fwd_t<128, 64>(tmQ, tmK, tmV, s, fwd_ptr, fwd_col, scale, O, lse, ctl, st);
  if (s.block == 64 && s.d == 128)
    return launch_fwd_t<64, 128>(tmQ, tmK, tmV, s, fwd_ptr, fwd_col, scale, O, lse, ctl, st);
  return launch_fwd_t<64, 64>(tmQ, tmK, tmV, s, fwd_ptr, fwd_col, scale, O, lse, ctl, st);
}

}  // namespace dsv
