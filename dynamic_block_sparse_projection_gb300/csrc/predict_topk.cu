// predict_topk.cu — the block-score predictor fused with the per-group top-k.
//
// DSV page [nl], "Technische samenvatting" 2B: the critical KV of a query
// group are estimated and selected in one custom kernel, so the memory of the
// estimate stays proportional to the selection instead of the full group x
// block score matrix ([hi] 2B says the same).  Here the pooled rank-r vectors
// (qbar_g, kbar_j, as in predict.cu) go through:
//
//   pool_project_kernel (predict.cu) writes, beside each pooled vector x,
//                       x_hi = tf32(x) and x_lo = tf32(x - x_hi), zero-padded
//                       to 32 rank columns.
//   kstats_*_kernel     per head, the mean and covariance of the pooled keys.
//   score_select_kernel one CTA per (b, h) and 128 consecutive groups.  The
//                       score tile S[g, j] = qbar_g . kbar_j of 128 groups x
//                       128 key blocks is q_hi k_hi + q_hi k_lo + q_lo k_hi:
//                       three tcgen05 kind::tf32 products accumulated in fp32
//                       in tensor memory (the dropped q_lo k_lo term and the
//                       tf32 rounding of the parts leave ~2^-21 of each
//                       product).  The tiles are recomputed in every pass
//                       (the tensor pipe is otherwise idle), so the scores
//                       never leave the SM.  Thread r of the four selection
//                       warps owns group row r (its tensor-memory lane) and
//                       selects that row's top k alone, with no CTA-wide
//                       reductions:
//     pass 0  mean and variance of the row, in closed form from the query's
//             pooled vector and the head's key mean and covariance (no tiles);
//     pass 1  a 128-bin histogram of the row over mean + (z_k -+ 1) sd, z_k
//             the normal quantile of 1 - k/nb (bins clamp at both ends, so the
//             range only decides how many scores share a bin, never which are
//             kept); the bin b* holding the k-th largest score follows;
//     pass 2  the selection bitmask: scores in bins above b* are kept, the
//             few in b* (at most kCand) are collected and ranked exactly by
//             (score desc, index asc) unless all of them are kept.
//   A row whose bin b* holds more than kCand scores and is only partly kept
//   (for example a row of equal scores) is finished by an exact radix select
//   on order-preserving 32-bit keys (five digit passes and an emit pass, run
//   by the CTA only when one of its rows needs it).  The four threads of a row
//   then write its ascending list, each a quarter of the row's bitmask words
//   after the counts of the quarters before it; the bitmask, in the layout of
//   the two-call top-k's workspace, feeds the same transpose kernels.
#include <cuda_runtime.h>

#include <type_traits>

#include "dsv_launch.h"

namespace dsv {

namespace {

constexpr int kRP = 32;                 // rank columns of the split operands (r <= 32, zero padded)
constexpr int kRows = 128;              // groups per CTA: tensor-memory lanes, MMA M
constexpr int kChunk = 128;             // key blocks per score tile: MMA N
constexpr int kNBuf = 4;                // score tiles in tensor memory (4 x 128 columns)
constexpr int kNSlot = 2;               // shared-memory slots of k_hi / k_lo tiles
constexpr int kBins = 128;              // value bins of a row (pass 1)
constexpr int kCand = 32;               // scores of the threshold bin ranked exactly per row
static_assert(kBins * 32 >= kPredictTopkMaxBlocks, "a row's bitmask words must fit its shared-memory column");
constexpr float kZHalf = 1.0f;          // half-width of the binned range, in standard deviations
constexpr int kColGroups = 4;           // threads per row: each takes 32 of a tile's 128 columns
constexpr int kSelWarp0 = 2;            // warps 2 .. 17 select
constexpr int kSelWarps = 4 * kColGroups;
constexpr int kThreads = 32 * (kSelWarp0 + kSelWarps);
constexpr int kTileBytes = kRows * kRP * 4;   // one 128 x 32 fp32 operand tile (16 KB)
constexpr int kNumMain = 3;             // passes 0..2 (pass 0: the row moments, in closed form, no tiles)
constexpr int kKStatSplits = 64;
constexpr int kKStat = kRP + kRP * kRP;   // per head: mu[32], then C[32][32]
constexpr int kNumRadix = 6;            // digit passes of the exact fallback (6, 6, 6, 6, 6, 2 bits)
constexpr int kRadixBins = 64;
constexpr int kFallbackDigit = -1;      // compile-time tag of the fallback's digit passes
// digit dp of a 32-bit key: bits [shift, shift + width) counted from the top
__host__ __device__ constexpr int radix_bits(int dp) { return dp < 5 ? 6 : 2; }
__host__ __device__ constexpr int radix_shift(int dp) { return dp < 5 ? 26 - 6 * dp : 0; }

enum : unsigned int { W_QF = 1, W_KF, W_KFREE, W_SF, W_TFREE, W_DRAIN };
constexpr unsigned int KID_SEL = 4;

struct SelArgs {
  CUtensorMap qh, ql, kh, kl;          // [B*H*G, 32] fp32, box 32 x 128, 128-byte swizzle
  int H, G, words, tiles;              // tiles = ceil(G / 128) per (b, h)
  long long item0;                     // CTA x takes item item0 + x (item = (b*H + h) * tiles + tile)
  long long rows;                      // B*H*G
  int nnz;
  int32_t* fwd_ptr;
  int32_t* fwd_col;
  uint32_t* mask;                      // [B*H][words][G]
  float* scores;                       // optional [B*H*G, G]: the scores the selection used
  const float* kstats;                 // [B*H][kKStat]: mu and C of the pooled keys of each head
  HeadK hk;
  Ctl ctl;
};

// Order-preserving map of a score to uint32: larger score, larger key; -0.0
// and +0.0 map to the same key; NaN maps below every number.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;
  uint32_t b = __float_as_uint(f);
  if ((b << 1) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Instruction descriptor of kind::tf32 with fp32 accumulation, both operands
// K-major: D format F32 (bits 4-5 = 1), A and B format TF32 (bits 7-9 and
// 10-12 = 2), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], tf32 operands; the whole warp calls it and
// one elected lane issues.
__device__ __forceinline__ void mma_tf32_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---------------------------------------------------------------------------
// Per-head statistics of the pooled keys: the mean and covariance of a row of
// scores are closed forms of them, S[g, .] = qbar_g . kbar_.:
//   mean_j S[g, j] = qbar_g . mu,   var_j S[g, j] = qbar_g^T C qbar_g,
// with mu the mean and C the covariance of the kbar_j over the row's nb key
// blocks.  Sums are taken about the head's first key block (shifted data) in
// fixed order: kKStatSplits partial sums per head, then one reduction.
// ---------------------------------------------------------------------------

// grid: (B*H, kKStatSplits), 256 threads: slice t / 64 of the split's rows,
// entries i = 4 ib .. 4 ib + 3, j = 4 jb .. 4 jb + 3 with ib = (t / 8) % 8,
// jb = t % 8 (a 4 x 4 register block: 16 fma per two vector loads); the four
// slices are summed in shared memory in fixed order.
constexpr int kStatRows = 64;           // rows of a split staged at a time
__global__ void __launch_bounds__(256) kstats_partial_kernel(const float* __restrict__ kp, int r, int G,
                                                             float* __restrict__ part) {
  __shared__ __align__(16) float tile[kStatRows][kRP];
  __shared__ float red[4][kKStat];
  __shared__ float k0[kRP];
  const long long bh = blockIdx.x;
  const int t = threadIdx.x, slice = t >> 6, ib = (t >> 3) & 7, jb = t & 7;
  const float* K = kp + bh * G * (long long)r;
  const int per = (G + kKStatSplits - 1) / kKStatSplits;
  const int g_begin = blockIdx.y * per, g_end = min(G, g_begin + per);
  if (t < kRP) k0[t] = t < r ? K[t] : 0.f;
  float acc[4][4], si[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    si[m] = 0.f;
#pragma unroll
    for (int n = 0; n < 4; ++n) acc[m][n] = 0.f;
  }
  for (int g0 = g_begin; g0 < g_end; g0 += kStatRows) {
    __syncthreads();
    for (int e = t; e < kStatRows * kRP; e += 256) {
      const int row = e / kRP, c = e % kRP;
      tile[row][c] = (g0 + row < g_end && c < r) ? K[(long long)(g0 + row) * r + c] - k0[c] : 0.f;
    }
    __syncthreads();
    const int nrow = min(kStatRows, g_end - g0);
    for (int row = slice; row < nrow; row += 4) {
      const float4 a = *reinterpret_cast<const float4*>(&tile[row][4 * ib]);
      const float4 b = *reinterpret_cast<const float4*>(&tile[row][4 * jb]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        si[m] += av[m];
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n] = fmaf(av[m], bv[n], acc[m][n]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (jb == 0) red[slice][4 * ib + m] = si[m];
#pragma unroll
    for (int n = 0; n < 4; ++n) red[slice][kRP + (4 * ib + m) * kRP + 4 * jb + n] = acc[m][n];
  }
  __syncthreads();
  float* P = part + (bh * kKStatSplits + blockIdx.y) * (long long)kKStat;
  for (int e = t; e < kKStat; e += 256) P[e] = ((red[0][e] + red[1][e]) + red[2][e]) + red[3][e];
}

// grid: B*H, 1024 threads: mu and C of each head from its partial sums
__global__ void __launch_bounds__(1024) kstats_reduce_kernel(const float* __restrict__ kp, int r, int G,
                                                             const float* __restrict__ part, float* __restrict__ stats) {
  __shared__ float s[kRP];
  const long long bh = blockIdx.x;
  const int t = threadIdx.x, i = t >> 5, j = t & 31;
  const float* P = part + bh * kKStatSplits * (long long)kKStat;
  float acc = 0.f, si = 0.f;
#pragma unroll 16
  for (int q = 0; q < kKStatSplits; ++q) {
    acc += P[q * kKStat + kRP + i * kRP + j];
    if (j == 0) si += P[q * kKStat + i];
  }
  if (j == 0) s[i] = si;
  __syncthreads();
  const float inv = 1.0f / (float)G;
  const float mi = s[i] * inv, mj = s[j] * inv;
  float* S = stats + bh * (long long)kKStat;
  S[kRP + i * kRP + j] = acc * inv - mi * mj;
  if (j == 0) S[i] = (i < r ? kp[bh * G * (long long)r + i] : 0.f) + mi;
}

// ---------------------------------------------------------------------------
// Score tiles on the tensor cores, selection one row per thread
// ---------------------------------------------------------------------------
constexpr float kB0 = 12582912.0f;      // 1.5 * 2^23: adding it leaves round(x) in the low mantissa bits

// fma with the result clamped to [0, 1] (one instruction)
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// x[e] for an index e that is the same in every lane of the warp (a jump on
// e, so that x stays in registers)
__device__ __forceinline__ uint32_t pick32(const uint32_t (&x)[32], int e) {
  switch (e) {
    case 0: return x[0];   case 1: return x[1];   case 2: return x[2];   case 3: return x[3];
    case 4: return x[4];   case 5: return x[5];   case 6: return x[6];   case 7: return x[7];
    case 8: return x[8];   case 9: return x[9];   case 10: return x[10]; case 11: return x[11];
    case 12: return x[12]; case 13: return x[13]; case 14: return x[14]; case 15: return x[15];
    case 16: return x[16]; case 17: return x[17]; case 18: return x[18]; case 19: return x[19];
    case 20: return x[20]; case 21: return x[21]; case 22: return x[22]; case 23: return x[23];
    case 24: return x[24]; case 25: return x[25]; case 26: return x[26]; case 27: return x[27];
    case 28: return x[28]; case 29: return x[29]; case 30: return x[30]; default: return x[31];
  }
}

// (w << 1) | sign bit of d: one funnel shift of the 64-bit value w:d
__device__ __forceinline__ uint32_t shift_in_sign(uint32_t w, float d) {
  return __funnelshift_l(__float_as_uint(d), w, 1);
}

// The bin map of a row: z = clamp(s * sc + c0, 0, 1) (scores below the binned
// range give 0, above it 1), bin = round(127 z), returned as the float bits
// B0 + bin (adding 1.5 * 2^23 leaves the rounded value in the low mantissa
// bits).  Two fma, both non-decreasing in s, so the map is monotone.
__device__ __forceinline__ uint32_t bin_bits(float s, float sc, float c0) {
  return __float_as_uint(fmaf(fma_sat(s, sc, c0), (float)(kBins - 1), kB0));
}

// inverse of order_key for the keys of numbers (not NaN)
__device__ __forceinline__ float key_float(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// The largest value (+inf included) whose bin is at most `bin`.  bin_bits is
// non-decreasing in its argument, so {s : bin(s) > bin} = {s : s > result}:
// a pass can compare scores with this value instead of recomputing bins.
// Binary search over the ordered keys of -inf .. +inf.
__device__ float bin_upper(float sc, float c0, uint32_t bin) {
  const uint32_t target = __float_as_uint(kB0) + bin;
  uint32_t lo = 0x007fffffu, hi = 0xff800000u;          // keys of -inf and +inf
  if (bin_bits(key_float(hi), sc, c0) <= target) return __uint_as_float(0x7f800000u);
  while (hi - lo > 1u) {                                // bin(key_float(lo)) <= target < bin(key_float(hi))
    const uint32_t mid = lo + ((hi - lo) >> 1);
    if (bin_bits(key_float(mid), sc, c0) <= target) lo = mid;
    else hi = mid;
  }
  return key_float(lo);
}

// Per-row state shared by the four threads of a row (shared memory).
struct RowShared {
  float mom_mean[kColGroups], mom_m2[kColGroups];   // pass 0: the four threads' parts of the mean and variance
  float keep_v;          // pass 2 keeps the scores above this value
  float coll_v;          // and collects the scores in (coll_v, keep_v] for exact ranking
  uint32_t kk;           // how many of that bin are kept
  int ccount;            // scores collected from that bin so far
  int fail;              // the row needs the exact fallback
  int cnt[kColGroups];   // output: kept blocks in each thread's range of words
};

// bitmask word wi of row r in the shared column region (XOR spread: a warp's
// rows, or a row's 32 consecutive words, fall in 32 different banks)
__device__ __forceinline__ int word_at(int wi, int r) { return wi * kRows + (r ^ (wi & 31)); }

// Fire-and-forget add to a shared-memory counter (32-bit shared address).
__device__ __forceinline__ void red_shared_add(uint32_t saddr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}
static_assert(kRows * 4 == 512, "histogram rows are 512 bytes apart (bin << 9)");

__device__ __forceinline__ void sel_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(kSelWarps * 32) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) score_select_kernel(const __grid_constant__ SelArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sbase = smem_align1024(smem_raw);             // accesses below stay in the shared space
  uint8_t* sQh = sbase;
  uint8_t* sQl = sQh + kTileBytes;
  uint8_t* sKh = sQl + kTileBytes;                       // [kNSlot] tiles
  uint8_t* sKl = sKh + kNSlot * kTileBytes;              // [kNSlot] tiles
  // [kBins][kRows]: per row (column r) its histogram (bin * kRows + r), later its bitmask words (word_at)
  uint32_t* hist = reinterpret_cast<uint32_t*>(sKl + kNSlot * kTileBytes);
  uint2* cand = reinterpret_cast<uint2*>(hist + kBins * kRows);             // [kCand][kRows]
  RowShared* rs = reinterpret_cast<RowShared*>(cand + kCand * kRows);      // [kRows]
  float* kst = reinterpret_cast<float*>(rs + kRows);                       // [kKStat]: mu, C of this head
  uint64_t* bars = reinterpret_cast<uint64_t*>(kst + kKStat);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_free = k_full + kNSlot;
  uint64_t* s_full = k_free + kNSlot;
  uint64_t* t_free = s_full + kNBuf;
  uint64_t* mma_drain = t_free + kNBuf;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_fail = const_cast<int*>(abort_flag + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Ctl& ctl = a.ctl;
  const unsigned int kid = KID_SEL << 8;
  const int G = a.G, nb = a.G, words = a.words;
  const long long item = a.item0 + blockIdx.x;
  const long long bh = item / a.tiles;
  const int g0 = (int)(item - bh * a.tiles) * kRows;
  const int h = (int)(bh % a.H), b = (int)(bh / a.H);
  const int k = a.hk.k[h];
  const int nc = (nb + kChunk - 1) / kChunk;             // score tiles of a row
  const bool select_all = k >= nb;                       // k = nb: every block, nothing to score

  // selection threads: row r (tensor-memory lane) and column group cg of each 128-column tile
  const bool sel = warp >= kSelWarp0;
  const int quarter = warp & 3;
  const int cg = sel ? (warp - kSelWarp0) >> 2 : 0;
  const int r = quarter * 32 + lane;
  const int g = g0 + r;
  const bool row_ok = sel && g < G;
  const long long grow = bh * G + g;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kNSlot; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_free[s], 1);
    }
    for (int s = 0; s < kNBuf; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&t_free[s], 4 * 32);                   // the four warps of the group that reads the tile
    }
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    *s_fail = 0;
    fence_mbar_init();
  }
  if (sel) {
    for (int i = threadIdx.x - kSelWarp0 * 32; i < kKStat; i += kSelWarps * 32) kst[i] = a.kstats[bh * kKStat + i];
    for (int i = cg * (kBins / kColGroups); i < (cg + 1) * (kBins / kColGroups); ++i) hist[i * kRows + r] = 0u;
    if (cg == 0) {
      rs[r].ccount = 0;
      rs[r].fail = 0;
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kNBuf * kChunk);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool tmem_ok = tmem_base == 0u;
  if (!tmem_ok && threadIdx.x == 0) set_error(ctl, DSV_ERR_INTERNAL, blockIdx.x);

  // per-thread row state
  float sc = 0.f, c0 = 0.f;                              // bin map
  float keep_v = 0.f, coll_v = __uint_as_float(0x7f800000u);
  bool fail = false;
  uint32_t prefix = 0u, hmask = 0u, rk = 0u;             // exact fallback (column group 0)

  uint32_t gc = 0;                                       // score tiles so far (all passes)
  int issued_q = 0;
  uint32_t issued_k = 0;
  bool ok = tmem_ok;

  auto ntiles = [&](int pass) { return pass == 0 ? 0 : nc; };     // pass 0: closed-form moments
  auto tile_of = [&](int pass, int t) { return t; };

  // One run of passes pass0 .. pass0 + npass - 1 over the score tiles; every
  // role walks the same tiles, so barrier phases follow gc.
  auto run_passes = [&](int pass0, int npass) {
    if (!ok || npass == 0) return;
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        if (issued_q == 0) {
          tma_prefetch_desc(&a.kh);
          tma_prefetch_desc(&a.kl);
          mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
          tma_load_2d(sQh, &a.qh, q_full, 0, (int)(bh * G + g0));
          tma_load_2d(sQl, &a.ql, q_full, 0, (int)(bh * G + g0));
          issued_q = 1;
        }
        uint32_t n = gc;
        for (int pass = pass0; ok && pass < pass0 + npass; ++pass) {
          for (int t = 0; t < ntiles(pass); ++t, ++n) {
            const int slot = (int)(n % kNSlot);
            if (n >= kNSlot &&
                !mbar_wait(&k_free[slot], ((n - kNSlot) / kNSlot) & 1u, abort_flag, ctl, kid | W_KFREE)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&k_full[slot], 2 * kTileBytes);
            const int y = (int)(bh * G + (long long)tile_of(pass, t) * kChunk);
            tma_load_2d(sKh + slot * kTileBytes, &a.kh, &k_full[slot], 0, y);
            tma_load_2d(sKl + slot * kTileBytes, &a.kl, &k_full[slot], 0, y);
            issued_k = n + 1;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t ID = idesc_tf32_f32(kRows, kChunk);
      if (!mbar_wait_warp(q_full, 0, abort_flag, ctl, kid | W_QF)) {
        ok = false;
      } else {
        const uint64_t dQh = sdesc_sw128(smem_u32(sQh), 16, 1024);
        const uint64_t dQl = sdesc_sw128(smem_u32(sQl), 16, 1024);
        const uint64_t dKh = sdesc_sw128(smem_u32(sKh), 16, 1024);
        const uint64_t dKl = sdesc_sw128(smem_u32(sKl), 16, 1024);
        uint32_t n = gc;
        for (int pass = pass0; ok && pass < pass0 + npass; ++pass) {
          for (int t = 0; t < ntiles(pass); ++t, ++n) {
            const int slot = (int)(n % kNSlot);
            const int buf = (int)(n % kNBuf);
            if (!mbar_wait_warp(&k_full[slot], (n / kNSlot) & 1u, abort_flag, ctl, kid | W_KF)) {
              ok = false;
              break;
            }
            if (n >= kNBuf &&
                !mbar_wait_warp(&t_free[buf], ((n - kNBuf) / kNBuf) & 1u, abort_flag, ctl, kid | W_TFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = (uint32_t)buf * kChunk;
            const uint32_t koff = (uint32_t)slot * kTileBytes;
#pragma unroll
            for (int p = 0; p < 3; ++p) {
              const uint64_t da = p == 2 ? dQl : dQh;               // q_hi k_hi, q_hi k_lo, q_lo k_hi
              const uint64_t db = desc_off(p == 1 ? dKl : dKh, koff);
#pragma unroll
              for (int kk = 0; kk < kRP / 8; ++kk)
                mma_tf32_w(d, desc_off(da, kk * 32), desc_off(db, kk * 32), ID, (p > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_w(&s_full[buf]);
            mma_commit_w(&k_free[slot]);
          }
        }
      }
    } else {
      // ---------------- selection: row r, columns cg*32 .. cg*32 + 31 of every tile ----------------
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      uint32_t* hcol = hist + r;
      const uint32_t hcol_s = smem_u32(hcol);            // shared address of this row's histogram column
      // address of bin b from the bin bits B0 + b: ((B0 + b) << 9) = (B0 << 9) + 512 b (mod 2^32)
      const uint32_t hbase = hcol_s - (__float_as_uint(kB0) << 9);
      uint32_t n = gc;
      for (int pass = pass0; pass < pass0 + npass; ++pass) {
        const bool fb = pass >= kNumMain;                  // exact fallback pass: column group 0 does the row
        const bool work = row_ok && (!fb || (fail && cg == 0));
        // the fallback's digit histograms live in the candidate region, [bin][row]: the
        // histogram region now holds bitmask words, spread over other rows' columns
        uint32_t* fcol = reinterpret_cast<uint32_t*>(cand) + r;
        const uint32_t fcol_s = smem_u32(fcol);
        if (fb && work && pass < kNumMain + kNumRadix)
          for (int i = 0; i < kRadixBins; ++i) fcol[i * kRows] = 0u;   // this digit's histogram
        const int nt = ntiles(pass);
        // the 32 scores of column group q of tile c (columns j0 .. j0 + 31, the first nvg valid)
          // P: the pass, known at compile time (kFallbackDigit: one of the fallback's digit passes)
          auto proc = [&](const uint32_t (&x)[32], int c, int nv, int q, auto full_tag, auto pass_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            constexpr int P = decltype(pass_tag)::value;
            const int j0 = c * kChunk + q * 32;
            const int nvg = nv - q * 32;
            const int wi = j0 >> 5;                       // bitmask word of these 32 columns
            if constexpr (P == 1) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (work && (FULL || e < nvg))
                  red_shared_add(hbase + (bin_bits(__uint_as_float(x[e]), sc, c0) << 9), 1u);
              if (work && a.scores != nullptr) {
                // check output: the scores this selection uses
                float* dst = a.scores + grow * (long long)nb + j0;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (FULL || e < nvg) dst[e] = __uint_as_float(x[e]);
              }
            } else if constexpr (P == 2) {
              // word: scores above keep_v; above: scores above coll_v (a superset);
              // the threshold bin's scores are the difference
              // bit e of a word is the sign of (threshold - score e): the difference
              // is negative exactly when the score is above the threshold (a
              // rounded difference keeps the sign of the exact one, equal values
              // give +0, the thresholds are never -0, and a NaN score gives the
              // canonical NaN, sign clear).  The sign bits are shifted in from the
              // top, last column first, so that column e lands on bit e.
              uint32_t word = 0u, above = 0u;
              if constexpr (FULL) {
                // two columns per packed subtraction (each lane of it rounds like
                // a scalar one)
                const uint64_t kk2 = f2_pack(keep_v, keep_v), cc2 = f2_pack(coll_v, coll_v);
#pragma unroll
                for (int e = 31; e >= 1; e -= 2) {
                  const uint64_t sv = f2_pack(__uint_as_float(x[e - 1]), __uint_as_float(x[e]));
                  float dk0, dk1, dc0, dc1;
                  f2_unpack(sub2(kk2, sv), dk0, dk1);
                  f2_unpack(sub2(cc2, sv), dc0, dc1);
                  word = shift_in_sign(shift_in_sign(word, dk1), dk0);
                  above = shift_in_sign(shift_in_sign(above, dc1), dc0);
                }
              } else {
#pragma unroll
                for (int e = 31; e >= 0; --e) {
                  if (e < nvg) {
                    const float s = __uint_as_float(x[e]);
                    word = shift_in_sign(word, __fsub_rn(keep_v, s));
                    above = shift_in_sign(above, __fsub_rn(coll_v, s));
                  } else {
                    word <<= 1;
                    above <<= 1;
                  }
                }
              }
              const uint32_t eq = work ? above & ~word : 0u;
              if (work) hist[word_at(wi, r)] = word;
              // the threshold bin's scores: one step per column where any row of
              // the warp has one (every lane of the warp takes part: the pass
              // runs for all 32 rows, those past the last group with no work),
              // the score picked from the registers by that column
              uint32_t ecols = __reduce_or_sync(0xffffffffu, eq);
              if (ecols) {
                // this row's slots, reserved at once (the row's four threads add
                // candidates concurrently)
                const int cnt = __popc(eq);
                int pos = cnt ? atomicAdd(&rs[r].ccount, cnt) : 0;
                while (ecols) {
                  const int e = __ffs(ecols) - 1;
                  ecols &= ecols - 1u;
                  if ((eq >> e) & 1u) {
                    if (pos < kCand) cand[pos * kRows + r] = make_uint2(order_key(__uint_as_float(pick32(x, e))), (uint32_t)(j0 + e));
                    ++pos;
                  }
                }
              }
            } else if constexpr (P == kNumMain + kNumRadix) {
              // exact fallback, emit: keys above T, then keys equal to T lowest index first
              uint32_t word = 0u;
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                if (FULL || e < nvg) {
                  const uint32_t u = order_key(__uint_as_float(x[e]));
                  const bool eqk = u == prefix;
                  word |= ((u > prefix) || (eqk && rk > 0u) ? 1u : 0u) << e;
                  if (eqk && rk > 0u) --rk;
                }
              }
              hist[word_at(wi, r)] = word;
            } else {
              // exact fallback, digit pass: histogram of this digit among keys matching the prefix
              const int dp = pass - kNumMain;
              const int sh = radix_shift(dp);
              const uint32_t dmask = (1u << radix_bits(dp)) - 1u;
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                if (FULL || e < nvg) {
                  const uint32_t u = order_key(__uint_as_float(x[e]));
                  if ((u & hmask) == prefix) red_shared_add(fcol_s + (((u >> sh) & dmask) << 9), 1u);
                }
              }
            }
          };
          auto run_group = [&](const uint32_t (&x)[32], int c, int q, auto pass_tag) {
            const int nv = min(kChunk, nb - c * kChunk);   // valid columns of tile c (uniform)
            if (nv - q * 32 >= 32) proc(x, c, nv, q, std::true_type{}, pass_tag);
            else if (nv - q * 32 > 0) proc(x, c, nv, q, std::false_type{}, pass_tag);
          };
        auto tile_addr = [&](uint32_t nn) { return tmem_base + lane_off + (uint32_t)(nn % kNBuf) * kChunk; };
        auto main_tiles = [&](auto pass_tag) {
          // tile t belongs to column group t % kColGroups: its four warps read all
          // 128 columns, so the warps sharing a scheduler (same lane quarter,
          // different groups) work on different tiles and hide each other's
          // latencies.  After an abort the warp still walks the pass (no waits, no
          // work) so that it reaches the barriers below.
#pragma unroll 1
          for (int t = cg; t < nt; t += kColGroups) {
            const uint32_t nn = n + (uint32_t)t;
            if (!ok) continue;
            const int buf = (int)(nn % kNBuf);
            if (!mbar_wait_warp(&s_full[buf], (nn / kNBuf) & 1u, abort_flag, ctl, kid | W_SF)) {
              ok = false;
              continue;
            }
            tc_fence_after();
#pragma unroll 1
            for (int q = 0; q < kColGroups; ++q) {
              uint32_t x[32];
              tmem_ld32(tile_addr(nn) + (uint32_t)q * 32, x);
              tmem_ld_wait();
              if (q == kColGroups - 1) {
                tc_fence_before();
                mbar_arrive(&t_free[buf]);
              }
              run_group(x, tile_of(pass, t), q, pass_tag);   // every lane (rows past G with no work):
                                                             // pass 2 has warp-wide steps
            }
          }
          n += (uint32_t)nt;
        };
        if (!fb) {
          if (pass == 1) main_tiles(std::integral_constant<int, 1>{});
          else if (pass == 2) main_tiles(std::integral_constant<int, 2>{});
        } else {
          for (int t = 0; t < nt; ++t, ++n) {
            if (!ok || cg != 0) continue;              // column group 0 reads every tile of a fallback pass
            const int buf = (int)(n % kNBuf);
            if (!mbar_wait_warp(&s_full[buf], (n / kNBuf) & 1u, abort_flag, ctl, kid | W_SF)) {
              ok = false;
              continue;
            }
            tc_fence_after();
            if (cg == 0) {
              // the fallback row's four column groups, in order, by one thread
#pragma unroll 1
              for (int q = 0; q < kColGroups; ++q) {
                uint32_t x[32];
                tmem_ld32(tile_addr(n) + (uint32_t)q * 32, x);
                tmem_ld_wait();
                if (q == kColGroups - 1) {
                  tc_fence_before();
                  mbar_arrive(&t_free[buf]);
                }
                if (work) {
                  if (pass == kNumMain + kNumRadix) run_group(x, t, q, std::integral_constant<int, kNumMain + kNumRadix>{});
                  else run_group(x, t, q, std::integral_constant<int, kFallbackDigit>{});
                }
              }
            }
          }
        }
        // ---- end of a pass ----
        if (pass == 0) {
          // the row's mean and variance in closed form: qbar . mu and qbar^T C qbar, the
          // four threads of a row each taking 8 of the 32 terms of the outer sum
          if (ok && !mbar_wait_warp(q_full, 0, abort_flag, ctl, kid | W_QF)) ok = false;
          if (row_ok && ok) {
            // element (r, c) of the 128-byte-swizzled tiles: 16-byte chunk c/4 of row r sits at chunk (c/4) ^ (r % 8)
            auto qval = [&](int c) {
              const int off = r * 128 + ((((c >> 2) ^ (r & 7))) << 4) + ((c & 3) << 2);
              return *reinterpret_cast<const float*>(sQh + off) + *reinterpret_cast<const float*>(sQl + off);
            };
            float q[kRP];
#pragma unroll
            for (int c = 0; c < kRP; ++c) q[c] = qval(c);
            float pm = 0.f, pv = 0.f;
#pragma unroll 1
            for (int ii = 0; ii < kRP / kColGroups; ++ii) {
              const int i = cg * (kRP / kColGroups) + ii;
              float ci = 0.f;
#pragma unroll
              for (int jj = 0; jj < kRP; ++jj) ci = fmaf(kst[kRP + i * kRP + jj], q[jj], ci);
              const float qi = qval(i);
              pm = fmaf(qi, kst[i], pm);
              pv = fmaf(qi, ci, pv);
            }
            rs[r].mom_mean[cg] = pm;
            rs[r].mom_m2[cg] = pv;
          }
          sel_barrier();
          if (row_ok && ok) {
            float mean = 0.f, var = 0.f;
            for (int qg = 0; qg < kColGroups; ++qg) {
              mean += rs[r].mom_mean[qg];
              var += rs[r].mom_m2[qg];
            }
            const float sd = sqrtf(fmaxf(var, 0.f));
            const float zk = normcdfinvf(1.0f - (float)k / (float)nb);
            const float lo = mean + (zk - kZHalf) * sd;
            sc = 1.0f / (2.0f * kZHalf * sd);
            c0 = -lo * sc;
            if (!(sc > 0.f && sc < 1e30f && isfinite(c0) && isfinite(zk))) {
              sc = 0.f;                                  // one bin: the exact fallback decides
              c0 = 0.f;
            }
          }
        } else if (pass == 1) {
          sel_barrier();                                 // every thread's histogram adds are in
          if (row_ok && cg == 0) {
            uint32_t above = 0u, bstar = 0u, cnt = 0u;
            for (int i = kBins - 1; i >= 0; --i) {
              const uint32_t ci = hcol[i * kRows];
              if (above + ci >= (uint32_t)k) {
                bstar = (uint32_t)i;
                cnt = ci;
                break;
              }
              above += ci;
            }
            const uint32_t kk = (uint32_t)k - above;
            rs[r].kk = kk;
            // value bounds of bin b*: (below, top]
            const float below = bstar > 0u ? bin_upper(sc, c0, bstar - 1u) : __uint_as_float(0xff800000u);
            if (cnt == kk) {
              rs[r].keep_v = below;                      // the whole bin is kept
              rs[r].coll_v = __uint_as_float(0x7f800000u);
            } else {
              rs[r].keep_v = bin_upper(sc, c0, bstar);
              rs[r].coll_v = below;
              rs[r].fail = cnt > (uint32_t)kCand ? 1 : 0;
            }
          }
          sel_barrier();                                 // decisions out; the histogram region becomes words
          if (row_ok) {
            keep_v = __fadd_rn(rs[r].keep_v, 0.0f);      // -0 becomes +0
            coll_v = __fadd_rn(rs[r].coll_v, 0.0f);
            fail = rs[r].fail != 0;
          }
        } else if (pass == 2) {
          sel_barrier();                                 // every word and candidate of the row is in
          if (row_ok && cg == 0) {
            if (coll_v < __uint_as_float(0x7f800000u) && !fail) {
              // rank the threshold bin's scores exactly and add the kept ones to the bitmask
              const int n2 = min(rs[r].ccount, kCand);
              const uint32_t kk = rs[r].kk;
              for (int i = 0; i < n2; ++i) {
                const uint2 ci = cand[i * kRows + r];
                uint32_t rank = 0u;
                for (int j = 0; j < n2; ++j) {
                  const uint2 cj = cand[j * kRows + r];
                  rank += (cj.x > ci.x || (cj.x == ci.x && cj.y < ci.y)) ? 1u : 0u;
                }
                if (rank < kk) hist[word_at((int)(ci.y >> 5), r)] |= 1u << (ci.y & 31u);
              }
            }
            if (fail) {
              prefix = 0u;
              hmask = 0u;
              rk = (uint32_t)k;
            }
          }
        } else if (work && pass < kNumMain + kNumRadix) {
          const int dp = pass - kNumMain;
          const int sh = radix_shift(dp);
          const int nbin = 1 << radix_bits(dp);
          uint32_t above = 0u;
          for (int i = nbin - 1; i >= 0; --i) {
            const uint32_t ci = fcol[i * kRows];
            if (above + ci >= rk) {
              prefix |= (uint32_t)i << sh;
              rk -= above;
              break;
            }
            above += ci;
          }
          hmask |= (uint32_t)(nbin - 1) << sh;
          // after the last digit: prefix = T, the k-th largest key; rk = keys equal to T to take
        }
      }
    }
    for (int pass = pass0; pass < pass0 + npass; ++pass) gc += (uint32_t)ntiles(pass);
  };

  if (!select_all) run_passes(0, kNumMain);

  // rows that need the exact fallback: the CTA runs its passes if any does
  if (row_ok && cg == 0 && fail) atomicOr(s_fail, 1);
  __syncthreads();
  if (ok && *s_fail && !*abort_flag) run_passes(kNumMain, kNumRadix + 1);

  // every copy and product this CTA issued must be done before it exits
  if (warp == 0 && lane == 0) {
    if (issued_q) mbar_wait(q_full, 0, nullptr, ctl, kid | W_DRAIN);
    for (uint32_t n = (issued_k > kNSlot ? issued_k - kNSlot : 0u); n < issued_k; ++n)
      mbar_wait(&k_full[n % kNSlot], (n / kNSlot) & 1u, nullptr, ctl, kid | W_DRAIN);
  } else if (warp == 1 && tmem_ok) {
    mma_commit_w(mma_drain);
    mbar_wait_warp(mma_drain, 0, nullptr, ctl, kid | W_DRAIN);
  }

  // outputs: the bitmask words (coalesced over consecutive rows), then the
  // ascending lists.  After this barrier every failed wait has raised the abort
  // flag, so out_ok is the same in every thread and the named barriers below
  // are reached by all selection warps or by none.
  __syncthreads();
  const bool out_ok = ok && !*abort_flag;
  if (sel && out_ok) {
    if (row_ok && select_all) {
      for (int wi = cg; wi < words; wi += kColGroups) {
        const int rem = nb - wi * 32;
        hist[word_at(wi, r)] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
      }
    }
    sel_barrier();                                       // every word of every row is final
    if (row_ok)
      for (int wi = cg; wi < words; wi += kColGroups) a.mask[(bh * words + wi) * (long long)G + g] = hist[word_at(wi, r)];
    // the ascending list of row r: thread cg writes the blocks of words
    // [cg * wpt, (cg + 1) * wpt), after the counts of the row's earlier threads
    const int wpt = (words + kColGroups - 1) / kColGroups;
    const int w0 = cg * wpt, w1 = min(words, w0 + wpt);
    if (row_ok) {
      int cnt = 0;
      for (int wi = w0; wi < w1; ++wi) cnt += __popc(hist[word_at(wi, r)]);
      rs[r].cnt[cg] = cnt;
    }
    sel_barrier();
    if (row_ok) {
      int pos = 0, total = 0;
#pragma unroll
      for (int q = 0; q < kColGroups; ++q) {
        const int c = rs[r].cnt[q];
        pos += q < cg ? c : 0;
        total += c;
      }
      const long long hbase = (long long)b * G * a.hk.kpre[a.H] + (long long)a.hk.kpre[h] * G;
      int32_t* dst = a.fwd_col + hbase + (long long)g * k;
      uint32_t mn = w0 < w1 ? hist[word_at(w0, r)] : 0u;
      for (int wi = w0; wi < w1; ++wi) {
        uint32_t m = mn;
        if (wi + 1 < w1) mn = hist[word_at(wi + 1, r)];   // next word in flight
        while (m) {
          const int b0 = __ffs(m) - 1;
          m &= m - 1u;
          const int b1 = __ffs(m) - 1;                    // -1 when m is now empty
          m &= m - 1u;
          if (pos < k) dst[pos] = wi * 32 + b0;
          if (b1 >= 0 && pos + 1 < k) dst[pos + 1] = wi * 32 + b1;
          pos += b1 >= 0 ? 2 : 1;
        }
      }
      if (cg == 0) {
        if (total != k) set_error(ctl, DSV_ERR_INTERNAL, (unsigned int)(grow & 0x7fffffff));
        a.fwd_ptr[grow] = (int32_t)(hbase + (long long)g * k);
        if (grow == a.rows - 1) a.fwd_ptr[a.rows] = a.nnz;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1 && tmem_ok) tmem_dealloc(tmem_base, kNBuf * kChunk);
}

constexpr int kSelSmem = 1024 + 2 * kTileBytes + 2 * kNSlot * kTileBytes + kBins * kRows * 4 + kCand * kRows * 8 +
                         kRows * (int)sizeof(RowShared) + kKStat * 4 + (1 + 2 * kNSlot + 2 * kNBuf + 1) * 8 + 16;
static_assert((kRows * (int)sizeof(RowShared) + kKStat * 4) % 8 == 0, "barriers must stay 8-byte aligned");
static_assert(kSelSmem <= 227 * 1024, "score/select tiles exceed shared memory");
static_assert(kRadixBins * 4 <= kCand * 8, "the fallback's digit histograms must fit the candidate region");

}  // namespace

size_t split_tf32_bytes(const dsv_shape& s) {
  const size_t bhs = (size_t)s.B * s.H;
  return 4 * align256(bhs * (size_t)(s.N / s.block) * kRP * sizeof(float)) +
         align256(bhs * kKStatSplits * kKStat * sizeof(float)) + align256(bhs * kKStat * sizeof(float));
}

long long select_tiles(const dsv_shape& s) { return (s.N / s.block + kRows - 1) / kRows; }

long long split_part_floats(const dsv_shape& s) {
  const size_t rows = (size_t)s.B * s.H * (size_t)(s.N / s.block);
  return (long long)(align256(rows * kRP * sizeof(float)) / sizeof(float));
}

cudaError_t launch_key_stats(const float* kp, const dsv_shape& s, float* split, cudaStream_t st) {
  // per-head key statistics after the four tf32 parts: partial sums, then mu and C
  const long long part = split_part_floats(s);
  const unsigned bhs = (unsigned)(s.B * s.H);
  float* kpart = split + 4 * part;
  float* kstats = kpart + align256((size_t)bhs * kKStatSplits * kKStat * sizeof(float)) / sizeof(float);
  kstats_partial_kernel<<<dim3(bhs, kKStatSplits), 256, 0, st>>>(kp, s.r, s.N / s.block, kpart);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kstats_reduce_kernel<<<bhs, 1024, 0, st>>>(kp, s.r, s.N / s.block, kpart, kstats);
  return cudaGetLastError();
}

cudaError_t launch_score_select(const PredictTopkMaps& maps, const dsv_shape& s, const HeadK& hk, int64_t nnz,
                                int32_t* fwd_ptr, int32_t* fwd_col, uint32_t* mask, float* scores, const float* split,
                                const Ctl& ctl, cudaStream_t st, long long item0, long long item1) {
  SelArgs a;
  a.qh = maps.qh;
  a.ql = maps.ql;
  a.kh = maps.kh;
  a.kl = maps.kl;
  a.H = s.H;
  a.G = s.N / s.block;
  a.words = (a.G + 31) / 32;
  a.tiles = (a.G + kRows - 1) / kRows;
  a.rows = (long long)s.B * s.H * a.G;
  a.nnz = (int)nnz;
  a.fwd_ptr = fwd_ptr;
  a.fwd_col = fwd_col;
  a.mask = mask;
  a.scores = scores;
  {
    const size_t bhs = (size_t)s.B * s.H;
    const size_t part = align256(bhs * (size_t)a.G * kRP * sizeof(float)) / sizeof(float);
    a.kstats = split + 4 * part + align256(bhs * kKStatSplits * kKStat * sizeof(float)) / sizeof(float);
  }
  a.hk = hk;
  a.ctl = ctl;
  cudaError_t e = cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmem);
  if (e != cudaSuccess) return e;
  const long long items = (long long)s.B * s.H * a.tiles;
  if (item1 < 0 || item1 > items) item1 = items;
  if (item0 < 0 || item0 >= item1) return cudaSuccess;
  a.item0 = item0;
  score_select_kernel<<<(unsigned)(item1 - item0), kThreads, kSelSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace dsv
