// topk.cu — per-group top-k critical key blocks and the transposed lists.
//
// DSV page [nl], "Technische samenvatting" 2B (estimation & selection of the
// critical KV per query group) and [hi] 2A (critical KV pairs).  For each row
// (b, h, g) the k_h blocks with the largest predicted score are kept, equal
// scores going to the lower block index; lists are written ascending.  The
// backward pass needs, per key block, the ascending list of groups that kept
// it; that transpose is built deterministically without atomics.
//
// Kernels:
//   topk_select    one CTA per row (32 ... 512 threads, 16 consecutive
//                  scores per thread in registers).  Scores are binned by
//                  value between the row's min and max; the bucket holding
//                  the k-th largest is ranked exactly on order-preserving
//                  uint32 keys (ties to the lower index), with an MSB-first
//                  radix select as the fallback.  Each thread writes its kept
//                  indices (ascending) and the row's bitmask words.
//   topk_colcount  per (b, h, 32-column slab), down all rows: 32x32 bit
//                  transposes of the mask (stored word column by word
//                  column, rows contiguous) give each column's count before
//                  every 128-row segment and its total.
//   topk_scan      per (b, h): exclusive scan of the column totals -> bwd_ptr.
//   topk_fill      per (slab, segment); per column with entries in a
//                  32-row chunk, one ballot and one coalesced store of
//                  those rows, in ascending g.
#include <algorithm>

#include "dsv_launch.h"

namespace dsv {

namespace {


// Order-preserving map float -> uint32 with -0.0 == +0.0 and NaN below -inf.
__device__ __forceinline__ uint32_t score_key(float f) {
  if (f != f) return 0u;               // NaN ranks lowest
  uint32_t b = __float_as_uint(f);
  if ((b << 1) == 0u) b = 0u;          // -0.0 -> +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkArgs {
  const float* scores;
  int32_t* fwd_ptr;
  int32_t* fwd_col;
  uint32_t* mask;
  int H, G, nb, words;
  long long rows;   // B*H*G
  int nnz;
  HeadK hk;
  // per-row list sizes (mass-threshold selection): k and the list start of
  // row r are row_k[r] and row_ptr[r] (fwd_ptr, already written), the head's
  // first entry row_ptr[bh * G] and the total row_ptr[rows]; null: k per head
  const int32_t* row_k;
  const int32_t* row_ptr;
  // the transposes cover heads bh0 .. bh0 + gridDim - 1 (slices of B*H)
  long long bh0;
};

// One CTA of RT threads per row.  Thread t holds kE consecutive scores
// (slots [kE*t - off, kE*t - off + kE), off = the row start's offset from a
// 16-byte boundary, so whole threads load with 16-byte vectors).
//
// Fast path (finite row with max > min): the scores are binned by value into
// BINS equal-width buckets between the row minimum and maximum (one FMA,
// rounded by the 1.5 * 2^23 trick, clamped: a monotone map, so a higher
// bucket holds only larger scores).  One shared-memory histogram gives the
// bucket b* holding the k-th largest score; every score in a higher bucket is
// kept, and the few scores of b* (at most kCandMax) are ranked exactly by
// (key desc, index asc) unless all of them are kept.  Each thread then writes
// its own kept indices (ascending) at its prefix position and 32-bit mask
// words are put together from the threads' E-bit slot masks.  Value binning
// spreads the scores over the buckets, so the shared-memory atomics rarely
// collide; radix digits of float bits would pile into the few bins of the
// common exponents.  Slots outside the row hold NaN: ignored by min / max,
// binned into bucket 0 and taken out of its count.  Real NaNs also land in
// bucket 0 and rank below every number there.
// Fallback (infinite scores, all equal, or a crowded b*): the row is re-read
// with element i in thread i % RT, and an MSB-first radix select on the
// order-preserving keys (11-bit digits, 2048-bin histogram; 8-bit for rows of
// at most 1024 keys) below their common prefix gives the k-th largest key T and
// how many keys equal to T to take (lowest index first); ballots per 32-index
// chunk give the mask words.

// Digit width of the radix passes and bucket count of the value binning: 11
// bits (2048 bins) for long rows, 8 bits for rows of at most 1024 keys, where
// clearing and scanning a large histogram would cost more than the keys.
template <int RT>
struct SelCfg {
  static constexpr int DIGIT = RT >= 128 ? 11 : 8;
  static constexpr int BINS = 1 << DIGIT;
};

constexpr int kE = 16;                   // scores per thread

template <int RT>
__device__ __forceinline__ void cta_find_bin(const uint32_t* hist, uint32_t kk, uint32_t* s_tot, uint32_t* s_res) {
  // the bin holding the kk-th largest key (counted from the top bin down) and its rank inside the bin
  constexpr int kBins = SelCfg<RT>::BINS;
  constexpr int BPT = kBins / RT;
  static_assert(BPT % 4 == 0, "bins per thread in 16-byte loads");
  constexpr int NW = RT / 32;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  uint32_t c[BPT];
#pragma unroll
  for (int q = 0; q < BPT / 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(hist)[t * (BPT / 4) + q];
    c[4 * q] = u.x;
    c[4 * q + 1] = u.y;
    c[4 * q + 2] = u.z;
    c[4 * q + 3] = u.w;
  }
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) tot += c[i];
  // suffix sum over threads above t: warp-level, then across warps
  uint32_t suf = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  if (NW > 1) {
    if (lane == 0) s_tot[w] = suf;  // total of warp w
    __syncthreads();
#pragma unroll
    for (int v = 1; v < NW; ++v)
      if (v > w) suf += s_tot[v];
  }
  uint32_t above = suf - tot;      // keys in bins above this thread's range
  if (above < kk && above + tot >= kk) {
#pragma unroll
    for (int i = BPT - 1; i >= 0; --i) {
      if (above < kk && above + c[i] >= kk) {
        s_res[0] = (uint32_t)(t * BPT + i);
        s_res[1] = kk - above;
      }
      above += c[i];
    }
  }
  __syncthreads();
}

constexpr int kCandMax = 256;            // keys tied for the threshold bucket, ranked exactly

// CTA-wide exclusive prefix of popc(words[ci]) over chunks ci < nw, into off[]
// (warp 0; MAXC chunks at most).
template <int MAXC>
__device__ __forceinline__ void chunk_prefix(const uint32_t* words, int nw, int32_t* off, int lane) {
  constexpr int CPL = (MAXC + 31) / 32;   // chunks per lane
  uint32_t c[CPL];
  uint32_t tot = 0;
#pragma unroll
  for (int q = 0; q < CPL; ++q) {
    const int ci = lane * CPL + q;
    c[q] = (ci < nw) ? (uint32_t)__popc(words[ci]) : 0u;
    tot += c[q];
  }
  uint32_t inc = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  uint32_t run = inc - tot;
#pragma unroll
  for (int q = 0; q < CPL; ++q) {
    const int ci = lane * CPL + q;
    if (ci < MAXC) off[ci] = (int32_t)run;
    run += c[q];
  }
}

// CTAs per SM the register budget is sized for (64 registers a thread at 128
// and 256 threads; more where fewer registers would spill)
constexpr int select_min_blocks(int rt) { return (rt == 128 || rt == 256) ? 1024 / rt : 1; }

template <int RT>
__global__ void __launch_bounds__(RT, select_min_blocks(RT)) topk_select_kernel(const __grid_constant__ TopkArgs a) {
  constexpr int E = kE;
  constexpr int kBins = SelCfg<RT>::BINS;
  constexpr int kDigit = SelCfg<RT>::DIGIT;
  constexpr int NW = RT / 32;
  constexpr int MAXC = RT * E / 32;      // 32-element chunks of the row
  __shared__ __align__(16) uint32_t hist[kBins];
  __shared__ uint32_t s_tot[NW];
  __shared__ uint32_t s_red[2 * NW];
  __shared__ uint32_t s_res[2];
  __shared__ uint32_t s_cnt;
  __shared__ uint32_t candk[kCandMax];
  __shared__ int32_t candi[kCandMax];
  __shared__ uint32_t gms[RT + 32 / E];  // fast path: kept slots of thread t (bit e = slot e); zero slots after
  __shared__ uint32_t eqw[MAXC];         // fallback: per-chunk words
  __shared__ uint32_t selw[MAXC];
  __shared__ int32_t offw[MAXC];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const long long row = blockIdx.x;
  const int nb = a.nb;
  const int words = (nb + 31) >> 5;
  const long long bh = row / a.G;
  const int g = (int)(row - bh * a.G);
  const int h = (int)(bh % a.H);
  const int b = (int)(bh / a.H);
  const uint32_t k = a.row_k ? (uint32_t)a.row_k[row] : (uint32_t)a.hk.k[h];
  const long long base = a.row_k ? (long long)a.row_ptr[row]
                                 : (long long)b * a.G * a.hk.kpre[a.H] + (long long)a.hk.kpre[h] * a.G + (long long)g * k;
  int32_t* dst = a.fwd_col + base;
  // mask word (b, h, ci, g): word columns contiguous over g for the transpose kernels
  uint32_t* mcol = a.mask + bh * (long long)a.words * a.G + g;

  const float* src = a.scores + row * (long long)nb;
  int off = (int)((reinterpret_cast<uintptr_t>(src) >> 2) & 3u);
  const bool vec = off + nb <= RT * E;   // else (rows of nearly RT * E keys) scalar loads from slot 0 = index 0
  if (!vec) off = 0;
  const int i0 = E * t - off;
  float x[E];
  float lo, hi;
  uint32_t vmask;                        // slots inside the row
  if (vec && i0 >= 0 && i0 + E <= nb) {
    const float4* p = reinterpret_cast<const float4*>(src + i0);
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      const float4 v = __ldcs(p + q);
      x[4 * q] = v.x;
      x[4 * q + 1] = v.y;
      x[4 * q + 2] = v.z;
      x[4 * q + 3] = v.w;
    }
    lo = fminf(x[0], x[E - 1]);
    hi = fmaxf(x[0], x[E - 1]);
#pragma unroll
    for (int e = 1; e + 1 < E - 1; e += 2) {
      lo = min3f(lo, x[e], x[e + 1]);
      hi = max3f(hi, x[e], x[e + 1]);
    }
    vmask = (1u << E) - 1u;
  } else {
    lo = INFINITY;
    hi = -INFINITY;
    vmask = 0u;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = i0 + e;
      const bool in = i >= 0 && i < nb;
      x[e] = in ? __ldcs(src + i) : __int_as_float(0x7fffffff);
      if (in) {
        lo = fminf(lo, x[e]);
        hi = fmaxf(hi, x[e]);
        vmask |= 1u << e;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    s_red[w] = __float_as_uint(lo);
    s_red[NW + w] = __float_as_uint(hi);
  }
  for (int i = 4 * t; i < kBins; i += 4 * RT) *reinterpret_cast<uint4*>(&hist[i]) = make_uint4(0u, 0u, 0u, 0u);
  if (t == 0) s_cnt = 0u;
  if (t < 32 / E) gms[RT + t] = 0u;
  __syncthreads();
#pragma unroll
  for (int v = 0; v < NW; ++v) {
    lo = fminf(lo, __uint_as_float(s_red[v]));
    hi = fmaxf(hi, __uint_as_float(s_red[NW + v]));
  }
  // any monotone bucket map will do, so a fast division: 0 (no fast path) when
  // hi - lo overflows or exceeds 2^126, huge when it is tiny
  const float scale = __fdividef((float)(kBins - 1), hi - lo);
  bool fast = hi > lo && scale > 0.f && scale < 1e30f;   // finite min < max (uniform over the CTA)

  if (fast) {
    // bucket = round((f - lo) * scale): adding 1.5 * 2^23 leaves the rounded
    // value in the low mantissa bits; NaN clamps to bucket 0
    const float B0 = 12582912.0f, B1 = B0 + (float)(kBins - 1);
    const float c0 = B0 - lo * scale;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = fminf(fmaxf(fmaf(x[e], scale, c0), B0), B1);
      atomicAdd(&hist[__float_as_uint(x[e]) - 0x4B400000u], 1u);
    }
    if (t == 0) atomicAdd(&hist[0], (uint32_t)nb - (uint32_t)(RT * E));   // the NaN slots outside the row
    __syncthreads();
    cta_find_bin<RT>(hist, k, s_tot, s_res);
    const uint32_t bstar = s_res[0];
    const uint32_t kk = s_res[1];                         // how many of bucket b* are kept
    const uint32_t C = hist[bstar];
    if (C <= (uint32_t)kCandMax) {
      const float xs = __uint_as_float(0x4B400000u + bstar);
      uint32_t gm = 0u;
      bool anyeq = false;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        gm |= (x[e] > xs) ? 1u << e : 0u;
        anyeq |= x[e] == xs;
      }
      uint32_t eqm = 0u;
      if (anyeq) {                                        // few threads
#pragma unroll
        for (int e = 0; e < E; ++e) eqm |= (x[e] == xs) ? 1u << e : 0u;
        eqm &= vmask;
      }
      if (C == kk) gm |= eqm;                             // the whole bucket is kept
      gms[t] = gm;
      if (C != kk) {                                      // uniform
        while (eqm) {
          const int i = i0 + __ffs(eqm) - 1;
          eqm &= eqm - 1u;
          const uint32_t pos = atomicAdd(&s_cnt, 1u);
          candk[pos] = score_key(__ldg(src + i));
          candi[pos] = i;
        }
        __syncthreads();
        for (uint32_t c = t; c < C; c += RT) {
          const uint32_t kc = candk[c];
          const int ic = candi[c];
          uint32_t rank = 0;
          for (uint32_t c2 = 0; c2 < C; ++c2) {
            const uint32_t k2 = candk[c2];
            rank += (k2 > kc || (k2 == kc && candi[c2] < ic)) ? 1u : 0u;
          }
          if (rank < kk) atomicOr(&gms[(ic + off) / E], 1u << ((ic + off) % E));
        }
      }
      __syncthreads();
      gm = gms[t];
      // list positions: exclusive prefix of the kept counts over threads
      const uint32_t cnt = (uint32_t)__popc(gm);
      uint32_t inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      if (lane == 31) s_tot[w] = inc;
      __syncthreads();
      uint32_t before = inc - cnt;
#pragma unroll
      for (int v = 0; v < NW - 1; ++v)
        if (v < w) before += s_tot[v];
      int32_t* d = dst + before;
      while (gm) {
        *d++ = i0 + __ffs(gm) - 1;
        gm &= gm - 1u;
      }
      // mask word m covers indices [32m, 32m + 32): the slot masks of threads
      // (32/E) m .. (32/E) (m + 1) shifted by off
      for (int m = t; m < words; m += RT) {
        constexpr int SPW = 32 / E;                       // threads per mask word
        uint64_t v = 0ull;
#pragma unroll
        for (int i = 0; i <= SPW; ++i) v |= (uint64_t)gms[SPW * m + i] << (E * i);
        mcol[(long long)m * a.G] = (uint32_t)(v >> off);
      }
    } else {
      fast = false;                                       // crowded bucket: exact radix select
    }
  }

  if (!fast) {
    // the row again, element i in thread i % RT (rare path)
    float f[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int i = j * RT + t;
      f[j] = (i < nb) ? __ldg(src + i) : 0.f;
    }
    uint32_t vand = 0xffffffffu, vor = 0u;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int i = j * RT + t;
      if (i < nb) {
        const uint32_t kj = score_key(f[j]);
        vand &= kj;
        vor |= kj;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vand &= __shfl_xor_sync(0xffffffffu, vand, o);
      vor |= __shfl_xor_sync(0xffffffffu, vor, o);
    }
    if (lane == 0) {
      s_red[w] = vand;
      s_red[NW + w] = vor;
    }
    __syncthreads();
    vand = 0xffffffffu;
    vor = 0u;
#pragma unroll
    for (int v = 0; v < NW; ++v) {
      vand &= s_red[v];
      vor |= s_red[NW + v];
    }
    const uint32_t diff = vand ^ vor;
    int remaining = diff ? 32 - __clz(diff) : 0;          // bits below the common prefix
    uint32_t hi_mask = remaining >= 32 ? 0u : ~((1u << remaining) - 1u);
    uint32_t prefix = vand & hi_mask;
    uint32_t kk = k;                                       // rank of the wanted key among those matching prefix
    while (remaining > 0) {
      const int nbits = remaining < kDigit ? remaining : kDigit;
      const int sh = remaining - nbits;
      const uint32_t dmask = (1u << nbits) - 1u;
      for (int i = t; i < kBins; i += RT) hist[i] = 0u;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int i = j * RT + t;
        const uint32_t kj = score_key(f[j]);
        const bool in = i < nb && (kj & hi_mask) == prefix;
        const uint32_t d = in ? (kj >> sh) & dmask : 0xffffffffu;
        const uint32_t same = __match_any_sync(0xffffffffu, d);
        if (in && lane == __ffs(same) - 1) atomicAdd(&hist[d], (uint32_t)__popc(same));
      }
      __syncthreads();
      cta_find_bin<RT>(hist, kk, s_tot, s_res);
      prefix |= s_res[0] << sh;
      kk = s_res[1];
      hi_mask |= dmask << sh;
      remaining = sh;
      __syncthreads();   // s_res / hist are reused
    }
    const uint32_t T = prefix;
    const uint32_t need_eq = kk;   // keys equal to T that are taken, lowest index first
    uint32_t gtw[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int i = j * RT + t;
      const bool valid = i < nb;
      const uint32_t kj = score_key(f[j]);
      gtw[j] = __ballot_sync(0xffffffffu, valid && kj > T);
      const uint32_t e = __ballot_sync(0xffffffffu, valid && kj == T);
      if (lane == 0) eqw[j * NW + w] = e;
    }
    __syncthreads();
    if (w == 0) chunk_prefix<MAXC>(eqw, words, offw, lane);   // equal keys before each chunk
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int ci = j * NW + w;
      if (ci < words) {
        const uint32_t e = eqw[ci];
        const uint32_t before = (uint32_t)offw[ci];
        uint32_t take = 0u;
        if (e != 0u && before < need_eq) {
          const uint32_t room = need_eq - before;
          if ((uint32_t)__popc(e) <= room) {
            take = e;
          } else {
            uint32_t x2 = e;
            for (uint32_t q = 0; q < room; ++q) {
              take |= x2 & (~x2 + 1u);
              x2 &= x2 - 1u;
            }
          }
        }
        if (lane == 0) selw[ci] = gtw[j] | take;
      }
    }
    __syncthreads();
    // ascending list (offsets per chunk) and the row's mask words
    if (w == 0) chunk_prefix<MAXC>(selw, words, offw, lane);
    __syncthreads();
    for (int ci = t; ci < words; ci += RT) {
      uint32_t sw = selw[ci];
      mcol[(long long)ci * a.G] = sw;
      int o = offw[ci];
      while (sw) {
        dst[o++] = ci * 32 + (__ffs(sw) - 1);
        sw &= sw - 1u;
      }
    }
  }

  if (t == 0) {
    if (!a.row_k) {
      a.fwd_ptr[row] = (int32_t)base;
      if (row == a.rows - 1) a.fwd_ptr[a.rows] = a.nnz;
    }
  }
}

// Lane i holds row i of a 32x32 bit block (bit j = column j); afterwards lane
// j holds column j (bit i = row i).  Block swaps of halves, quarters, ...
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  const uint32_t masks[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int t = 0; t < 5; ++t) {
    const int s = 16 >> t;
    const uint32_t m = masks[t];
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
    x = (lane & s) ? ((x & ~m) | ((y & ~m) >> s)) : ((x & m) | ((y & m) << s));
  }
  return x;
}

// The G rows of a (b, h) slice are cut into segments of kSeg rows so that the
// column walks below run in parallel: counts[bh][seg][col] is the number of
// rows of segment seg that selected column col.  Short segments keep the walk
// of a column that most rows select (a hub) short.
constexpr int kSeg = 128;

constexpr int kSegChunks = kSeg / 32;

// grid: (ceil(words / 8), heads); warp w walks word column blockIdx.x*8 + w of
// one (b, h) from the first row to the last, segment by segment (the next
// segment's loads issued before the current one is counted).  Lane l keeps the
// count of column wc*32 + l so far: counts[bh][seg][col] gets the entries of
// the column in the segments before seg, tot[bh][col] the column's total.
__global__ void __launch_bounds__(256) topk_colcount_kernel(const uint32_t* __restrict__ mask, int G, int nb,
                                                            int words, int nseg, int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ tot, long long bh0) {
  const int wc = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wc >= words) return;
  const int lane = threadIdx.x & 31;
  const long long bh = bh0 + blockIdx.y;
  const uint32_t* M = mask + (bh * words + wc) * (long long)G;   // this word column, rows contiguous
  const int col = wc * 32 + lane;
  auto load = [&](int seg, uint32_t (&xs)[kSegChunks]) {
#pragma unroll
    for (int i = 0; i < kSegChunks; ++i) {
      const int g = seg * kSeg + 32 * i + lane;
      xs[i] = g < G ? __ldg(M + g) : 0u;
    }
  };
  uint32_t xn[kSegChunks];
  load(0, xn);
  int run = 0;
  for (int seg = 0; seg < nseg; ++seg) {
    uint32_t xs[kSegChunks];
#pragma unroll
    for (int i = 0; i < kSegChunks; ++i) xs[i] = xn[i];
    if (seg + 1 < nseg) load(seg + 1, xn);
    if (col < nb) counts[(bh * nseg + seg) * nb + col] = run;
#pragma unroll
    for (int i = 0; i < kSegChunks; ++i) run += __popc(warp_transpose32(xs[i], lane));
  }
  if (col < nb) tot[bh * nb + col] = run;
}

// One CTA (1024 threads) per (b, h): bwd_ptr = slice base + exclusive scan of
// the column totals (read coalesced into shared memory, scanned there).
__global__ void __launch_bounds__(1024) topk_scan_kernel(const int32_t* __restrict__ tot,
                                                         const __grid_constant__ TopkArgs a,
                                                         int32_t* __restrict__ bwd_ptr, long long nslices) {
  __shared__ int warp_tot[32];
  __shared__ int col[kMaxBlocksPerRow];
  const long long bh = a.bh0 + blockIdx.x;
  const int h = (int)(bh % a.H), b = (int)(bh / a.H);
  const int nb = a.nb;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  for (int j = t; j < nb; j += 1024) col[j] = tot[bh * nb + j];
  __syncthreads();
  // thread t takes `per` consecutive columns
  const int per = (nb + 1023) / 1024;
  const int j0 = t * per, j1 = min(nb, j0 + per);
  int loc = 0;
  for (int j = j0; j < j1; ++j) loc += col[j];
  int inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += v;
    }
    warp_tot[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  const long long base = a.row_k ? (long long)a.row_ptr[bh * a.G]
                                 : (long long)b * a.G * a.hk.kpre[a.H] + (long long)a.hk.kpre[h] * a.G;
  int run = (int)base + (w > 0 ? warp_tot[w - 1] : 0) + inc - loc;
  for (int j = j0; j < j1; ++j) {
    const int c = col[j];
    col[j] = run;
    run += c;
  }
  __syncthreads();
  for (int j = t; j < nb; j += 1024) bwd_ptr[bh * nb + j] = col[j];
  if (bh == nslices - 1 && t == 0) bwd_ptr[nslices * nb] = a.row_k ? a.row_ptr[a.rows] : a.nnz;
}

// Each warp walks the rows of one segment of 32 mask columns (one word column),
// 32 rows at a time (lane i holds row g0 + i's word).  For every column with an
// entry among these rows (in ascending order) a ballot gives the rows that
// selected it, and those lanes store their row at the column's next output
// positions, consecutive in lane order: one coalesced store per (column,
// 32-row chunk), however many rows selected the column.  Lane l keeps the next
// output position of column wc * 32 + l.
constexpr int kFillWarps = 4;
// grid: (ceil(words / kFillWarps), nseg, B*H); the column's entries of segment
// seg start at bwd_ptr[col] + pos[seg][col] (pos = colcount's in-column counts).
__global__ void __launch_bounds__(kFillWarps * 32) topk_fill_kernel(const uint32_t* __restrict__ mask, int G, int nb,
                                                                    int words, const int32_t* __restrict__ pos,
                                                                    const int32_t* __restrict__ bwd_ptr,
                                                                    int32_t* __restrict__ bwd_col, long long bh0) {
  const int warp = threadIdx.x >> 5;
  const int wc = blockIdx.x * kFillWarps + warp;
  if (wc >= words) return;
  const int lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;             // lanes before this one
  const int seg = blockIdx.y, nseg = gridDim.y;
  const long long bh = bh0 + blockIdx.z;
  const uint32_t* M = mask + (bh * words + wc) * (long long)G;   // this word column, rows contiguous
  const int col = wc * 32 + lane;
  int cur = (col < nb) ? bwd_ptr[bh * nb + col] + pos[(bh * nseg + seg) * nb + col] : 0;
  const int gs = seg * kSeg, g1 = min(G, gs + kSeg);
  uint32_t xn = (gs + lane < g1) ? M[gs + lane] : 0u;
  for (int g0 = gs; g0 < g1; g0 += 32) {
    const uint32_t x = xn;
    if (g0 + 32 < g1) xn = (g0 + 32 + lane < g1) ? M[g0 + 32 + lane] : 0u;   // next chunk in flight
    uint32_t cols = __reduce_or_sync(0xffffffffu, x);   // columns with an entry in these rows
    if (cols == 0u) continue;
    // the columns' positions advance once per chunk (from the transposed bits),
    // so the per-column steps below do not depend on one another
    const uint32_t t = warp_transpose32(x, lane);       // lane l: the rows that selected column l
    while (cols) {
      const int c = __ffs(cols) - 1;
      cols &= cols - 1u;
      const uint32_t rows = __shfl_sync(0xffffffffu, t, c);
      const int base = __shfl_sync(0xffffffffu, cur, c);
      if ((rows >> lane) & 1u) bwd_col[base + __popc(rows & below)] = g0 + lane;
    }
    cur += __popc(t);
  }
}

// ---------------------------------------------------------------------------
// Mass-threshold selection: the list size m of each row.
//
// DSV pages [nl] 2A and [hi] 2A: the critical KV pairs are those that carry
// about 90 % of the attention score.  The predicted mass of block j in row r
// is p_j = softmax(temperature * S_r)_j; with the blocks in rank order
// (larger score first, equal scores by lower index) m is the smallest count
// whose leading blocks carry mass >= tau, clamped to [kmin, kmax]; the row
// then keeps its top m blocks (topk_select with per-row k).
//
// One CTA per row, 16 consecutive scores per thread as in topk_select.  The
// masses are fixed-point integers, P_j = round(2^40 exp2((s_j - max) c)), so
// every sum is exact and independent of the order of the atomics; the target
// is ceil(tau * sum P).  A histogram of counts and masses over value buckets
// finds the bucket where the leading mass reaches the target; if it holds at
// most kCandMax scores they are ranked exactly, else the search goes on
// inside that bucket with 11-bit radix digits of the order-preserving keys
// below their common prefix, until the remaining scores are all equal (then
// m follows by division).  A row holding a non-finite score gets m = kmax.
// ---------------------------------------------------------------------------
struct MassArgs {
  const float* scores;
  int32_t* m_out;
  int nb;
  long long rows;
  float coef;                            // temperature * log2(e)
  double tau;
  int kmin, kmax;
};

constexpr float kMassOne = 1099511627776.0f;   // 2^40: fixed-point unit of a mass

// 128 registers a thread: the 16 keys, masses (64-bit) and buckets stay in registers
constexpr int mass_min_blocks(int rt) { return rt >= 128 ? 512 / rt : 1; }

template <int RT>
__global__ void __launch_bounds__(RT, mass_min_blocks(RT)) topk_mass_count_kernel(const __grid_constant__ MassArgs a) {
  using u64 = unsigned long long;
  constexpr int E = kE;
  constexpr int kBins = SelCfg<RT>::BINS;
  constexpr int kDigit = SelCfg<RT>::DIGIT;
  constexpr int NW = RT / 32;
  constexpr int BPT = kBins / RT;
  __shared__ uint32_t hcnt[kBins];
  __shared__ u64 hmass[kBins];
  __shared__ u64 s_u[NW];
  __shared__ uint32_t s_w[2 * NW];
  __shared__ uint32_t s_bin, s_cnt;
  __shared__ u64 s_above, s_above_cnt;
  __shared__ uint32_t candk[kCandMax];
  __shared__ int32_t candi[kCandMax];
  __shared__ u64 candp[kCandMax];
  __shared__ u64 sortedp[kCandMax];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const long long row = blockIdx.x;
  const int nb = a.nb;
  const float* src = a.scores + row * (long long)nb;
  const int i0 = E * t;
  float x[E];
  uint32_t inplay = 0u;                  // slots in the search
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = i0 + e;
    x[e] = i < nb ? __ldg(src + i) : 0.f;
    if (i < nb) inplay |= 1u << e;
  }
  // CTA-wide helpers (every thread calls them)
  auto cta_max = [&](float v) -> float {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) s_w[w] = __float_as_uint(v);
    __syncthreads();
    float r = __uint_as_float(s_w[0]);
    for (int q = 1; q < NW; ++q) r = fmaxf(r, __uint_as_float(s_w[q]));
    return r;
  };
  auto cta_sum64 = [&](u64 v) -> u64 {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) s_u[w] = v;
    __syncthreads();
    u64 r = 0;
    for (int q = 0; q < NW; ++q) r += s_u[q];
    return r;
  };
  auto cta_and_or = [&](uint32_t& va, uint32_t& vo) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      va &= __shfl_xor_sync(0xffffffffu, va, o);
      vo |= __shfl_xor_sync(0xffffffffu, vo, o);
    }
    __syncthreads();
    if (lane == 0) {
      s_w[w] = va;
      s_w[NW + w] = vo;
    }
    __syncthreads();
    va = 0xffffffffu;
    vo = 0u;
    for (int q = 0; q < NW; ++q) {
      va &= s_w[q];
      vo |= s_w[NW + q];
    }
  };

  // a non-finite score: m = kmax
  bool bad = false;
#pragma unroll
  for (int e = 0; e < E; ++e) bad |= ((inplay >> e) & 1u) && !isfinite(x[e]);
  if (__syncthreads_or(bad)) {
    if (t == 0) a.m_out[row] = a.kmax;
    return;
  }
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((inplay >> e) & 1u) mx = fmaxf(mx, x[e]);
  const float hi = cta_max(mx);
  u64 P[E];
  u64 zs = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    P[e] = ((inplay >> e) & 1u) ? (u64)__float2ull_rn(exp2f((x[e] - hi) * a.coef) * kMassOne) : 0ull;
    zs += P[e];
  }
  const u64 Z = cta_sum64(zs);
  u64 target = (u64)ceil(a.tau * (double)Z);
  if (target > Z) target = Z;
  if (target == 0) target = 1;
  u64 mass_above = 0, cnt_above = 0;     // of the scores ranked above those still in play
  long long m = -1;
  uint32_t keys[E];
#pragma unroll
  for (int e = 0; e < E; ++e) keys[e] = score_key(x[e]);
  for (int level = 0; level < 5 && m < 0; ++level) {
    // bucket of every score in play: value buckets first, then radix digits
    uint32_t va = 0xffffffffu, vo = 0u;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if ((inplay >> e) & 1u) {
        va &= keys[e];
        vo |= keys[e];
      }
    cta_and_or(va, vo);
    const uint32_t diff = va ^ vo;
    if (diff == 0u) {
      // all scores in play are equal (equal masses): take as many as needed
      u64 pe = 0;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((inplay >> e) & 1u) pe = P[e];
      for (int o = 16; o > 0; o >>= 1) pe = max(pe, __shfl_xor_sync(0xffffffffu, pe, o));
      __syncthreads();
      if (lane == 0) s_u[w] = pe;
      __syncthreads();
      for (int q = 0; q < NW; ++q) pe = max(pe, s_u[q]);
      const u64 need = target - mass_above;
      m = (long long)cnt_above + (long long)((need + pe - 1) / (pe > 0 ? pe : 1));
      break;
    }
    const int remaining = 32 - __clz(diff);
    const int nbits = remaining < kDigit ? remaining : kDigit;
    const int sh = remaining - nbits;
    float scale = 0.f, c0 = 0.f, lo = 0.f, hv = 0.f;
    bool by_value = false;
    if (level == 0) {
      float mn = INFINITY;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((inplay >> e) & 1u) mn = fminf(mn, x[e]);
      lo = -cta_max(-mn);
      hv = hi;
      scale = __fdividef((float)(kBins - 1), hv - lo);
      by_value = hv > lo && scale > 0.f && scale < 1e30f;
      c0 = 12582912.0f - lo * scale;
    }
    uint32_t bk[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (by_value) {
        bk[e] = __float_as_uint(fminf(fmaxf(fmaf(x[e], scale, c0), 12582912.0f), 12582912.0f + (float)(kBins - 1))) -
                0x4B400000u;
      } else {
        bk[e] = (keys[e] >> sh) & ((1u << nbits) - 1u);
      }
    }
    for (int i = t; i < kBins; i += RT) {
      hcnt[i] = 0u;
      hmass[i] = 0ull;
    }
    if (t == 0) {
      s_cnt = 0u;
      s_bin = 0u;               // always overwritten below (the target lies in play); never read uninitialised
      s_above = mass_above;
      s_above_cnt = cnt_above;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e)
      if ((inplay >> e) & 1u) {
        atomicAdd(&hcnt[bk[e]], 1u);
        atomicAdd(&hmass[bk[e]], P[e]);
      }
    __syncthreads();
    // the bucket where the leading mass reaches the target: suffix sums from the top bucket down
    u64 tm = 0;
    uint32_t tc = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      tm += hmass[t * BPT + i];
      tc += hcnt[t * BPT + i];
    }
    u64 sm = tm;
    uint32_t sc = tc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const u64 vm = __shfl_down_sync(0xffffffffu, sm, o);
      const uint32_t vc = __shfl_down_sync(0xffffffffu, sc, o);
      if (lane + o < 32) {
        sm += vm;
        sc += vc;
      }
    }
    if (lane == 0) {
      s_u[w] = sm;
      s_w[w] = sc;
    }
    __syncthreads();
    for (int q = w + 1; q < NW; ++q) {
      sm += s_u[q];
      sc += s_w[q];
    }
    u64 above = mass_above + (sm - tm);          // mass of the buckets above this thread's range
    uint32_t above_c = sc - tc;
    if (above < target && above + tm >= target) {
      for (int i = BPT - 1; i >= 0; --i) {
        const u64 c = hmass[t * BPT + i];
        if (above + c >= target) {
          s_bin = (uint32_t)(t * BPT + i);
          s_above = above;
          s_above_cnt = cnt_above + above_c;
          break;
        }
        above += c;
        above_c += hcnt[t * BPT + i];
      }
    }
    __syncthreads();
    const uint32_t bstar = s_bin;
    mass_above = s_above;
    cnt_above = s_above_cnt;
    const uint32_t C = hcnt[bstar];
    // only the scores of bucket b* stay in play
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (bk[e] != bstar) inplay &= ~(1u << e);
    if (C <= (uint32_t)kCandMax) {
      // rank the bucket exactly by (key desc, index asc) and walk its masses in that order
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((inplay >> e) & 1u) {
          const uint32_t pos = atomicAdd(&s_cnt, 1u);
          candk[pos] = keys[e];
          candi[pos] = i0 + e;
          candp[pos] = P[e];
        }
      __syncthreads();
      for (uint32_t c = t; c < C; c += RT) {
        const uint32_t kc = candk[c];
        const int ic = candi[c];
        uint32_t rank = 0;
        for (uint32_t c2 = 0; c2 < C; ++c2) {
          const uint32_t k2 = candk[c2];
          rank += (k2 > kc || (k2 == kc && candi[c2] < ic)) ? 1u : 0u;
        }
        sortedp[rank] = candp[c];
      }
      __syncthreads();
      if (t == 0) {
        u64 run = mass_above;
        uint32_t r = 0;
        while (r + 1 < C && run + sortedp[r] < target) run += sortedp[r++];
        s_w[0] = r + 1;                          // how many of the bucket are needed
      }
      __syncthreads();
      m = (long long)cnt_above + (long long)s_w[0];
    }
    __syncthreads();                             // s_* and the histograms are reused
  }
  if (m < 0) m = a.kmax;                         // not reached: the digits run out first
  if (t == 0) a.m_out[row] = (int32_t)(m < a.kmin ? a.kmin : (m > a.kmax ? a.kmax : m));
}

// fwd_ptr[r] = sum of m over rows before r, fwd_ptr[rows] = the total (one CTA)
__global__ void __launch_bounds__(1024) topk_row_scan_kernel(const int32_t* __restrict__ m, long long rows,
                                                             int32_t* __restrict__ fwd_ptr) {
  __shared__ long long warp_tot[32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const long long per = (rows + 1023) / 1024;
  const long long j0 = t * per, j1 = j0 + per < rows ? j0 + per : rows;
  long long loc = 0;
  for (long long j = j0; j < j1; ++j) loc += m[j];
  long long inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[w] = inc;
  __syncthreads();
  if (w == 0) {
    long long v = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    warp_tot[lane] = v;
  }
  __syncthreads();
  long long run = (w > 0 ? warp_tot[w - 1] : 0) + inc - loc;
  for (long long j = j0; j < j1; ++j) {
    fwd_ptr[j] = (int32_t)run;
    run += m[j];
  }
  if (t == 1023) fwd_ptr[rows] = (int32_t)warp_tot[31];
}

}  // namespace

size_t topk_ws_bytes(const dsv_shape& s) {
  const size_t G = (size_t)(s.N / s.block);
  const size_t words = (G + 31) / 32;
  const size_t bhs = (size_t)s.B * s.H;
  const size_t nseg = (G + kSeg - 1) / kSeg;
  return align256(bhs * G * words * sizeof(uint32_t)) + align256(bhs * nseg * G * sizeof(int32_t)) +
         align256(bhs * G * sizeof(int32_t));
}

namespace {

cudaError_t run_topk_transpose(const TopkArgs& a, int32_t* bwd_ptr, int32_t* bwd_col, int32_t* counts,
                               cudaStream_t st, long long bh1);

// the select kernel and the transposed lists, for fixed (a.row_k == null) or per-row k
cudaError_t run_topk(const TopkArgs& a, int32_t* bwd_ptr, int32_t* bwd_col, int32_t* counts, cudaStream_t st) {
  const int G = a.G, words = a.words;
  const long long bhs = a.rows / G;
  // threads per row: the smallest of 32 ... 512 holding the row in 16 keys per
  // thread (32 keys per thread measured slower on 4050-block rows: half the
  // threads per SM for the load latency)
  cudaError_t e;
  const unsigned grid = (unsigned)a.rows;
  if (G <= 32 * kE) topk_select_kernel<32><<<grid, 32, 0, st>>>(a);
  else if (G <= 64 * kE) topk_select_kernel<64><<<grid, 64, 0, st>>>(a);
  else if (G <= 128 * kE) topk_select_kernel<128><<<grid, 128, 0, st>>>(a);
  else if (G <= 256 * kE) topk_select_kernel<256><<<grid, 256, 0, st>>>(a);
  else topk_select_kernel<512><<<grid, 512, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return run_topk_transpose(a, bwd_ptr, bwd_col, counts, st, -1);
}

// The transposed lists from the selection bitmask a.mask: per-segment column
// counts, their scan into bwd_ptr and output positions, then the fill.
// Heads a.bh0 .. bh1 - 1 only (bh1 < 0: to the last).
cudaError_t run_topk_transpose(const TopkArgs& a, int32_t* bwd_ptr, int32_t* bwd_col, int32_t* counts,
                               cudaStream_t st, long long bh1) {
  const int G = a.G, words = a.words;
  const long long bhs = a.rows / G;
  const long long nh = (bh1 < 0 ? bhs : bh1) - a.bh0;
  if (nh <= 0) return cudaSuccess;
  cudaError_t e;
  const int nseg = (G + kSeg - 1) / kSeg;
  int32_t* tot = counts + align256((size_t)bhs * nseg * G * sizeof(int32_t)) / sizeof(int32_t);
  dim3 g2((unsigned)((words + 7) / 8), (unsigned)nh);
  topk_colcount_kernel<<<g2, 256, 0, st>>>(a.mask, G, G, words, nseg, counts, tot, a.bh0);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_scan_kernel<<<(unsigned)nh, 1024, 0, st>>>(tot, a, bwd_ptr, bhs);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dim3 g3((unsigned)((words + kFillWarps - 1) / kFillWarps), (unsigned)nseg, (unsigned)nh);
  topk_fill_kernel<<<g3, kFillWarps * 32, 0, st>>>(a.mask, G, G, words, counts, bwd_ptr, bwd_col, a.bh0);
  return cudaGetLastError();
}

TopkArgs topk_args(const float* scores, const dsv_shape& s, int32_t* fwd_ptr, int32_t* fwd_col, void* ws) {
  const int G = s.N / s.block;
  TopkArgs a{};
  a.scores = scores;
  a.fwd_ptr = fwd_ptr;
  a.fwd_col = fwd_col;
  a.mask = static_cast<uint32_t*>(ws);
  a.H = s.H;
  a.G = G;
  a.nb = G;
  a.words = (G + 31) / 32;
  a.rows = (long long)s.B * s.H * G;
  a.row_k = nullptr;
  a.row_ptr = nullptr;
  a.bh0 = 0;
  return a;
}

int32_t* topk_counts(void* ws, const dsv_shape& s) {
  const size_t G = (size_t)(s.N / s.block);
  return reinterpret_cast<int32_t*>(static_cast<char*>(ws) +
                                    align256((size_t)s.B * s.H * G * ((G + 31) / 32) * sizeof(uint32_t)));
}

}  // namespace

cudaError_t launch_topk(const float* scores, const dsv_shape& s, const HeadK& hk, int64_t nnz, int32_t* fwd_ptr,
                        int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col, void* ws, cudaStream_t st) {
  TopkArgs a = topk_args(scores, s, fwd_ptr, fwd_col, ws);
  a.nnz = (int)nnz;
  a.hk = hk;
  return run_topk(a, bwd_ptr, bwd_col, topk_counts(ws, s), st);
}

cudaError_t launch_topk_transpose(const dsv_shape& s, const HeadK& hk, int64_t nnz, int32_t* bwd_ptr,
                                  int32_t* bwd_col, void* ws, cudaStream_t st, long long bh0, long long bh1) {
  TopkArgs a = topk_args(nullptr, s, nullptr, nullptr, ws);
  a.nnz = (int)nnz;
  a.hk = hk;
  a.bh0 = bh0;
  return run_topk_transpose(a, bwd_ptr, bwd_col, topk_counts(ws, s), st, bh1);
}

size_t topk_mass_ws_bytes(const dsv_shape& s) {
  return topk_ws_bytes(s) + align256((size_t)s.B * s.H * (size_t)(s.N / s.block) * sizeof(int32_t));
}

cudaError_t launch_topk_mass(const float* scores, const dsv_shape& s, float tau, float temperature, int kmin,
                             int kmax, int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col,
                             void* ws, cudaStream_t st) {
  TopkArgs a = topk_args(scores, s, fwd_ptr, fwd_col, ws);
  int32_t* m = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + topk_ws_bytes(s));
  MassArgs ma;
  ma.scores = scores;
  ma.m_out = m;
  ma.nb = a.nb;
  ma.rows = a.rows;
  ma.coef = temperature * 1.4426950408889634f;
  ma.tau = (double)tau;
  ma.kmin = kmin;
  ma.kmax = kmax;
  const unsigned grid = (unsigned)a.rows;
  const int G = a.G;
  if (G <= 32 * kE) topk_mass_count_kernel<32><<<grid, 32, 0, st>>>(ma);
  else if (G <= 64 * kE) topk_mass_count_kernel<64><<<grid, 64, 0, st>>>(ma);
  else if (G <= 128 * kE) topk_mass_count_kernel<128><<<grid, 128, 0, st>>>(ma);
  else if (G <= 256 * kE) topk_mass_count_kernel<256><<<grid, 256, 0, st>>>(ma);
  else topk_mass_count_kernel<512><<<grid, 512, 0, st>>>(ma);
  cudaError_t e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_row_scan_kernel<<<1, 1024, 0, st>>>(m, a.rows, fwd_ptr);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  a.row_k = m;
  a.row_ptr = fwd_ptr;
  return run_topk(a, bwd_ptr, bwd_col, topk_counts(ws, s), st);
}

}  // namespace dsv
