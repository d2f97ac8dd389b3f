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
//   topk_colcount  per (b, h, 32-column slab): 32x32 bit transposes of the
//                  mask (stored word column by word column, rows contiguous)
//                  give each column's population.
//   topk_scan      per (b, h): exclusive scan of the column counts -> bwd_ptr.
//   topk_fill      same walk as colcount; each lane appends the set rows of
//                  its column in ascending g.
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
// words are put together from the threads' 16-bit slot masks.  Value binning
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
  __shared__ uint32_t gms[RT + 2];       // fast path: kept slots of thread t (bit e = slot e); two zero slots after
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
  const uint32_t k = (uint32_t)a.hk.k[h];
  const long long base = (long long)b * a.G * a.hk.kpre[a.H] + (long long)a.hk.kpre[h] * a.G + (long long)g * k;
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
  if (t < 2) gms[RT + t] = 0u;
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
      // mask word m covers indices [32m, 32m + 32): slots 2m .. 2m + 2 shifted by off
      for (int m = t; m < words; m += RT) {
        const uint64_t v = (uint64_t)gms[2 * m] | ((uint64_t)gms[2 * m + 1] << 16) | ((uint64_t)gms[2 * m + 2] << 32);
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
    a.fwd_ptr[row] = (int32_t)base;
    if (row == a.rows - 1) a.fwd_ptr[a.rows] = a.nnz;
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
// rows of segment seg that selected column col.
constexpr int kSeg = 512;

// grid: (ceil(words / 8), nseg, B*H); warp w handles mask word column blockIdx.x*8 + w.
__global__ void __launch_bounds__(256) topk_colcount_kernel(const uint32_t* __restrict__ mask, int G, int nb,
                                                            int words, int32_t* __restrict__ counts) {
  const int wc = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wc >= words) return;
  const int lane = threadIdx.x & 31;
  const int seg = blockIdx.y, nseg = gridDim.y;
  const long long bh = blockIdx.z;
  const uint32_t* M = mask + (bh * words + wc) * (long long)G;   // this word column, rows contiguous
  const int g1 = min(G, (seg + 1) * kSeg);
  int cnt = 0;
#pragma unroll 4
  for (int g0 = seg * kSeg; g0 < g1; g0 += 32) {
    const int g = g0 + lane;
    const uint32_t x = (g < g1) ? M[g] : 0u;
    cnt += __popc(warp_transpose32(x, lane));
  }
  const int col = wc * 32 + lane;
  if (col < nb) counts[(bh * nseg + seg) * nb + col] = cnt;
}

// One CTA (1024 threads) per (b, h): bwd_ptr = slice base + exclusive scan of
// the column totals; counts[bh][seg][col] becomes the output position of the
// first entry of segment seg in column col.
__global__ void __launch_bounds__(1024) topk_scan_kernel(int32_t* __restrict__ counts, int nseg,
                                                         const __grid_constant__ TopkArgs a,
                                                         int32_t* __restrict__ bwd_ptr, long long nslices) {
  __shared__ int warp_tot[32];
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H), b = (int)(bh / a.H);
  const int nb = a.nb;
  int32_t* C = counts + bh * (long long)nseg * nb;
  const int per = (nb + 1023) / 1024;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int j0 = t * per;
  int loc = 0;
  for (int j = j0; j < min(nb, j0 + per); ++j)
    for (int sg = 0; sg < nseg; ++sg) loc += C[sg * nb + j];
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
  const long long base = (long long)b * a.G * a.hk.kpre[a.H] + (long long)a.hk.kpre[h] * a.G;
  int run = (int)base + (w > 0 ? warp_tot[w - 1] : 0) + inc - loc;
  for (int j = j0; j < min(nb, j0 + per); ++j) {
    bwd_ptr[bh * nb + j] = run;
    for (int sg = 0; sg < nseg; ++sg) {
      const int c = C[sg * nb + j];
      C[sg * nb + j] = run;
      run += c;
    }
  }
  if (bh == nslices - 1 && t == 0) bwd_ptr[nslices * nb] = a.nnz;
}

// Each warp walks the G rows of 32 mask columns (one word column), 32 rows at a
// time; after a 32x32 bit transpose lane l holds column l's bits.  The rows
// found are staged per column in shared memory and written out 33..64 at a
// time by the whole warp (coalesced), not one 4-byte store per lane.
constexpr int kFillWarps = 4;
constexpr int kFillCap = 64;             // staged entries per column
// grid: (ceil(words / kFillWarps), nseg, B*H); pos = counts after topk_scan.
__global__ void __launch_bounds__(kFillWarps * 32) topk_fill_kernel(const uint32_t* __restrict__ mask, int G, int nb,
                                                                    int words, const int32_t* __restrict__ pos,
                                                                    int32_t* __restrict__ bwd_col) {
  __shared__ int32_t stage[kFillWarps][32][kFillCap + 1];   // +1: lanes at the same depth hit different banks
  const int warp = threadIdx.x >> 5;
  const int wc = blockIdx.x * kFillWarps + warp;
  if (wc >= words) return;
  const int lane = threadIdx.x & 31;
  const int seg = blockIdx.y, nseg = gridDim.y;
  const long long bh = blockIdx.z;
  const uint32_t* M = mask + (bh * words + wc) * (long long)G;   // this word column, rows contiguous
  const int col = wc * 32 + lane;
  int32_t (*buf)[kFillCap + 1] = stage[warp];
  int cur = (col < nb) ? pos[(bh * nseg + seg) * nb + col] : 0;   // next output position of this lane's column
  int cnt = 0;                                          // staged entries of this lane's column
  auto flush = [&](unsigned who) {
    while (who) {
      const int l = __ffs(who) - 1;
      who &= who - 1u;
      const int n = __shfl_sync(0xffffffffu, cnt, l);
      const int base = __shfl_sync(0xffffffffu, cur, l);
      for (int i = lane; i < n; i += 32) bwd_col[base + i] = buf[l][i];
      if (lane == l) {
        cur += cnt;
        cnt = 0;
      }
    }
    __syncwarp();
  };
  const int gs = seg * kSeg, g1 = min(G, gs + kSeg);
  uint32_t xn = (gs + lane < g1) ? M[gs + lane] : 0u;
  for (int g0 = gs; g0 < g1; g0 += 32) {
    const uint32_t x = xn;
    if (g0 + 32 < g1) xn = (g0 + 32 + lane < g1) ? M[g0 + 32 + lane] : 0u;   // next chunk in flight
    uint32_t t = warp_transpose32(x, lane);
    flush(__ballot_sync(0xffffffffu, cnt + __popc(t) > kFillCap));
    while (t) {
      const int bit = __ffs(t) - 1;
      buf[lane][cnt++] = g0 + bit;
      t &= t - 1u;
    }
    __syncwarp();
  }
  flush(__ballot_sync(0xffffffffu, cnt > 0));
}

}  // namespace

size_t topk_ws_bytes(const dsv_shape& s) {
  const size_t G = (size_t)(s.N / s.block);
  const size_t words = (G + 31) / 32;
  const size_t bhs = (size_t)s.B * s.H;
  const size_t nseg = (G + kSeg - 1) / kSeg;
  return align256(bhs * G * words * sizeof(uint32_t)) + align256(bhs * nseg * G * sizeof(int32_t));
}

cudaError_t launch_topk(const float* scores, const dsv_shape& s, const HeadK& hk, int64_t nnz, int32_t* fwd_ptr,
                        int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col, void* ws, cudaStream_t st) {
  const int G = s.N / s.block;
  const int words = (G + 31) / 32;
  const long long bhs = (long long)s.B * s.H;
  uint32_t* mask = static_cast<uint32_t*>(ws);
  int32_t* counts =
      reinterpret_cast<int32_t*>(static_cast<char*>(ws) + align256((size_t)bhs * G * words * sizeof(uint32_t)));
  TopkArgs a;
  a.scores = scores;
  a.fwd_ptr = fwd_ptr;
  a.fwd_col = fwd_col;
  a.mask = mask;
  a.H = s.H;
  a.G = G;
  a.nb = G;
  a.words = words;
  a.rows = bhs * G;
  a.nnz = (int)nnz;
  a.hk = hk;
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
  const int nseg = (G + kSeg - 1) / kSeg;
  dim3 g2((unsigned)((words + 7) / 8), (unsigned)nseg, (unsigned)bhs);
  topk_colcount_kernel<<<g2, 256, 0, st>>>(mask, G, G, words, counts);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_scan_kernel<<<(unsigned)bhs, 1024, 0, st>>>(counts, nseg, a, bwd_ptr, bhs);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dim3 g3((unsigned)((words + kFillWarps - 1) / kFillWarps), (unsigned)nseg, (unsigned)bhs);
  topk_fill_kernel<<<g3, kFillWarps * 32, 0, st>>>(mask, G, G, words, counts, bwd_col);
  return cudaGetLastError();
}

}  // namespace dsv
