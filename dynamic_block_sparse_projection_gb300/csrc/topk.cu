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
//   topk_rows      one warp per row.  Scores become order-preserving uint32
//                  keys in shared memory; an MSB-first radix select (4 x 8
//                  bits) finds the k-th largest key T and how many keys equal
//                  to T to take; one pass in index order then emits the list
//                  (ballot + prefix) and the row's bitmask word by word.
//   topk_colcount  per (b, h, 32-column slab): 32x32 bit transposes of the
//                  mask give each column's population.
//   topk_scan      per (b, h): exclusive scan of the column counts -> bwd_ptr.
//   topk_fill      same walk as colcount; each lane appends the set rows of
//                  its column in ascending g.
#include <algorithm>

#include "dsv_launch.h"

namespace dsv {

namespace {

constexpr int kRowWarps = 8;
constexpr size_t kTopkSmemBudget = 200 * 1024;  // rows kernel: keys + histogram per warp

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

__global__ void __launch_bounds__(kRowWarps * 32) topk_rows_kernel(const __grid_constant__ TopkArgs a) {
  extern __shared__ uint32_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= a.rows) return;
  const int nb = a.nb;
  const int nbp = (nb + 31) & ~31;
  uint32_t* keys = sm + warp * (nbp + 256);
  uint32_t* hist = keys + nbp;
  const long long bh = row / a.G;
  const int g = (int)(row - bh * a.G);
  const int h = (int)(bh % a.H);
  const int b = (int)(bh / a.H);
  const int k = a.hk.k[h];

  const float* src = a.scores + row * (long long)nb;
#pragma unroll 8
  for (int i = lane; i < nbp; i += 32) keys[i] = (i < nb) ? score_key(__ldcs(src + i)) : 0u;
  __syncwarp();

  // MSB-first radix select of the k-th largest key.
  uint32_t prefix = 0u, pmask = 0u;
  int kk = k;  // rank of the wanted key among the keys that match `prefix`
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
#pragma unroll
    for (int i = lane; i < 256; i += 32) hist[i] = 0u;
    __syncwarp();
    for (int i = lane; i < nb; i += 32) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    int c[8];
    int tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = (int)hist[8 * lane + e];
      tot += c[e];
    }
    int suf = tot;  // sum of tot over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += v;
    }
    int cum = suf - tot;  // keys in bins above this lane's 8 bins
    int found = -1, newkk = 0;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
      if (found < 0 && cum < kk && cum + c[e] >= kk) {
        found = 8 * lane + e;
        newkk = kk - cum;
      }
      cum += c[e];
    }
    const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
    const int src_lane = __ffs(bal) - 1;
    const int digit = __shfl_sync(0xffffffffu, found, src_lane);
    kk = __shfl_sync(0xffffffffu, newkk, src_lane);
    prefix |= (uint32_t)digit << shift;
    pmask |= 255u << shift;
    __syncwarp();
  }
  const uint32_t T = prefix;
  const int need_eq = kk;  // how many keys equal to T are taken, lowest index first

  // Emit in index order; the selection ballot of each 32-element chunk is the mask word.
  const long long base = (long long)b * a.G * a.hk.kpre[a.H] + (long long)a.hk.kpre[h] * a.G + (long long)g * k;
  int32_t* dst = a.fwd_col + base;
  uint32_t* mrow = a.mask + row * (long long)a.words;
  const unsigned lt = (1u << lane) - 1u;
  int n_eq = 0, n_sel = 0;
  for (int c0 = 0; c0 < nbp; c0 += 32) {
    const int i = c0 + lane;
    const bool valid = i < nb;
    const uint32_t key = keys[i];
    const bool eq = valid && key == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const bool sel = valid && (key > T || (eq && (n_eq + __popc(beq & lt)) < need_eq));
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    if (sel) dst[n_sel + __popc(bsel & lt)] = i;
    if (lane == 0) mrow[c0 >> 5] = bsel;
    n_eq += __popc(beq);
    n_sel += __popc(bsel);
  }
  if (lane == 0) {
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

// grid: (ceil(words / 8), B*H); warp w handles mask word column blockIdx.x*8 + w.
__global__ void __launch_bounds__(256) topk_colcount_kernel(const uint32_t* __restrict__ mask, int G, int nb,
                                                            int words, int32_t* __restrict__ counts) {
  const int wc = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wc >= words) return;
  const int lane = threadIdx.x & 31;
  const long long bh = blockIdx.y;
  const uint32_t* M = mask + bh * (long long)G * words;
  int cnt = 0;
  for (int g0 = 0; g0 < G; g0 += 32) {
    const int g = g0 + lane;
    const uint32_t x = (g < G) ? M[(long long)g * words + wc] : 0u;
    cnt += __popc(warp_transpose32(x, lane));
  }
  const int col = wc * 32 + lane;
  if (col < nb) counts[bh * nb + col] = cnt;
}

// One CTA (1024 threads) per (b, h): bwd_ptr = slice base + exclusive scan of counts.
__global__ void __launch_bounds__(1024) topk_scan_kernel(const int32_t* __restrict__ counts,
                                                         const __grid_constant__ TopkArgs a,
                                                         int32_t* __restrict__ bwd_ptr, long long nslices) {
  __shared__ int warp_tot[32];
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H), b = (int)(bh / a.H);
  const int nb = a.nb;
  const int per = (nb + 1023) / 1024;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int j0 = t * per;
  int loc = 0;
  for (int j = j0; j < min(nb, j0 + per); ++j) loc += counts[bh * nb + j];
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
    run += counts[bh * nb + j];
  }
  if (bh == nslices - 1 && t == 0) bwd_ptr[nslices * nb] = a.nnz;
}

__global__ void __launch_bounds__(256) topk_fill_kernel(const uint32_t* __restrict__ mask, int G, int nb, int words,
                                                        const int32_t* __restrict__ bwd_ptr,
                                                        int32_t* __restrict__ bwd_col) {
  const int wc = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wc >= words) return;
  const int lane = threadIdx.x & 31;
  const long long bh = blockIdx.y;
  const uint32_t* M = mask + bh * (long long)G * words;
  const int col = wc * 32 + lane;
  int cur = (col < nb) ? bwd_ptr[bh * nb + col] : 0;
  for (int g0 = 0; g0 < G; g0 += 32) {
    const int g = g0 + lane;
    const uint32_t x = (g < G) ? M[(long long)g * words + wc] : 0u;
    uint32_t t = warp_transpose32(x, lane);
    while (t) {
      const int bit = __ffs(t) - 1;
      bwd_col[cur++] = g0 + bit;
      t &= t - 1u;
    }
  }
}

}  // namespace

size_t topk_ws_bytes(const dsv_shape& s) {
  const size_t G = (size_t)(s.N / s.block);
  const size_t words = (G + 31) / 32;
  const size_t bhs = (size_t)s.B * s.H;
  return align256(bhs * G * words * sizeof(uint32_t)) + align256(bhs * G * sizeof(int32_t));
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
  const int nbp = (G + 31) & ~31;
  const size_t per_warp = (size_t)(nbp + 256) * sizeof(uint32_t);
  const int warps = (int)std::max<size_t>(1, std::min<size_t>(kRowWarps, kTopkSmemBudget / per_warp));
  const size_t smem = (size_t)warps * per_warp;
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<(unsigned)((a.rows + warps - 1) / warps), warps * 32, smem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dim3 g2((unsigned)((words + 7) / 8), (unsigned)bhs);
  topk_colcount_kernel<<<g2, 256, 0, st>>>(mask, G, G, words, counts);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_scan_kernel<<<(unsigned)bhs, 1024, 0, st>>>(counts, a, bwd_ptr, bhs);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_fill_kernel<<<g2, 256, 0, st>>>(mask, G, G, words, bwd_ptr, bwd_col);
  return cudaGetLastError();
}

}  // namespace dsv
