// cube.cu — 3D cube query grouping as a token permutation.
//
// DSV pages [nl] 2B and [hi] 2B (query grouping): adjacent tokens in 3D space
// share their critical KV, so queries are grouped in small cubes (the pages
// name 2x2x2) that share one proxy's critical-KV indices.  The hot path
// groups `block` consecutive tokens; regrouping the token order so that each
// run of `block` consecutive tokens is one ct x cy x cx cube of the T x Hl x Wl
// latent grid makes those groups cubes.  The permutation is applied by the
// caller before the path (Q, K, V, dO) and undone after it (O, dQ, dK, dV);
// the path itself is unchanged.
//
// Order: raster n = (t*Hl + y)*Wl + x; cube order walks the cube grid
// (T/ct, Hl/cy, Wl/cx) in raster order and the tokens of a cube in raster
// order (lt, ly, lx).  perm(n_cube) = n_raster.
//
// A token row of d bf16 is moved by d/8 threads, 16 bytes each, read and
// written whole; each thread moves 4 rows' chunks with all loads issued first
// (HBM-bound: 2 * B*H*N*d*2 bytes per call).
#include "dsv_launch.h"

namespace dsv {
namespace {

struct CubeGeom {
  int Hl, Wl, ct, cy, cx;
  int CY, CX;            // cubes along y and x
  int block;             // ct * cy * cx
};

// raster index of the token at cube-order position n
__device__ __forceinline__ int cube_to_raster(int n, const CubeGeom& g) {
  const int c = n / g.block, l = n - c * g.block;
  const int bx = c % g.CX, cyx = c / g.CX;
  const int by = cyx % g.CY, bt = cyx / g.CY;
  const int lx = l % g.cx, lyt = l / g.cx;
  const int ly = lyt % g.cy, lt = lyt / g.cy;
  return ((bt * g.ct + lt) * g.Hl + by * g.cy + ly) * g.Wl + bx * g.cx + lx;
}

constexpr int kRowsPerThread = 4;       // 16-byte moves in flight per thread

template <int D>
__global__ void __launch_bounds__(256) cube_permute_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           long long rows, int N, CubeGeom g, int inverse) {
  constexpr int TPR = D / 8;             // threads per token row (16 bytes each)
  constexpr int RPC = 256 / TPR;         // rows per CTA and pass
  const int c = threadIdx.x % TPR;
  long long from[kRowsPerThread], to[kRowsPerThread];
  uint4 v[kRowsPerThread];
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) {
    const long long r = ((long long)blockIdx.x * kRowsPerThread + i) * RPC + threadIdx.x / TPR;
    const bool valid = r < rows;
    const long long bh = valid ? r / N : 0;
    const int n = valid ? (int)(r - bh * N) : 0;
    // the first thread of a row works out its raster index and hands it to
    // the row's other TPR - 1 threads
    int m = (c == 0 && valid) ? cube_to_raster(n, g) : 0;
    m = __shfl_sync(0xffffffffu, m, 0, TPR);
    const long long other = bh * N + m;
    // forward: row n of the cube order comes from raster row perm(n); inverse: the other way
    from[i] = valid ? (inverse ? r : other) : -1;
    to[i] = inverse ? other : r;
  }
  // all loads first, so that each thread keeps kRowsPerThread moves in flight
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i)
    if (from[i] >= 0) v[i] = __ldcs(src + from[i] * TPR + c);
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i)
    if (from[i] >= 0) __stcs(dst + to[i] * TPR + c, v[i]);
}

}  // namespace

cudaError_t launch_cube_permute(const void* src, void* dst, const dsv_shape& s, int T, int Hl, int Wl, int ct, int cy,
                                int cx, int inverse, cudaStream_t st) {
  (void)T;
  CubeGeom g{Hl, Wl, ct, cy, cx, Hl / cy, Wl / cx, ct * cy * cx};
  const long long rows = (long long)s.B * s.H * s.N;
  const uint4* a = static_cast<const uint4*>(src);
  uint4* b = static_cast<uint4*>(dst);
  if (s.d == 128) {
    constexpr int RPB = 256 / 16 * kRowsPerThread;   // rows per CTA
    cube_permute_kernel<128><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, st>>>(a, b, rows, s.N, g, inverse);
  } else {
    constexpr int RPB = 256 / 8 * kRowsPerThread;
    cube_permute_kernel<64><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, st>>>(a, b, rows, s.N, g, inverse);
  }
  return cudaGetLastError();
}

}  // namespace dsv
