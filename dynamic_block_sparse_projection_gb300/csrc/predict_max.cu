// predict_max.cu — max-pooled block scores of the low-rank predictor.
//
// DSV page [nl], "Technische samenvatting" 2A (low-rank predictors W^Q_lr,
// W^K_lr whose logits approximate Q K^T) and 2B (one proxy per query group).
// The pages leave open how a (group, key block) tile of logits is reduced to
// one score; predict.cu takes the mean, this file the largest logit:
//   S[g, j] = max over i in group g, l in key block j of (Q_i W^Q) . (K_l W^K).
// A maximum does not commute with pooling, so every token is projected and
// every tile is formed: block^2 r FMAs per (g, j), on the CUDA cores in fp32.
//
// Kernel 1 projects 64 token rows of Q (or K) of one (b, h) per CTA to rank r,
// the head's W staged once in shared memory, into the workspace
// ([B*H*N, r] fp32 for each tensor).  Kernel 2 takes one query group and a run
// of kJPerCta key blocks per CTA: the group's rank-r rows stay in shared
// memory, each key tile is staged [rank][token] while the next one loads into
// registers, a thread owns a (block/16) x (block/16) register tile of logits
// summed by packed two-lane FMAs (per-lane rounding of fmaf), and the tile
// maximum goes through warp shuffles and one shared-memory step.  fmaxf drops
// a NaN logit.
#include <cuda_bf16.h>

#include "dsv_launch.h"

namespace dsv {
namespace {

constexpr int kProjRows = 64;            // token rows per projection CTA (N is a multiple)
constexpr int kJPerCta = 16;             // key blocks per tile CTA

// grid (B*H*N / kProjRows, 2): blockIdx.y = 0 projects Q with W^Q, 1 projects K with W^K.
// Thread t computes row t % 64 and the r/4 columns (t / 64) * r/4 ...
template <int D, int R>
__global__ void __launch_bounds__(256) lowrank_project_kernel(const __nv_bfloat16* __restrict__ Q,
                                                              const __nv_bfloat16* __restrict__ K,
                                                              const float* __restrict__ Wq,
                                                              const float* __restrict__ Wk, int H, int N,
                                                              float* __restrict__ qlr, float* __restrict__ klr) {
  constexpr int XS = D + 1;              // padded row: a warp's 32 rows hit 32 banks
  constexpr int RC = R / 4;              // output columns per thread (even: R % 8 == 0)
  extern __shared__ float4 sm4[];
  float* w_s = reinterpret_cast<float*>(sm4);   // [D][R]
  float* x_s = w_s + D * R;                     // [kProjRows][XS]
  const int t = threadIdx.x;
  const long long row0 = (long long)blockIdx.x * kProjRows;
  const int which = blockIdx.y;
  const int h = (int)((row0 / N) % H);          // 64 rows never straddle a (b, h): N % 64 == 0
  const uint4* X = reinterpret_cast<const uint4*>((which ? K : Q) + row0 * D);
  const float4* W = reinterpret_cast<const float4*>((which ? Wk : Wq) + (long long)h * D * R);
  float* out = (which ? klr : qlr) + row0 * R;
  for (int i = t; i < D * R / 4; i += 256) reinterpret_cast<float4*>(w_s)[i] = __ldg(W + i);
  for (int i = t; i < kProjRows * D / 8; i += 256) {
    const int row = i / (D / 8), c8 = (i - row * (D / 8)) * 8;
    const uint4 v = __ldcs(X + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x_s[row * XS + c8 + 2 * e] = __uint_as_float(w[e] << 16);
      x_s[row * XS + c8 + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  __syncthreads();
  const int row = t % kProjRows, c0 = (t / kProjRows) * RC;
  float acc[RC];
#pragma unroll
  for (int m = 0; m < RC; ++m) acc[m] = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; ++c) {
    const float x = x_s[row * XS + c];
    const float2* wr = reinterpret_cast<const float2*>(w_s + c * R + c0);
#pragma unroll
    for (int m = 0; m < RC / 2; ++m) {
      const float2 wv = wr[m];
      acc[2 * m] = fmaf(x, wv.x, acc[2 * m]);
      acc[2 * m + 1] = fmaf(x, wv.y, acc[2 * m + 1]);
    }
  }
  float2* dst = reinterpret_cast<float2*>(out + (long long)row * R + c0);
#pragma unroll
  for (int m = 0; m < RC / 2; ++m) dst[m] = make_float2(acc[2 * m], acc[2 * m + 1]);
}

// One [BLOCK, R] fp32 tile of rank-r rows, moved through registers into a
// [R][BLOCK] shared tile.  Slot i of the tile is row i % BLOCK, ranks
// 4*(i / BLOCK) .. +3, so a warp's stores cover 32 consecutive rows of one
// rank: 32 banks.
template <int BLOCK, int R>
struct TileIO {
  static constexpr int NV = BLOCK * R / 4;                 // float4 slots
  static constexpr int LPT = (NV + 255) / 256;             // slots per thread
  float4 v[LPT];
  __device__ __forceinline__ void load(const float4* __restrict__ src) {
#pragma unroll
    for (int p = 0; p < LPT; ++p) {
      const int i = threadIdx.x + 256 * p;
      if (i < NV) {
        const int row = i % BLOCK, k4 = (i / BLOCK) * 4;
        v[p] = __ldg(src + row * (R / 4) + k4 / 4);
      }
    }
  }
  __device__ __forceinline__ void store(float* __restrict__ dst) const {
#pragma unroll
    for (int p = 0; p < LPT; ++p) {
      const int i = threadIdx.x + 256 * p;
      if (i < NV) {
        const int row = i % BLOCK, k4 = (i / BLOCK) * 4;
        dst[(k4 + 0) * BLOCK + row] = v[p].x;
        dst[(k4 + 1) * BLOCK + row] = v[p].y;
        dst[(k4 + 2) * BLOCK + row] = v[p].z;
        dst[(k4 + 3) * BLOCK + row] = v[p].w;
      }
    }
  }
};

// grid (G * ceil(G / kJPerCta), 1, B*H).  CTA: query group g = blockIdx.x / chunks,
// key blocks j0 .. j1-1.  Thread (tr, tc) = (t / 16, t % 16) owns tile rows
// TM*tr .. TM*tr+TM-1 and columns 4*tc + 64*q .. +3 for q < TN/4.
template <int BLOCK, int R>
__global__ void __launch_bounds__(256) tile_max_kernel(const float* __restrict__ qlr, const float* __restrict__ klr,
                                                       int G, int chunks, float* __restrict__ S) {
  constexpr int TM = BLOCK / 16;         // rows per thread
  constexpr int TN = BLOCK / 16;         // columns per thread
  constexpr int NP = TN / 2;             // packed column pairs per row
  extern __shared__ float4 sm4[];
  float* qs = reinterpret_cast<float*>(sm4);   // [R][BLOCK]
  float* ks = qs + R * BLOCK;                  // [R][BLOCK]
  __shared__ float red[8];
  __shared__ float s_out[kJPerCta];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const long long bh = blockIdx.z;
  const int g = (int)(blockIdx.x / chunks);
  const int j0 = (int)(blockIdx.x - (long long)g * chunks) * kJPerCta;
  const int j1 = min(G, j0 + kJPerCta);
  const float4* qsrc = reinterpret_cast<const float4*>(qlr + (bh * G + g) * (long long)BLOCK * R);
  const float4* kbase = reinterpret_cast<const float4*>(klr + bh * G * (long long)BLOCK * R);
  {
    TileIO<BLOCK, R> q;
    q.load(qsrc);
    q.store(qs);
  }
  TileIO<BLOCK, R> kt;
  kt.load(kbase + (long long)j0 * (BLOCK * R / 4));
  const int tc = t & 15, tr = t >> 4;
  for (int j = j0; j < j1; ++j) {
    __syncthreads();                       // the previous tile's products are done with ks
    kt.store(ks);
    __syncthreads();
    if (j + 1 < j1) kt.load(kbase + (long long)(j + 1) * (BLOCK * R / 4));
    uint64_t acc[TM][NP];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int m = 0; m < NP; ++m) acc[i][m] = 0ull;
#pragma unroll 4
    for (int kk = 0; kk < R; ++kk) {
      float a[TM];
#pragma unroll
      for (int p = 0; p < TM / 4; ++p) {
        const float4 av = *reinterpret_cast<const float4*>(qs + kk * BLOCK + tr * TM + 4 * p);
        a[4 * p] = av.x;
        a[4 * p + 1] = av.y;
        a[4 * p + 2] = av.z;
        a[4 * p + 3] = av.w;
      }
      uint64_t b2[NP];
#pragma unroll
      for (int q = 0; q < TN / 4; ++q) {
        const float4 bv = *reinterpret_cast<const float4*>(ks + kk * BLOCK + 64 * q + 4 * tc);
        b2[2 * q] = f2_pack(bv.x, bv.y);
        b2[2 * q + 1] = f2_pack(bv.z, bv.w);
      }
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const uint64_t a2 = f2_pack(a[i], a[i]);
#pragma unroll
        for (int m = 0; m < NP; ++m) acc[i][m] = fma2(a2, b2[m], acc[i][m]);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int m = 0; m < NP; ++m) {
        float lo, hi;
        f2_unpack(acc[i][m], lo, hi);
        mx = fmaxf(mx, fmaxf(lo, hi));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[w] = mx;
    __syncthreads();
    if (t == 0) {
      float r = red[0];
#pragma unroll
      for (int q = 1; q < 8; ++q) r = fmaxf(r, red[q]);
      s_out[j - j0] = r;
    }
  }
  __syncthreads();
  if (t < j1 - j0) S[(bh * G + g) * (long long)G + j0 + t] = s_out[t];
}

template <int BLOCK, int R>
cudaError_t launch_tile_max(const float* qlr, const float* klr, const dsv_shape& s, float* scores, cudaStream_t st) {
  const int G = s.N / BLOCK;
  const int chunks = (G + kJPerCta - 1) / kJPerCta;
  const int smem = 2 * R * BLOCK * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(tile_max_kernel<BLOCK, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((long long)G * chunks), 1, (unsigned)(s.B * s.H));
  tile_max_kernel<BLOCK, R><<<grid, 256, smem, st>>>(qlr, klr, G, chunks, scores);
  return cudaGetLastError();
}

template <int D, int R>
cudaError_t launch_project(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                           float* qlr, float* klr, cudaStream_t st) {
  const int smem = (D * R + kProjRows * (D + 1)) * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(lowrank_project_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)s.B * s.H * s.N;
  dim3 grid((unsigned)(rows / kProjRows), 2);
  lowrank_project_kernel<D, R><<<grid, 256, smem, st>>>(static_cast<const __nv_bfloat16*>(Q),
                                                        static_cast<const __nv_bfloat16*>(K), Wq, Wk, s.H, s.N, qlr,
                                                        klr);
  return cudaGetLastError();
}

template <int R>
cudaError_t launch_predict_max_r(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                                 float* qlr, float* klr, float* scores, cudaStream_t st) {
  cudaError_t e = s.d == 128 ? launch_project<128, R>(Q, K, Wq, Wk, s, qlr, klr, st)
                             : launch_project<64, R>(Q, K, Wq, Wk, s, qlr, klr, st);
  if (e != cudaSuccess) return e;
  return s.block == 128 ? launch_tile_max<128, R>(qlr, klr, s, scores, st)
                        : launch_tile_max<64, R>(qlr, klr, s, scores, st);
}

}  // namespace

size_t predict_max_ws_bytes(const dsv_shape& s) {
  const size_t rows = (size_t)s.B * s.H * (size_t)s.N;
  return 2 * align256(rows * (size_t)s.r * sizeof(float));
}

cudaError_t launch_predict_max(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                               float* scores, void* ws, cudaStream_t st) {
  const size_t rows = (size_t)s.B * s.H * (size_t)s.N;
  float* qlr = static_cast<float*>(ws);
  float* klr = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows * (size_t)s.r * sizeof(float)));
  switch (s.r) {
    case 8: return launch_predict_max_r<8>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    case 16: return launch_predict_max_r<16>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    case 24: return launch_predict_max_r<24>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    case 32: return launch_predict_max_r<32>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    case 40: return launch_predict_max_r<40>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    case 48: return launch_predict_max_r<48>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    case 56: return launch_predict_max_r<56>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
    default: return launch_predict_max_r<64>(Q, K, Wq, Wk, s, qlr, klr, scores, st);
  }
}

}  // namespace dsv
