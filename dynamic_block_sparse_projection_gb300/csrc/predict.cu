// predict.cu — low-rank block-score predictor.
//
// DSV page [nl], "Technische samenvatting" 2A (per-head low-rank predictors
// W^Q_lr, W^K_lr approximating Q K^T) and 2B (query grouping: one proxy query
// per group of adjacent tokens).  A group's proxy is the mean of its
// low-rank queries and a key block is scored by the mean of its low-rank
// keys; by linearity the mean can be taken before the projection:
//   qbar_g = (mean_{i in g} Q_i) W^Q,   kbar_j = (mean_{i in j} K_i) W^K,
//   S[g, j] = qbar_g . kbar_j.
//
// Kernel 1 (HBM-bound) streams Q and K once: one CTA per (tensor, b, h,
// group) sums its `block` rows with 16-byte loads, then projects the mean to
// rank r.  Kernel 2 writes the G x nb score matrix of each (b, h) from the
// pooled vectors with an r-deep fp32 FMA tile.
#include <cuda_bf16.h>

#include "dsv_launch.h"

namespace dsv {

namespace {

constexpr int kPoolThreads = 256;

__device__ __forceinline__ uint4 ld_stream_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void add_bf16x8(float* acc, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(w[i] << 16);
    acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// grid: (B*H*G, 2); blockIdx.y = 0 pools Q with W^Q, 1 pools K with W^K.
// out: [B*H*G, r] fp32 (qp for Q, kp for K).
template <int D, int BLOCK>
__global__ void __launch_bounds__(kPoolThreads) pool_project_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                    const __nv_bfloat16* __restrict__ K,
                                                                    const float* __restrict__ Wq,
                                                                    const float* __restrict__ Wk, int H, int G, int r,
                                                                    float* __restrict__ qp, float* __restrict__ kp) {
  constexpr int VEC = D / 8;                   // 16-byte vectors per row
  constexpr int RPP = kPoolThreads / VEC;      // rows per pass
  constexpr int PASSES = BLOCK / RPP;
  static_assert(BLOCK % RPP == 0, "block must be a multiple of rows per pass");
  __shared__ float4 part[RPP][VEC * 2];        // partial column sums
  __shared__ float mean[D];
  __shared__ float proj[kPoolThreads];

  const long long row = blockIdx.x;            // (b*H + h)*G + g
  const int which = blockIdx.y;
  const __nv_bfloat16* X = which ? K : Q;
  const float* W = which ? Wk : Wq;
  float* out = which ? kp : qp;
  const int h = (int)((row / G) % H);

  const uint4* src = reinterpret_cast<const uint4*>(X + row * (long long)BLOCK * D);
  const int c = threadIdx.x % VEC;
  const int rl = threadIdx.x / VEC;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  uint4 v[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) v[p] = ld_stream_u4(src + (p * RPP + rl) * VEC + c);
#pragma unroll
  for (int p = 0; p < PASSES; ++p) add_bf16x8(acc, v[p]);
  part[rl][2 * c] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  part[rl][2 * c + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (threadIdx.x < D) {
    const float* pf = reinterpret_cast<const float*>(&part[0][0]);
    float sum = 0.f;
#pragma unroll 8
    for (int i = 0; i < RPP; ++i) sum += pf[i * D + threadIdx.x];
    mean[threadIdx.x] = sum * (1.0f / BLOCK);
  }
  __syncthreads();
  // projection: thread t handles output column t % r over a slice of the d inputs
  const int parts = kPoolThreads / r;
  const int t = threadIdx.x;
  float s = 0.f;
  if (t < parts * r) {
    const int col = t % r;
    const int sl = t / r;
    const int per = (D + parts - 1) / parts;
    const int c0 = sl * per;
    const int c1 = min(D, c0 + per);
    const float* Wh = W + (long long)h * D * r;
    for (int cc = c0; cc < c1; ++cc) s = fmaf(mean[cc], __ldg(Wh + cc * r + col), s);
  }
  proj[t] = s;
  __syncthreads();
  if (t < r) {
    float tot = 0.f;
    for (int sl = 0; sl < parts; ++sl) tot += proj[sl * r + t];
    out[row * r + t] = tot;
  }
}

// S tile of 64 groups x 128 blocks for one (b, h).  Thread t owns 8 rows and
// 4 columns; VW selects how the 4 columns map to stores (16, 8 or 4 bytes).
constexpr int kTM = 64, kTN = 128;

template <int VW>
__device__ __forceinline__ int score_col(int tc, int m) {
  if (VW == 4) return 4 * tc + m;
  if (VW == 2) return 64 * (m >> 1) + 2 * tc + (m & 1);
  return 32 * m + tc;
}

template <int VW>
__global__ void __launch_bounds__(256) score_kernel(const float* __restrict__ qp, const float* __restrict__ kp, int G,
                                                    int nb, int r, float* __restrict__ S) {
  extern __shared__ float sm[];
  float* qs = sm;                 // [r][kTM]
  float* ks = sm + r * kTM;       // [r][kTN]
  const long long bh = blockIdx.z;
  const int g0 = blockIdx.y * kTM;
  const int j0 = blockIdx.x * kTN;
  const float* qsrc = qp + (bh * G + g0) * (long long)r;
  const float* ksrc = kp + (bh * nb + j0) * (long long)r;
  for (int i = threadIdx.x; i < kTM * r; i += 256) {
    const int gi = i / r, kk = i % r;
    qs[kk * kTM + gi] = (g0 + gi < G) ? qsrc[i] : 0.f;
  }
  for (int i = threadIdx.x; i < kTN * r; i += 256) {
    const int ji = i / r, kk = i % r;
    ks[kk * kTN + ji] = (j0 + ji < nb) ? ksrc[i] : 0.f;
  }
  __syncthreads();
  const int tc = threadIdx.x & 31;
  const int tr = threadIdx.x >> 5;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[i][m] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < r; ++kk) {
    const float4 a0 = *reinterpret_cast<const float4*>(qs + kk * kTM + tr * 8);
    const float4 a1 = *reinterpret_cast<const float4*>(qs + kk * kTM + tr * 8 + 4);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    float b[4];
    if (VW == 4) {
      const float4 b4 = *reinterpret_cast<const float4*>(ks + kk * kTN + 4 * tc);
      b[0] = b4.x;
      b[1] = b4.y;
      b[2] = b4.z;
      b[3] = b4.w;
    } else {
#pragma unroll
      for (int m = 0; m < 4; ++m) b[m] = ks[kk * kTN + score_col<VW>(tc, m)];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m) acc[i][m] = fmaf(a[i], b[m], acc[i][m]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int g = g0 + tr * 8 + i;
    if (g >= G) break;
    float* dst = S + (bh * G + g) * (long long)nb;
    if (VW == 4) {
      const int j = j0 + 4 * tc;
      if (j + 3 < nb) {
        __stcs(reinterpret_cast<float4*>(dst + j), make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
      } else {
        for (int m = 0; m < 4; ++m)
          if (j + m < nb) dst[j + m] = acc[i][m];
      }
    } else if (VW == 2) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int j = j0 + 64 * h2 + 2 * tc;
        if (j + 1 < nb) {
          __stcs(reinterpret_cast<float2*>(dst + j), make_float2(acc[i][2 * h2], acc[i][2 * h2 + 1]));
        } else if (j < nb) {
          dst[j] = acc[i][2 * h2];
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int j = j0 + 32 * m + tc;
        if (j < nb) dst[j] = acc[i][m];
      }
    }
  }
}

template <int D, int BLOCK>
cudaError_t launch_pool(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s, float* qp,
                        float* kp, cudaStream_t st) {
  const long long rows = (long long)s.B * s.H * (s.N / s.block);
  dim3 grid((unsigned)rows, 2);
  pool_project_kernel<D, BLOCK><<<grid, kPoolThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K), Wq, Wk, s.H, s.N / s.block, s.r,
      qp, kp);
  return cudaGetLastError();
}

}  // namespace

size_t predict_ws_bytes(const dsv_shape& s) {
  const size_t rows = (size_t)s.B * s.H * (size_t)(s.N / s.block);
  return 2 * align256(rows * (size_t)s.r * sizeof(float));
}

cudaError_t launch_predict(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                           float* scores, void* ws, cudaStream_t st) {
  const int G = s.N / s.block;
  const size_t rows = (size_t)s.B * s.H * G;
  float* qp = static_cast<float*>(ws);
  float* kp = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows * (size_t)s.r * sizeof(float)));
  cudaError_t e;
  if (s.d == 128 && s.block == 128) e = launch_pool<128, 128>(Q, K, Wq, Wk, s, qp, kp, st);
  else if (s.d == 128 && s.block == 64) e = launch_pool<128, 64>(Q, K, Wq, Wk, s, qp, kp, st);
  else if (s.d == 64 && s.block == 128) e = launch_pool<64, 128>(Q, K, Wq, Wk, s, qp, kp, st);
  else e = launch_pool<64, 64>(Q, K, Wq, Wk, s, qp, kp, st);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((G + kTN - 1) / kTN), (unsigned)((G + kTM - 1) / kTM), (unsigned)(s.B * s.H));
  const size_t smem = (size_t)s.r * (kTM + kTN) * sizeof(float);
  if (G % 4 == 0) score_kernel<4><<<grid, 256, smem, st>>>(qp, kp, G, G, s.r, scores);
  else if (G % 2 == 0) score_kernel<2><<<grid, 256, smem, st>>>(qp, kp, G, G, s.r, scores);
  else score_kernel<1><<<grid, 256, smem, st>>>(qp, kp, G, G, s.r, scores);
  return cudaGetLastError();
}

}  // namespace dsv
