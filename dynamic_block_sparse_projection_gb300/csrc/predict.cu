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
// Kernel 1 (HBM-bound) streams Q and K once: one CTA per (tensor, b, h, 8
// consecutive groups) sums each group's `block` rows with 16-byte loads, then
// projects the 8 means to rank r with the head's W staged once in shared
// memory (for the fused predictor + top-k it also writes the tf32 hi / lo
// parts of each projected vector, the operands of its tensor-core scores).  Kernel 2 writes the G x nb score matrix of each (b, h) from the
// pooled vectors with r-deep fp32 FMA register tiles (8 x 8 per thread).
#include <cuda_bf16.h>

#include <type_traits>

#include "dsv_launch.h"

namespace dsv {

namespace {

constexpr int kPoolThreads = 256;
constexpr int kGPC = 8;                  // groups pooled per CTA (one W load per CTA)
constexpr int kSplitCols = 32;           // columns of the fused predictor's tf32 operand rows (r <= 32)

// x rounded to tf32 (10 mantissa bits, to nearest, ties away from zero), as fp32 bits
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

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

// grid: (B*H*ceil(G/kGPC), 2); blockIdx.y = 0 pools Q with W^Q, 1 pools K with W^K.
// A CTA takes kGPC consecutive groups of one (b, h): the group means, then the
// projection of all of them with this head's W held in shared memory.  Loads
// of the next group are issued before the current one is reduced.
// out: [B*H*G, R] fp32 (qp for Q, kp for K).
template <int D, int BLOCK, int R>
__global__ void __launch_bounds__(kPoolThreads) pool_project_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                    const __nv_bfloat16* __restrict__ K,
                                                                    const float* __restrict__ Wq,
                                                                    const float* __restrict__ Wk, int H, int G,
                                                                    float* __restrict__ qp, float* __restrict__ kp,
                                                                    float* __restrict__ split, long long split_stride) {
  constexpr int VEC = D / 8;                   // 16-byte vectors per row
  constexpr int RPP = kPoolThreads / VEC;      // rows per pass
  constexpr int PASSES = BLOCK / RPP;
  static_assert(BLOCK % RPP == 0, "block must be a multiple of rows per pass");
  __shared__ float4 part[RPP][VEC * 2];        // partial column sums of one group
  __shared__ float mean[kGPC][D];
  __shared__ float w_s[D * R];

  const int cpb = (G + kGPC - 1) / kGPC;       // CTAs per (b, h)
  const long long bh = blockIdx.x / cpb;
  const int g0 = (int)(blockIdx.x - bh * cpb) * kGPC;
  const int ng = min(kGPC, G - g0);
  const int which = blockIdx.y;
  const __nv_bfloat16* X = which ? K : Q;
  const int h = (int)(bh % H);
  const float* W = (which ? Wk : Wq) + (long long)h * D * R;
  float* out = which ? kp : qp;

  const int c = threadIdx.x % VEC;
  const int rl = threadIdx.x / VEC;
  const uint4* src = reinterpret_cast<const uint4*>(X + (bh * G + g0) * (long long)BLOCK * D);
  uint4 v[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) v[p] = ld_stream_u4(src + (p * RPP + rl) * VEC + c);
  for (int i = threadIdx.x; i < D * R / 4; i += kPoolThreads)
    reinterpret_cast<float4*>(w_s)[i] = __ldg(reinterpret_cast<const float4*>(W) + i);
  for (int gi = 0; gi < ng; ++gi) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) add_bf16x8(acc, v[p]);
    if (gi + 1 < ng) {
      const uint4* nsrc = src + (long long)(gi + 1) * BLOCK * VEC;
#pragma unroll
      for (int p = 0; p < PASSES; ++p) v[p] = ld_stream_u4(nsrc + (p * RPP + rl) * VEC + c);
    }
    part[rl][2 * c] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    part[rl][2 * c + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
    if (threadIdx.x < D) {
      const float* pf = reinterpret_cast<const float*>(&part[0][0]);
      float sum = 0.f;
#pragma unroll 8
      for (int i = 0; i < RPP; ++i) sum += pf[i * D + threadIdx.x];
      mean[gi][threadIdx.x] = sum * (1.0f / BLOCK);
    }
    __syncthreads();
  }
  // projection: output (gi, col) = mean[gi] . W[:, col] for gi < ng, col < R
  for (int o = threadIdx.x; o < ng * R; o += kPoolThreads) {
    const int gi = o / R, col = o - gi * R;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int cc = 0; cc < D; cc += 2) {
      s0 = fmaf(mean[gi][cc], w_s[cc * R + col], s0);
      s1 = fmaf(mean[gi][cc + 1], w_s[(cc + 1) * R + col], s1);
    }
    const float v = s0 + s1;
    const long long row = bh * G + g0 + gi;
    out[row * R + col] = v;
    if (split != nullptr) {
      // the tf32 parts of the fused predictor: hi = tf32(v), lo = tf32(v - hi),
      // rows of kSplitCols columns (zero beyond R); parts q hi, q lo, k hi, k lo
      float* hi = split + (2 * which) * split_stride + row * kSplitCols;
      const float h = tf32_rna(v);
      hi[col] = h;
      hi[split_stride + col] = tf32_rna(v - h);
    }
  }
  if (split != nullptr && R < kSplitCols) {
    for (int o = threadIdx.x; o < ng * (kSplitCols - R); o += kPoolThreads) {
      const int gi = o / (kSplitCols - R), col = R + o - gi * (kSplitCols - R);
      float* hi = split + (2 * which) * split_stride + (bh * G + g0 + gi) * kSplitCols;
      hi[col] = 0.f;
      hi[split_stride + col] = 0.f;
    }
  }
}

// Scores of one (b, h): a 128 x 128 tile of S per CTA, r-deep fp32 FMAs.
// Thread (tr, tc) owns rows 8*tr .. 8*tr+7 and columns 4*tc .. 4*tc+3 and
// 64 + 4*tc .. 64 + 4*tc+3: per rank step 4 vector shared loads feed 64 FMAs,
// issued as 32 packed two-lane FMAs (each lane rounds like fmaf, so the sums
// are those of the scalar loop).  VW = 4, 2 or 1: the widest store the row
// length allows.
constexpr int kST = 128;

template <int R, int VW>
__global__ void __launch_bounds__(256) score_kernel(const float* __restrict__ qp, const float* __restrict__ kp, int G,
                                                    int nb, float* __restrict__ S) {
  extern __shared__ float4 sm4[];
  float* qs = reinterpret_cast<float*>(sm4);   // [R][kST]
  float* ks = qs + R * kST;                    // [R][kST]
  const long long bh = blockIdx.z;
  const int g0 = blockIdx.y * kST;
  const int j0 = blockIdx.x * kST;
  const float4* qsrc = reinterpret_cast<const float4*>(qp + (bh * G + g0) * (long long)R);
  const float4* ksrc = reinterpret_cast<const float4*>(kp + (bh * nb + j0) * (long long)R);
  // transpose the pooled vectors into [rank][row] tiles: a warp takes 32
  // consecutive rows of one 4-rank slice, so its shared stores hit 32 banks
  for (int i = threadIdx.x; i < kST * R / 4; i += 256) {
    const int row = i % kST, k4 = (i / kST) * 4;
    const float4 a = (g0 + row < G) ? __ldg(qsrc + row * (R / 4) + k4 / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    qs[(k4 + 0) * kST + row] = a.x;
    qs[(k4 + 1) * kST + row] = a.y;
    qs[(k4 + 2) * kST + row] = a.z;
    qs[(k4 + 3) * kST + row] = a.w;
    const float4 b = (j0 + row < nb) ? __ldg(ksrc + row * (R / 4) + k4 / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    ks[(k4 + 0) * kST + row] = b.x;
    ks[(k4 + 1) * kST + row] = b.y;
    ks[(k4 + 2) * kST + row] = b.z;
    ks[(k4 + 3) * kST + row] = b.w;
  }
  __syncthreads();
  const int tc = threadIdx.x & 15;
  const int tr = threadIdx.x >> 4;
  uint64_t acc[8][4];                          // column pairs (2m, 2m + 1) of row i
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[i][m] = 0ull;
#pragma unroll
  for (int kk = 0; kk < R; ++kk) {
    const float4 a0 = *reinterpret_cast<const float4*>(qs + kk * kST + tr * 8);
    const float4 a1 = *reinterpret_cast<const float4*>(qs + kk * kST + tr * 8 + 4);
    const float4 b0 = *reinterpret_cast<const float4*>(ks + kk * kST + 4 * tc);
    const float4 b1 = *reinterpret_cast<const float4*>(ks + kk * kST + 64 + 4 * tc);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint64_t b2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y), f2_pack(b1.z, b1.w)};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t a2 = f2_pack(a[i], a[i]);
#pragma unroll
      for (int m = 0; m < 4; ++m) acc[i][m] = fma2(a2, b2[m], acc[i][m]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int g = g0 + tr * 8 + i;
    if (g >= G) break;
    float* dst = S + (bh * G + g) * (long long)nb;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int j = j0 + 64 * hh + 4 * tc;
      float v[4];
      f2_unpack(acc[i][2 * hh], v[0], v[1]);
      f2_unpack(acc[i][2 * hh + 1], v[2], v[3]);
      if (j + 3 < nb) {
        if (VW == 4) {
          __stcs(reinterpret_cast<float4*>(dst + j), make_float4(v[0], v[1], v[2], v[3]));
        } else if (VW == 2) {
          __stcs(reinterpret_cast<float2*>(dst + j), make_float2(v[0], v[1]));
          __stcs(reinterpret_cast<float2*>(dst + j + 2), make_float2(v[2], v[3]));
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) __stcs(dst + j + m, v[m]);
        }
      } else {
        for (int m = 0; m < 4; ++m)
          if (j + m < nb) dst[j + m] = v[m];
      }
    }
  }
}

template <int D, int BLOCK, int R>
cudaError_t launch_pool(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s, float* qp,
                        float* kp, cudaStream_t st, float* split = nullptr, long long part = 0) {
  if (split != nullptr && R > kSplitCols) return cudaErrorInvalidValue;
  const int G = s.N / s.block;
  const long long ctas = (long long)s.B * s.H * ((G + kGPC - 1) / kGPC);
  dim3 grid((unsigned)ctas, 2);
  pool_project_kernel<D, BLOCK, R><<<grid, kPoolThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(Q),
                                                                  static_cast<const __nv_bfloat16*>(K), Wq, Wk, s.H,
                                                                  G, qp, kp, split, part);
  return cudaGetLastError();
}

template <int R>
cudaError_t launch_predict_r(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                             float* qp, float* kp, float* scores, cudaStream_t st) {
  cudaError_t e;
  if (s.d == 128 && s.block == 128) e = launch_pool<128, 128, R>(Q, K, Wq, Wk, s, qp, kp, st);
  else if (s.d == 128 && s.block == 64) e = launch_pool<128, 64, R>(Q, K, Wq, Wk, s, qp, kp, st);
  else if (s.d == 64 && s.block == 128) e = launch_pool<64, 128, R>(Q, K, Wq, Wk, s, qp, kp, st);
  else e = launch_pool<64, 64, R>(Q, K, Wq, Wk, s, qp, kp, st);
  if (e != cudaSuccess) return e;
  const int G = s.N / s.block;
  dim3 grid((unsigned)((G + kST - 1) / kST), (unsigned)((G + kST - 1) / kST), (unsigned)(s.B * s.H));
  const int smem = 2 * R * kST * (int)sizeof(float);
  auto k4 = score_kernel<R, 4>;
  auto k2 = score_kernel<R, 2>;
  auto k1 = score_kernel<R, 1>;
  auto kern = G % 4 == 0 ? k4 : (G % 2 == 0 ? k2 : k1);
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  kern<<<grid, 256, smem, st>>>(qp, kp, G, G, scores);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pool_project(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                                float* qp, float* kp, cudaStream_t st, float* split, long long part) {
  auto pool = [&](auto rtag) -> cudaError_t {
    constexpr int R = decltype(rtag)::value;
    if (s.d == 128 && s.block == 128) return launch_pool<128, 128, R>(Q, K, Wq, Wk, s, qp, kp, st, split, part);
    if (s.d == 128 && s.block == 64) return launch_pool<128, 64, R>(Q, K, Wq, Wk, s, qp, kp, st, split, part);
    if (s.d == 64 && s.block == 128) return launch_pool<64, 128, R>(Q, K, Wq, Wk, s, qp, kp, st, split, part);
    return launch_pool<64, 64, R>(Q, K, Wq, Wk, s, qp, kp, st, split, part);
  };
  switch (s.r) {
    case 8: return pool(std::integral_constant<int, 8>{});
    case 16: return pool(std::integral_constant<int, 16>{});
    case 24: return pool(std::integral_constant<int, 24>{});
    default: return pool(std::integral_constant<int, 32>{});
  }
}

size_t predict_ws_bytes(const dsv_shape& s) {
  const size_t rows = (size_t)s.B * s.H * (size_t)(s.N / s.block);
  return 2 * align256(rows * (size_t)s.r * sizeof(float));
}

cudaError_t launch_predict(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                           float* scores, void* ws, cudaStream_t st) {
  const size_t rows = (size_t)s.B * s.H * (size_t)(s.N / s.block);
  float* qp = static_cast<float*>(ws);
  float* kp = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows * (size_t)s.r * sizeof(float)));
  switch (s.r) {
    case 8: return launch_predict_r<8>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    case 16: return launch_predict_r<16>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    case 24: return launch_predict_r<24>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    case 32: return launch_predict_r<32>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    case 40: return launch_predict_r<40>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    case 48: return launch_predict_r<48>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    case 56: return launch_predict_r<56>(Q, K, Wq, Wk, s, qp, kp, scores, st);
    default: return launch_predict_r<64>(Q, K, Wq, Wk, s, qp, kp, scores, st);
  }
}

}  // namespace dsv
