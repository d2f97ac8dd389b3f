// dsv_launch.h — host-side launchers shared between the C ABI and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsv.h"
#include "dsv_device.cuh"

namespace dsv {

constexpr int kMaxHeads = 1024;
constexpr int kMaxBlocksPerRow = 8192;

// Per-head top-k sizes and their prefix sums (kernel parameter by value).
struct HeadK {
  int32_t k[kMaxHeads];
  int32_t kpre[kMaxHeads + 1];  // kpre[h] = k[0] + ... + k[h-1]
};

// Predictor: pooled low-rank vectors into `ws`, then the score tile kernel.
cudaError_t launch_predict(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                           float* scores, void* ws, cudaStream_t st);
size_t predict_ws_bytes(const dsv_shape& s);
// Max-pooled predictor: per-token rank-r projections into `ws`, then the tile-maximum kernel.
cudaError_t launch_predict_max(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                               float* scores, void* ws, cudaStream_t st);
size_t predict_max_ws_bytes(const dsv_shape& s);

// Top-k, transposed lists.
cudaError_t launch_topk(const float* scores, const dsv_shape& s, const HeadK& hk, int64_t nnz, int32_t* fwd_ptr,
                        int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col, void* ws, cudaStream_t st);
size_t topk_ws_bytes(const dsv_shape& s);
// Mass-threshold selection: per row the smallest top set carrying >= tau of
// the predicted softmax mass (temperature * scores), clamped to [kmin, kmax].
cudaError_t launch_topk_mass(const float* scores, const dsv_shape& s, float tau, float temperature, int kmin,
                             int kmax, int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col,
                             void* ws, cudaStream_t st);
size_t topk_mass_ws_bytes(const dsv_shape& s);

// Attention forward.  Tensor maps cover [B*H*N, d] bf16 with a 64-column box.
cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col, float scale,
                            void* O, float* lse, const Ctl& ctl, cudaStream_t st);

// Attention backward.
cudaError_t launch_attn_bwd(const void* Q, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmdO, const void* O, const void* dO, const float* lse,
                            const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col,
                            const int32_t* bwd_ptr, const int32_t* bwd_col, float scale, void* dQ, void* dK,
                            void* dV, void* ws, const Ctl& ctl, cudaStream_t st);
// The stages of launch_attn_bwd (preprocess; dK/dV; dQ).
cudaError_t launch_attn_bwd_pre(const void* O, const void* dO, const float* lse, const dsv_shape& s, void* ws,
                                cudaStream_t st);
cudaError_t launch_attn_bwd_kv(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const CUtensorMap& tmdO, const dsv_shape& s, const int32_t* bwd_ptr,
                               const int32_t* bwd_col, float scale, void* dK, void* dV, void* ws,
                               const Ctl& ctl, cudaStream_t st);
cudaError_t launch_attn_bwd_q(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmdO,
                              const dsv_shape& s, const int32_t* fwd_ptr, const int32_t* fwd_col, float scale,
                              void* dQ, const void* ws, const Ctl& ctl, cudaStream_t st);
size_t attn_bwd_ws_bytes(const dsv_shape& s);

// 3D cube query grouping: token rows moved between raster and cube order.
cudaError_t launch_cube_permute(const void* src, void* dst, const dsv_shape& s, int T, int Hl, int Wl, int ct, int cy,
                                int cx, int inverse, cudaStream_t st);

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace dsv
