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
constexpr int kPredictTopkMaxBlocks = 4096;   // key blocks per row of the fused predictor + top-k

// Per-head top-k sizes and their prefix sums (kernel parameter by value).
struct HeadK {
  int32_t k[kMaxHeads];
  int32_t kpre[kMaxHeads + 1];  // kpre[h] = k[0] + ... + k[h-1]
};

// Predictor: pooled low-rank vectors into `ws`, then the score tile kernel.
cudaError_t launch_predict(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                           float* scores, void* ws, cudaStream_t st);
size_t predict_ws_bytes(const dsv_shape& s);
// Max-pooled predictor: per-token rank-r projections, split into bf16 parts in
// the MMA layout, into `ws`; then the tile-maximum kernel (tcgen05).
cudaError_t launch_predict_max(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                               float* scores, void* ws, const Ctl& ctl, cudaStream_t st);
size_t predict_max_ws_bytes(const dsv_shape& s);

// Top-k, transposed lists.
cudaError_t launch_topk(const float* scores, const dsv_shape& s, const HeadK& hk, int64_t nnz, int32_t* fwd_ptr,
                        int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col, void* ws, cudaStream_t st);
size_t topk_ws_bytes(const dsv_shape& s);
// The transposed lists only, from a selection bitmask already in `ws` (the
// layout launch_topk's select kernel writes: word (b, h, w, g) at
// ((b*H + h) * words + w) * G + g).
// Heads (slices b*H + h) bh0 .. bh1 - 1 only (bh1 < 0: to the last).
cudaError_t launch_topk_transpose(const dsv_shape& s, const HeadK& hk, int64_t nnz, int32_t* bwd_ptr,
                                  int32_t* bwd_col, void* ws, cudaStream_t st, long long bh0 = 0,
                                  long long bh1 = -1);
// Pooled rank-r projections only (qp, kp: [B*H*G, r] fp32), the first kernel of launch_predict.
// split != null (r <= 32): also the tf32 hi / lo parts of every projected
// vector, zero-padded to 32 columns: four [B*H*G, 32] fp32 arrays (q hi, q lo,
// k hi, k lo), `part` floats apart.
cudaError_t launch_pool_project(const void* Q, const void* K, const float* Wq, const float* Wk, const dsv_shape& s,
                                float* qp, float* kp, cudaStream_t st, float* split = nullptr, long long part = 0);
// Fused predictor + top-k: the tf32 operand splits of the pooled vectors
// (written by launch_pool_project), the per-head key statistics, then one
// kernel that scores every (group, key block) pair on the tensor cores and
// selects each group's top k without writing the score matrix (unless
// `scores` is given); the forward lists and the selection bitmask (in the
// top-k workspace layout) come out of it.  `split` holds 4 arrays of
// [B*H*G, 32] fp32 (q hi, q lo, k hi, k lo), then the per-head key statistics
// (partial sums, then mean and covariance), each part 256-byte aligned.
struct PredictTopkMaps {
  CUtensorMap qh, ql, kh, kl;
};
long long split_part_floats(const dsv_shape& s);
// Score/select items: (b*H + h) * select_tiles(s) + tile, tile = 128 groups; a
// launch covers items item0 .. item1 - 1 (item1 < 0: to the last).
long long select_tiles(const dsv_shape& s);
cudaError_t launch_key_stats(const float* kp, const dsv_shape& s, float* split, cudaStream_t st);
cudaError_t launch_score_select(const PredictTopkMaps& maps, const dsv_shape& s, const HeadK& hk, int64_t nnz,
                                int32_t* fwd_ptr, int32_t* fwd_col, uint32_t* mask, float* scores, const float* split,
                                const Ctl& ctl, cudaStream_t st, long long item0 = 0,
                                long long item1 = -1);
size_t split_tf32_bytes(const dsv_shape& s);
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
