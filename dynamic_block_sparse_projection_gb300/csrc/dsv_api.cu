// dsv_api.cu — the C ABI of libdsv: argument checks, TMA descriptors, dispatch.
//
// Every entry point validates its arguments on the host before any launch
// (returning DSV_ERR_INVALID_ARG / DSV_ERR_UNSUPPORTED and writing nothing),
// then enqueues its kernels on the caller's stream without synchronising
// (dsv_predict_topk_blocks also forks part of its work onto a library-owned
// side stream and joins it back with events).
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "dsv_launch.h"

namespace dsv {

// One error word per device: the first device-side error since the last clear.
static __device__ DeviceErr g_err_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 1000000000ULL;

std::mutex g_mu;
DeviceErr* g_err_addr[kMaxDevices] = {};
unsigned long long g_limit_ns[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

dsv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DSV_OK : DSV_ERR_CUDA; }

// A second stream (and two events) per device for the fused predictor +
// top-k: the transposed lists of the heads whose rows are all selected are
// built there while the select kernel's last, partly filled wave runs on the
// caller's stream.  g_fork_mu keeps one call's record / wait / launch
// sequence on these objects from interleaving with another's.
struct ForkRes {
  cudaStream_t side = nullptr;
  cudaEvent_t main_done = nullptr, side_done = nullptr;
  int nsm = 0;
};
ForkRes g_fork[kMaxDevices];
std::mutex g_fork_mu;

cudaError_t fork_res(ForkRes** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  ForkRes& f = g_fork[dev];
  if (f.side == nullptr) {
    ForkRes n;
    if ((e = cudaDeviceGetAttribute(&n.nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&n.side, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&n.main_done, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&n.side_done, cudaEventDisableTiming)) != cudaSuccess) return e;
    f = n;
  }
  *out = &f;
  return cudaSuccess;
}

// Control block of the current device (error word address, wait limit).
cudaError_t current_ctl(Ctl* ctl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_err_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_err_word);
    if (e != cudaSuccess) return e;
    g_err_addr[dev] = static_cast<DeviceErr*>(p);
  }
  ctl->err = g_err_addr[dev];
  ctl->wait_limit_ns = g_limit_ns[dev] ? g_limit_ns[dev] : kDefaultWaitNs;
  return cudaSuccess;
}

cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return cudaSuccess;
}

// 2D map over a [rows, d] bf16 tensor, box = [box_rows, 64 columns], 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, const void* base, long long rows, int d, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encode(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2D map over a [rows, 32] fp32 array, box = [32 columns, box_rows], 128-byte swizzle
// (the tf32 operand tiles of the fused predictor + top-k).
cudaError_t make_map_f32x32(CUtensorMap* map, const void* base, long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encode(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {32u, (cuuint64_t)rows};
  cuuint64_t strides[1] = {32u * 4u};
  cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// Common shape rules.  Returns DSV_OK, or the status to return.
dsv_status check_shape(const dsv_shape& s, bool need_r) {
  if (s.B < 0 || s.H < 0 || s.N < 0) return DSV_ERR_INVALID_ARG;
  if (s.block != 64 && s.block != 128) return DSV_ERR_UNSUPPORTED;
  if (s.d != 64 && s.d != 128) return DSV_ERR_UNSUPPORTED;
  if (s.N % s.block != 0) return DSV_ERR_INVALID_ARG;
  if (need_r && (s.r < 8 || s.r > 64 || s.r % 8 != 0)) return DSV_ERR_UNSUPPORTED;
  if (s.H > kMaxHeads) return DSV_ERR_UNSUPPORTED;
  if ((long long)s.B * s.H > 65535) return DSV_ERR_UNSUPPORTED;
  if ((long long)s.B * s.H * s.N >= (1LL << 31)) return DSV_ERR_UNSUPPORTED;
  return DSV_OK;
}

bool empty(const dsv_shape& s) { return (long long)s.B * s.H * s.N == 0; }

float resolve_scale(const dsv_shape& s, float scale) {
  return (scale > 0.f && isfinite(scale)) ? scale : 1.0f / sqrtf((float)s.d);
}

// One thread waits on a barrier that nothing arrives at: phase 0 of a freshly
// initialised barrier never completes, so the bounded wait runs out, records
// DSV_ERR_TIMEOUT and returns.  Nothing else is in flight in this CTA.
__global__ void selftest_wait_kernel(Ctl ctl) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait(&bar, 0, &abort_flag, ctl, DSV_SELFTEST_WAIT_ID);
}

}  // namespace
}  // namespace dsv

using namespace dsv;

extern "C" {

int32_t dsv_version(void) { return 10000; }


const char* dsv_status_string(dsv_status st) {
  switch (st) {
    case DSV_OK: return "ok";
    case DSV_ERR_INVALID_ARG: return "invalid argument";
    case DSV_ERR_UNSUPPORTED: return "unsupported size";
    case DSV_ERR_CUDA: return "CUDA error";
    case DSV_ERR_BAD_INDEX: return "out-of-range block index in a CSR list";
    case DSV_ERR_TIMEOUT: return "a kernel wait ran past its time limit";
    case DSV_ERR_INTERNAL: return "a kernel consistency check failed";
  }
  return "unknown status";
}

dsv_status dsv_set_wait_limit_ns(uint64_t limit_ns) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  g_limit_ns[dev] = limit_ns;
  return DSV_OK;
}

dsv_status dsv_get_device_error(dsv_stream_t stream, uint32_t* info) {
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DSV_ERR_CUDA;
  DeviceErr h{};
  if (cudaMemcpy(&h, ctl.err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return DSV_ERR_CUDA;
  if (info) *info = h.info;
  return static_cast<dsv_status>(h.code);
}

dsv_status dsv_selftest_wait_timeout(dsv_stream_t stream) {
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  selftest_wait_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ctl);
  return from_cuda(cudaGetLastError());
}

dsv_status dsv_clear_device_error(dsv_stream_t stream) {
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  return from_cuda(cudaMemsetAsync(ctl.err, 0, sizeof(DeviceErr), reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsv_predict_workspace_bytes(dsv_shape s) {
  if (check_shape(s, true) != DSV_OK || empty(s)) return 0;
  return predict_ws_bytes(s);
}

dsv_status dsv_predict_scores(const void* Q, const void* K, const float* Wq, const float* Wk, dsv_shape s,
                              float* scores, void* workspace, size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, true);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!Q || !K || !Wq || !Wk || !scores || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(Wq) || !al16(Wk) || !al16(scores) || !al256(workspace))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < predict_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  return from_cuda(launch_predict(Q, K, Wq, Wk, s, scores, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsv_predict_max_workspace_bytes(dsv_shape s) {
  if (check_shape(s, true) != DSV_OK || empty(s)) return 0;
  return predict_max_ws_bytes(s);
}

dsv_status dsv_predict_scores_max(const void* Q, const void* K, const float* Wq, const float* Wk, dsv_shape s,
                                  float* scores, void* workspace, size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, true);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!Q || !K || !Wq || !Wk || !scores || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(Wq) || !al16(Wk) || !al16(scores) || !al256(workspace))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < predict_max_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  return from_cuda(
      launch_predict_max(Q, K, Wq, Wk, s, scores, workspace, ctl, reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsv_topk_workspace_bytes(dsv_shape s) {
  if (check_shape(s, false) != DSV_OK || empty(s)) return 0;
  return topk_ws_bytes(s);
}

dsv_status dsv_topk_blocks(const float* scores, dsv_shape s, const int32_t* k_per_head, int32_t* fwd_ptr,
                           int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col, void* workspace,
                           size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!fwd_ptr || !bwd_ptr) return DSV_ERR_INVALID_ARG;
  if (empty(s)) {
    cudaError_t e = cudaMemsetAsync(fwd_ptr, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(bwd_ptr, 0, sizeof(int32_t), st);
    return from_cuda(e);
  }
  const int nb = s.N / s.block;
  if (nb > kMaxBlocksPerRow) return DSV_ERR_UNSUPPORTED;
  if (!scores || !k_per_head || !fwd_col || !bwd_col || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(scores) || !al16(fwd_ptr) || !al16(fwd_col) || !al16(bwd_ptr) || !al16(bwd_col) || !al256(workspace))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < topk_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  HeadK hk;
  hk.kpre[0] = 0;
  for (int h = 0; h < s.H; ++h) {
    const int k = k_per_head[h];
    if (k < 1 || k > nb) return DSV_ERR_INVALID_ARG;
    hk.k[h] = k;
    hk.kpre[h + 1] = hk.kpre[h] + k;
  }
  for (int h = s.H; h < kMaxHeads; ++h) {
    hk.k[h] = 0;
    hk.kpre[h + 1] = hk.kpre[h];
  }
  const long long nnz = (long long)s.B * nb * hk.kpre[s.H];
  if (nnz > INT32_MAX) return DSV_ERR_UNSUPPORTED;
  return from_cuda(launch_topk(scores, s, hk, nnz, fwd_ptr, fwd_col, bwd_ptr, bwd_col, workspace, st));
}

size_t dsv_predict_topk_workspace_bytes(dsv_shape s) {
  if (check_shape(s, true) != DSV_OK || empty(s) || s.r > 32) return 0;
  return predict_ws_bytes(s) + split_tf32_bytes(s) + topk_ws_bytes(s);
}

dsv_status dsv_predict_topk_blocks(const void* Q, const void* K, const float* Wq, const float* Wk, dsv_shape s,
                                   const int32_t* k_per_head, int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr,
                                   int32_t* bwd_col, float* scores, void* workspace, size_t workspace_bytes,
                                   dsv_stream_t stream) {
  dsv_status v = check_shape(s, true);
  if (v != DSV_OK) return v;
  if (s.r > 32) return DSV_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!fwd_ptr || !bwd_ptr) return DSV_ERR_INVALID_ARG;
  if (empty(s)) {
    cudaError_t e = cudaMemsetAsync(fwd_ptr, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(bwd_ptr, 0, sizeof(int32_t), st);
    return from_cuda(e);
  }
  const int nb = s.N / s.block;
  if (nb > kPredictTopkMaxBlocks) return DSV_ERR_UNSUPPORTED;
  if (!Q || !K || !Wq || !Wk || !k_per_head || !fwd_col || !bwd_col || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(Wq) || !al16(Wk) || !al16(fwd_ptr) || !al16(fwd_col) || !al16(bwd_ptr) ||
      !al16(bwd_col) || !al256(workspace) || (scores && !al16(scores)))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < predict_ws_bytes(s) + split_tf32_bytes(s) + topk_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  HeadK hk;
  hk.kpre[0] = 0;
  for (int h = 0; h < s.H; ++h) {
    const int k = k_per_head[h];
    if (k < 1 || k > nb) return DSV_ERR_INVALID_ARG;
    hk.k[h] = k;
    hk.kpre[h + 1] = hk.kpre[h] + k;
  }
  for (int h = s.H; h < kMaxHeads; ++h) {
    hk.k[h] = 0;
    hk.kpre[h + 1] = hk.kpre[h];
  }
  const long long nnz = (long long)s.B * nb * hk.kpre[s.H];
  if (nnz > INT32_MAX) return DSV_ERR_UNSUPPORTED;
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  // workspace: pooled vectors | tf32 parts | top-k bitmask and transpose counts
  char* w = static_cast<char*>(workspace);
  const size_t rows = (size_t)s.B * s.H * nb;
  float* qp = reinterpret_cast<float*>(w);
  float* kp = reinterpret_cast<float*>(w + align256(rows * (size_t)s.r * sizeof(float)));
  float* split = reinterpret_cast<float*>(w + predict_ws_bytes(s));
  void* tws = w + predict_ws_bytes(s) + split_tf32_bytes(s);
  const size_t part = align256(rows * 32 * sizeof(float));
  PredictTopkMaps maps;
  const char* sp = reinterpret_cast<const char*>(split);
  if (make_map_f32x32(&maps.qh, sp, (long long)rows, 128) != cudaSuccess ||
      make_map_f32x32(&maps.ql, sp + part, (long long)rows, 128) != cudaSuccess ||
      make_map_f32x32(&maps.kh, sp + 2 * part, (long long)rows, 128) != cudaSuccess ||
      make_map_f32x32(&maps.kl, sp + 3 * part, (long long)rows, 128) != cudaSuccess)
    return DSV_ERR_CUDA;
  ForkRes* fr = nullptr;
  cudaError_t e = fork_res(&fr);
  if (e == cudaSuccess) e = launch_pool_project(Q, K, Wq, Wk, s, qp, kp, st, split, split_part_floats(s));
  if (e == cudaSuccess) e = launch_key_stats(kp, s, split, st);
  if (e != cudaSuccess) return from_cuda(e);
  uint32_t* mask = static_cast<uint32_t*>(tws);
  // The select kernel runs one CTA per SM; the items of a last, partly filled
  // wave go into a launch of their own, and the transposes of the heads done
  // before it run beside it on the side stream.
  const long long tiles = select_tiles(s), bhs = (long long)s.B * s.H, items = bhs * tiles;
  const long long tail = items % fr->nsm, n1 = items - tail, heads1 = n1 / tiles;
  if (tail == 0 || items < 2LL * fr->nsm || heads1 == 0) {
    e = launch_score_select(maps, s, hk, nnz, fwd_ptr, fwd_col, mask, scores, split, ctl, st);
    if (e == cudaSuccess) e = launch_topk_transpose(s, hk, nnz, bwd_ptr, bwd_col, tws, st);
    return from_cuda(e);
  }
  std::lock_guard<std::mutex> lock(g_fork_mu);
  e = launch_score_select(maps, s, hk, nnz, fwd_ptr, fwd_col, mask, scores, split, ctl, st, 0, n1);
  if (e == cudaSuccess) e = cudaEventRecord(fr->main_done, st);
  if (e == cudaSuccess) e = launch_score_select(maps, s, hk, nnz, fwd_ptr, fwd_col, mask, scores, split, ctl, st, n1, items);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(fr->side, fr->main_done, 0);
  if (e == cudaSuccess) e = launch_topk_transpose(s, hk, nnz, bwd_ptr, bwd_col, tws, fr->side, 0, heads1);
  if (e == cudaSuccess) e = cudaEventRecord(fr->side_done, fr->side);
  if (e == cudaSuccess) e = launch_topk_transpose(s, hk, nnz, bwd_ptr, bwd_col, tws, st, heads1, -1);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, fr->side_done, 0);
  return from_cuda(e);
}

dsv_status dsv_dispatch_heads(const int32_t* k_per_head, int32_t H, int32_t nb, const float* rho,
                              const float* ratio, int32_t n, int32_t* k_out, int32_t* dense_out) {
  if (!k_per_head || !rho || !ratio || !k_out || !dense_out || H < 1 || nb < 1 || n < 1) return DSV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    if (!(rho[i] > 0.f && rho[i] <= 1.f) || !(ratio[i] > 0.f) || !isfinite(ratio[i])) return DSV_ERR_INVALID_ARG;
    if (i > 0 && !(rho[i] > rho[i - 1])) return DSV_ERR_INVALID_ARG;
  }
  for (int32_t h = 0; h < H; ++h)
    if (k_per_head[h] < 1 || k_per_head[h] > nb) return DSV_ERR_INVALID_ARG;
  for (int32_t h = 0; h < H; ++h) {
    const double x = (double)k_per_head[h] / (double)nb;
    double y;
    if (x <= rho[0]) {
      y = ratio[0];
    } else if (x >= rho[n - 1]) {
      y = ratio[n - 1];
    } else {
      int32_t i = 1;
      while (rho[i] < x) ++i;                     // rho[i-1] < x <= rho[i]
      const double t = (x - rho[i - 1]) / ((double)rho[i] - rho[i - 1]);
      y = ratio[i - 1] + t * ((double)ratio[i] - ratio[i - 1]);
    }
    const int dense = y >= 1.0 ? 1 : 0;
    dense_out[h] = dense;
    k_out[h] = dense ? nb : k_per_head[h];
  }
  return DSV_OK;
}

size_t dsv_topk_mass_workspace_bytes(dsv_shape s) {
  if (check_shape(s, false) != DSV_OK || empty(s)) return 0;
  return topk_mass_ws_bytes(s);
}

dsv_status dsv_topk_mass_blocks(const float* scores, dsv_shape s, float tau, float temperature, int32_t kmin,
                                int32_t kmax, int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col,
                                size_t col_capacity, void* workspace, size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!fwd_ptr || !bwd_ptr) return DSV_ERR_INVALID_ARG;
  if (!(tau > 0.f && tau <= 1.f) || !(temperature > 0.f) || !isfinite(temperature)) return DSV_ERR_INVALID_ARG;
  if (empty(s)) {
    cudaError_t e = cudaMemsetAsync(fwd_ptr, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(bwd_ptr, 0, sizeof(int32_t), st);
    return from_cuda(e);
  }
  const int nb = s.N / s.block;
  if (nb > kMaxBlocksPerRow) return DSV_ERR_UNSUPPORTED;
  if (kmin < 1 || kmin > kmax || kmax > nb) return DSV_ERR_INVALID_ARG;
  if (!scores || !fwd_col || !bwd_col || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(scores) || !al16(fwd_ptr) || !al16(fwd_col) || !al16(bwd_ptr) || !al16(bwd_col) || !al256(workspace))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < topk_mass_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  const long long cap = (long long)s.B * s.H * nb * kmax;   // every row at most kmax entries
  if (cap > INT32_MAX) return DSV_ERR_UNSUPPORTED;
  if ((long long)col_capacity < cap) return DSV_ERR_INVALID_ARG;
  return from_cuda(
      launch_topk_mass(scores, s, tau, temperature, kmin, kmax, fwd_ptr, fwd_col, bwd_ptr, bwd_col, workspace, st));
}

dsv_status dsv_sparse_attn_fwd(const void* Q, const void* K, const void* V, dsv_shape s, const int32_t* fwd_ptr,
                               const int32_t* fwd_col, float softmax_scale, void* O, float* lse,
                               dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!Q || !K || !V || !fwd_ptr || !fwd_col || !O || !lse) return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(V) || !al16(O) || !al16(lse)) return DSV_ERR_INVALID_ARG;
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  const long long rows = (long long)s.B * s.H * s.N;
  CUtensorMap tq, tk, tv;
  if (make_map(&tq, Q, rows, s.d, s.block) != cudaSuccess || make_map(&tk, K, rows, s.d, s.block) != cudaSuccess ||
      make_map(&tv, V, rows, s.d, s.block) != cudaSuccess)
    return DSV_ERR_CUDA;
  return from_cuda(launch_attn_fwd(tq, tk, tv, s, fwd_ptr, fwd_col, resolve_scale(s, softmax_scale), O, lse, ctl,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsv_attn_bwd_workspace_bytes(dsv_shape s) {
  if (check_shape(s, false) != DSV_OK || empty(s)) return 0;
  return attn_bwd_ws_bytes(s);
}

dsv_status dsv_sparse_attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                               const float* lse, dsv_shape s, const int32_t* fwd_ptr, const int32_t* fwd_col,
                               const int32_t* bwd_ptr, const int32_t* bwd_col, float softmax_scale, void* dQ,
                               void* dK, void* dV, void* workspace, size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!Q || !K || !V || !O || !dO || !lse || !fwd_ptr || !fwd_col || !bwd_ptr || !bwd_col || !dQ || !dK || !dV ||
      !workspace)
    return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(V) || !al16(O) || !al16(dO) || !al16(lse) || !al16(dQ) || !al16(dK) ||
      !al16(dV) || !al256(workspace))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  const long long rows = (long long)s.B * s.H * s.N;
  CUtensorMap tq, tk, tv, tdo;
  if (make_map(&tq, Q, rows, s.d, s.block) != cudaSuccess || make_map(&tk, K, rows, s.d, s.block) != cudaSuccess ||
      make_map(&tv, V, rows, s.d, s.block) != cudaSuccess || make_map(&tdo, dO, rows, s.d, s.block) != cudaSuccess)
    return DSV_ERR_CUDA;
  return from_cuda(launch_attn_bwd(Q, tq, tk, tv, tdo, O, dO, lse, s, fwd_ptr, fwd_col, bwd_ptr, bwd_col,
                                   resolve_scale(s, softmax_scale), dQ, dK, dV, workspace, ctl,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

dsv_status dsv_cube_permute(const void* src, void* dst, dsv_shape s, int T, int Hl, int Wl, int ct, int cy, int cx,
                            int inverse, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  if (T <= 0 || Hl <= 0 || Wl <= 0 || ct <= 0 || cy <= 0 || cx <= 0) return DSV_ERR_INVALID_ARG;
  if ((long long)T * Hl * Wl != s.N || ct * cy * cx != s.block) return DSV_ERR_INVALID_ARG;
  if (T % ct != 0 || Hl % cy != 0 || Wl % cx != 0) return DSV_ERR_INVALID_ARG;
  if (inverse != 0 && inverse != 1) return DSV_ERR_INVALID_ARG;
  if (empty(s)) return DSV_OK;
  if (!src || !dst || !al16(src) || !al16(dst)) return DSV_ERR_INVALID_ARG;
  const size_t bytes = (size_t)s.B * s.H * s.N * s.d * 2;
  const char* a = static_cast<const char*>(src);
  const char* b = static_cast<const char*>(dst);
  if (a < b + bytes && b < a + bytes) return DSV_ERR_INVALID_ARG;   // overlapping buffers
  return from_cuda(launch_cube_permute(src, dst, s, T, Hl, Wl, ct, cy, cx, inverse,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

dsv_status dsv_attn_bwd_preprocess(const void* O, const void* dO, const float* lse, dsv_shape s, void* workspace,
                                   size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!O || !dO || !lse || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(O) || !al16(dO) || !al16(lse) || !al256(workspace)) return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  return from_cuda(launch_attn_bwd_pre(O, dO, lse, s, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

dsv_status dsv_attn_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO, dsv_shape s,
                             const int32_t* bwd_ptr, const int32_t* bwd_col, float softmax_scale, void* dK, void* dV,
                             void* workspace, size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!Q || !K || !V || !dO || !bwd_ptr || !bwd_col || !dK || !dV || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(V) || !al16(dO) || !al16(dK) || !al16(dV) || !al256(workspace))
    return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  const long long rows = (long long)s.B * s.H * s.N;
  CUtensorMap tq, tk, tv, tdo;
  if (make_map(&tq, Q, rows, s.d, s.block) != cudaSuccess || make_map(&tk, K, rows, s.d, s.block) != cudaSuccess ||
      make_map(&tv, V, rows, s.d, s.block) != cudaSuccess || make_map(&tdo, dO, rows, s.d, s.block) != cudaSuccess)
    return DSV_ERR_CUDA;
  return from_cuda(launch_attn_bwd_kv(tq, tk, tv, tdo, s, bwd_ptr, bwd_col, resolve_scale(s, softmax_scale), dK, dV,
                                      workspace, ctl, reinterpret_cast<cudaStream_t>(stream)));
}

dsv_status dsv_attn_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, dsv_shape s,
                           const int32_t* fwd_ptr, const int32_t* fwd_col, float softmax_scale, void* dQ,
                           const void* workspace, size_t workspace_bytes, dsv_stream_t stream) {
  dsv_status v = check_shape(s, false);
  if (v != DSV_OK) return v;
  if (empty(s)) return DSV_OK;
  if (!Q || !K || !V || !dO || !fwd_ptr || !fwd_col || !dQ || !workspace) return DSV_ERR_INVALID_ARG;
  if (!al16(Q) || !al16(K) || !al16(V) || !al16(dO) || !al16(dQ) || !al256(workspace)) return DSV_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_ws_bytes(s)) return DSV_ERR_INVALID_ARG;
  Ctl ctl;
  if (current_ctl(&ctl) != cudaSuccess) return DSV_ERR_CUDA;
  const long long rows = (long long)s.B * s.H * s.N;
  CUtensorMap tq, tk, tv, tdo;
  if (make_map(&tq, Q, rows, s.d, s.block) != cudaSuccess || make_map(&tk, K, rows, s.d, s.block) != cudaSuccess ||
      make_map(&tv, V, rows, s.d, s.block) != cudaSuccess || make_map(&tdo, dO, rows, s.d, s.block) != cudaSuccess)
    return DSV_ERR_CUDA;
  return from_cuda(launch_attn_bwd_q(tq, tk, tv, tdo, s, fwd_ptr, fwd_col, resolve_scale(s, softmax_scale), dQ,
                                     workspace, ctl, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
