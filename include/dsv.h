/*
 * dsv.h — C ABI of the DSV dynamic sparse 3D attention hot path on GB300 (sm_103a).
 *
 * Source pages (cited by title and section):
 *   [nl] "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
 *        Training", gist.science/nl/paper/2502.07590, "Technische samenvatting".
 *   [hi] the same title, gist.science/hi/paper/2502.07590, technical summary.
 *
 * The path: a low-rank predictor scores (query group, key block) pairs
 * ([nl] 2A, 2B), a per-group top-k picks the critical key blocks ([nl] 2B,
 * [hi] 2A "critical KV"), and block-sparse softmax attention runs forward and
 * backward over only those blocks ([nl] 2A stage 2, [hi] 2A/2B).
 *
 * Conventions shared by every call
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16, shape [B, H, N, d],
 *     contiguous (d fastest).  Token n of a video latent t x Hl x Wl is in
 *     raster order n = (t*Hl + y)*Wl + x.
 *   - A group (queries) and a key block are `block` consecutive tokens:
 *     G = nb = N / block per (b, h).
 *   - All pointers except `k_per_head` are DEVICE pointers owned by the
 *     caller.  The library allocates no device memory; scratch space is
 *     passed in as `workspace` (size from the *_workspace_bytes query).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream) and never synchronises the host.
 *   - Argument errors are detected on the host before any launch and
 *     returned as DSV_ERR_INVALID_ARG / DSV_ERR_UNSUPPORTED; nothing is
 *     written then.  A failed launch returns DSV_ERR_CUDA.  Errors found by
 *     the kernels themselves (an out-of-range index in a caller's list, a
 *     wait that ran out of time) are recorded in a per-device error word read
 *     by dsv_get_device_error().
 *   - Empty problems (B*H*N == 0) are valid: only the CSR row-pointer heads
 *     are written.
 *   - Outputs are fully overwritten and bit-identical from run to run (no
 *     atomics on any output).
 */
#ifndef DSV_H_
#define DSV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t. */
typedef struct CUstream_st* dsv_stream_t;

typedef enum {
  DSV_OK = 0,
  DSV_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, k out of range */
  DSV_ERR_UNSUPPORTED = 2,  /* a size the library has no kernel for */
  DSV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  DSV_ERR_BAD_INDEX = 4,    /* a kernel met an out-of-range CSR entry */
  DSV_ERR_TIMEOUT = 5,      /* a kernel wait ran past its time limit */
  DSV_ERR_INTERNAL = 6      /* a kernel's own consistency check failed */
} dsv_status;

/* Problem shape.  Supported: d in {64, 128}; block in {64, 128};
 * r a multiple of 8 in [8, 64]; N a multiple of block; H <= 1024;
 * B*H <= 65535; B*H*N < 2^31; N / block <= 8192 for the top-k. */
typedef struct {
  int32_t B, H, N, d, block, r;
} dsv_shape;

/* ------------------------------------------------------------------------
 * dsv_predict_scores — low-rank block-score predictor
 * ([nl] 2A low-rank predictors W^Q_lr, W^K_lr; 2B query grouping / proxy query)
 *
 *   qbar[b,h,g] = mean over the `block` tokens i of group g of Q[b,h,i] W^Q[h]
 *   kbar[b,h,j] = mean over the tokens of key block j of K[b,h,i] W^K[h]
 *   scores[b,h,g,j] = qbar[b,h,g] . kbar[b,h,j]        (fp32, no scale)
 *
 * Q, K      bf16 [B,H,N,d], 16-byte aligned.
 * Wq, Wk    fp32 [H,d,r] (row-major: r fastest), 16-byte aligned.
 * scores    fp32 [B,H,G,nb] row-major, 16-byte aligned; overwritten.
 * workspace >= dsv_predict_workspace_bytes(s) bytes, 256-byte aligned
 *           (holds the pooled rank-r vectors).
 * ------------------------------------------------------------------------ */
size_t dsv_predict_workspace_bytes(dsv_shape s);
dsv_status dsv_predict_scores(const void* Q, const void* K, const float* Wq, const float* Wk,
                              dsv_shape s, float* scores, void* workspace, size_t workspace_bytes,
                              dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_predict_scores_max — max-pooled block scores of the same predictor
 * ([nl] 2A low-rank logits approximating Q K^T; 2B one proxy per group).
 * The pages do not fix how a (group, key block) tile of low-rank logits
 * becomes one score; dsv_predict_scores takes the tile mean, this call the
 * tile maximum:
 *
 *   scores[b,h,g,j] = max over tokens i of group g and l of key block j of
 *                     (Q[b,h,i] W^Q[h]) . (K[b,h,l] W^K[h])     (fp32, no scale)
 *
 * Every token is projected and every tile formed: an [N, N] x r contraction
 * per (b, h), on the tensor cores.  Each fp32 projection is split into two
 * bf16 parts (v = hi + lo to 2^-18 relative) and a logit is taken as
 * hi.hi + hi.lo + lo.hi, one bf16 contraction of length 3r with fp32
 * accumulation (~1e-5 of the logit scale against the fp32 value).  A NaN
 * logit is dropped by the maximum.
 * Arguments and layout as dsv_predict_scores, except:
 * workspace >= dsv_predict_max_workspace_bytes(s) bytes, 256-byte aligned
 *           (holds every token's split rank-r row of Q and of K in the MMA
 *           layout: 2 * B*H*ceil(N/128)*128 rows of round_up(3r, 16) bf16).
 * Waits inside the kernel are bounded like the attention kernels'
 * (dsv_set_wait_limit_ns); one that runs out is reported as DSV_ERR_TIMEOUT
 * through dsv_get_device_error.
 * The scores feed dsv_topk_blocks or dsv_topk_mass_blocks unchanged.
 * ------------------------------------------------------------------------ */
size_t dsv_predict_max_workspace_bytes(dsv_shape s);
dsv_status dsv_predict_scores_max(const void* Q, const void* K, const float* Wq, const float* Wk,
                                  dsv_shape s, float* scores, void* workspace, size_t workspace_bytes,
                                  dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_topk_blocks — per-group top-k critical key blocks and their transpose
 * ([nl] 2B fused estimation & selection; [hi] 2B top-k selection)
 *
 * For every row (b,h,g): the k_per_head[h] block indices j with the largest
 * scores[b,h,g,j]; equal scores go to the lower j; -0.0 equals +0.0; NaN
 * ranks below every number.  Lists are written in ascending j.
 *
 * scores     fp32 [B,H,G,nb] (device), 16-byte aligned.
 * k_per_head HOST array [H], 1 <= k <= nb.
 * fwd_ptr    int32 [B*H*G + 1]: row (b*H + h)*G + g holds fwd_col[fwd_ptr[row] .. fwd_ptr[row+1]).
 * fwd_col    int32 [nnz], nnz = B*G*sum_h k_per_head[h]: block index j within (b,h).
 * bwd_ptr    int32 [B*H*nb + 1]: row (b*H + h)*nb + j lists the groups whose list holds j.
 * bwd_col    int32 [nnz]: group index g within (b,h), ascending.
 * workspace  >= dsv_topk_workspace_bytes(s) bytes, 256-byte aligned
 *            (a G x nb bitmask per (b,h) and per-block counts).
 * ------------------------------------------------------------------------ */
size_t dsv_topk_workspace_bytes(dsv_shape s);
dsv_status dsv_topk_blocks(const float* scores, dsv_shape s, const int32_t* k_per_head,
                           int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col,
                           void* workspace, size_t workspace_bytes, dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_topk_mass_blocks — mass-threshold selection of the critical key blocks
 * ([nl] 2A and [hi] 2A: the critical KV pairs carry about 90 % of the
 * attention score)
 *
 * For every row (b,h,g): p_j = softmax(temperature * scores[b,h,g,:])_j is
 * the predicted attention mass of block j; with the blocks in rank order
 * (larger score first, equal scores to the lower j) m is the smallest count
 * whose leading blocks carry mass >= tau, clamped to [kmin, kmax], and the row
 * keeps its top m blocks, listed in ascending j.  A row holding a non-finite
 * score gets m = kmax.  The masses are summed in fixed point (2^-40 units,
 * exact and independent of order, fp32 exponentials), so m can differ from an
 * exact-arithmetic count only where the leading mass passes tau within about
 * 1e-6.
 *
 * Arguments and outputs as dsv_topk_blocks, except that the rows have
 * variable lengths: nnz = fwd_ptr[B*H*G] = bwd_ptr[B*H*nb] (device).
 * fwd_col, bwd_col   int32 arrays of col_capacity >= B*H*G*kmax entries.
 * tau                in (0, 1]; temperature > 0, finite; 1 <= kmin <= kmax <= nb.
 * workspace          >= dsv_topk_mass_workspace_bytes(s) bytes, 256-byte aligned
 *                    (that of dsv_topk_blocks plus the row sizes).
 * DSV_ERR_UNSUPPORTED if B*H*G*kmax >= 2^31 (or as dsv_topk_blocks).
 * ------------------------------------------------------------------------ */
size_t dsv_topk_mass_workspace_bytes(dsv_shape s);
dsv_status dsv_topk_mass_blocks(const float* scores, dsv_shape s, float tau, float temperature,
                                int32_t kmin, int32_t kmax, int32_t* fwd_ptr, int32_t* fwd_col,
                                int32_t* bwd_ptr, int32_t* bwd_col, size_t col_capacity,
                                void* workspace, size_t workspace_bytes, dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_topk_blocks_noalloc — dsv_topk_blocks for callers that cannot allocate
 * (the DSV pages have no counterpart: this is a deployment convenience)
 *
 * Same arguments, lists and results as dsv_topk_blocks, minus the workspace.
 * For callers that must not call cudaMalloc or any allocating routine (for
 * example while another thread captures a CUDA graph, inside a plug-in whose
 * host framework owns the device heap, or in a loop where an allocation may
 * block): the scratch comes from a fixed device array inside libdsv of
 * DSV_TOPK_NOALLOC_SCRATCH_BYTES, held on every GPU that loads the library
 * until the process exits.  Problems whose dsv_topk_workspace_bytes() exceed
 * it return DSV_ERR_UNSUPPORTED before any launch.  The first call on a
 * device looks up the array's device address (make it before any stream
 * capture).  All calls share the array, so calls that overlap on the GPU race;
 * serialise them (one stream, or events).
 * ------------------------------------------------------------------------ */
#define DSV_TOPK_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
dsv_status dsv_topk_blocks_noalloc(const float* scores, dsv_shape s, const int32_t* k_per_head,
                                   int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr, int32_t* bwd_col,
                                   dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_sparse_attn_fwd — block-sparse softmax attention forward
 * ([nl] 2A stage 2: only the critical KV subset is computed; [hi] 2A)
 *
 * For query i in group g, over the keys of the blocks in g's list only:
 *   s_ij = scale * q_i . k_j,  O_i = sum_j softmax(s_i)_j v_j,
 *   lse_i = ln sum_j exp(s_ij)  (natural log).
 * A group with an empty list gets O_i = 0 and lse_i = -inf.
 *
 * Q, K, V   bf16 [B,H,N,d], 16-byte aligned.
 * fwd_ptr/fwd_col  the forward CSR (any valid lists, e.g. from dsv_topk_blocks).
 * softmax_scale    <= 0 selects 1/sqrt(d).
 * O         bf16 [B,H,N,d]; lse fp32 [B,H,N]; both overwritten.
 * ------------------------------------------------------------------------ */
dsv_status dsv_sparse_attn_fwd(const void* Q, const void* K, const void* V, dsv_shape s,
                               const int32_t* fwd_ptr, const int32_t* fwd_col, float softmax_scale,
                               void* O, float* lse, dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_sparse_attn_bwd — gradient of dsv_sparse_attn_fwd over the same blocks
 *
 *   D_i = sum_c dO_ic O_ic;  P_ij = exp(s_ij - lse_i);  dP_ij = dO_i . v_j;
 *   dS_ij = P_ij (dP_ij - D_i);  dV_j = sum_i P_ij dO_i;
 *   dQ_i = scale sum_j dS_ij k_j;  dK_j = scale sum_i dS_ij q_i.
 * Sums run over the selected (group, block) pairs only; key blocks that no
 * group selected get dK = dV = 0.  dQ uses the forward lists, dK/dV the
 * transposed lists; every output tile has exactly one writer (no atomics).
 *
 * Q, K, V, O, dO bf16 [B,H,N,d]; lse fp32 [B,H,N] from the forward.
 * dQ, dK, dV bf16 [B,H,N,d]; overwritten.
 * workspace >= dsv_attn_bwd_workspace_bytes(s) bytes, 256-byte aligned: D_i,
 * -lse_i*log2(e) and the dK/dV kernel's block order.
 * ------------------------------------------------------------------------ */
size_t dsv_attn_bwd_workspace_bytes(dsv_shape s);
dsv_status dsv_sparse_attn_bwd(const void* Q, const void* K, const void* V, const void* O,
                               const void* dO, const float* lse, dsv_shape s,
                               const int32_t* fwd_ptr, const int32_t* fwd_col,
                               const int32_t* bwd_ptr, const int32_t* bwd_col, float softmax_scale,
                               void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                               dsv_stream_t stream);

/* The three stages dsv_sparse_attn_bwd runs, one kernel each, for callers
 * that schedule or time them separately; in this order on one stream (or
 * with the ordering made explicit) they give results bitwise equal to the
 * single call, and dsv_attn_bwd_dkdv / dsv_attn_bwd_dq may run in either
 * order once the preprocess is done.  Arguments mean what they mean above.
 *   dsv_attn_bwd_preprocess  D_i and -lse_i * log2(e) into the workspace.
 *   dsv_attn_bwd_dkdv        dK, dV (one CTA per key block, transposed lists, the
 *                            blocks with the longest lists first; the order is
 *                            kept in the workspace's last part).
 *   dsv_attn_bwd_dq          dQ (persistent CTAs over the query groups, forward
 *                            lists).
 * Errors as for dsv_sparse_attn_bwd; a stage does not check that the
 * preprocess ran. */
dsv_status dsv_attn_bwd_preprocess(const void* O, const void* dO, const float* lse, dsv_shape s,
                                   void* workspace, size_t workspace_bytes, dsv_stream_t stream);
dsv_status dsv_attn_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO, dsv_shape s,
                             const int32_t* bwd_ptr, const int32_t* bwd_col, float softmax_scale,
                             void* dK, void* dV, void* workspace, size_t workspace_bytes,
                             dsv_stream_t stream);
dsv_status dsv_attn_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, dsv_shape s,
                           const int32_t* fwd_ptr, const int32_t* fwd_col, float softmax_scale,
                           void* dQ, const void* workspace, size_t workspace_bytes, dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_cube_permute — 3D cube query grouping as a token permutation
 * ([nl] 2B and [hi] 2B query grouping: adjacent tokens in 3D space share
 * critical KV, so queries are grouped in small cubes, e.g. 2x2x2)
 *
 * The hot path groups s.block consecutive tokens.  This call reorders the
 * tokens of every (b, h) so that each run of s.block consecutive tokens is
 * one ct x cy x cx cube of the T x Hl x Wl latent grid: the caller applies
 * it to Q, K, V, dO before the path and its inverse to O, dQ, dK, dV after.
 * Raster order n = (t*Hl + y)*Wl + x; cube order walks the cube grid
 * (T/ct, Hl/cy, Wl/cx) in raster order and the tokens inside a cube in
 * raster order (lt, ly, lx); perm(n_cube) = n_raster.
 *   inverse = 0:  dst[b,h,n] = src[b,h,perm(n)]   (raster -> cube order)
 *   inverse = 1:  dst[b,h,perm(n)] = src[b,h,n]   (cube -> raster order)
 *
 * src, dst  bf16 [B,H,N,d] device, 16-byte aligned, not overlapping; dst is
 *           overwritten.  s.r is ignored.
 * Requires s.N == T*Hl*Wl, s.block == ct*cy*cx and T % ct == Hl % cy ==
 * Wl % cx == 0 (DSV_ERR_INVALID_ARG otherwise).
 * ------------------------------------------------------------------------ */
dsv_status dsv_cube_permute(const void* src, void* dst, dsv_shape s, int T, int Hl, int Wl, int ct, int cy,
                            int cx, int inverse, dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_predict_topk_blocks — the predictor fused with the top-k
 * ([nl] 2B: the critical KV of a query group are estimated and selected in
 * one kernel, so the group x block score matrix is never stored; [hi] 2B)
 *
 * Same result as dsv_predict_scores followed by dsv_topk_blocks, with the
 * score matrix kept on chip: the lists hold, for every row (b, h, g), the
 * k_h blocks with the largest score qbar_g . kbar_j (ties to the lower block
 * index), ascending, and the transposed lists as dsv_topk_blocks writes them.
 * The scores are computed on the tensor cores from tf32 hi / lo parts of the
 * pooled fp32 vectors (three products, ~2^-21 relative to each product), so
 * they agree with dsv_predict_scores' fp32 sums to about 1e-6 of the row's
 * scale, not bit for bit; near-ties may therefore select differently from the
 * two-call path.  The selection is exact for the scores this call computed.
 *
 * Q, K, Wq, Wk  as dsv_predict_scores.  Requires r <= 32 and
 *               N / block <= 4096 (else DSV_ERR_UNSUPPORTED).
 * k_per_head, fwd_ptr, fwd_col, bwd_ptr, bwd_col  as dsv_topk_blocks.
 * scores        optional (NULL: not written).  If given, fp32 [B,H,G,nb],
 *               16-byte aligned: the scores the selection used (a check
 *               output; writing it costs the score matrix's HBM traffic).
 * workspace     >= dsv_predict_topk_workspace_bytes(s) bytes, 256-byte aligned.
 *
 * Streams: the work is ordered on `stream`.  When the select kernel's items
 * (one per 128 groups of a head, one CTA per SM) leave a partly filled last
 * wave, that wave is a launch of its own and the transposed lists of the
 * heads already selected are built meanwhile on a second, library-owned
 * stream of the current device.  That stream first waits on an event
 * recorded in `stream`, and at the end `stream` waits on an event recorded
 * after its work, so everything enqueued on `stream` after the call runs
 * after all of the call's work: the call stays stream-ordered (and can be
 * captured into a CUDA graph).  A host mutex keeps calls from several threads
 * from interleaving these event records.
 * ------------------------------------------------------------------------ */
size_t dsv_predict_topk_workspace_bytes(dsv_shape s);
dsv_status dsv_predict_topk_blocks(const void* Q, const void* K, const float* Wq, const float* Wk, dsv_shape s,
                                   const int32_t* k_per_head, int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr,
                                   int32_t* bwd_col, float* scores, void* workspace, size_t workspace_bytes,
                                   dsv_stream_t stream);

/* ------------------------------------------------------------------------
 * dsv_dispatch_heads — the OP dispatcher ([nl] 2A, [hi] 2A: each block goes
 * sparse or dense by a sparsity threshold found by offline profiling)
 *
 * Host-only; touches no device memory.  For every head h, with kept fraction
 * rho_h = k_per_head[h] / nb, the measured profile gives the time of the
 * sparse path (predictor, top-k and sparse attention with k_h blocks per
 * group) relative to the dense path (the same attention kernels with every
 * block: k = nb, no predictor): ratio(rho), piecewise linear between the
 * profile points and constant beyond its ends.  The head goes dense when
 * ratio(rho_h) >= 1: k_out[h] = nb and dense_out[h] = 1; otherwise
 * k_out[h] = k_per_head[h] and dense_out[h] = 0.
 *
 * k_per_head  host [H], each in [1, nb].
 * rho, ratio  host [n], n >= 1: rho strictly increasing in (0, 1], ratio
 *             finite and > 0 (a profile such as bench.py --dispatch-profile
 *             writes).
 * k_out, dense_out  host [H], written.
 * Returns DSV_ERR_INVALID_ARG (nothing written) on a null pointer, H < 1,
 * nb < 1, a k outside [1, nb] or a malformed profile.
 * ------------------------------------------------------------------------ */
dsv_status dsv_dispatch_heads(const int32_t* k_per_head, int32_t H, int32_t nb, const float* rho,
                              const float* ratio, int32_t n, int32_t* k_out, int32_t* dense_out);

/* ------------------------------------------------------------------------
 * Status and device-side error reporting.
 * ------------------------------------------------------------------------ */
const char* dsv_status_string(dsv_status status);

/* Synchronises `stream`, then returns the first device-side error recorded
 * on the current device since the last clear (DSV_OK if none).  `info`, if
 * not NULL, receives a kernel-specific detail word (which wait or index). */
dsv_status dsv_get_device_error(dsv_stream_t stream, uint32_t* info);

/* Resets the current device's error word (asynchronous on `stream`). */
dsv_status dsv_clear_device_error(dsv_stream_t stream);

/* Time limit, in nanoseconds, of every wait inside the kernels on the
 * current device (default 1e9).  A wait past it records DSV_ERR_TIMEOUT and
 * the kernel returns without finishing.  0 restores the default.  The waits
 * with which a kernel drains the copies and tensor-core products it has
 * already issued (before it exits, or frees its tensor memory) keep a limit
 * of at least 2 s whatever is set here: that work finishes on its own. */
dsv_status dsv_set_wait_limit_ns(uint64_t limit_ns);

/* Failure-detection self-test (the pages have no counterpart; it checks the
 * library's own error reporting).  Enqueues on `stream` one single-thread
 * kernel that waits, through the same bounded barrier wait the attention
 * kernels use, on a shared-memory barrier nothing ever arrives at.  The wait
 * gives up after the limit set by dsv_set_wait_limit_ns, records
 * DSV_ERR_TIMEOUT with info DSV_SELFTEST_WAIT_ID in the device error word
 * (unless an earlier error is already recorded) and the kernel returns: no
 * fault, and the context stays usable.  Returns DSV_ERR_CUDA if the launch
 * fails; read the outcome with dsv_get_device_error(). */
#define DSV_SELFTEST_WAIT_ID 0xD5F0u
dsv_status dsv_selftest_wait_timeout(dsv_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int32_t dsv_version(void);


#ifdef __cplusplus
}
#endif

#endif /* DSV_H_ */
