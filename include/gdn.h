/*
 * gdn.h -- C ABI of libgdn.so: chunkwise forward of the gated delta rule (GDN),
 * its DeltaProduct generalisation, and the camera-branch prep, for one
 * NVIDIA GB300 (sm_103a).
 *
 * General rules for every entry point below:
 *  - All tensor arguments are DEVICE pointers to contiguous, row-major
 *    buffers owned by the caller.  The library never allocates, frees or
 *    keeps a pointer after the call returns, and never synchronises.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns an error status and enqueues nothing.
 *  - Tensor base pointers must be 16-byte aligned (GDN_ERR_MISALIGNED).
 *  - A launch failure returns GDN_ERR_CUDA.  A device-side bounded wait that
 *    gives up (it never spins forever) records GDN_ERR_TIMEOUT in a device
 *    word that gdn_get_device_error() reads back.
 *  - No C++ exception crosses this interface.
 *
 * State convention (fixed by this library): the per-(batch, head) state S is
 * Dk x Dv, rows indexed by the key dimension, columns by the value dimension,
 * stored row-major as fp32 [B,H,Dk,Dv], and
 *
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * (gated_deltaproduct test.py: `gated_chunk_delta_rule_fwd_kernel_h`, the
 * state is [K, V] and `b_v -= dot(w, h)` predicts with the decayed state;
 * `gated_chunk_linear_attn_fwd_kernel_o` includes token t's own update via
 * the `>=` causal mask.  fused_cam_gdn.py, `_cam_scan_kernel`: decay the
 * state, then predict, then correct.)
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_F32 = 0,  /* fp32 tensors; all arithmetic in fp32                  */
    GDN_BF16 = 1  /* bf16 tensors; fp32 state and accumulation             */
} gdn_dtype_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null required pointer, bad size or shape   */
    GDN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. Dk=96)     */
    GDN_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned    */
    GDN_ERR_WORKSPACE = 4,    /* workspace missing or smaller than queried  */
    GDN_ERR_CUDA = 5,         /* a CUDA launch or runtime call failed       */
    GDN_ERR_TIMEOUT = 6       /* a bounded device wait gave up             */
} gdn_status_t;

/* flags */
#define GDN_QK_L2NORM 1u /* normalise q_t and k_t to unit L2 norm at load,
                            q <- q / max(||q||, 1e-12) per (token, head)   */
#define GDN_PATH_SIMT 2u /* use the CUDA-core path even where the tensor-core
                            path applies (bf16, Dk = Dv = 128, chunk 64,
                            r in {1, 2, 4})                                */
#define GDN_CAM_REVERSE 4u /* cam_scan_fwd only: the anti-causal mode        */

/* Human-readable name of a status code; never NULL. */
const char *gdn_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int gdn_version(void);

/*
 * Bytes of device workspace gdn_chunk_fwd / deltaproduct_chunk_fwd need for
 * these sizes (r = 1 for GDN) on the current device.  May be 0.  Returns
 * (size_t)-1 for sizes the library rejects.
 */
size_t gdn_chunk_fwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int chunk,
                                     int dtype);

/*
 * gdn_chunk_fwd -- chunkwise GDN forward (gated_deltaproduct test.py: the
 * decay-masked KK^T kernel `gated_chunk_scaled_dot_kkt_fwd_kernel`, the
 * 16x16 triangular solve and merge kernels, `gated_fwd_recompute_w_u_kernel`,
 * the state scan `gated_chunk_delta_rule_fwd_kernel_h` and the output kernel
 * `gated_chunk_linear_attn_fwd_kernel_o`, run as one pass).
 *
 *   q, k    [B,H,T,Dk]  dtype
 *   v, o    [B,H,T,Dv]  dtype (o is written; it may not alias an input)
 *   beta    [B,H,T]     dtype
 *   g       [B,H,T]     fp32, natural-log decay: the state is multiplied by
 *                       exp(g_t) before token t's correction
 *   initial_state [B,H,Dk,Dv] fp32 or NULL (NULL = zero state)
 *   final_state   [B,H,Dk,Dv] fp32 or NULL (written when given)
 *   chunk   rows per chunk: 16, 32 or 64.  Results do not depend on it beyond
 *           rounding.  T need not be a multiple of it.
 *   scale   multiplies every output (1.0 for the plain definition)
 *   flags   0 or a combination of GDN_QK_L2NORM and GDN_PATH_SIMT
 *   dtype   GDN_F32 or GDN_BF16
 *   Dk, Dv  64 or 128 each
 *   workspace / workspace_bytes: device scratch of at least
 *           gdn_chunk_fwd_workspace_bytes(...) bytes (NULL if that is 0),
 *           16-byte aligned.  The tensor-core path uses it, for B*H up to
 *           min(80, SMs/2) heads, as a ring through which the chunk-local
 *           results travel to the state scan (about 205 KB per head).  Its
 *           contents need no initialisation and are not meaningful after
 *           the call; calls that may overlap on the GPU need separate
 *           workspaces.  A call that completes leaves the ring's tags zeroed,
 *           so a workspace may be reused by launches that carry the same tag
 *           epoch (replays of one captured CUDA graph); after a call that
 *           ended in GDN_ERR_TIMEOUT, zero the workspace before such reuse.
 *           A smaller workspace is GDN_ERR_WORKSPACE; one that is not
 *           16-byte aligned makes the call run without the ring.
 * T = 0 or B*H = 0 is valid and enqueues nothing (final_state, if given,
 * receives initial_state or zeros).
 */
int gdn_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                  const float *g, const float *initial_state, void *o, float *final_state,
                  int B, int H, int T, int Dk, int Dv, int chunk, float scale,
                  unsigned flags, int dtype, void *workspace, size_t workspace_bytes,
                  void *stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate
 * device memory: code running where cudaMalloc is off limits (inside a host
 * callback, from a plug-in whose host owns every allocation, or under a memory
 * budget fixed in advance) cannot provide the workspace that gdn_chunk_fwd may
 * ask for.  This entry point takes no workspace and allocates nothing; when
 * the tensor-core path needs scratch it uses an array inside the library, of
 * fixed size (13.1 MB, enough for B*H <= 64 heads), which every GPU that loads
 * the library holds until the process exits.  The paper has no counterpart:
 * this is a deployment convenience only.
 *
 * Arguments, layouts and results are those of gdn_chunk_fwd.  For head
 * counts whose ring would not fit the array (more than 64 heads), the
 * tensor-core path runs in its cluster mode, which needs no scratch; no size
 * that gdn_chunk_fwd accepts is refused for want of scratch.
 * The first call on a device looks up the array's device address with that
 * device current (no allocation); make that first call before any stream
 * capture.  All calls share the one array, which keeps the last call's
 * contents; nothing in it has to start at zero (every tag it holds names the
 * launch that wrote it, and a call that completes zeroes the tags it used).
 * Two calls that overlap on the GPU, on different streams, race on it:
 * serialise them.
 */
int gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *beta,
                          const float *g, const float *initial_state, void *o, float *final_state,
                          int B, int H, int T, int Dk, int Dv, int chunk, float scale,
                          unsigned flags, int dtype, void *stream);

/*
 * deltaproduct_chunk_fwd -- DeltaProduct forward: per token the decay exp(g_t)
 * is applied once, then r corrections in order j = 0..r-1,
 *     S <- (I - beta_{t,j} k_{t,j} k_{t,j}^T) S + beta_{t,j} k_{t,j} v_{t,j}^T,
 * and o_t = scale * S^T q_t reads the state after the last one.  Each
 * sub-step has its own key, value and beta (the rows (t,j) form one sequence
 * of r*T rows; gated_deltaproduct test.py interleaves them the same way, as
 * BT*r rows per chunk).
 *
 *   q, o    [B,H,T,Dk] / [B,H,T,Dv]   dtype
 *   k       [B,H,T,r,Dk]              dtype
 *   v       [B,H,T,r,Dv]              dtype
 *   beta    [B,H,T,r]                 dtype
 *   g       [B,H,T]                   fp32
 *   chunk   row capacity of a chunk (16, 32 or 64); each chunk holds
 *           floor(chunk / r) whole tokens, i.e. r*floor(chunk/r) rows
 *   r       1..8
 * Everything else as gdn_chunk_fwd.  r = 1 computes exactly gdn_chunk_fwd.
 */
int deltaproduct_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                           const float *g, const float *initial_state, void *o,
                           float *final_state, int B, int H, int T, int r, int Dk, int Dv,
                           int chunk, float scale, unsigned flags, int dtype, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * masked_deltaproduct_chunk_fwd -- block-masked DeltaProduct forward
 * (gated_deltaproduct test.py: the mask_ij coupling of
 * `gated_chunk_scaled_dot_kkt_fwd_kernel` and `gated_fwd_recompute_w_u_kernel`,
 * the per-slice state update of `gated_chunk_delta_rule_fwd_kernel_h`, and the
 * sum over r of `gated_chunk_fwd_o_fn`).  The key dimension is cut into r
 * slices of Dk/r; per token the decay is applied once, then each sub-row
 * i < r predicts from that same state with k_t masked slice-wise by
 * mask[i][:] and corrects the state's slice-i rows with slice i of k_t; one
 * value and one beta per token:
 *     S <- exp(g_t) S;   z_j = S_(j)^T k_t,(j);   d_i = beta_t (v_t - sum_j mask[i][j] z_j)
 *     S_(i) <- S_(i) + k_t,(i) d_i^T   (every i from the same z);   o_t = scale * S^T q_t
 * i.e. S_t = exp(g_t) (I - beta_t (k_t k_t^T) o M) S_{t-1} + beta_t k_t v_t^T with M
 * the mask expanded to Dk/r x Dk/r blocks.  An all-ones mask is gdn_chunk_fwd.
 *
 *   q, k [B,H,T,Dk]; v, o [B,H,T,Dv]; beta [B,H,T] (all dtype); g [B,H,T] fp32
 *   mask [r][r] fp32 (device), shared by all heads; r in {1, 2, 4, 8}, r | Dk
 *   chunk   16, 32 or 64, a multiple of r (accepted for symmetry with the other
 *           entry points: the kernels work on 64 sub-rows, 64 / r tokens, per
 *           chunk, and results do not depend on the chunk beyond rounding)
 *   flags   0, or GDN_QK_L2NORM and GDN_PATH_SIMT.  Three launches: the
 *           chunks' WY factors in parallel (CUDA cores, fp32), the state
 *           chain, then the outputs in parallel (CUDA cores, fp32).  With bf16
 *           tensors at Dk = Dv = 128 the chain runs on tcgen05 (one CTA per
 *           head, fp32 state in tensor memory, bf16 hi / lo split products of
 *           about 2^-16 relative error); otherwise, or with GDN_PATH_SIMT, on
 *           the CUDA cores by 32 value columns per CTA.
 *   workspace: masked_deltaproduct_chunk_fwd_workspace_bytes(...) bytes,
 *           16-byte aligned (GDN_ERR_WORKSPACE when missing or short); no
 *           initialisation needed, contents not meaningful afterwards.
 * State, scale, dtype and the empty cases as gdn_chunk_fwd.
 */
size_t masked_deltaproduct_chunk_fwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int dtype);
int masked_deltaproduct_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                                  const float *g, const float *mask, const float *initial_state, void *o,
                                  float *final_state, int B, int H, int T, int r, int Dk, int Dv, int chunk,
                                  float scale, unsigned flags, int dtype, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Bytes of device workspace masked_deltaproduct_chunk_bwd needs: per head and
 * chunk of 64 / r tokens the chunk's WY factors, the state entering it and the
 * gradient of the state leaving it (about 370 KB at Dk = Dv = 128).  0 when
 * T = 0; (size_t)-1 for sizes it rejects.
 */
size_t masked_deltaproduct_chunk_bwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int dtype);

/*
 * masked_deltaproduct_chunk_bwd -- backward of masked_deltaproduct_chunk_fwd
 * (gated_deltaproduct test.py: `gated_chunk_delta_rule_bwd_kernel_dhu`,
 * `gated_chunk_delta_rule_bwd_kernel_dqkw`, `gated_bwd_prepare_wy_repr_kernel`).
 * Per token, with D the decayed state, the sub-rows' read keys kr_i and write
 * keys kw_i as in the forward, e_i = v - D^T kr_i and G the gradient of the
 * state after the token:
 *     w_i = G^T kw_i;  dv = beta sum_i w_i;  dbeta = sum_i kw_i . (G e_i)
 *     dkw_i = beta G e_i;  dkr_i = -beta D w_i;  dD = G - beta sum_i kr_i w_i^T
 * slice j of dk = slice j of (dkw_j + sum_i mask[i][j] dkr_i), dg = <dD, D>,
 * and the state entering the token gets exp(g) dD; computed chunk-wise in
 * three launches as gdn_chunk_bwd (flags: GDN_QK_L2NORM, GDN_PATH_SIMT).
 *   q, k, v, beta, g, mask, initial_state, scale, flags, dtype, Dk, Dv, r: as
 *           given to masked_deltaproduct_chunk_fwd (r in {1, 2, 4, 8})
 *   dout [B,H,T,Dv] dtype;  dfinal_state [B,H,Dk,Dv] fp32 or NULL (= zero)
 *   dq, dk [B,H,T,Dk], dv [B,H,T,Dv] dtype;  dbeta, dg [B,H,T] fp32;
 *   dinitial_state [B,H,Dk,Dv] fp32 or NULL (not wanted)
 *   workspace: masked_deltaproduct_chunk_bwd_workspace_bytes(...) bytes,
 *           16-byte aligned.
 * The empty cases as gdn_chunk_bwd.
 */
int masked_deltaproduct_chunk_bwd(const void *q, const void *k, const void *v, const void *beta, const float *g,
                                  const float *mask, const float *initial_state, const void *dout,
                                  const float *dfinal_state, void *dq, void *dk, void *dv, float *dbeta, float *dg,
                                  float *dinitial_state, int B, int H, int T, int r, int Dk, int Dv, float scale,
                                  unsigned flags, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace cam_scan_fwd needs for these sizes on the current
 * device (0 on the CUDA-core path).  (size_t)-1 for sizes it rejects.
 */
size_t cam_scan_fwd_workspace_bytes(int B, int H, int F, int S, int Dk, int Dv, int dtype);

/*
 * cam_scan_fwd -- frame-level, numerator-only camera scan (fused_cam_gdn.py:
 * `_cam_scan_kernel`, `_torch_cam_scan_single_chunk`; the reverse mode is
 * `_torch_cam_scan_reference` with `_flip_and_shift`).  The N = F*S tokens of
 * each (batch, head) form F frames of S tokens.  Forward, for f = 0 .. F-1:
 *     S <- decay_f S                                   (once per frame)
 *     S <- S + K_f^T diag(beta_f) (V_f - K_f S)        (every token of the frame
 *                                                       predicts from the same S)
 *     o_s = scale * S^T q_s   for the frame's tokens    (after the update, so a
 *                                                       frame sees all of itself)
 * Reverse (flags & GDN_CAM_REVERSE): frames from last to first with a zero
 * start; frame f's tokens read the state built from frames f+1 .. F-1 only
 * (the last frame reads zero), frame j's factor decay_j decaying the state as
 * frame j is taken in.
 *
 *   q, k    [B,H,N,Dk]  dtype (the layout cam_prep_fwd writes)
 *   v, o    [B,H,N,Dv]  dtype
 *   beta    [B,H,N]     dtype
 *   decay   [B,H,F]     fp32 factors (not logs) of each frame
 *   initial_state / final_state [B,H,Dk,Dv] fp32 or NULL: forward only
 *           (GDN_ERR_UNSUPPORTED with GDN_CAM_REVERSE)
 *   F >= 0 frames of S >= 1 tokens; Dk, Dv 64 or 128; flags: GDN_QK_L2NORM
 *   (unit q and k per token and head), GDN_PATH_SIMT, GDN_CAM_REVERSE.
 *   workspace: at least cam_scan_fwd_workspace_bytes(...) bytes, 16-byte
 *           aligned (128 KB per head and frame on the tensor-core path: the
 *           frame products K^T diag(beta) [K | V] and each frame's state).
 * The page's scan takes [B,H,D,N] fp32 tensors; this library keeps the
 * token-major layout of its other entry points.
 */
int cam_scan_fwd(const void *q, const void *k, const void *v, const void *beta, const float *decay,
                 const float *initial_state, void *o, float *final_state, int B, int H, int F, int S,
                 int Dk, int Dv, float scale, unsigned flags, int dtype, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace cam_prep_scan_fwd needs; (size_t)-1 for sizes it
 * rejects.
 */
size_t cam_prep_scan_fwd_workspace_bytes(int B, int N, int H, int D, int F, int dtype);

/*
 * cam_prep_scan_fwd -- the camera prep fused into the frame scan
 * (fused_cam_gdn.py: `cam_prep_func`, whose `_precompute_cam_inv_rms` is the
 * separate reduction pass, then `_cam_scan_kernel`): computes
 * cam_scan_fwd(cam_prep_fwd(raw ...)) without writing the prepped q, k, v.
 * A pre-pass forms each token's full-C inverse RMS of q and k; the frame
 * scan then reads the raw rows and applies the norm (with the weights), ReLU
 * and K-scale, the 4 x 4 projection and the rotation at load.
 *
 *   q_raw, k_raw, v_raw [B,N,H,D] bf16; q_norm_w, k_norm_w [H*D] fp32 or NULL;
 *   proj_q, proj_kv [B,N,4,4] fp32;
 *   rope_base > 0: the rotation angles th_i = n * rope_base^(-2i/(D/2)) of
 *   cam_prep_fwd without tables (this path takes no tables);
 *   beta [B,H,N] bf16, decay [B,H,F] fp32 factors, o [B,H,N,D] bf16,
 *   initial_state / final_state as cam_scan_fwd (forward only);
 *   N = F * S; D = 128, H*D <= 4096, bf16 only; flags: GDN_QK_L2NORM (unit
 *   prepped q and k), GDN_CAM_REVERSE; workspace of
 *   cam_prep_scan_fwd_workspace_bytes bytes, 16-byte aligned.
 * The k norms before and after the projection (cam_prep_fwd's k_pre_sq and
 * k_post_sq) are not produced.
 */
int cam_prep_scan_fwd(const void *q_raw, const void *k_raw, const void *v_raw, const float *q_norm_w,
                      const float *k_norm_w, const float *proj_q, const float *proj_kv, float rope_base,
                      const void *beta, const float *decay, const float *initial_state, void *o,
                      float *final_state, int B, int N, int H, int D, int F, float k_scale, float eps, float scale,
                      unsigned flags, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * cam_prep_fwd -- fused camera-branch prep (fused_cam_gdn.py, `_cam_prep_kernel`
 * and `_torch_cam_prep_reference`), one pass over q, k, v:
 *   1. full-C RMSNorm of q and k per token, C = H*D:
 *        x <- x * rsqrt(sum_{h,d} x^2 / C + eps) * w[h*D+d]
 *   2. ReLU on q and k; k additionally times k_scale.  v gets neither.
 *   3. first D/2 dims, each group of 4: out_i = sum_j P[i][j] in_j with
 *      P = proj_q[b,n] for q and P = proj_kv[b,n] for k and v;
 *   4. last D/2 dims, interleaved pairs: y[d] = x[d] cos[d] + x[d^1] sin[d]
 *      with the tables' encoding cos[2i] = cos[2i+1] = cos(th_i),
 *      sin[2i] = -sin(th_i), sin[2i+1] = +sin(th_i);
 *   5. optional ||k||^2 per (b,h,n) after step 2 (k_pre_sq) and after 4
 *      (k_post_sq).
 *
 *   q_raw, k_raw, v_raw  [B,N,H,D]  dtype
 *   q_norm_w, k_norm_w   [H*D] fp32 or NULL (= all ones)
 *   proj_q, proj_kv      [B,N,4,4] fp32 row-major
 *   rope_cos, rope_sin   [N,D/2] fp32 in the encoding above, or both NULL:
 *                        then th_i = n * rope_base^(-2i/(D/2)), n = token index
 *   q_out, k_out, v_out  [B,H,N,D]  dtype (head-major, ready for the scan)
 *   k_pre_sq, k_post_sq  [B,H,N] fp32 or NULL
 *   D a multiple of 16 with D/8 dividing 32 (16, 32, 64, 128 or 256);
 *   H*D <= 4096.
 */
int cam_prep_fwd(const void *q_raw, const void *k_raw, const void *v_raw, const float *q_norm_w,
                 const float *k_norm_w, const float *proj_q, const float *proj_kv,
                 const float *rope_cos, const float *rope_sin, float rope_base, void *q_out,
                 void *k_out, void *v_out, float *k_pre_sq, float *k_post_sq, int B, int N,
                 int H, int D, float k_scale, float eps, int dtype, void *stream);

/*
 * Bytes of device workspace gdn_chunk_bwd / deltaproduct_chunk_bwd need
 * (r = 1 for GDN): per head and chunk of floor(64 / r) tokens, the chunk's
 * WY factors, the states entering it and their gradients (about 370 KB at
 * Dk = Dv = 128).  0 when T = 0; (size_t)-1 for sizes they reject.
 */
size_t gdn_chunk_bwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int dtype);

/*
 * gdn_chunk_bwd -- backward of gdn_chunk_fwd (gated_deltaproduct test.py: the
 * state-gradient kernel `gated_chunk_delta_rule_bwd_kernel_dhu`, the
 * chunk-local `gated_chunk_delta_rule_bwd_kernel_dqkw` and the WY backward
 * `gated_bwd_prepare_wy_repr_kernel`): the gradients of q, k, v, beta, g and
 * the initial state, given the gradient of o and (optionally) of the final
 * state.  Per token, with G the gradient of the state after the token and X
 * the decayed state the correction starts from:
 *     G += scale q do^T;  dq = scale S do;  e = v - X^T k,  w = G^T k
 *     dv = beta w;  dbeta = k.(G e);  dk = beta (G e - X w);  G <- G - beta k w^T
 *     dg = <G, X>;  G <- exp(g) G
 * computed chunk-wise in the WY form (64-row chunks) in three launches: the
 * chunk factors (CUDA cores, fp32); the forward state chain and the reverse
 * gradient chain side by side; the input gradients (CUDA cores, fp32).  With
 * bf16 tensors at Dk = Dv = 128 the two chains run on tcgen05 (one CTA per
 * head and chain, fp32 state in tensor memory, bf16 hi / lo split products of
 * about 2^-16 relative error); otherwise, or with GDN_PATH_SIMT, on the CUDA
 * cores in fp32 by 64 value columns per CTA.
 *
 *   q, k, v, beta, g, initial_state, scale, dtype, Dk, Dv: as given to
 *           gdn_chunk_fwd (flags: GDN_QK_L2NORM and GDN_PATH_SIMT)
 *   dout    [B,H,T,Dv] dtype;  dfinal_state [B,H,Dk,Dv] fp32 or NULL (= zero)
 *   dq, dk [B,H,T,Dk], dv [B,H,T,Dv] dtype (written);  dbeta [B,H,T] fp32;
 *   dg [B,H,T] fp32;  dinitial_state [B,H,Dk,Dv] fp32 or NULL (not wanted)
 *   workspace: gdn_chunk_bwd_workspace_bytes(...) bytes, 16-byte aligned
 *           (GDN_ERR_WORKSPACE when missing or short); its contents need no
 *           initialisation and are not meaningful afterwards.
 * T = 0 or B*H = 0 enqueues at most the copy of dfinal_state (or zeros) into
 * dinitial_state.
 */
int gdn_chunk_bwd(const void *q, const void *k, const void *v, const void *beta, const float *g,
                  const float *initial_state, const void *dout, const float *dfinal_state, void *dq, void *dk,
                  void *dv, float *dbeta, float *dg, float *dinitial_state, int B, int H, int T, int Dk, int Dv,
                  float scale, unsigned flags, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * deltaproduct_chunk_bwd -- backward of deltaproduct_chunk_fwd: per token the
 * r sub-steps are undone last first, then the decay (gdn_chunk_bwd's step per
 * sub-step).  k, dk [B,H,T,r,Dk]; v, dv [B,H,T,r,Dv]; beta, dbeta [B,H,T,r];
 * 1 <= r <= 8; each chunk holds floor(64 / r) tokens.  Everything else as
 * gdn_chunk_bwd; r = 1 computes exactly gdn_chunk_bwd.
 */
int deltaproduct_chunk_bwd(const void *q, const void *k, const void *v, const void *beta, const float *g,
                           const float *initial_state, const void *dout, const float *dfinal_state, void *dq,
                           void *dk, void *dv, float *dbeta, float *dg, float *dinitial_state, int B, int H, int T,
                           int r, int Dk, int Dv, float scale, unsigned flags, int dtype, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace cam_scan_bwd needs ((size_t)-1 for sizes it
 * rejects): per head and frame, the frame's products K^T diag(beta) K,
 * K^T diag(beta) V and scale Q^T dO, the state entering it and the gradient
 * of the state after it (fp32), and one float per 64-token tile.
 */
size_t cam_scan_bwd_workspace_bytes(int B, int H, int F, int S, int Dk, int Dv, int dtype);

/*
 * cam_scan_bwd -- backward of cam_scan_fwd, forward direction
 * (fused_cam_gdn.py, `_cam_scan_bwd_kernel`): the gradients of q, k, v, beta,
 * each frame's decay and the initial state, given the gradient of o (and of
 * the final state).  With S' the state entering frame f and S_f the state
 * after it, R = diag(beta)(V - d K S'), S_f = d S' + K^T R, O = scale Q S_f; the
 * frames are taken from last to first with dS the gradient of S_f:
 *     dS += scale Q^T dO;   dq_t = scale S_f do_t
 *     dR = K dS;   dv_t = beta_t dR_t;   dbeta_t = dR_t . (v_t - d S'^T k_t)
 *     dk_t = dS r_t - d beta_t S' dR_t;   ddecay_f = <dS, S'> - sum_t beta_t dR_t . S'^T k_t
 *     dS <- d (dS - K^T diag(beta) dR)
 * and, with GDN_QK_L2NORM, the unit-norm map's adjoint on q and k.
 *
 *   q, k, v, beta, decay, initial_state, scale, flags, dtype: as given to
 *           cam_scan_fwd (GDN_CAM_REVERSE is GDN_ERR_UNSUPPORTED)
 *   dout    [B,H,N,Dv] dtype;  dfinal_state [B,H,Dk,Dv] fp32 or NULL (= zero)
 *   dq, dk [B,H,N,Dk], dv [B,H,N,Dv] dtype;  dbeta [B,H,N] fp32;
 *   ddecay [B,H,F] fp32;  dinitial_state [B,H,Dk,Dv] fp32 or NULL
 *   flags   GDN_QK_L2NORM, and GDN_PATH_SIMT to keep every product on the
 *           CUDA cores
 *   workspace: cam_scan_bwd_workspace_bytes bytes, 16-byte aligned.
 * Four launches: the frame products (one CTA per frame, head and product),
 * the forward state chain and the reverse gradient chain side by side, the
 * token gradients, then each frame's ddecay.  For bf16 with Dk = Dv = 128 on
 * an sm_10x device the frame products, the chains (one CTA per head and
 * chain) and the token gradients run on tcgen05 (fp32 accumulators in TMEM;
 * the fp32 operands split into bf16 hi + lo, products formed as
 * hi.hi + hi.lo + lo.hi; the token kernel persistent over 128-token tiles);
 * otherwise on the CUDA cores in fp32 (chains by 32 value columns per CTA,
 * 64-token tiles).
 */
int cam_scan_bwd(const void *q, const void *k, const void *v, const void *beta, const float *decay,
                 const float *initial_state, const void *dout, const float *dfinal_state, void *dq, void *dk,
                 void *dv, float *dbeta, float *ddecay, float *dinitial_state, int B, int H, int F, int S, int Dk,
                 int Dv, float scale, unsigned flags, int dtype, void *workspace, size_t workspace_bytes,
                 void *stream);

/*
 * cam_prep_bwd -- backward of cam_prep_fwd (fused_cam_gdn.py,
 * `_cam_prep_bwd_kernel`, continued through the full-C RMSNorm that the page
 * leaves to torch): the gradients of the raw rows given those of the outputs.
 * In reverse order of the forward, per token: the rotation and the 4 x 4
 * projection transposed (dx[d] = dy[d] cos[d] + dy[d^1] sin[d^1];
 * dx_j = sum_i P[i][j] dy_i), the ||k_out||^2 and ||k||^2 terms, K-scale, the
 * ReLU mask, and the RMSNorm backward
 *     dx_j = r w_j dxhat_j - (r^3 / C) x_j sum_c w_c x_c dxhat_c,
 *     r = (sum_c x_c^2 / C + eps)^(-1/2).
 *
 *   q_raw, k_raw, norm weights, projections, rotary tables / rope_base,
 *   k_scale, eps: as given to cam_prep_fwd (v_raw is not needed)
 *   dq_out, dk_out, dv_out  [B,H,N,D] dtype
 *   dk_pre_sq, dk_post_sq   [B,H,N] fp32 or NULL (= zero)
 *   dq_raw, dk_raw, dv_raw  [B,N,H,D] dtype (written)
 * Gradients of the norm weights and projections are not formed.  fp32
 * arithmetic; H*D <= 4096.
 */
int cam_prep_bwd(const void *q_raw, const void *k_raw, const float *q_norm_w, const float *k_norm_w,
                 const float *proj_q, const float *proj_kv, const float *rope_cos, const float *rope_sin,
                 float rope_base, const void *dq_out, const void *dk_out, const void *dv_out,
                 const float *dk_pre_sq, const float *dk_post_sq, void *dq_raw, void *dk_raw, void *dv_raw, int B,
                 int N, int H, int D, float k_scale, float eps, int dtype, void *stream);

/*
 * Reads and clears the device error word of the current device after
 * synchronising `stream`.  Returns GDN_OK, GDN_ERR_TIMEOUT, or GDN_ERR_CUDA if
 * the synchronisation itself failed.
 */
int gdn_get_device_error(void *stream);

/*
 * Number of kernels this library has launched in this process (all devices,
 * all entry points) since it was loaded.  Host-side counter; never blocks.
 */
unsigned long long gdn_launch_count(void);

/*
 * Test hook for the bounded-wait path: sets the wall-clock limit, in
 * microseconds, of the bounded device waits in later launches of the
 * tensor-core scan (gdn_chunk_fwd, deltaproduct_chunk_fwd) and of the
 * tensor-core state chains (the chunk backward passes
 * and the block-masked forward); 0 restores the default of one second.  The
 * other tensor-core kernels keep a one-second limit.  A wait that runs out
 * sets GDN_ERR_TIMEOUT in the device error word and its kernel stops early;
 * the outputs of that call are then undefined, but the context stays usable.
 */
int gdn_set_wait_limit(unsigned long long polls);

/*
 * Cluster shape of the tcgen05 path for later calls on this process: each
 * thread-block cluster holds heads_per_cluster scan CTAs (one (batch, head)
 * each) and wy_ctas_per_cluster CTAs that compute the chunk-local WY products
 * for them (two pipelines each, taking the cluster's (head, chunk) items in
 * turn).  A forced shape also turns off the ring mode (one cooperative grid
 * whose WY results travel through the workspace), which is otherwise the
 * default up to min(80, SMs/2) heads.  0, 0 restores the automatic choice:
 * the ring mode where it applies, else the cluster shape with the most WY
 * pipelines per head whose clusters are all resident on the device at once.
 * Returns GDN_ERR_INVALID_ARG unless 1 <= heads_per_cluster <= 4,
 * wy_ctas_per_cluster >= 1 and their sum <= 16.  A shape whose clusters cannot
 * be scheduled makes the next launch fail with GDN_ERR_CUDA.
 */
int gdn_set_cluster_shape(int heads_per_cluster, int wy_ctas_per_cluster);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
