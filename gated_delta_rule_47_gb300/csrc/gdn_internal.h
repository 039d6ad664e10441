// Internal host-side declarations shared by the translation units of libgdn.so.
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {

// Arguments of one scan call.  r = 1 for GDN; for DeltaProduct the r
// sub-steps of token t are rows t*r .. t*r+r-1 of one sequence of T*r rows.
struct ScanArgs {
    const void *q, *k, *v, *beta;
    const float *g;
    const float *s0;
    void *o;
    float *sf;
    int B, H, T, r, Dk, Dv, chunk;
    float scale;
    unsigned flags;
    int dtype;
    void *ws;
    size_t ws_bytes;
};

struct CamArgs {
    const void *q_raw, *k_raw, *v_raw;
    const float *q_norm_w, *k_norm_w, *proj_q, *proj_kv, *rope_cos, *rope_sin;
    float rope_base;
    void *q_out, *k_out, *v_out;
    float *k_pre_sq, *k_post_sq;
    int B, N, H, D;
    float k_scale, eps;
    int dtype;
};

// SIMT chunkwise path (any supported dtype, Dk/Dv in {64,128}, chunk in {16,32,64}).
int launch_scan_simt(const ScanArgs &a, cudaStream_t stream);

// tcgen05 path (bf16, Dk = Dv = 128, chunk 64).  Returns GDN_ERR_UNSUPPORTED
// for anything else so that the caller can pick the SIMT path.
bool scan_tc_supported(const ScanArgs &a);
size_t scan_tc_workspace_bytes(const ScanArgs &a);
int launch_scan_tc(const ScanArgs &a, cudaStream_t stream);
int scan_tc_read_clear_error(cudaStream_t stream);
int scan_tc_set_wait_limit(unsigned long long polls);
// The bounded-wait limit gdn_set_wait_limit last set, in ns.
unsigned long long wait_limit_ns();
// Cluster shape of the tcgen05 path (heads and WY CTAs per cluster); 0, 0 = automatic.
int scan_tc_set_cluster_shape(int hc, int nwy);
// Device address and size of the fixed scratch array behind
// gdn_chunk_fwd_noalloc (set up on the current device at the first call).
int scan_tc_noalloc_scratch(void **ptr, size_t *bytes);

// Arguments of one frame-level camera scan call: q,k [B,H,F*S,Dk], v,o
// [B,H,F*S,Dv], beta [B,H,F*S], decay [B,H,F] factors.
struct CamScanArgs {
    const void *q, *k, *v, *beta;
    const float *decay;
    const float *s0;
    void *o;
    float *sf;
    int B, H, F, S, Dk, Dv;
    float scale;
    unsigned flags;
    int dtype;
    void *ws;
    size_t ws_bytes;
};

// Arguments of one block-masked DeltaProduct call: q,k [B,H,T,Dk], v,o
// [B,H,T,Dv], beta,g [B,H,T], mask [r][r]; chunk counts sub-rows (tokens x r).
struct MaskedDpArgs {
    const void *q, *k, *v, *beta;
    const float *g, *mask, *s0;
    void *o;
    float *sf;
    int B, H, T, r, Dk, Dv, chunk;
    float scale;
    unsigned flags;
    int dtype;
    void *ws;
    size_t ws_bytes;
};
size_t masked_dp_workspace_bytes(const MaskedDpArgs &a);
int launch_masked_dp(const MaskedDpArgs &a, cudaStream_t stream);

// Frame scan: the tensor-core path (bf16, Dk = Dv = 128) needs a workspace of
// cam_scan_workspace_bytes; everything else runs on the CUDA cores.
bool cam_scan_tc_supported(const CamScanArgs &a);
size_t cam_scan_workspace_bytes(const CamScanArgs &a);
int launch_cam_scan(const CamScanArgs &a, cudaStream_t stream);
int cam_scan_read_clear_error();

// The camera prep fused into the frame scan (bf16, D = 128, rotary angles
// from the base): raw q, k, v [B,N,H,128]; the scan's beta [B,H,N], decay [B,H,F].
struct CamFusedArgs {
    const void *q_raw, *k_raw, *v_raw;
    const float *q_norm_w, *k_norm_w, *proj_q, *proj_kv;
    float rope_base;
    const void *beta;
    const float *decay, *s0;
    void *o;
    float *sf;
    int B, H, F, S;
    float k_scale, eps, scale;
    unsigned flags;
    void *ws;
    size_t ws_bytes;
};
size_t cam_fused_workspace_bytes(const CamFusedArgs &a);

// Backward of the frame scan (forward direction): q,k [B,H,N,Dk], v [B,H,N,Dv],
// beta [B,H,N], decay [B,H,F], dout [B,H,N,Dv], dsf [B,H,Dk,Dv] or null.
struct CamScanBwdArgs {
    const void *q, *k, *v, *beta;
    const float *decay, *s0;
    const void *dout;
    const float *dsf;
    void *dq, *dk, *dv;
    float *dbeta, *ddecay, *ds0;
    int B, H, F, S, Dk, Dv;
    float scale;
    unsigned flags;
    int dtype;
    void *ws;
    size_t ws_bytes;
};
size_t cam_scan_bwd_workspace_bytes(const CamScanBwdArgs &a);
int launch_cam_scan_bwd(const CamScanBwdArgs &a, cudaStream_t stream);
// Reads and clears the error word of the frame scan's backward (GDN_OK or GDN_ERR_TIMEOUT).
int cam_scan_bwd_read_clear_error();
int launch_cam_fused(const CamFusedArgs &a, cudaStream_t stream);

// 3-D TMA map (128-byte swizzle) over a [heads][rows][128] bf16 tensor with a
// {box0, box1, 1} box; false if the driver entry point is missing or rejects it.
bool make_bf16_map(CUtensorMap *m, const void *base, int heads, long rows, int box0, int box1);
// 4-D TMA map (128-byte swizzle) over a [heads][frames][frame_rows][128] bf16
// tensor with a {box0, box1, 1, 1} box: a box that runs past a frame's last
// row is clipped there (zero-filled on loads, not written on stores).
bool make_bf16_frame_map(CUtensorMap *m, const void *base, int heads, int frames, int frame_rows, int box0,
                         int box1);
// As make_bf16_frame_map over a [outer][frames][frame_rows][cols] tensor with
// rows of `cols` bf16 (cols a multiple of 64).
bool make_bf16_frame_map_wide(CUtensorMap *m, const void *base, int outer, int frames, int frame_rows, int cols,
                              int box0, int box1);
// True on an sm_10x device (tcgen05 available); cached.
bool sm100_family();
int device_sm_count();

int launch_cam_prep(const CamArgs &a, cudaStream_t stream);

// Backward of the camera prep: the gradients of the raw q, k, v from those of
// q_out, k_out, v_out and of k_pre_sq, k_post_sq.
struct CamBwdArgs {
    const void *q_raw, *k_raw;
    const float *q_norm_w, *k_norm_w, *proj_q, *proj_kv, *rope_cos, *rope_sin;
    float rope_base;
    const void *dq_out, *dk_out, *dv_out;
    const float *dpre, *dpost;
    void *dq_raw, *dk_raw, *dv_raw;
    int B, N, H, D;
    float k_scale, eps;
    int dtype;
};
int launch_cam_prep_bwd(const CamBwdArgs &a, cudaStream_t stream);
// Reads and clears the error word of the streamed camera prep (GDN_OK or GDN_ERR_TIMEOUT).
int cam_prep_read_clear_error();

// Backward of the chunkwise GDN / DeltaProduct forward (r = 1 for GDN).
struct ChunkBwdArgs {
    const void *q, *k, *v, *beta;
    const float *g, *s0;
    const void *dout;
    const float *dsf;
    void *dq, *dk, *dv;
    float *dbeta, *dg, *ds0;
    int B, H, T, r, Dk, Dv;
    float scale;
    unsigned flags;
    int dtype;
    void *ws;
    size_t ws_bytes;
};
size_t chunk_bwd_workspace_bytes(const ChunkBwdArgs &a);
int launch_chunk_bwd(const ChunkBwdArgs &a, cudaStream_t stream);

// Backward of the block-masked DeltaProduct forward.
struct MaskedBwdArgs {
    const void *q, *k, *v, *beta;
    const float *g, *mask, *s0;
    const void *dout;
    const float *dsf;
    void *dq, *dk, *dv;
    float *dbeta, *dg, *ds0;
    int B, H, T, r, Dk, Dv;
    float scale;
    unsigned flags;
    int dtype;
    void *ws;
    size_t ws_bytes;
};
size_t masked_bwd_workspace_bytes(const MaskedBwdArgs &a);
int launch_masked_bwd(const MaskedBwdArgs &a, cudaStream_t stream);

// The sequential chains of the chunkwise WY form on tcgen05 (wy_chain_tc.cu),
// for Dk = Dv = 128 and 64-row chunks; per (head, chunk) ci = head * NT + c.
// roles = 1 runs the forward state chain only, 2 also the reverse gradient
// chain (a second CTA per head).
struct WyChainTcArgs {
    const float *s0, *dsf;  // [BH][128][128] initial state / final state's gradient, or null (zero)
    float *sf, *ds0;        // [BH][128][128] final state / initial state's gradient, or null (not wanted)
    float *Sw, *dSw;        // [ci][128][128] state entering / gradient leaving each chunk
    float *Vnw;             // [ci][64][128] Vn of each chunk (forward chain)
    const unsigned char *Wimg, *Kdimg;  // [ci] 32 KB bf16 hi | lo images of W and Kd (write_chain_image)
    const float *Uw, *Bw, *Gw;          // [ci][64][128] U, [ci][128][128] B (reverse), [ci][64] gamma
    // or null: [ci] Y = Kd dS' of each chunk ([64][128], reverse chain), written over the first half
    // of that chunk's B once the chain has read it
    float *Yw;
    int BH, NT, roles;
    unsigned long long timeout_ns;  // bounded-wait limit (set by the launcher)
};
int launch_wy_chain_tc(const WyChainTcArgs &a, cudaStream_t stream);
// The products the backward's gradient kernels need, on tcgen05
// (wy_chain_tc.cu), per (head, chunk) ci after both chains, written over
// slots that nothing reads afterwards:
//   dS' slot: t1 = dO S^T [Ct][128] (floats 8192..)
//   S slot:   dR = T^T dVn [64][128] (0..8191)
//   Vn slot:  dR Vn^T [64][64] (0..4095), DOV = dO Vn^T [64][64] (4096..; rows
//             past the chunk's queries undefined)
//   B slot:   the rows' dk share [64][128] (0..8191, below), <dS', S> at float
//             8192, each row's Y . Vn at 8256..8319 and kr . t2 at 8320..8383
//   W slot:   P~ Kw [Ct][128]
// with dk's share = ww (e^{gl-gamma} Z + X1) + wr (X2 - diag(beta e^gamma) t2),
// Z = Vn dS'^T, t2 = dR S^T, X1 = P~^T Q + L^T Kr, X2 = L Kw (ww = wr = 1 but
// for the block-masked variant's slice weights),
// dVn = Y + P^^T dO, Y = Kd dS' (the first half of the B slot, from the
// reverse chain), P^ and T from the WY kernel, and the gradient kernel's
// P~ = the decay-masked scale dO Vn^T and L = -(dR Vn^T) diag(beta) E below
// the diagonal (earlier tokens for the block-masked variant); Q, Kr and Kw
// the unit-normalised queries, read keys and write keys when asked.
struct ChunkProductsTcArgs {
    float *Sw, *Vnw, *dSw, *Bw, *Uw, *Ww;  // [ci][128][128], [ci][64][128], [ci][128][128] x 2, [ci][64][128] x 2
    const float *Pw, *Tw, *Gw;             // [ci][64][64] x 2, [ci][64]
    const unsigned short *q, *k, *beta;    // bf16 bits: k and beta per sub-row (GDN / DeltaProduct) or per token
    const unsigned short *dout;            // [BH][T][128] bf16 bits of dO
    const float *mask;                     // [r][r] (block-masked)
    int BH, NT, T, Ct, r, masked, l2;      // Ct: query rows (tokens) per chunk, Ct = 64 / r
    float scale;
    int nq2;                               // set by the launcher
    unsigned long long timeout_ns;         // set by the launcher
};
int launch_chunk_products_tc(const ChunkProductsTcArgs &a, cudaStream_t stream);

// Chunk-local WY factors on tcgen05 (bf16, Dk = Dv = 128, 64-row chunks of
// Ct = 64 / r tokens, r in {1, 2, 4, 8}), for the block-masked DeltaProduct
// forward (masked = 1, bwd = 0) and for the backward passes of the chunk GDN /
// DeltaProduct (masked = 0, bwd = 1) and of the block-masked variant (masked =
// 1, bwd = 1).  Per (head, chunk) ci it writes W and Kd as the tensor-core
// chain's bf16 hi | lo operand images (32 KB each, in the W and Kd slots), U
// [64][128], P [64][64] and gamma [64] in fp32; the backward also T [64][64],
// K K^T (read keys against write keys) [64][64] and B [128][128].  The
// output kernel of the block-masked forward reads S [128][128], Vn [64][128],
// P and gamma and writes o.
struct WyTcArgs {
    const unsigned short *q, *k, *v, *beta;  // bf16 bits; k, v, beta per sub-row (GDN / DeltaProduct) or per token
    const unsigned short *dout;              // [BH][T][128] bf16 bits (backward)
    const float *g, *mask;                   // [BH][T] log-decays, [r][r] (block-masked)
    unsigned short *o;                       // [BH][T][128] bf16 bits (block-masked output kernel)
    float *Tw, *Ww, *Uw, *Kdw, *Bw, *Vnw, *Sw, *Pw, *KKw, *Gw;
    int BH, T, r, Ct, NT, l2, masked, bwd;
    float scale;
    unsigned long long timeout_ns;  // set by the launchers
};
int launch_wy_tc(const WyTcArgs &a, cudaStream_t stream);
int launch_masked_out_tc(const WyTcArgs &a, cudaStream_t stream);
// Reads and clears the error word of the chain kernel (GDN_OK or GDN_ERR_TIMEOUT).
int wy_chain_tc_read_clear_error();

// Counts one kernel launch (thread-safe); read by gdn_launch_count().
void note_launch();

}  // namespace gdn
