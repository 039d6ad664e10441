// gdn_api.cu -- the extern "C" boundary of libgdn.so: host-side argument
// checks, dispatch between the tcgen05 and SIMT scan paths, status strings.
// No allocation, no synchronisation, no exception crosses this file.  Every
// compute entry point opens an NVTX range named after itself around its
// checks and launches (header-only NVTX 3: a no-op unless a tool such as
// Nsight Compute or Nsight Systems is attached), so a profiler can select a
// call's kernels by range (ncu --nvtx --nvtx-include "gdn_chunk_fwd/").
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <atomic>

#include "gdn_internal.h"

namespace gdn {
namespace {
std::atomic<unsigned long long> g_launches{0};
}
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace gdn

namespace {

// An NVTX range over the enclosing scope.
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_scan(const gdn::ScanArgs &a) {
    if (a.B < 0 || a.H < 0 || a.T < 0 || a.r < 1) return GDN_ERR_INVALID_ARG;
    if (a.dtype != GDN_F32 && a.dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (a.flags & ~(GDN_QK_L2NORM | GDN_PATH_SIMT)) return GDN_ERR_INVALID_ARG;
    if (a.chunk <= 0) return GDN_ERR_INVALID_ARG;
    if (a.chunk != 16 && a.chunk != 32 && a.chunk != 64) return GDN_ERR_UNSUPPORTED;
    if (a.r > 8) return GDN_ERR_UNSUPPORTED;
    if ((a.Dk != 64 && a.Dk != 128) || (a.Dv != 64 && a.Dv != 128)) return GDN_ERR_UNSUPPORTED;
    if ((long long)a.B * a.H > 65535) return GDN_ERR_UNSUPPORTED;  // grid.y limit
    if ((long long)a.T * a.r > (1LL << 30)) return GDN_ERR_UNSUPPORTED;
    const bool empty = (long long)a.B * a.H * a.T == 0;
    if (!empty) {
        if (!a.q || !a.k || !a.v || !a.beta || !a.g || !a.o) return GDN_ERR_INVALID_ARG;
        const void *ps[] = {a.q, a.k, a.v, a.beta, a.g, a.o};
        for (const void *p : ps)
            if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    }
    if ((a.s0 && !aligned16(a.s0)) || (a.sf && !aligned16(a.sf))) return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

size_t scan_workspace(const gdn::ScanArgs &a) {
    return gdn::scan_tc_supported(a) ? gdn::scan_tc_workspace_bytes(a) : 0;
}

// need_ws = false lets a call without enough workspace run anyway: the
// tensor-core path then takes its cluster mode, which needs no scratch.
int run_scan(gdn::ScanArgs &a, void *stream_v, bool need_ws = true) {
    int st = check_scan(a);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const size_t need = scan_workspace(a);
    if (need_ws && need > 0 && (a.ws == nullptr || a.ws_bytes < need)) return GDN_ERR_WORKSPACE;
    if ((long long)a.B * a.H == 0) return GDN_OK;
    if (a.T == 0) {
        if (a.sf) {
            const size_t bytes = sizeof(float) * (size_t)a.B * a.H * a.Dk * a.Dv;
            cudaError_t e = a.s0 ? cudaMemcpyAsync(a.sf, a.s0, bytes, cudaMemcpyDeviceToDevice, stream)
                                 : cudaMemsetAsync(a.sf, 0, bytes, stream);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    if (gdn::scan_tc_supported(a)) return gdn::launch_scan_tc(a, stream);
    return gdn::launch_scan_simt(a, stream);
}

int check_cam_scan(const gdn::CamScanArgs &a) {
    if (a.B < 0 || a.H < 0 || a.F < 0 || a.S < 0) return GDN_ERR_INVALID_ARG;
    if (a.F > 0 && a.S == 0) return GDN_ERR_INVALID_ARG;  // a frame holds at least one token
    if (a.dtype != GDN_F32 && a.dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (a.flags & ~(GDN_QK_L2NORM | GDN_PATH_SIMT | GDN_CAM_REVERSE)) return GDN_ERR_INVALID_ARG;
    if ((a.Dk != 64 && a.Dk != 128) || (a.Dv != 64 && a.Dv != 128)) return GDN_ERR_UNSUPPORTED;
    if ((a.flags & GDN_CAM_REVERSE) && (a.s0 || a.sf)) return GDN_ERR_UNSUPPORTED;
    if ((long long)a.B * a.H > 65535 || (long long)a.F * a.S >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if ((long long)a.B * a.H * a.F != 0) {
        if (!a.q || !a.k || !a.v || !a.beta || !a.decay || !a.o) return GDN_ERR_INVALID_ARG;
        const void *ps[] = {a.q, a.k, a.v, a.beta, a.decay, a.o};
        for (const void *p : ps)
            if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    }
    if ((a.s0 && !aligned16(a.s0)) || (a.sf && !aligned16(a.sf))) return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
        default: return "GDN_ERR_UNKNOWN";
    }
}

int gdn_version(void) { return 100; }

size_t gdn_chunk_fwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int chunk,
                                     int dtype) {
    gdn::ScanArgs a{};
    a.B = B; a.H = H; a.T = T; a.r = r; a.Dk = Dk; a.Dv = Dv; a.chunk = chunk;
    a.dtype = dtype; a.scale = 1.f;
    // pointer checks do not apply to a size query
    if (B < 0 || H < 0 || T < 0 || r < 1 || chunk <= 0) return (size_t)-1;
    if ((chunk != 16 && chunk != 32 && chunk != 64) || r > 8) return (size_t)-1;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return (size_t)-1;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return (size_t)-1;
    return scan_workspace(a);
}

int gdn_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                  const float *g, const float *initial_state, void *o, float *final_state,
                  int B, int H, int T, int Dk, int Dv, int chunk, float scale,
                  unsigned flags, int dtype, void *workspace, size_t workspace_bytes,
                  void *stream) {
    const Range nvtx_range("gdn_chunk_fwd");
    gdn::ScanArgs a{q, k, v, beta, g, initial_state, o, final_state, B, H, T, 1, Dk, Dv,
                    chunk, scale, flags, dtype, workspace, workspace_bytes};
    return run_scan(a, stream);
}

int gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *beta,
                          const float *g, const float *initial_state, void *o, float *final_state,
                          int B, int H, int T, int Dk, int Dv, int chunk, float scale,
                          unsigned flags, int dtype, void *stream) {
    const Range nvtx_range("gdn_chunk_fwd_noalloc");
    // gdn_chunk_fwd with the library's own fixed scratch in place of a
    // caller-provided workspace; nothing is allocated
    gdn::ScanArgs a{q, k, v, beta, g, initial_state, o, final_state, B, H, T, 1, Dk, Dv,
                    chunk, scale, flags, dtype, nullptr, 0};
    const int st = check_scan(a);
    if (st != GDN_OK) return st;
    if (scan_workspace(a) > 0) {
        void *ws = nullptr;
        size_t bytes = 0;
        const int ss = gdn::scan_tc_noalloc_scratch(&ws, &bytes);
        if (ss != GDN_OK) return ss;
        // more heads than the array's ring serves: no scratch, so the
        // tensor-core path runs in its cluster mode
        if (scan_workspace(a) <= bytes) {
            a.ws = ws;
            a.ws_bytes = bytes;
        }
    }
    return run_scan(a, stream, false);
}

int deltaproduct_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                           const float *g, const float *initial_state, void *o,
                           float *final_state, int B, int H, int T, int r, int Dk, int Dv,
                           int chunk, float scale, unsigned flags, int dtype, void *workspace,
                           size_t workspace_bytes, void *stream) {
    const Range nvtx_range("deltaproduct_chunk_fwd");
    gdn::ScanArgs a{q, k, v, beta, g, initial_state, o, final_state, B, H, T, r, Dk, Dv,
                    chunk, scale, flags, dtype, workspace, workspace_bytes};
    return run_scan(a, stream);
}

size_t masked_deltaproduct_chunk_fwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int dtype) {
    if (B < 0 || H < 0 || T < 0 || r < 1 || r > 8 || 64 % r != 0) return (size_t)-1;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128) || Dk % r != 0) return (size_t)-1;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return (size_t)-1;
    gdn::MaskedDpArgs a{};
    a.B = B; a.H = H; a.T = T; a.r = r; a.Dk = Dk; a.Dv = Dv; a.dtype = dtype;
    return gdn::masked_dp_workspace_bytes(a);
}

int masked_deltaproduct_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                                  const float *g, const float *mask, const float *initial_state, void *o,
                                  float *final_state, int B, int H, int T, int r, int Dk, int Dv, int chunk,
                                  float scale, unsigned flags, int dtype, void *workspace, size_t workspace_bytes,
                                  void *stream_v) {
    const Range nvtx_range("masked_deltaproduct_chunk_fwd");
    if (B < 0 || H < 0 || T < 0 || r < 1) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (flags & ~(GDN_QK_L2NORM | GDN_PATH_SIMT)) return GDN_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return chunk <= 0 ? GDN_ERR_INVALID_ARG : GDN_ERR_UNSUPPORTED;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return GDN_ERR_UNSUPPORTED;
    if (r > 8 || Dk % r != 0 || chunk % r != 0) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H * T != 0) {
        if (!q || !k || !v || !beta || !g || !mask || !o) return GDN_ERR_INVALID_ARG;
        const void *ps[] = {q, k, v, beta, g, mask, o};
        for (const void *p : ps)
            if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    }
    if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
        return GDN_ERR_MISALIGNED;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if ((long long)B * H == 0) return GDN_OK;
    if (T == 0) {
        if (final_state) {
            const size_t bytes = sizeof(float) * (size_t)B * H * Dk * Dv;
            cudaError_t e = initial_state
                                ? cudaMemcpyAsync(final_state, initial_state, bytes, cudaMemcpyDeviceToDevice, stream)
                                : cudaMemsetAsync(final_state, 0, bytes, stream);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    gdn::MaskedDpArgs a{q, k, v, beta, g, mask, initial_state, o, final_state, B, H, T, r, Dk, Dv, chunk,
                        scale, flags, dtype, workspace, workspace_bytes};
    const size_t need = gdn::masked_dp_workspace_bytes(a);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return GDN_ERR_WORKSPACE;
    return gdn::launch_masked_dp(a, stream);
}

size_t cam_scan_fwd_workspace_bytes(int B, int H, int F, int S, int Dk, int Dv, int dtype) {
    gdn::CamScanArgs a{};
    a.B = B; a.H = H; a.F = F; a.S = S; a.Dk = Dk; a.Dv = Dv; a.dtype = dtype; a.scale = 1.f;
    if (B < 0 || H < 0 || F < 0 || S < 0 || (F > 0 && S == 0)) return (size_t)-1;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return (size_t)-1;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return (size_t)-1;
    return gdn::cam_scan_workspace_bytes(a);
}

int cam_scan_fwd(const void *q, const void *k, const void *v, const void *beta, const float *decay,
                 const float *initial_state, void *o, float *final_state, int B, int H, int F, int S,
                 int Dk, int Dv, float scale, unsigned flags, int dtype, void *workspace,
                 size_t workspace_bytes, void *stream_v) {
    const Range nvtx_range("cam_scan_fwd");
    gdn::CamScanArgs a{q, k, v, beta, decay, initial_state, o, final_state, B, H, F, S, Dk, Dv,
                       scale, flags, dtype, workspace, workspace_bytes};
    const int st = check_cam_scan(a);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const size_t need = gdn::cam_scan_workspace_bytes(a);
    if (need > 0 && (a.ws == nullptr || a.ws_bytes < need || !aligned16(a.ws))) return GDN_ERR_WORKSPACE;
    if ((long long)B * H == 0) return GDN_OK;
    if (F == 0) {
        if (final_state) {
            const size_t bytes = sizeof(float) * (size_t)B * H * Dk * Dv;
            cudaError_t e = initial_state
                                ? cudaMemcpyAsync(final_state, initial_state, bytes, cudaMemcpyDeviceToDevice, stream)
                                : cudaMemsetAsync(final_state, 0, bytes, stream);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    return gdn::launch_cam_scan(a, stream);
}

size_t cam_prep_scan_fwd_workspace_bytes(int B, int N, int H, int D, int F, int dtype) {
    if (B < 0 || N < 0 || H < 1 || F < 1 || N % F != 0) return (size_t)-1;
    if (dtype != GDN_BF16 || D != 128 || (long long)H * D > 4096) return (size_t)-1;
    gdn::CamFusedArgs a{};
    a.B = B; a.H = H; a.F = F; a.S = N / F;
    return gdn::cam_fused_workspace_bytes(a);
}

int cam_prep_scan_fwd(const void *q_raw, const void *k_raw, const void *v_raw, const float *q_norm_w,
                      const float *k_norm_w, const float *proj_q, const float *proj_kv, float rope_base,
                      const void *beta, const float *decay, const float *initial_state, void *o,
                      float *final_state, int B, int N, int H, int D, int F, float k_scale, float eps, float scale,
                      unsigned flags, int dtype, void *workspace, size_t workspace_bytes, void *stream_v) {
    const Range nvtx_range("cam_prep_scan_fwd");
    if (B < 0 || N < 0 || H < 1 || F < 1) return GDN_ERR_INVALID_ARG;
    if (N % F != 0 || (N > 0 && N / F == 0)) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (flags & ~(GDN_QK_L2NORM | GDN_CAM_REVERSE)) return GDN_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (!(rope_base > 0.f)) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 || D != 128 || (long long)H * D > 4096) return GDN_ERR_UNSUPPORTED;
    if ((flags & GDN_CAM_REVERSE) && (initial_state || final_state)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535 || (long long)N * H * D >= (1LL << 40)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * N != 0) {
        if (!q_raw || !k_raw || !v_raw || !proj_q || !proj_kv || !beta || !decay || !o) return GDN_ERR_INVALID_ARG;
    }
    const void *ps[] = {q_raw, k_raw, v_raw, q_norm_w, k_norm_w, proj_q, proj_kv, beta, decay, initial_state, o,
                        final_state};
    for (const void *p : ps)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::CamFusedArgs a{q_raw, k_raw, v_raw, q_norm_w, k_norm_w, proj_q, proj_kv, rope_base, beta, decay,
                        initial_state, o, final_state, B, H, F, N / F, k_scale, eps, scale, flags, workspace,
                        workspace_bytes};
    const size_t need = gdn::cam_fused_workspace_bytes(a);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return GDN_ERR_WORKSPACE;
    if ((long long)B * N == 0) return GDN_OK;
    return gdn::launch_cam_fused(a, static_cast<cudaStream_t>(stream_v));
}

int cam_prep_fwd(const void *q_raw, const void *k_raw, const void *v_raw, const float *q_norm_w,
                 const float *k_norm_w, const float *proj_q, const float *proj_kv,
                 const float *rope_cos, const float *rope_sin, float rope_base, void *q_out,
                 void *k_out, void *v_out, float *k_pre_sq, float *k_post_sq, int B, int N,
                 int H, int D, float k_scale, float eps, int dtype, void *stream) {
    const Range nvtx_range("cam_prep_fwd");
    if (B < 0 || N < 0 || H < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if ((rope_cos == nullptr) != (rope_sin == nullptr)) return GDN_ERR_INVALID_ARG;
    if (D % 2 != 0 || (D / 2) % 4 != 0) return GDN_ERR_INVALID_ARG;  // page's own rule
    if (D % 16 != 0 || 32 % (D / 8) != 0 || D > 256) return GDN_ERR_UNSUPPORTED;
    if ((long long)H * D > 4096 || H > 64) return GDN_ERR_UNSUPPORTED;
    if (!(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if ((long long)B * N == 0 || H == 0) return GDN_OK;
    if (!q_raw || !k_raw || !v_raw || !proj_q || !proj_kv || !q_out || !k_out || !v_out)
        return GDN_ERR_INVALID_ARG;
    const void *ps[] = {q_raw, k_raw, v_raw, proj_q, proj_kv, q_out, k_out, v_out,
                        q_norm_w, k_norm_w, rope_cos, rope_sin, k_pre_sq, k_post_sq};
    for (const void *p : ps)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if (rope_cos == nullptr && !(rope_base > 0.f)) return GDN_ERR_INVALID_ARG;
    gdn::CamArgs a{q_raw, k_raw, v_raw, q_norm_w, k_norm_w, proj_q, proj_kv, rope_cos, rope_sin,
                   rope_base, q_out, k_out, v_out, k_pre_sq, k_post_sq, B, N, H, D, k_scale, eps,
                   dtype};
    return gdn::launch_cam_prep(a, static_cast<cudaStream_t>(stream));
}

size_t cam_scan_bwd_workspace_bytes(int B, int H, int F, int S, int Dk, int Dv, int dtype) {
    if (B < 0 || H < 0 || F < 0 || S < 0 || (F > 0 && S == 0)) return (size_t)-1;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return (size_t)-1;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return (size_t)-1;
    gdn::CamScanBwdArgs a{};
    a.B = B; a.H = H; a.F = F; a.S = S; a.Dk = Dk; a.Dv = Dv; a.dtype = dtype;
    return gdn::cam_scan_bwd_workspace_bytes(a);
}

int cam_scan_bwd(const void *q, const void *k, const void *v, const void *beta, const float *decay,
                 const float *initial_state, const void *dout, const float *dfinal_state, void *dq, void *dk,
                 void *dv, float *dbeta, float *ddecay, float *dinitial_state, int B, int H, int F, int S, int Dk,
                 int Dv, float scale, unsigned flags, int dtype, void *workspace, size_t workspace_bytes,
                 void *stream) {
    const Range nvtx_range("cam_scan_bwd");
    if (B < 0 || H < 0 || F < 0 || S < 0 || (F > 0 && S == 0)) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (flags & ~(GDN_QK_L2NORM | GDN_CAM_REVERSE | GDN_PATH_SIMT)) return GDN_ERR_INVALID_ARG;
    if (flags & GDN_CAM_REVERSE) return GDN_ERR_UNSUPPORTED;  // forward direction only
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535 || (long long)F * S >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H * F != 0) {
        if (!q || !k || !v || !beta || !decay || !dout || !dq || !dk || !dv || !dbeta || !ddecay)
            return GDN_ERR_INVALID_ARG;
    }
    const void *ps[] = {q, k, v, beta, decay, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, ddecay,
                        dinitial_state};
    for (const void *p : ps)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::CamScanBwdArgs a{q, k, v, beta, decay, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, ddecay,
                          dinitial_state, B, H, F, S, Dk, Dv, scale, flags, dtype, workspace, workspace_bytes};
    const size_t need = gdn::cam_scan_bwd_workspace_bytes(a);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return GDN_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((long long)B * H == 0) return GDN_OK;
    if (F == 0) {  // nothing depends on the inputs: the initial state's gradient is the final state's
        if (dinitial_state) {
            const size_t bytes = sizeof(float) * (size_t)B * H * Dk * Dv;
            cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, bytes,
                                                           cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(dinitial_state, 0, bytes, st);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    return gdn::launch_cam_scan_bwd(a, st);
}

int cam_prep_bwd(const void *q_raw, const void *k_raw, const float *q_norm_w, const float *k_norm_w,
                 const float *proj_q, const float *proj_kv, const float *rope_cos, const float *rope_sin,
                 float rope_base, const void *dq_out, const void *dk_out, const void *dv_out,
                 const float *dk_pre_sq, const float *dk_post_sq, void *dq_raw, void *dk_raw, void *dv_raw, int B,
                 int N, int H, int D, float k_scale, float eps, int dtype, void *stream) {
    const Range nvtx_range("cam_prep_bwd");
    if (B < 0 || N < 0 || H < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if ((rope_cos == nullptr) != (rope_sin == nullptr)) return GDN_ERR_INVALID_ARG;
    if (D % 2 != 0 || (D / 2) % 4 != 0) return GDN_ERR_INVALID_ARG;
    if (D % 16 != 0 || (long long)H * D > 4096) return GDN_ERR_UNSUPPORTED;
    if (!(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (rope_cos == nullptr && !(rope_base > 0.f)) return GDN_ERR_INVALID_ARG;
    if ((long long)B * N == 0 || H == 0) return GDN_OK;
    if ((long long)B * N > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    if (!q_raw || !k_raw || !proj_q || !proj_kv || !dq_out || !dk_out || !dv_out || !dq_raw || !dk_raw || !dv_raw)
        return GDN_ERR_INVALID_ARG;
    const void *ps[] = {q_raw, k_raw, q_norm_w, k_norm_w, proj_q, proj_kv, rope_cos, rope_sin, dq_out, dk_out,
                        dv_out, dk_pre_sq, dk_post_sq, dq_raw, dk_raw, dv_raw};
    for (const void *p : ps)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::CamBwdArgs a{q_raw, k_raw, q_norm_w, k_norm_w, proj_q, proj_kv, rope_cos, rope_sin, rope_base, dq_out,
                      dk_out, dv_out, dk_pre_sq, dk_post_sq, dq_raw, dk_raw, dv_raw, B, N, H, D, k_scale, eps, dtype};
    return gdn::launch_cam_prep_bwd(a, static_cast<cudaStream_t>(stream));
}

size_t gdn_chunk_bwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int dtype) {
    if (B < 0 || H < 0 || T < 0 || r < 1 || r > 8) return (size_t)-1;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return (size_t)-1;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return (size_t)-1;
    gdn::ChunkBwdArgs a{};
    a.B = B; a.H = H; a.T = T; a.r = r; a.Dk = Dk; a.Dv = Dv;
    return gdn::chunk_bwd_workspace_bytes(a);
}

int deltaproduct_chunk_bwd(const void *q, const void *k, const void *v, const void *beta, const float *g,
                           const float *initial_state, const void *dout, const float *dfinal_state, void *dq,
                           void *dk, void *dv, float *dbeta, float *dg, float *dinitial_state, int B, int H, int T,
                           int r, int Dk, int Dv, float scale, unsigned flags, int dtype, void *workspace,
                           size_t workspace_bytes, void *stream) {
    const Range nvtx_range("deltaproduct_chunk_bwd");
    if (B < 0 || H < 0 || T < 0 || r < 1 || r > 8) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (flags & ~(GDN_QK_L2NORM | GDN_PATH_SIMT)) return GDN_ERR_INVALID_ARG;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535 || (long long)T * r >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H * T != 0) {
        if (!q || !k || !v || !beta || !g || !dout || !dq || !dk || !dv || !dbeta || !dg)
            return GDN_ERR_INVALID_ARG;
    }
    const void *ps[] = {q, k, v, beta, g, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, dg,
                        dinitial_state};
    for (const void *p : ps)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::ChunkBwdArgs a{q, k, v, beta, g, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, dg,
                        dinitial_state, B, H, T, r, Dk, Dv, scale, flags, dtype, workspace, workspace_bytes};
    const size_t need = gdn::chunk_bwd_workspace_bytes(a);
    if ((long long)B * H * T != 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return GDN_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((long long)B * H == 0) return GDN_OK;
    if (T == 0) {  // the initial state's gradient is the final state's
        if (dinitial_state) {
            const size_t bytes = sizeof(float) * (size_t)B * H * Dk * Dv;
            cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, bytes,
                                                           cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(dinitial_state, 0, bytes, st);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    return gdn::launch_chunk_bwd(a, st);
}

int gdn_chunk_bwd(const void *q, const void *k, const void *v, const void *beta, const float *g,
                  const float *initial_state, const void *dout, const float *dfinal_state, void *dq, void *dk,
                  void *dv, float *dbeta, float *dg, float *dinitial_state, int B, int H, int T, int Dk, int Dv,
                  float scale, unsigned flags, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
    const Range nvtx_range("gdn_chunk_bwd");
    return deltaproduct_chunk_bwd(q, k, v, beta, g, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, dg,
                                  dinitial_state, B, H, T, 1, Dk, Dv, scale, flags, dtype, workspace,
                                  workspace_bytes, stream);
}

size_t masked_deltaproduct_chunk_bwd_workspace_bytes(int B, int H, int T, int r, int Dk, int Dv, int dtype) {
    if (B < 0 || H < 0 || T < 0 || r < 1 || r > 8 || 64 % r != 0) return (size_t)-1;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128) || Dk % r != 0) return (size_t)-1;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return (size_t)-1;
    gdn::MaskedBwdArgs a{};
    a.B = B; a.H = H; a.T = T; a.r = r; a.Dk = Dk; a.Dv = Dv; a.dtype = dtype;
    return gdn::masked_bwd_workspace_bytes(a);
}

int masked_deltaproduct_chunk_bwd(const void *q, const void *k, const void *v, const void *beta, const float *g,
                                  const float *mask, const float *initial_state, const void *dout,
                                  const float *dfinal_state, void *dq, void *dk, void *dv, float *dbeta, float *dg,
                                  float *dinitial_state, int B, int H, int T, int r, int Dk, int Dv, float scale,
                                  unsigned flags, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
    const Range nvtx_range("masked_deltaproduct_chunk_bwd");
    if (B < 0 || H < 0 || T < 0 || r < 1) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (flags & ~(GDN_QK_L2NORM | GDN_PATH_SIMT)) return GDN_ERR_INVALID_ARG;
    if ((Dk != 64 && Dk != 128) || (Dv != 64 && Dv != 128)) return GDN_ERR_UNSUPPORTED;
    if (r > 8 || 64 % r != 0 || Dk % r != 0) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535 || (long long)T * r >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H * T != 0) {
        if (!q || !k || !v || !beta || !g || !mask || !dout || !dq || !dk || !dv || !dbeta || !dg)
            return GDN_ERR_INVALID_ARG;
    }
    const void *ps[] = {q, k, v, beta, g, mask, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, dg,
                        dinitial_state};
    for (const void *p : ps)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::MaskedBwdArgs a{q, k, v, beta, g, mask, initial_state, dout, dfinal_state, dq, dk, dv, dbeta, dg,
                         dinitial_state, B, H, T, r, Dk, Dv, scale, flags, dtype, workspace, workspace_bytes};
    const size_t need = gdn::masked_bwd_workspace_bytes(a);
    if ((long long)B * H * T != 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return GDN_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((long long)B * H == 0) return GDN_OK;
    if (T == 0) {  // the initial state's gradient is the final state's
        if (dinitial_state) {
            const size_t bytes = sizeof(float) * (size_t)B * H * Dk * Dv;
            cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, bytes,
                                                           cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(dinitial_state, 0, bytes, st);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    return gdn::launch_masked_bwd(a, st);
}

int gdn_get_device_error(void *stream) {
    const int a = gdn::scan_tc_read_clear_error(static_cast<cudaStream_t>(stream));
    const int b = gdn::cam_prep_read_clear_error();
    const int c = gdn::cam_scan_read_clear_error();
    const int d = gdn::cam_scan_bwd_read_clear_error();
    const int e = gdn::wy_chain_tc_read_clear_error();
    const int r[] = {a, b, c, d, e};
    for (int x : r)
        if (x != GDN_OK) return x;
    return GDN_OK;
}

unsigned long long gdn_launch_count(void) { return gdn::g_launches.load(); }

int gdn_set_wait_limit(unsigned long long us) { return gdn::scan_tc_set_wait_limit(us); }

int gdn_set_cluster_shape(int heads_per_cluster, int wy_ctas_per_cluster) {
    return gdn::scan_tc_set_cluster_shape(heads_per_cluster, wy_ctas_per_cluster);
}

}  // extern "C"
