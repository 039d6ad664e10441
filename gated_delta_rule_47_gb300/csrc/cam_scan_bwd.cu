// cam_scan_bwd.cu -- backward of the frame-level camera scan, forward direction
// (fused_cam_gdn.py, `_cam_scan_bwd_kernel`), on the CUDA cores in fp32.
//
// Per (batch, head) the N = F*S tokens form F frames of S tokens.  With E_f
// the state entering frame f, d_f its decay factor, G_f = K^T diag(beta) K
// and H_f = K^T diag(beta) V over the frame's tokens, the frame's update is
//     X_f = d_f (I - G_f) E_f + H_f      (= E_{f+1}),   o_t = scale X_f^T q_t.
// With dX_f the gradient of X_f, dE_F the final state's gradient and
// P_f = scale Q_f^T dO_f:
//     dX_f = dE_{f+1} + P_f,   dE_f = d_f (I - G_f) dX_f      (G_f is symmetric)
// and per token t of frame f, with dR_t = dX_f^T k_t and KE_t = E_f^T k_t:
//     dv_t = beta_t dR_t;   dbeta_t = dR_t . (v_t - d_f KE_t)
//     dk_t = dX_f r_t - d_f beta_t E_f dR_t,   r_t = beta_t (v_t - d_f KE_t)
//     dq_t = scale X_f do_t
//     ddecay_f = <dX_f, E_f> - sum_t beta_t dR_t . KE_t
// and, with the unit-norm flag, the unit-norm map's adjoint on q and k.
//
// Four launches:
//   1. fb_frame_kernel (one CTA per frame, head and product): G_f, H_f and P_f
//      as sums over the frame's 64-token tiles.
//   2. fb_chain_kernel: the states E_f (forward) and the gradients dX_f
//      (reverse, down to the initial state's) side by side, each CTA holding
//      32 value columns of one head.
//   3. fb_token_kernel (one CTA per 64-token tile of a frame): every token's
//      gradients, and the tile's share of ddecay.
//   4. fb_decay_kernel: each frame's ddecay, its tiles' shares summed in order.
#include "gdn_internal.h"
#include "simt_tile.cuh"

namespace gdn {
namespace {

using namespace tile;
constexpr int kFChainThr = 256;
constexpr int kSl = 32;  // value columns per chain CTA
constexpr int LSl = kSl + 1;

struct FbParams {
    const void *q, *k, *v, *beta, *dout;
    const float *decay, *s0, *dsf;
    void *dq, *dk, *dv;
    float *dbeta, *ddecay, *ds0;
    // workspace: G [BH][F][Dk][Dk], H and P [BH][F][Dk][Dv], E [BH][F+1][Dk][Dv],
    // dX [BH][F][Dk][Dv], ddecay shares [BH][F][tiles per frame]
    float *Gw, *Hw, *Pw, *Ew, *dXw, *part;
    int F, S, N, tiles;
    float scale;
    int l2;
};

// ======================================== 1. the frame products G, H and P
// blockIdx.x: frame; blockIdx.y: head; blockIdx.z: 0 = G, 1 = H, 2 = P.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) fb_frame_kernel(FbParams p) {
    extern __shared__ float sm[];
    constexpr int LK = DK + 1, LV = DV + 1;
    float *As = sm;             // [64][LK]  k (G, H) or q (P) rows
    float *Bs = As + kC * LK;   // [64][LK or LV]  beta k, beta v or do rows
    float *bet = Bs + kC * LK;  // [64]
    float *nrm = bet + kC;      // [64]
    const int f = blockIdx.x, bh = blockIdx.y, part = blockIdx.z, tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const size_t tok0 = (size_t)bh * p.N + (size_t)f * p.S;
    const bool l2 = p.l2 != 0;
    if (part == 0) {
        float acc[DK / 32][DK / 16];
        zero(acc);
        for (int t0 = 0; t0 < p.S; t0 += kC) {
            const int n = min(kC, p.S - t0);
            load_rows<T, DK>(As, (const T *)p.k + (tok0 + t0) * DK, n, l2, nrm);
            if (tid < kC) bet[tid] = tid < n ? ld_f((const T *)p.beta + tok0 + t0 + tid) : 0.f;
            __syncthreads();
            for (int e = tid; e < kC * DK; e += kThr) Bs[(e / DK) * LK + e % DK] = bet[e / DK] * As[(e / DK) * LK + e % DK];
            __syncthreads();
            mm<kThr, DK / 32, DK / 16>(acc, As, 1, LK, Bs, LK, 1, kC);
            __syncthreads();
        }
        float *out = p.Gw + ((size_t)bh * p.F + f) * DK * DK;
#pragma unroll
        for (int i = 0; i < DK / 32; ++i)
#pragma unroll
            for (int j = 0; j < DK / 16; ++j) out[(ty + 32 * i) * DK + tx + 16 * j] = acc[i][j];
    } else {
        float acc[DK / 32][DV / 16];
        zero(acc);
        for (int t0 = 0; t0 < p.S; t0 += kC) {
            const int n = min(kC, p.S - t0);
            if (part == 1) {
                load_rows<T, DK>(As, (const T *)p.k + (tok0 + t0) * DK, n, l2, nrm);
                load_rows<T, DV>(Bs, (const T *)p.v + (tok0 + t0) * DV, n, false, nullptr);
                if (tid < kC) bet[tid] = tid < n ? ld_f((const T *)p.beta + tok0 + t0 + tid) : 0.f;
                __syncthreads();
                for (int e = tid; e < kC * DV; e += kThr) Bs[(e / DV) * LV + e % DV] *= bet[e / DV];
            } else {
                load_rows<T, DK>(As, (const T *)p.q + (tok0 + t0) * DK, n, l2, nrm);
                load_rows<T, DV>(Bs, (const T *)p.dout + (tok0 + t0) * DV, n, false, nullptr);
            }
            __syncthreads();
            mm<kThr, DK / 32, DV / 16>(acc, As, 1, LK, Bs, LV, 1, kC);
            __syncthreads();
        }
        const float s = part == 2 ? p.scale : 1.f;
        float *out = (part == 1 ? p.Hw : p.Pw) + ((size_t)bh * p.F + f) * DK * DV;
#pragma unroll
        for (int i = 0; i < DK / 32; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) out[(ty + 32 * i) * DV + tx + 16 * j] = s * acc[i][j];
    }
}

// ================================================================ 2. chains
// blockIdx.x: 32-column slice; blockIdx.y: head; blockIdx.z: 0 = states,
// 1 = gradients.
template <int DK, int DV>
__global__ void __launch_bounds__(kFChainThr) fb_chain_kernel(FbParams p) {
    extern __shared__ float sm[];
    constexpr int LK = DK + 1;
    float *Gs = sm;             // [DK][LK]
    float *St = Gs + DK * LK;   // [DK][LSl]
    const int col0 = blockIdx.x * kSl, bh = blockIdx.y, role = blockIdx.z;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, F = p.F;
    const float *init = role == 0 ? p.s0 : p.dsf;
    for (int e = tid; e < DK * kSl; e += kFChainThr) {
        const int m = e / kSl, n = e % kSl;
        St[m * LSl + n] = init ? init[((size_t)bh * DK + m) * DV + col0 + n] : 0.f;
    }
    __syncthreads();
    for (int s = 0; s < F; ++s) {
        const int f = role == 0 ? s : F - 1 - s;
        const size_t fi = (size_t)bh * F + f;
        const float d = p.decay[fi];
        if (role == 0) {  // E_f out
            float *Eg = p.Ew + ((size_t)bh * (F + 1) + f) * DK * DV;
            for (int e = tid; e < DK * kSl; e += kFChainThr) {
                const int m = e / kSl, n = e % kSl;
                Eg[(size_t)m * DV + col0 + n] = St[m * LSl + n];
            }
        } else {  // dX_f = dE_{f+1} + P_f, out
            const float *Pg = p.Pw + fi * DK * DV;
            float *dXg = p.dXw + fi * DK * DV;
            for (int e = tid; e < DK * kSl; e += kFChainThr) {
                const int m = e / kSl, n = e % kSl;
                const float x = St[m * LSl + n] + Pg[(size_t)m * DV + col0 + n];
                St[m * LSl + n] = x;
                dXg[(size_t)m * DV + col0 + n] = x;
            }
        }
        const float *Gg = p.Gw + fi * DK * DK;
        for (int e = tid; e < DK * DK; e += kFChainThr) Gs[(e / DK) * LK + e % DK] = Gg[e];
        __syncthreads();
        float acc[DK / 16][2];
        zero(acc);
        mm<kFChainThr, DK / 16, 2>(acc, Gs, LK, 1, St, LSl, 1, DK);
        __syncthreads();
        const float *Hg = p.Hw + fi * DK * DV;
#pragma unroll
        for (int i = 0; i < DK / 16; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int m = ty + 16 * i, n = tx + 16 * j;
                const float x = d * (St[m * LSl + n] - acc[i][j]);
                St[m * LSl + n] = role == 0 ? x + Hg[(size_t)m * DV + col0 + n] : x;
            }
        __syncthreads();
    }
    if (role == 0) {  // the state after the last frame
        float *Eg = p.Ew + ((size_t)bh * (F + 1) + F) * DK * DV;
        for (int e = tid; e < DK * kSl; e += kFChainThr) {
            const int m = e / kSl, n = e % kSl;
            Eg[(size_t)m * DV + col0 + n] = St[m * LSl + n];
        }
    } else if (p.ds0) {
        for (int e = tid; e < DK * kSl; e += kFChainThr) {
            const int m = e / kSl, n = e % kSl;
            p.ds0[((size_t)bh * DK + m) * DV + col0 + n] = St[m * LSl + n];
        }
    }
}

// =================================================== 3. the token gradients
// blockIdx.x: frame * tiles + tile; blockIdx.y: head.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) fb_token_kernel(FbParams p) {
    extern __shared__ float sm[];
    constexpr int LK = DK + 1, LV = DV + 1, TK = DK / 16, TV = DV / 16, NH = DK / 64;
    float *Ks = sm, *Qs = Ks + kC * LK, *dOs = Qs + kC * LK, *Rs = dOs + kC * LV, *dRs = Rs + kC * LV;
    float *Hs = dRs + kC * LV;                 // [64][LV] a 64-row block of E_f, dX_f or X_f
    float *bet = Hs + kC * LV, *nk = bet + kC, *nq = nk + kC, *dbr = nq + kC, *ddr = dbr + kC;
    float *red = ddr + kC;                     // [16]
    const int f = blockIdx.x / p.tiles, tl = blockIdx.x % p.tiles, bh = blockIdx.y;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = tl * kC, n = min(kC, p.S - t0);
    const size_t tok = (size_t)bh * p.N + (size_t)f * p.S + t0, fi = (size_t)bh * p.F + f;
    const float d = p.decay[fi];
    const float *Eg = p.Ew + ((size_t)bh * (p.F + 1) + f) * DK * DV;
    const float *Xg = Eg + (size_t)DK * DV;  // E_{f+1} = X_f
    const float *dXg = p.dXw + fi * DK * DV;
    const T *vp = (const T *)p.v + tok * DV;

    load_rows<T, DK>(Ks, (const T *)p.k + tok * DK, n, p.l2 != 0, nk);
    load_rows<T, DK>(Qs, (const T *)p.q + tok * DK, n, p.l2 != 0, nq);
    load_rows<T, DV>(dOs, (const T *)p.dout + tok * DV, n, false, nullptr);
    if (tid < kC) bet[tid] = tid < n ? ld_f((const T *)p.beta + tok + tid) : 0.f;

    // 1. KE = K E_f and dR = K dX_f
    float accKE[2][TV], accdR[2][TV];
    zero(accKE);
    zero(accdR);
    for (int h = 0; h < NH; ++h) {
        __syncthreads();
        for (int e = tid; e < 64 * DV; e += kThr) Hs[(e / DV) * LV + e % DV] = Eg[(size_t)64 * h * DV + e];
        __syncthreads();
        mm<kThr, 2, TV>(accKE, Ks + 64 * h, LK, 1, Hs, LV, 1, 64);
        __syncthreads();
        for (int e = tid; e < 64 * DV; e += kThr) Hs[(e / DV) * LV + e % DV] = dXg[(size_t)64 * h * DV + e];
        __syncthreads();
        mm<kThr, 2, TV>(accdR, Ks + 64 * h, LK, 1, Hs, LV, 1, 64);
    }
    // 2. r, dR to shared memory; dv; dbeta and the decay shares per row
    T *dvp = (T *)p.dv + tok * DV;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = ty + 32 * i;
        float sb = 0.f, sd = 0.f;
#pragma unroll
        for (int j = 0; j < TV; ++j) {
            const int c = tx + 16 * j;
            const float vv = t < n ? ld_f(vp + (size_t)t * DV + c) : 0.f;
            const float u = vv - d * accKE[i][j];
            Rs[t * LV + c] = bet[t] * u;
            dRs[t * LV + c] = accdR[i][j];
            sb += accdR[i][j] * u;
            sd += accdR[i][j] * accKE[i][j];
            if (t < n) st_f(dvp + (size_t)t * DV + c, bet[t] * accdR[i][j]);
        }
        sb = row_sum16(sb);
        sd = row_sum16(sd);
        if (tx == 0) {
            dbr[t] = sb;
            ddr[t] = bet[t] * sd;
        }
    }
    if (tl == 0) {  // <dX_f, E_f>, once per frame
        float s = 0.f;
        for (int e = tid; e < DK * DV; e += kThr) s += dXg[e] * Eg[e];
        s = warp_sum(s);
        if ((tid & 31) == 0) red[tid >> 5] = s;
    }
    // 3. dk = R dX^T - d diag(beta) dR E^T;  dq = scale dO X^T (by 64-row blocks of Dk)
    float accDK[2][TK], accDQ[2][TK];
    zero(accDK);
    zero(accDQ);
    for (int h = 0; h < NH; ++h) {
        float t1[2][4];
        __syncthreads();
        for (int e = tid; e < 64 * DV; e += kThr) Hs[(e / DV) * LV + e % DV] = dXg[(size_t)64 * h * DV + e];
        __syncthreads();
        zero(t1);
        mm<kThr, 2, 4>(t1, Rs, LV, 1, Hs, 1, LV, DV);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) accDK[i][4 * h + j] += t1[i][j];
        __syncthreads();
        for (int e = tid; e < 64 * DV; e += kThr) Hs[(e / DV) * LV + e % DV] = Eg[(size_t)64 * h * DV + e];
        __syncthreads();
        zero(t1);
        mm<kThr, 2, 4>(t1, dRs, LV, 1, Hs, 1, LV, DV);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float sk = d * bet[ty + 32 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) accDK[i][4 * h + j] -= sk * t1[i][j];
        }
        __syncthreads();
        for (int e = tid; e < 64 * DV; e += kThr) Hs[(e / DV) * LV + e % DV] = Xg[(size_t)64 * h * DV + e];
        __syncthreads();
        zero(t1);
        mm<kThr, 2, 4>(t1, dOs, LV, 1, Hs, 1, LV, DV);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) accDQ[i][4 * h + j] += p.scale * t1[i][j];
    }
    __syncthreads();
    // 4. dbeta, the tile's decay share, dk and dq through the unit-norm map
    if (tid < n) p.dbeta[tok + tid] = dbr[tid];
    if (tid == 0) {
        float s = 0.f;
        for (int t = 0; t < kC; ++t) s -= ddr[t];
        if (tl == 0)
            for (int w = 0; w < kThr / 32; ++w) s += red[w];
        p.part[fi * p.tiles + tl] = s;
    }
    T *dkp = (T *)p.dk + tok * DK;
    T *dqp = (T *)p.dq + tok * DK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = ty + 32 * i;
        float kd = 0.f, qd = 0.f;
#pragma unroll
        for (int j = 0; j < TK; ++j) {
            kd += Ks[t * LK + tx + 16 * j] * accDK[i][j];
            qd += Qs[t * LK + tx + 16 * j] * accDQ[i][j];
        }
        kd = row_sum16(kd);
        qd = row_sum16(qd);
#pragma unroll
        for (int j = 0; j < TK; ++j) {
            const int c = tx + 16 * j;
            float xk = accDK[i][j], xq = accDQ[i][j];
            if (p.l2) {
                xk = nk[t] < 1e-12f ? xk * 1e12f : (xk - Ks[t * LK + c] * kd) / nk[t];
                xq = nq[t] < 1e-12f ? xq * 1e12f : (xq - Qs[t * LK + c] * qd) / nq[t];
            }
            if (t < n) {
                st_f(dkp + (size_t)t * DK + c, xk);
                st_f(dqp + (size_t)t * DK + c, xq);
            }
        }
    }
}

// ======================================================= 4. ddecay per frame
__global__ void fb_decay_kernel(FbParams p) {
    const int bh = blockIdx.x;
    for (int f = threadIdx.x; f < p.F; f += blockDim.x) {
        const size_t fi = (size_t)bh * p.F + f;
        float s = 0.f;
        for (int t = 0; t < p.tiles; ++t) s += p.part[fi * p.tiles + t];
        p.ddecay[fi] = s;
    }
}

constexpr size_t frame_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)kC * (DK + 1) + kC * ((DK > DV ? DK : DV) + 1) + 2 * kC);
}
constexpr size_t fchain_smem(int DK) { return sizeof(float) * ((size_t)DK * (DK + 1) + DK * LSl); }
constexpr size_t token_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)2 * kC * (DK + 1) + 4 * kC * (DV + 1) + 5 * kC + 16);
}

size_t ws_floats(const CamScanBwdArgs &a) {
    const size_t BH = (size_t)a.B * a.H, F = (size_t)a.F, DK = (size_t)a.Dk, DV = (size_t)a.Dv;
    const size_t tiles = (size_t)(a.S + kC - 1) / kC;
    return BH * F * DK * DK + 3 * BH * F * DK * DV + BH * (F + 1) * DK * DV + BH * F * tiles;
}

template <typename T, int DK, int DV>
int run(const CamScanBwdArgs &a, cudaStream_t st) {
    const int BH = a.B * a.H, tiles = (a.S + kC - 1) / kC;
    const size_t nf = (size_t)BH * a.F;
    float *w = static_cast<float *>(a.ws);
    FbParams p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.beta = a.beta;
    p.dout = a.dout;
    p.decay = a.decay;
    p.s0 = a.s0;
    p.dsf = a.dsf;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.dbeta = a.dbeta;
    p.ddecay = a.ddecay;
    p.ds0 = a.ds0;
    p.Gw = w;
    p.Hw = p.Gw + nf * DK * DK;
    p.Pw = p.Hw + nf * DK * DV;
    p.dXw = p.Pw + nf * DK * DV;
    p.Ew = p.dXw + nf * DK * DV;
    p.part = p.Ew + (size_t)BH * (a.F + 1) * DK * DV;
    p.F = a.F;
    p.S = a.S;
    p.N = a.F * a.S;
    p.tiles = tiles;
    p.scale = a.scale;
    p.l2 = (a.flags & GDN_QK_L2NORM) ? 1 : 0;
    constexpr size_t s1 = frame_smem(DK, DV), s2 = fchain_smem(DK), s3 = token_smem(DK, DV);
    if (cudaFuncSetAttribute(fb_frame_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fb_chain_kernel<DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fb_token_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3) !=
            cudaSuccess)
        return GDN_ERR_CUDA;
    fb_frame_kernel<T, DK, DV><<<dim3((unsigned)a.F, (unsigned)BH, 3), kThr, s1, st>>>(p);
    note_launch();
    fb_chain_kernel<DK, DV><<<dim3((unsigned)(DV / kSl), (unsigned)BH, 2), kFChainThr, s2, st>>>(p);
    note_launch();
    fb_token_kernel<T, DK, DV><<<dim3((unsigned)(a.F * tiles), (unsigned)BH), kThr, s3, st>>>(p);
    note_launch();
    fb_decay_kernel<<<(unsigned)BH, 32, 0, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int run_t(const CamScanBwdArgs &a, cudaStream_t st) {
    if (a.Dk == 128 && a.Dv == 128) return run<T, 128, 128>(a, st);
    if (a.Dk == 128 && a.Dv == 64) return run<T, 128, 64>(a, st);
    if (a.Dk == 64 && a.Dv == 128) return run<T, 64, 128>(a, st);
    if (a.Dk == 64 && a.Dv == 64) return run<T, 64, 64>(a, st);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace

size_t cam_scan_bwd_workspace_bytes(const CamScanBwdArgs &a) { return sizeof(float) * ws_floats(a); }

int launch_cam_scan_bwd(const CamScanBwdArgs &a, cudaStream_t stream) {
    return a.dtype == GDN_BF16 ? run_t<__nv_bfloat16>(a, stream) : run_t<float>(a, stream);
}

}  // namespace gdn
