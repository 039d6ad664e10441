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
//   2. the states E_f (forward) and the gradients dX_f (reverse, down to the
//      initial state's) side by side: fb_chain_tc_kernel (bf16, Dk = Dv = 128,
//      one CTA per head and chain, the product G_f X on tcgen05 with G_f as
//      the bf16 hi | lo image the frame kernel writes), else fb_chain_kernel
//      (CUDA cores, each CTA holding 32 value columns of one head).
//   3. the token gradients, and each tile's share of ddecay:
//      fb_token_tc_kernel (bf16, Dk = Dv = 128, one CTA per 128-token tile):
//      K and dO tiles by TMA, the frame's E_f, dX_f and X_f as bf16 hi / lo
//      operand images (written by the chain kernel) by bulk copies; K E and
//      K dX, then dk += R dX^T + (-d diag(beta) dR) E^T and dq = dO X^T, all on
//      tcgen05 with fp32 accumulators in TMEM, each fp32 operand split into
//      bf16 hi + lo (products hi.hi + hi.lo + lo.hi, about 2^-16 relative);
//      fb_token_kernel (every other shape, CUDA cores, 64-token tiles).
//   4. fb_decay_kernel: each frame's ddecay, its tiles' shares summed in order.
#include <cuda.h>
#include <stdint.h>

#include <algorithm>

#include "gdn_internal.h"
#include "simt_tile.cuh"
#include "tc_util.cuh"

namespace gdn {
namespace {

using namespace tile;
constexpr int kFChainThr = 256;
constexpr uint32_t kImg = 65536;  // a 128 x 128 matrix as bf16 hi | lo operand images (2 x 32 KB)
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
    // tensor-core path only (else null): E_f (f <= F) and dX_f as bf16 hi | lo
    // images, [BH][F+1][kImg] and [BH][F][kImg]; each image holds the 128 x 128
    // matrix row-major as two 64-column blocks of 128-byte swizzled rows
    uint8_t *Eimg, *dXimg;
    int F, S, N, tiles, BH;
    float scale;
    int l2;
    // 1 when the frame kernel writes G_f as the tensor-core chain's bf16 hi | lo
    // operand image (K-major: two 64-column blocks of 128 swizzled rows, hi then
    // lo) in place of its fp32 copy
    int gimg;
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

// This CTA's 32 columns (col0 ..) of a 128 x 128 fp32 matrix St [128][LSl]
// into its bf16 hi | lo operand images: element (m, c) at block c / 64, row m,
// 16-byte chunk (c % 64) / 8 of the row swizzled by m % 8; lo = x - hi.
__device__ __forceinline__ void write_image(uint8_t *img, const float *St, int col0) {
    for (int e = threadIdx.x; e < 128 * (kSl / 8); e += kFChainThr) {
        const int m = e / (kSl / 8), c8 = (e % (kSl / 8)) * 8, col = col0 + c8;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = St[m * LSl + c8 + 2 * i], x1 = St[m * LSl + c8 + 2 * i + 1];
            hi[i] = tc::pack_bf16(x0, x1);
            lo[i] = tc::pack_bf16(x0 - __uint_as_float(hi[i] << 16), x1 - __uint_as_float(hi[i] & 0xffff0000u));
        }
        const uint32_t off = (uint32_t)(col >> 6) * 16384u + tc::sw128_offset((uint32_t)m, (uint32_t)(col & 63));
        *reinterpret_cast<uint4 *>(img + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(img + 32768 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
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
            if (p.Eimg) write_image(p.Eimg + ((size_t)bh * (F + 1) + f) * kImg, St, col0);
        } else {  // dX_f = dE_{f+1} + P_f, out
            const float *Pg = p.Pw + fi * DK * DV;
            float *dXg = p.dXw + fi * DK * DV;
            for (int e = tid; e < DK * kSl; e += kFChainThr) {
                const int m = e / kSl, n = e % kSl;
                const float x = St[m * LSl + n] + Pg[(size_t)m * DV + col0 + n];
                St[m * LSl + n] = x;
                dXg[(size_t)m * DV + col0 + n] = x;
            }
            if (p.dXimg) {
                __syncthreads();
                write_image(p.dXimg + fi * kImg, St, col0);
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
        if (p.Eimg) write_image(p.Eimg + ((size_t)bh * (F + 1) + F) * kImg, St, col0);
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

// ====================================== 3a. token gradients on the tensor cores
// Persistent CTAs over the (head, frame, 128-token tile) items, bf16,
// Dk = Dv = 128.  Warp 0 loads (TMA for the K and dO tiles, bulk copies for
// the operand images), warp 1 issues the MMAs, warps 2..9 form r, -d beta dR,
// dv, dbeta and the outputs (two warps per TMEM lane quarter, thread = token
// row, each warp half of the columns).  The products, all M = N = 128 with
// fp32 accumulators in TMEM:
//   KE = K E_f,  dR' = K dX_f                          (E, dX images MN-major)
//   DK = R dX_f^T + W E_f^T,  W = -d diag(beta) dR     (by 64-column halves of Dv)
//   DQ = dO X_f^T                                      (X_f = E_{f+1})
// The next item's loads and first products (columns 0..255) start as soon as
// the current item's last product has read its operands, while the epilogue
// still reads DK and DQ (columns 256..511).  With the unit-norm flag the raw K
// tile is the operand and its rows' scale 1/|k| is applied to KE and dR' in
// the epilogue (k-hat = k / |k|).
constexpr int kTcThr = 320;
constexpr int kTcEpi = 256;  // epilogue threads
constexpr int kTcRows = 128;
constexpr uint32_t TB_A = 0;        // K tile, then dO tile: two 64-column blocks of 128 swizzled rows
constexpr uint32_t TB_E = 32768;    // E_f image (hi | lo), then the X_f image
constexpr uint32_t TB_DX = 98304;   // dX_f image (hi | lo)
constexpr uint32_t TB_R = 163840;   // R, one 64-column half: hi (16 KB) | lo; row exchange at the end
constexpr uint32_t TB_W = 196608;   // W = -d beta dR, one half: hi | lo
constexpr uint32_t TB_BAR = 229376;
// Every barrier but OPND completes once per item, so a wait for item j uses
// parity j & 1; OPND completes twice per item (the two halves of Dv).
enum { TBB_K = 0, TBB_E, TBB_DX, TBB_DO, TBB_X, TBB_MMA1, TBB_OPND, TBB_MMA2A, TBB_MMA2B, TBB_MMA3, TBB_DRAIN, TBB_NUM };
constexpr uint32_t TB_MISC = TB_BAR + 8 * TBB_NUM;  // TMEM address, then 16 reduction floats
constexpr uint32_t TB_SMEM = TB_MISC + 80 + 1024;    // + alignment of the base to 1024 bytes
static_assert(TB_SMEM <= 232448, "token kernel fits the shared memory of one CTA");
constexpr uint32_t TM_KE = 0, TM_DR = 128, TM_DK = 256, TM_DQ = 384;

__device__ unsigned int g_fb_error = 0;  // set when a bounded wait of the token kernel gives up
constexpr unsigned long long kFbWaitNs = 1000000000ull;

__device__ __forceinline__ bool fb_wait(uint64_t *bar, uint32_t parity, unsigned code) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::global_timer_ns();
    while (true) {
        if (tc::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile unsigned *>(&g_fb_error) != 0u) return false;
        if (tc::global_timer_ns() - t0 > kFbWaitNs) {
            atomicOr(&g_fb_error, code);
            return false;
        }
    }
}

// A wait's outcome made uniform across the warp, so that the warp's
// .sync.aligned TMEM loads that follow are reached by all of its lanes.
__device__ __forceinline__ bool warp_all_ok(bool ok) { return __all_sync(0xffffffffu, ok) != 0; }

__device__ __forceinline__ void split8(const float (&x)[8], uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = tc::pack_bf16(x[2 * i], x[2 * i + 1]);
        l[i] = tc::pack_bf16(x[2 * i] - __uint_as_float(h[i] << 16), x[2 * i + 1] - __uint_as_float(h[i] & 0xffff0000u));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(tc::pack_bf16(x[0], x[1]), tc::pack_bf16(x[2], x[3]), tc::pack_bf16(x[4], x[5]),
                      tc::pack_bf16(x[6], x[7]));
}

// |row| of a 128-wide bf16 row in global memory
__device__ __forceinline__ float row_norm128(const __nv_bfloat16 *row) {
    float s = 0.f;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        float x[8];
        unpack8(*reinterpret_cast<const uint4 *>(row + 8 * j), x);
#pragma unroll
        for (int i = 0; i < 8; ++i) s += x[i] * x[i];
    }
    return sqrtf(s);
}

__global__ void __launch_bounds__(kTcThr, 1)
    fb_token_tc_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mDO, FbParams p) {
    using namespace tc;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + TB_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + TB_MISC);
    float *red = reinterpret_cast<float *>(sm + TB_MISC + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int items = p.F * p.tiles * p.BH;

    if (threadIdx.x == 0) {
        for (int i = 0; i < TBB_NUM; ++i) mbar_init(&bars[i], i == TBB_OPND ? (uint32_t)kTcEpi : 1u);
        fence_mbar_init();
        prefetch_tensormap(&mK);
        prefetch_tensormap(&mDO);
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    // item it -> (head, frame, tile), tiles fastest so that a frame's tiles run together
    auto decode = [&](int it, int &bh, int &f, int &tl) {
        tl = it % p.tiles;
        f = (it / p.tiles) % p.F;
        bh = it / (p.tiles * p.F);
    };

    if (warp == 0) {
        if (lane == 0) {
            int j = 0;
            for (int it = blockIdx.x; it < items; it += gridDim.x, ++j) {
                int bh, f, tl;
                decode(it, bh, f, tl);
                const uint8_t *Ei = p.Eimg + ((size_t)bh * (p.F + 1) + f) * kImg;
                const uint8_t *dXi = p.dXimg + ((size_t)bh * p.F + f) * kImg;
                // the previous item's last product has read K / dO, E / X and dX
                if (j > 0 && !fb_wait(&bars[TBB_MMA3], (j - 1) & 1, 1u)) break;
                mbar_arrive_expect_tx(&bars[TBB_K], 32768);
                tma_load_4d(sm + TB_A, &mK, &bars[TBB_K], 0, tl * kTcRows, f, bh);
                tma_load_4d(sm + TB_A + 16384, &mK, &bars[TBB_K], 64, tl * kTcRows, f, bh);
                mbar_arrive_expect_tx(&bars[TBB_E], kImg);
                bulk_load_global(sm + TB_E, Ei, 32768, &bars[TBB_E]);
                bulk_load_global(sm + TB_E + 32768, Ei + 32768, 32768, &bars[TBB_E]);
                mbar_arrive_expect_tx(&bars[TBB_DX], kImg);
                bulk_load_global(sm + TB_DX, dXi, 32768, &bars[TBB_DX]);
                bulk_load_global(sm + TB_DX + 32768, dXi + 32768, 32768, &bars[TBB_DX]);
                // dO over K once the first products have read it
                if (!fb_wait(&bars[TBB_MMA1], j & 1, 1u)) break;
                mbar_arrive_expect_tx(&bars[TBB_DO], 32768);
                tma_load_4d(sm + TB_A, &mDO, &bars[TBB_DO], 0, tl * kTcRows, f, bh);
                tma_load_4d(sm + TB_A + 16384, &mDO, &bars[TBB_DO], 64, tl * kTcRows, f, bh);
                // X_f over E_f once both halves of the dk products have read it
                if (!fb_wait(&bars[TBB_MMA2B], j & 1, 1u)) break;
                mbar_arrive_expect_tx(&bars[TBB_X], kImg);
                bulk_load_global(sm + TB_E, Ei + kImg, 32768, &bars[TBB_X]);
                bulk_load_global(sm + TB_E + 32768, Ei + kImg + 32768, 32768, &bars[TBB_X]);
            }
            // every copy issued has landed before the CTA may exit (the last item's dq product has read them)
            if (j > 0) fb_wait(&bars[TBB_MMA3], (j - 1) & 1, 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idMN = idesc_bf16(128, 128, false, true);  // B MN-major
            const uint32_t idK = idesc_bf16(128, 128, false, false);  // both K-major
            int j = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++j) {
                const uint32_t par = (uint32_t)(j & 1);
                ok = fb_wait(&bars[TBB_K], par, 2u) && fb_wait(&bars[TBB_E], par, 2u);
                if (!ok) break;
                tc_fence_after_sync();
                {
                    int nmm = 0;
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_bf16_ss(tmem + TM_KE,
                                        smem_desc(sb + TB_A + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                        smem_desc(sb + TB_E + part * 32768 + ks * 2048, 16384, 1024), idMN,
                                        (nmm++) > 0);
                }
                ok = fb_wait(&bars[TBB_DX], par, 2u);
                if (!ok) break;
                tc_fence_after_sync();
                {
                    int nmm = 0;
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_bf16_ss(tmem + TM_DR,
                                        smem_desc(sb + TB_A + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                        smem_desc(sb + TB_DX + part * 32768 + ks * 2048, 16384, 1024), idMN,
                                        (nmm++) > 0);
                }
                mma_commit(&bars[TBB_MMA1]);
                for (int h = 0; h < 2 && ok; ++h) {
                    ok = fb_wait(&bars[TBB_OPND], (uint32_t)h, 3u);
                    if (!ok) break;
                    tc_fence_after_sync();
                    // DK += R_h dX_h^T + W_h E_h^T, each as hi.hi + hi.lo + lo.hi
#pragma unroll
                    for (int term = 0; term < 2; ++term) {
                        const uint32_t abase = sb + (term ? TB_W : TB_R);
                        const uint32_t bbase = sb + (term ? TB_E : TB_DX) + h * 16384;
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint32_t a = abase + (c == 2 ? 16384 : 0);
                            const uint32_t b = bbase + (c == 1 ? 32768 : 0);
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                mma_bf16_ss(tmem + TM_DK, smem_desc(a + ks * 32, 16, 1024),
                                            smem_desc(b + ks * 32, 16, 1024), idK, (h | term | c | ks) != 0);
                        }
                    }
                    mma_commit(&bars[h ? TBB_MMA2B : TBB_MMA2A]);
                }
                ok = ok && fb_wait(&bars[TBB_DO], par, 2u) && fb_wait(&bars[TBB_X], par, 2u);
                if (!ok) break;
                tc_fence_after_sync();
                {
                    int nmm = 0;
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_bf16_ss(tmem + TM_DQ,
                                        smem_desc(sb + TB_A + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                        smem_desc(sb + TB_E + part * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32, 16,
                                                  1024),
                                        idK, (nmm++) > 0);
                }
                mma_commit(&bars[TBB_MMA3]);
            }
            // every MMA issued has completed before TMEM is released
            mma_commit(&bars[TBB_DRAIN]);
            fb_wait(&bars[TBB_DRAIN], 0, 2u);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 2;                    // 0..7
        const int q = warp & 3, half = ew >> 2;     // TMEM lane quarter; column half
        const int t = 32 * q + lane;                // token row = TMEM lane
        const uint32_t lb = (uint32_t)(32 * q) << 16;
        float *xch = reinterpret_cast<float *>(sm + TB_R);  // [2][128][4] row exchange at the end of an item
        int j = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items; it += gridDim.x, ++j) {
            int bh, f, tl;
            decode(it, bh, f, tl);
            const int n = min(kTcRows, p.S - tl * kTcRows);
            const size_t fi = (size_t)bh * p.F + f;
            const size_t tok = (size_t)bh * p.N + (size_t)f * p.S + tl * kTcRows + t;
            const float d = p.decay[fi];
            const bool valid = t < n;
            const __nv_bfloat16 *vrow = static_cast<const __nv_bfloat16 *>(p.v) + tok * 128;
            const __nv_bfloat16 *krow = static_cast<const __nv_bfloat16 *>(p.k) + tok * 128;
            const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(p.q) + tok * 128;
            const float bt = valid ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.beta)[tok]) : 0.f;
            float nk = 1.f, nq = 1.f;
            if (p.l2 && valid) {
                nk = row_norm128(krow);
                nq = row_norm128(qrow);
            }
            const float sk = p.l2 ? 1.f / fmaxf(nk, 1e-12f) : 1.f;
            float dbeta = 0.f, dec = 0.f;
            // this row's v values for both halves, loaded before the products are waited for
            uint4 vpre[2][2][2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int ci = 0; ci < 2; ++ci)
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj)
                        vpre[h][ci][jj] = valid ? *reinterpret_cast<const uint4 *>(vrow + 64 * h + 16 * (2 * half + ci) + 8 * jj)
                                                : make_uint4(0u, 0u, 0u, 0u);
            ok = ok && warp_all_ok(fb_wait(&bars[TBB_MMA1], j & 1, 4u));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 1) ok = ok && warp_all_ok(fb_wait(&bars[TBB_MMA2A], j & 1, 4u));
                if (ok) {
                    tc_fence_after_sync();
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) {  // 16 columns at a time
                        const int cc = 2 * half + ci;
                        uint32_t ke[16], dr[16];
                        tmem_ld16(tmem + lb + TM_KE + 64 * h + 16 * cc, ke);
                        tmem_ld16(tmem + lb + TM_DR + 64 * h + 16 * cc, dr);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int c8 = 16 * cc + 8 * jj;  // column within the half
                            float vv[8];
                            unpack8(vpre[h][ci][jj], vv);
                            float rr[8], ww[8], dv8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float kt = __uint_as_float(ke[8 * jj + e]) * sk;
                                const float drt = __uint_as_float(dr[8 * jj + e]) * sk;
                                const float u = vv[e] - d * kt;
                                rr[e] = bt * u;
                                ww[e] = -d * bt * drt;
                                dv8[e] = bt * drt;
                                dbeta += drt * u;
                                dec += bt * drt * kt;
                            }
                            if (valid)
                                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dv) + tok * 128 + 64 * h +
                                                           c8) = pack8(dv8);
                            uint4 hi, lo;
                            const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)c8);
                            split8(rr, hi, lo);
                            *reinterpret_cast<uint4 *>(sm + TB_R + off) = hi;
                            *reinterpret_cast<uint4 *>(sm + TB_R + 16384 + off) = lo;
                            split8(ww, hi, lo);
                            *reinterpret_cast<uint4 *>(sm + TB_W + off) = hi;
                            *reinterpret_cast<uint4 *>(sm + TB_W + 16384 + off) = lo;
                        }
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before_sync();
                mbar_arrive(&bars[TBB_OPND]);
            }
            // the tile's share of ddecay (and <dX_f, E_f> on the frame's first tile)
            float dot = 0.f;
            if (tl == 0) {
                const float *Eg = p.Ew + ((size_t)bh * (p.F + 1) + f) * 16384, *dXg = p.dXw + fi * 16384;
                for (int e = threadIdx.x - 64; e < 16384; e += kTcEpi) dot += dXg[e] * Eg[e];
            }
            dec = warp_sum(dec);
            dot = warp_sum(dot);
            // the last product has completed: R and W are free for the row exchange
            ok = ok && warp_all_ok(fb_wait(&bars[TBB_MMA3], j & 1, 4u));
            if (lane == 0) {
                red[ew] = dec;
                red[8 + ew] = dot;
            }
            float kd = 0.f, qd = 0.f;
            if (ok) {
                tc_fence_after_sync();
                if (p.l2) {
#pragma unroll 1
                    for (int cc = 4 * half; cc < 4 * half + 4; ++cc) {
                        uint32_t gk[16], gq[16];
                        tmem_ld16(tmem + lb + TM_DK + 16 * cc, gk);
                        tmem_ld16(tmem + lb + TM_DQ + 16 * cc, gq);
                        tmem_wait_ld();
                        if (valid) {
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj) {
                                float kx[8], qx[8];
                                unpack8(*reinterpret_cast<const uint4 *>(krow + 16 * cc + 8 * jj), kx);
                                unpack8(*reinterpret_cast<const uint4 *>(qrow + 16 * cc + 8 * jj), qx);
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    kd += kx[e] * __uint_as_float(gk[8 * jj + e]);
                                    qd += qx[e] * __uint_as_float(gq[8 * jj + e]);
                                }
                            }
                        }
                    }
                }
            }
            xch[(half * 128 + t) * 4 + 0] = dbeta;
            xch[(half * 128 + t) * 4 + 1] = kd;
            xch[(half * 128 + t) * 4 + 2] = qd;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            dbeta += xch[((half ^ 1) * 128 + t) * 4 + 0];
            kd += xch[((half ^ 1) * 128 + t) * 4 + 1];
            qd += xch[((half ^ 1) * 128 + t) * 4 + 2];
            if (ew == 0 && lane == 0) {
                float s = 0.f;
                for (int w = 0; w < 8; ++w) s += red[8 + w] - red[w];
                p.part[fi * p.tiles + tl] = s;
            }
            if (ok && valid && half == 0) p.dbeta[tok] = dbeta;
            if (ok) {
                kd *= sk;                           // k-hat . dk
                qd *= p.scale / fmaxf(nq, 1e-12f);  // q-hat . dq
                const float sq = 1.f / fmaxf(nq, 1e-12f);
#pragma unroll 1
                for (int cc = 4 * half; cc < 4 * half + 4; ++cc) {
                    uint32_t gk[16], gq[16];
                    tmem_ld16(tmem + lb + TM_DK + 16 * cc, gk);
                    tmem_ld16(tmem + lb + TM_DQ + 16 * cc, gq);
                    tmem_wait_ld();
                    if (valid) {
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            float kx[8], qx[8], ok8[8], oq8[8];
                            if (p.l2) {
                                unpack8(*reinterpret_cast<const uint4 *>(krow + 16 * cc + 8 * jj), kx);
                                unpack8(*reinterpret_cast<const uint4 *>(qrow + 16 * cc + 8 * jj), qx);
                            }
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                float xk = __uint_as_float(gk[8 * jj + e]);
                                float xq = p.scale * __uint_as_float(gq[8 * jj + e]);
                                if (p.l2) {
                                    xk = nk < 1e-12f ? xk * 1e12f : (xk - kx[e] * sk * kd) / nk;
                                    xq = nq < 1e-12f ? xq * 1e12f : (xq - qx[e] * sq * qd) / nq;
                                }
                                ok8[e] = xk;
                                oq8[e] = xq;
                            }
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dk) + tok * 128 + 16 * cc +
                                                       8 * jj) = pack8(ok8);
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dq) + tok * 128 + 16 * cc +
                                                       8 * jj) = pack8(oq8);
                        }
                    }
                }
            }
            tc_fence_before_sync();
            // the exchange area is R / W again for the next item, and red is reused
            asm volatile("bar.sync 1, 256;" ::: "memory");
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// ======================================== 1a. frame products on the tensor cores
// One CTA per (frame, head, product), bf16, Dk = Dv = 128: the frame's tokens
// stream through TMA in 128-token tiles (the last clipped at the frame's end
// and zero-filled); four builder warps (thread = token row) scale the A-side
// tile's rows and split them into bf16 hi + lo; the MMAs accumulate
// D = sum_t a_t b_t^T in TMEM with M = N = 128 and K = the tile's tokens,
// both operands MN-major (the tiles as loaded):
//   G: a_t = beta_t n_t^2 k_t,  b_t = k_t      (n_t = 1 / |k_t| with the
//   H: a_t = beta_t n_t k_t,    b_t = v_t       unit-norm flag, else 1)
//   P: a_t = m_t q_t,           b_t = do_t     (m_t = 1 / |q_t| or 1; times scale)
constexpr int kFrThr = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 builders then epilogue
constexpr uint32_t FR_STAGE = 65536;   // A-side tile | B-side tile (32 KB each)
constexpr uint32_t FR_A = 2 * FR_STAGE;  // A hi (32 KB) | lo
constexpr uint32_t FR_BAR = FR_A + 65536;
enum { FRB_FULL = 0, FRB_EMPTY = 2, FRB_AREADY = 4, FRB_AFREE = 5, FRB_DONE = 6, FRB_NUM = 7 };
constexpr uint32_t FR_MISC = FR_BAR + 8 * FRB_NUM;
constexpr uint32_t FR_SMEM = FR_MISC + 16 + 1024;
static_assert(FR_SMEM <= 232448, "frame-product kernel fits the shared memory of one CTA");

__global__ void __launch_bounds__(kFrThr, 1)
    fb_frame_tc_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                       const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mDO, FbParams p) {
    using namespace tc;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + FR_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + FR_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int f = blockIdx.x, bh = blockIdx.y, part = blockIdx.z;  // 0 = G, 1 = H, 2 = P
    const int nt = (p.S + 127) / 128;
    const size_t fi = (size_t)bh * p.F + f;
    const CUtensorMap *ma = part == 2 ? &mQ : &mK;
    const CUtensorMap *mb = part == 0 ? &mK : (part == 1 ? &mV : &mDO);
    const bool same = part == 0;  // G: the A side and the B side are the same tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < FRB_NUM; ++i) mbar_init(&bars[i], i == FRB_AREADY ? 128u : 1u);
        fence_mbar_init();
        prefetch_tensormap(ma);
        prefetch_tensormap(mb);
    }
    if (warp == 1) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            int armed[2] = {0, 0};
            for (int i = 0; i < nt; ++i) {
                const int s = i & 1;
                if (i >= 2 && !fb_wait(&bars[FRB_EMPTY + s], ((i - 2) >> 1) & 1, 16u)) break;
                uint8_t *st = sm + s * FR_STAGE;
                mbar_arrive_expect_tx(&bars[FRB_FULL + s], same ? 32768 : 65536);
                tma_load_4d(st, ma, &bars[FRB_FULL + s], 0, 128 * i, f, bh);
                tma_load_4d(st + 16384, ma, &bars[FRB_FULL + s], 64, 128 * i, f, bh);
                if (!same) {
                    tma_load_4d(st + 32768, mb, &bars[FRB_FULL + s], 0, 128 * i, f, bh);
                    tma_load_4d(st + 49152, mb, &bars[FRB_FULL + s], 64, 128 * i, f, bh);
                }
                armed[s]++;
            }
            for (int s = 0; s < 2; ++s)
                if (armed[s]) fb_wait(&bars[FRB_FULL + s], (armed[s] - 1) & 1, 16u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16(128, 128, true, true);
            bool ok = true;
            for (int i = 0; i < nt && ok; ++i) {
                const int s = i & 1;
                ok = fb_wait(&bars[FRB_AREADY], i & 1, 17u);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t bt = sb + s * FR_STAGE + (same ? 0 : 32768);
#pragma unroll
                for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ss(tmem, smem_desc(sb + FR_A + hl * 32768 + ks * 2048, 16384, 1024),
                                    smem_desc(bt + ks * 2048, 16384, 1024), id, (i | hl | ks) != 0);
                mma_commit(&bars[FRB_EMPTY + s]);
                mma_commit(&bars[FRB_AFREE]);
            }
            mma_commit(&bars[FRB_DONE]);
            fb_wait(&bars[FRB_DONE], 0, 17u);
        }
    } else {
        // ------------------------------------- builders (thread = token row)
        const int r = 32 * (warp & 3) + lane;
        const size_t tok_f = (size_t)bh * p.N + (size_t)f * p.S;
        bool ok = true;
        for (int i = 0; i < nt; ++i) {
            const int s = i & 1, t = 128 * i + r;
            const bool valid = t < p.S;
            float fac = 0.f;
            if (valid) fac = part == 2 ? 1.f : __bfloat162float(static_cast<const __nv_bfloat16 *>(p.beta)[tok_f + t]);
            ok = ok && warp_all_ok(fb_wait(&bars[FRB_FULL + s], (i >> 1) & 1, 18u));
            if (i >= 1) ok = ok && warp_all_ok(fb_wait(&bars[FRB_AFREE], (i - 1) & 1, 18u));
            if (ok) {
                const uint8_t *src = sm + s * FR_STAGE;
                if (p.l2) {
                    float ss = 0.f;
#pragma unroll 4
                    for (int c = 0; c < 16; ++c) {
                        float x[8];
                        unpack8(*reinterpret_cast<const uint4 *>(src + (c >> 3) * 16384 + sw128_offset(r, 8 * (c & 7))), x);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss += x[e] * x[e];
                    }
                    const float nrm = 1.f / fmaxf(sqrtf(ss), 1e-12f);
                    fac *= part == 0 ? nrm * nrm : nrm;
                }
#pragma unroll 4
                for (int c = 0; c < 16; ++c) {
                    const uint32_t off = (c >> 3) * 16384 + sw128_offset(r, 8 * (c & 7));
                    float x[8];
                    unpack8(*reinterpret_cast<const uint4 *>(src + off), x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] *= fac;
                    uint4 hi, lo;
                    split8(x, hi, lo);
                    *reinterpret_cast<uint4 *>(sm + FR_A + off) = hi;
                    *reinterpret_cast<uint4 *>(sm + FR_A + 32768 + off) = lo;
                }
                fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            mbar_arrive(&bars[FRB_AREADY]);
        }
        // ---------------------------------------- epilogue (thread = row of D)
        ok = ok && warp_all_ok(fb_wait(&bars[FRB_DONE], 0, 18u));
        if (ok) {
            tc_fence_after_sync();
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            const float sc = part == 2 ? p.scale : 1.f;
            float *out = (part == 0 ? p.Gw : (part == 1 ? p.Hw : p.Pw)) + fi * 16384 + (size_t)r * 128;
            if (part == 0 && p.gimg) {
                // G_f as the chain's operand image: row r, 16-byte chunks of 8 columns
                uint8_t *img = reinterpret_cast<uint8_t *>(p.Gw + fi * 16384);
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t x[16];
                    tmem_ld16(tmem + lb + 16 * cc, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = __uint_as_float(x[8 * g + e]);
                        uint4 hi, lo;
                        split8(y, hi, lo);
                        const int c = 16 * cc + 8 * g;
                        const uint32_t off = (uint32_t)(c >> 6) * 16384u + sw128_offset((uint32_t)r, (uint32_t)(c & 63));
                        *reinterpret_cast<uint4 *>(img + off) = hi;
                        *reinterpret_cast<uint4 *>(img + 32768 + off) = lo;
                    }
                }
            } else {
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t x[16];
                    tmem_ld16(tmem + lb + 16 * cc, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<float4 *>(out + 16 * cc + 4 * j) =
                            make_float4(sc * __uint_as_float(x[4 * j]), sc * __uint_as_float(x[4 * j + 1]),
                                        sc * __uint_as_float(x[4 * j + 2]), sc * __uint_as_float(x[4 * j + 3]));
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 128);
    }
}

// ================================== 2'. the chains on tcgen05 (bf16, D = 128)
// fb_chain_tc_kernel: one CTA per head and direction (blockIdx.y: 0 = the
// states E_f, 1 = the gradients dX_f), the 128 x 128 state held transposed in
// the registers of sixteen epilogue warps (thread = value index dv, and a
// quarter hh of the key indices).  Per frame each thread writes its part of the fp32
// snapshot, of the token kernel's bf16 hi | lo image and of the state's own
// hi | lo operand (K-major, value rows); one thread issues
// Z^T = X^T G_f^T as hi.hi + hi.lo + lo.hi (24 MMAs, M = N = 128) into TMEM,
// and the threads form E_{f+1} = d_f (E_f - G_f E_f) + H_f, or
// dE_f = d_f (dX_f - G_f dX_f) with dX_f = dE_{f+1} + P_f.  G_f arrives as the
// bf16 hi | lo image the frame kernel writes in place of its fp32 copy,
// double-buffered with bulk copies.
constexpr int kFcThr = 640;           // warp 0 issues, warp 1 holds TMEM, warp 2 loads, warps 4..19 epilogue
constexpr int kFcEpi = 512;           // epilogue threads
constexpr uint32_t FC_G = 0;          // two slots of G_f hi | lo (64 KB each)
constexpr uint32_t FC_X = 131072;     // X^T hi | lo: K-major [2 key blocks][128 value rows][128 B]
constexpr uint32_t FC_BAR = FC_X + 65536;
enum { FCB_FULL = 0, FCB_FREE = 2, FCB_XREADY = 4, FCB_ZDONE, FCB_DRAIN, FCB_NUM };
constexpr uint32_t FC_TSLOT = FC_BAR + 8 * FCB_NUM;
constexpr uint32_t FC_SMEM = FC_TSLOT + 16 + 1024;  // + alignment of the base to 1024 bytes
static_assert(FC_SMEM <= 232448, "frame chain kernel fits the shared memory of one CTA");

// This thread's column dv of rows 32 hh .. 32 hh + 31 of a 128 x 128 matrix
// into its bf16 hi | lo image (as write_image lays it out).
__device__ __forceinline__ void write_col_image(uint8_t *img, const float (&x)[32], int hh, int dv) {
    uint8_t *base = img + (uint32_t)(dv >> 6) * 16384u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t off = tc::sw128_offset((uint32_t)(32 * hh + i), (uint32_t)(dv & 63));
        const __nv_bfloat16 h = __float2bfloat16_rn(x[i]);
        *reinterpret_cast<__nv_bfloat16 *>(base + off) = h;
        *reinterpret_cast<__nv_bfloat16 *>(base + 32768 + off) = __float2bfloat16_rn(x[i] - __bfloat162float(h));
    }
}

__global__ void __launch_bounds__(kFcThr, 1) fb_chain_tc_kernel(FbParams p) {
    using namespace tc;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + FC_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + FC_TSLOT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, role = blockIdx.y, F = p.F;

    if (threadIdx.x == 0) {
        for (int i = 0; i < FCB_NUM; ++i) mbar_init(&bars[i], i == FCB_XREADY ? (uint32_t)kFcEpi : 1u);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id = idesc_bf16(128, 128, false, false);
            for (int s = 0; s < F; ++s) {
                const int b = s & 1;
                if (!fb_wait(&bars[FCB_FULL + b], (s >> 1) & 1, 32u)) break;
                if (!fb_wait(&bars[FCB_XREADY], s & 1, 32u)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int pr = 0; pr < 3; ++pr) {
                    const uint32_t xa = sb + FC_X + (pr == 2 ? 32768u : 0u);
                    const uint32_t gb = sb + FC_G + (uint32_t)b * 65536u + (pr == 1 ? 32768u : 0u);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ss(tmem, smem_desc(xa + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                    smem_desc(gb + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), id, (pr | ks) != 0);
                }
                mma_commit(&bars[FCB_ZDONE]);
                mma_commit(&bars[FCB_FREE + b]);
            }
            mma_commit(&bars[FCB_DRAIN]);
            mbar_wait(&bars[FCB_DRAIN], 0, 200000000ull);
        }
    } else if (warp == 2) {
        // ---------------------------------------------- G_f images, bulk copies
        if (lane == 0) {
            int armed[2] = {0, 0};
            for (int s = 0; s < F; ++s) {
                const int b = s & 1;
                // slot b held frame s-2, whose MMAs are complete when FCB_FREE + b completes
                if (s >= 2 && !fb_wait(&bars[FCB_FREE + b], ((s - 2) >> 1) & 1, 33u)) break;
                const size_t fi = (size_t)bh * F + (role == 0 ? s : F - 1 - s);
                const uint8_t *g = reinterpret_cast<const uint8_t *>(p.Gw + fi * 16384);
                mbar_arrive_expect_tx(&bars[FCB_FULL + b], 65536u);
                bulk_load_global(sm + FC_G + b * 65536, g, 32768u, &bars[FCB_FULL + b]);
                bulk_load_global(sm + FC_G + b * 65536 + 32768, g + 32768, 32768u, &bars[FCB_FULL + b]);
                armed[b]++;
            }
            for (int b = 0; b < 2; ++b)
                if (armed[b]) mbar_wait(&bars[FCB_FULL + b], (armed[b] - 1) & 1, 200000000ull);
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3, hh = (warp - 4) >> 2;
        const int dv = 32 * q + lane;
        const uint32_t lb = (uint32_t)(32 * q) << 16;
        const float *init = role == 0 ? p.s0 : p.dsf;
        float x[32], pre[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = init ? init[((size_t)bh * 128 + 32 * hh + i) * 128 + dv] : 0.f;
        // H_f (states: added after this frame's product) or P_f (gradients: added
        // before it, so loaded one frame ahead), rows 32 hh.., column dv
        auto load_pre = [&](int f) {
            const float *src = (role == 0 ? p.Hw : p.Pw) + ((size_t)bh * F + f) * 16384 + (size_t)(32 * hh) * 128 + dv;
#pragma unroll
            for (int i = 0; i < 32; ++i) pre[i] = src[(size_t)i * 128];
        };
        if (role == 1 && F > 0) load_pre(F - 1);
        bool ok = true;
        for (int s = 0; s < F; ++s) {
            const int f = role == 0 ? s : F - 1 - s;
            const size_t fi = (size_t)bh * F + f;
            const float d = p.decay[fi];
            if (role == 1) {
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] += pre[i];  // dX_f = dE_{f+1} + P_f
            }
            {  // the snapshot, the token kernel's image, and X^T as the MMA operand
                const size_t slot = role == 0 ? (size_t)bh * (F + 1) + f : fi;
                float *sn = (role == 0 ? p.Ew : p.dXw) + slot * 16384 + (size_t)(32 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 32; ++i) sn[(size_t)i * 128] = x[i];
                write_col_image((role == 0 ? p.Eimg : p.dXimg) + slot * kImg, x, hh, dv);
                uint8_t *xo = sm + FC_X + (hh >> 1) * 16384;  // key block of rows 32 hh..
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] = x[8 * c + e];
                    uint4 hi, lo;
                    split8(y, hi, lo);
                    const uint32_t off = sw128_offset((uint32_t)dv, (uint32_t)(32 * (hh & 1) + 8 * c));
                    *reinterpret_cast<uint4 *>(xo + off) = hi;
                    *reinterpret_cast<uint4 *>(xo + 32768 + off) = lo;
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bars[FCB_XREADY]);
            }
            if (role == 0)
                load_pre(f);
            else if (s + 1 < F)
                load_pre(f - 1);
            ok = warp_all_ok(fb_wait(&bars[FCB_ZDONE], s & 1, 34u));
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t z[16];
                tmem_ld16(tmem + lb + 32 * hh + 16 * j, z);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float gx = __uint_as_float(z[i]);
                    x[16 * j + i] = role == 0 ? d * (x[16 * j + i] - gx) + pre[16 * j + i] : d * (x[16 * j + i] - gx);
                }
            }
            tc_fence_before_sync();  // the TMEM reads complete before the next frame's MMAs (after FCB_XREADY)
        }
        if (ok) {
            if (role == 0) {  // the state after the last frame
                const size_t slot = (size_t)bh * (F + 1) + F;
                float *sn = p.Ew + slot * 16384 + (size_t)(32 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 32; ++i) sn[(size_t)i * 128] = x[i];
                write_col_image(p.Eimg + slot * kImg, x, hh, dv);
            } else if (p.ds0) {
#pragma unroll
                for (int i = 0; i < 32; ++i) p.ds0[((size_t)bh * 128 + 32 * hh + i) * 128 + dv] = x[i];
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 128);
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

// The shapes the tensor-core token kernel serves (bf16, Dk = Dv = 128); the
// workspace holds its operand images for these whatever the flags.
bool tc_shape(const CamScanBwdArgs &a) { return a.dtype == GDN_BF16 && a.Dk == 128 && a.Dv == 128; }

size_t ws_floats(const CamScanBwdArgs &a) {
    const size_t BH = (size_t)a.B * a.H, F = (size_t)a.F, DK = (size_t)a.Dk, DV = (size_t)a.Dv;
    const size_t tiles = (size_t)(a.S + kC - 1) / kC;
    const size_t imgs = tc_shape(a) ? BH * (2 * F + 1) * (kImg / sizeof(float)) : 0;
    const size_t shares = (BH * F * tiles + 63) / 64 * 64;  // keeps the images 256-byte aligned
    return BH * F * DK * DK + 3 * BH * F * DK * DV + BH * (F + 1) * DK * DV + shares + imgs;
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
    // the tensor-core token kernel: its operand images after the shares
    CUtensorMap mK, mDO;
    const bool tc = tc_shape(a) && !(a.flags & GDN_PATH_SIMT) && sm100_family() &&
                    make_bf16_frame_map(&mK, a.k, BH, a.F, a.S, 64, 128) &&
                    make_bf16_frame_map(&mDO, a.dout, BH, a.F, a.S, 64, 128);
    if (tc) {
        uint8_t *img = reinterpret_cast<uint8_t *>(p.part + (nf * tiles + 63) / 64 * 64);
        p.Eimg = img;
        p.dXimg = img + (size_t)BH * (a.F + 1) * kImg;
    }
    p.F = a.F;
    p.S = a.S;
    p.N = a.F * a.S;
    p.tiles = tiles;
    p.BH = BH;
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
    CUtensorMap mV, mQ;
    if (tc && make_bf16_frame_map(&mV, a.v, BH, a.F, a.S, 64, 128) &&
        make_bf16_frame_map(&mQ, a.q, BH, a.F, a.S, 64, 128)) {
        if (cudaFuncSetAttribute(fb_frame_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FR_SMEM) !=
            cudaSuccess)
            return GDN_ERR_CUDA;
        p.gimg = 1;  // G_f as the tensor-core chain's operand image
        fb_frame_tc_kernel<<<dim3((unsigned)a.F, (unsigned)BH, 3), kFrThr, FR_SMEM, st>>>(mK, mV, mQ, mDO, p);
    } else {
        fb_frame_kernel<T, DK, DV><<<dim3((unsigned)a.F, (unsigned)BH, 3), kThr, s1, st>>>(p);
    }
    note_launch();
    if (p.gimg) {
        if (cudaFuncSetAttribute(fb_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FC_SMEM) !=
            cudaSuccess)
            return GDN_ERR_CUDA;
        fb_chain_tc_kernel<<<dim3((unsigned)BH, 2), kFcThr, FC_SMEM, st>>>(p);
    } else {
        fb_chain_kernel<DK, DV><<<dim3((unsigned)(DV / kSl), (unsigned)BH, 2), kFChainThr, s2, st>>>(p);
    }
    note_launch();
    if (tc) {
        p.tiles = (a.S + kTcRows - 1) / kTcRows;
        if (cudaFuncSetAttribute(fb_token_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TB_SMEM) !=
            cudaSuccess)
            return GDN_ERR_CUDA;
        const long long items = (long long)a.F * p.tiles * BH;
        const int grid = (int)std::min<long long>(items, (long long)device_sm_count());
        fb_token_tc_kernel<<<(unsigned)grid, kTcThr, TB_SMEM, st>>>(mK, mDO, p);
    } else {
        fb_token_kernel<T, DK, DV><<<dim3((unsigned)(a.F * tiles), (unsigned)BH), kThr, s3, st>>>(p);
    }
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

int cam_scan_bwd_read_clear_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fb_error, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_fb_error, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
    return v ? GDN_ERR_TIMEOUT : GDN_OK;
}

}  // namespace gdn
