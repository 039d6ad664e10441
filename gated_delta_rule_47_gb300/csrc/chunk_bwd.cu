// chunk_bwd.cu -- backward of the chunkwise GDN / DeltaProduct forward, the
// chunk-local kernels on the CUDA cores in fp32 (gated_deltaproduct test.py computes the same
// gradients with `gated_chunk_delta_rule_bwd_kernel_dhu` for the state
// gradient, `gated_chunk_delta_rule_bwd_kernel_dqkw` and
// `gated_bwd_prepare_wy_repr_kernel` for the chunk-local ones).
//
// The rows of a head are the r*T sub-steps (t, j) in order; a chunk holds
// Ct = floor(64 / r) whole tokens, i.e. r*Ct <= 64 rows, padded to 64 with
// inert rows (k = v = beta = g = 0).  Row a of a chunk carries the log-decay
// g_t when j = 0 and 0 otherwise; gamma is the inclusive cumulative sum over
// the chunk's rows and gl its last value.  Query i reads the state after row
// rho(i) = i r + r - 1.  With S the state entering the chunk:
//
//   A[a][b] = beta_a e^{gamma_a - gamma_b} k_a.k_b (b < a),  T = (I + A)^-1
//   W = T diag(beta e^gamma) K,  U = T diag(beta) V,  Vn = U - W S
//   o_i = scale (e^{gamma_rho} S^T q_i + sum_{b <= rho} e^{gamma_rho - gamma_b} (q_i.k_b) vn_b)
//   S_next = e^{gl} S + Kd^T Vn,   Kd = diag(e^{gl - gamma}) K
//
// and, with dS' the gradient of S_next and P^[i][b] = scale e^{gamma_rho - gamma_b} q_i.k_b
// (b <= rho(i)):
//
//   dVn = Kd dS' + P^^T dO,  dR = T^T dVn,  dv = beta dR
//   dS  = e^{gl} dS' - W^T Kd dS' + B,   B = scale Q^T diag(e^{gamma_rho}) dO - W^T P^^T dO
//   dA  = -dR Vn^T (strictly lower);  dbeta_a = dR_a.(v_a - e^{gamma_a} S^T k_a) + sum_b dA E KK
//   dk  = P~^T Q + (L + L^T) K + diag(e^{gl-gamma}) Vn dS'^T - diag(beta e^gamma) dR S^T
//   dq  = P~ K + diag(scale e^{gamma_rho}) dO S^T
//   with P~[i][b] = scale e^{gamma_rho - gamma_b} do_i.vn_b (b <= rho), L = dA o beta E,
//   and dgamma collected term by term, then dg the reverse cumulative sum.
//
// Three launches (four with the tensor-core chains):
//   1. bwd_wy_kernel (one CTA per chunk): T, W, U, Kd, gamma and B to the workspace.
//   2. the forward state chain (S entering each chunk, and Vn) and the
//      reverse gradient chain (dS' of each chunk, and the initial state's
//      gradient) side by side: for bf16 at Dk = Dv = 128 wy_chain_tc_kernel
//      (tcgen05, one CTA per head and chain, the fp32 state in tensor memory;
//      the WY kernel then writes W and Kd as its bf16 hi / lo operand images
//      instead of fp32), otherwise wy_chain_kernel (CUDA cores, fp32; each CTA
//      holds 64 value columns of one head's state, since the columns of both
//      chains are independent).
//   3. (tensor-core chains only) chunk_products_tc_kernel: Z = Vn dS'^T,
//      t1 = dO S^T, dR = T^T dVn, dR Vn^T, t2 = dR S^T, dO Vn^T, <dS', S> and
//      each row's (Kd dS') . Vn per chunk on tcgen05, over dead slots.
//   4. bwd_grad_kernel (one CTA per chunk): every input gradient.
#include <cuda_bf16.h>

#include <type_traits>

#include "gdn_internal.h"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"
#include "wy_chain.cuh"

namespace gdn {
namespace {

using namespace tile;
constexpr int LC = kC + 1;      // leading dimension of the 64 x 64 tiles
constexpr int kSlice = 64;      // value columns per chain CTA

struct BwdParams {
    const void *q, *k, *v, *beta, *dout;
    const float *g, *s0, *dsf;
    void *dq, *dk, *dv;
    float *dbeta, *dg, *ds0;
    // workspace, per (head, chunk): T [64][64], W [64][Dk], U [64][Dv], Kd [64][Dk],
    // B [Dk][Dv], S [Dk][Dv], dS' [Dk][Dv], Vn [64][Dv], gamma [64], and the
    // products P^ [64][64] and K K^T [64][64] for the gradient kernel; with the
    // tensor-core chains (img) the first half of B then holds Y = Kd dS' [64][Dv]
    float *Tw, *Ww, *Uw, *Kdw, *Bw, *Sw, *dSw, *Vnw, *Gw, *Pw, *KKw;
    int T, r, Ct, NT;
    float scale;
    int l2;
    int img;  // W and Kd stored as the tensor-core chain's bf16 hi | lo images, not in fp32
};

// Chunk geometry shared by the per-chunk kernels.
struct Chunk {
    int c, bh, ntok, nrows;
    size_t hrow, htok, ci;
};

__device__ __forceinline__ Chunk chunk_of(const BwdParams &p) {
    Chunk ch;
    ch.c = blockIdx.x;
    ch.bh = blockIdx.y;
    const int t0 = ch.c * p.Ct;
    ch.ntok = min(p.Ct, p.T - t0);
    ch.nrows = ch.ntok * p.r;
    ch.htok = (size_t)ch.bh * p.T + t0;
    ch.hrow = ch.htok * p.r;
    ch.ci = (size_t)ch.bh * p.NT + ch.c;
    return ch;
}

// ============================================================ 1. WY products
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) bwd_wy_kernel(BwdParams p) {
    extern __shared__ float sm[];
    constexpr int LK = DK + 4, LV = DV + 1;  // the key-side tiles are read by mm_nt
    float *Ks = sm, *Vs = Ks + kC * LK, *Qs = Vs + kC * LV, *dOs = Qs + kC * LK, *Ws = dOs + kC * LV;
    float *Xa = Ws + kC * LK, *Xb = Xa + kC * LC, *X4 = Xb + kC * LC;
    float *gam = X4 + kC * kC / 4, *eg = gam + kC, *bet = eg + kC, *nrm = bet + kC;
    const Chunk ch = chunk_of(p);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, r = p.r;

    load_rows<T, DK, LK>(Ks, (const T *)p.k + ch.hrow * DK, ch.nrows, p.l2 != 0, nrm);
    load_rows<T, DV>(Vs, (const T *)p.v + ch.hrow * DV, ch.nrows, false, nullptr);
    load_rows<T, DK, LK>(Qs, (const T *)p.q + ch.htok * DK, ch.ntok, p.l2 != 0, nrm);
    load_rows<T, DV>(dOs, (const T *)p.dout + ch.htok * DV, ch.ntok, false, nullptr);
    if (tid < kC) bet[tid] = tid < ch.nrows ? ld_f((const T *)p.beta + ch.hrow + tid) : 0.f;
    if (tid < 32) {  // gamma: inclusive cumulative sum of the rows' log-decays
        const int a0 = tid, a1 = tid + 32;
        float x0 = (a0 < ch.nrows && a0 % r == 0) ? p.g[ch.htok + a0 / r] : 0.f;
        float x1 = (a1 < ch.nrows && a1 % r == 0) ? p.g[ch.htok + a1 / r] : 0.f;
        for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (tid >= o) {
                x0 += y0;
                x1 += y1;
            }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        gam[a0] = x0;
        gam[a1] = x1;
        eg[a0] = expf(x0);
        eg[a1] = expf(x1);
    }
    for (int e = tid; e < kC * LC; e += kThr) Xb[e] = 0.f;
    __syncthreads();

    // A = beta_a e^{gamma_a - gamma_b} k_a.k_b below the diagonal
    {
        float acc[2][4];
        zero(acc);
        mm_nt<kThr, 2, 4>(acc, Ks, LK, Ks, LK, DK);
        float *KKg = p.KKw + ch.ci * kC * kC;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int a = ty + 32 * i, b = tx + 16 * j;
                KKg[a * kC + b] = acc[i][j];
                Xa[a * LC + b] = b < a ? bet[a] * expf(gam[a] - gam[b]) * acc[i][j] : 0.f;
            }
    }
    __syncthreads();
    unit_lower_inverse<kC, kThr>(Xa, Xb, X4, LC);  // Xb = T (upper part stays 0)

    // T to the workspace; Xa = T diag(beta e^gamma), Xb = T diag(beta)
    {
        float *Tg = p.Tw + ch.ci * kC * kC;
        for (int e = tid; e < kC * kC; e += kThr) {
            const int m = e / kC, b = e % kC;
            const float t = Xb[m * LC + b];
            Tg[e] = t;
            Xa[m * LC + b] = t * bet[b] * eg[b];
            Xb[m * LC + b] = t * bet[b];
        }
    }
    __syncthreads();
    {
        float acc[2][DK / 16];
        zero(acc);
        mm<kThr, 2, DK / 16>(acc, Xa, LC, 1, Ks, LK, 1, kC);
        float *Wg = p.Ww + ch.ci * kC * DK;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < DK / 16; ++j) {
                const int m = ty + 32 * i, n = tx + 16 * j;
                if (!p.img) Wg[m * DK + n] = acc[i][j];
                Ws[m * LK + n] = acc[i][j];
            }
    }
    {
        float acc[2][DV / 16];
        zero(acc);
        mm<kThr, 2, DV / 16>(acc, Xb, LC, 1, Vs, LV, 1, kC);
        float *Ug = p.Uw + ch.ci * kC * DV;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) Ug[(ty + 32 * i) * DV + tx + 16 * j] = acc[i][j];
    }
    {
        const float gl = gam[kC - 1];
        float *Kdg = p.Kdw + ch.ci * kC * DK;
        if (!p.img) {
            for (int e = tid; e < kC * DK; e += kThr) {
                const int m = e / DK, n = e % DK;
                Kdg[e] = expf(gl - gam[m]) * Ks[m * LK + n];
            }
        }
        if (tid < kC) p.Gw[ch.ci * kC + tid] = gam[tid];
    }
    __syncthreads();
    if constexpr (DK == 128) {
        if (p.img) {  // W and Kd (= diag(e^{gl - gamma}) K) as the chain's operand images
            const float gl = gam[kC - 1];
            write_chain_image<kThr>(reinterpret_cast<unsigned char *>(p.Ww + ch.ci * kC * DK), Ws, LK,
                                    [](int) { return 1.f; });
            write_chain_image<kThr>(reinterpret_cast<unsigned char *>(p.Kdw + ch.ci * kC * DK), Ks, LK,
                                    [&](int m) { return expf(gl - gam[m]); });
        }
    }

    // P^ = scale e^{gamma_rho - gamma_b} q_i.k_b (b <= rho(i)) into Xa
    {
        float acc[2][4];
        zero(acc);
        mm_nt<kThr, 2, 4>(acc, Qs, LK, Ks, LK, DK);
        float *Pg = p.Pw + ch.ci * kC * kC;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int qi = ty + 32 * i, b = tx + 16 * j, rho = qi * r + r - 1;
                const float x =
                    (qi < ch.ntok && b <= rho) ? p.scale * expf(gam[rho] - gam[b]) * acc[i][j] : 0.f;
                Xa[qi * LC + b] = x;
                Pg[qi * kC + b] = x;
            }
    }
    __syncthreads();
    // Vs = -P^^T dO; dO rows scaled by scale e^{gamma_rho}
    {
        float acc[2][DV / 16];
        zero(acc);
        mm<kThr, 2, DV / 16>(acc, Xa, 1, LC, dOs, LV, 1, kC);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) Vs[(ty + 32 * i) * LV + tx + 16 * j] = -acc[i][j];
        for (int e = tid; e < kC * DV; e += kThr) {
            const int i = e / DV, n = e % DV;
            if (i < ch.ntok) dOs[i * LV + n] *= p.scale * eg[i * r + r - 1];
        }
    }
    __syncthreads();
    // B = Q^T (scaled dO) - W^T P^^T dO
    {
        float acc[DK / 32][DV / 16];
        zero(acc);
        mm<kThr, DK / 32, DV / 16>(acc, Qs, 1, LK, dOs, LV, 1, kC);
        mm<kThr, DK / 32, DV / 16>(acc, Ws, 1, LK, Vs, LV, 1, kC);
        float *Bg = p.Bw + ch.ci * DK * DV;
#pragma unroll
        for (int i = 0; i < DK / 32; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) Bg[(ty + 32 * i) * DV + tx + 16 * j] = acc[i][j];
    }
}

// ===================================================== 3. the input gradients
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) bwd_grad_kernel(BwdParams p) {
    extern __shared__ float sm[];
    // the value-side tiles are read by mm_nt (row stride 4 mod 32 words)
    constexpr int LK = DK + 1, LV = DV + 4, TK = DK / 16, TV = DV / 16, NH = DK / 64;
    float *Ks = sm, *Qs = Ks + kC * LK, *Vns = Qs + kC * LK, *dOs = Vns + kC * LV, *Hs = dOs + kC * LV;
    float *Xa = Hs + kC * LV, *Xb = Xa + kC * LC;
    float *gam = Xb + kC * LC, *eg = gam + kC, *bet = eg + kC, *nk = bet + kC, *nq = nk + kC;
    // decay and beta gradients, each slot written by one owner thread so that
    // the sums are formed in a fixed order (no atomics): rowg[a] by row a's
    // owner, qg[i] by query i's owner (added to row rho(i) at the end), lastg[b]
    // the share of the last row from row b, colg[ty][a] the column sums of
    // thread row ty, red[w] warp w's part of <dS', S>
    float *rowg = nq + kC, *dbet = rowg + kC, *qg = dbet + kC, *lastg = qg + kC, *colg = lastg + kC;
    float *red = colg + 32 * kC;
    const Chunk ch = chunk_of(p);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, r = p.r, ntok = ch.ntok, nrows = ch.nrows;
    const T *vp = (const T *)p.v + ch.hrow * DV;
    const float *Sg = p.Sw + ch.ci * DK * DV, *dSg = p.dSw + ch.ci * DK * DV;

    load_rows<T, DK>(Ks, (const T *)p.k + ch.hrow * DK, nrows, p.l2 != 0, nk);
    load_rows<T, DK>(Qs, (const T *)p.q + ch.htok * DK, ntok, p.l2 != 0, nq);
    if (!p.img) {  // with the tensor-core products, dO and Vn enter only through them
        load_rows<T, DV, LV>(dOs, (const T *)p.dout + ch.htok * DV, ntok, false, nullptr);
        load_rows<float, DV, LV>(Vns, p.Vnw + ch.ci * kC * DV, kC, false, nullptr);
    }
    if (tid < kC) {
        gam[tid] = p.Gw[ch.ci * kC + tid];
        eg[tid] = expf(gam[tid]);
        bet[tid] = tid < nrows ? ld_f((const T *)p.beta + ch.hrow + tid) : 0.f;
        rowg[tid] = 0.f;
        dbet[tid] = 0.f;
        qg[tid] = 0.f;
    }
    for (int e = tid; e < 32 * kC; e += kThr) colg[e] = 0.f;
    __syncthreads();
    const float gl = gam[kC - 1];

    // 1. through the state leaving the chunk: Kd dS' and Z = Vn dS'^T into dk.
    //    With the tensor-core chains the products kernel has left (layout with
    //    ChunkProductsTcArgs): Z and t1 = dO S^T in the dS' slot, dR and t2 = dR S^T
    //    in the S slot, dR Vn^T and DOV = dO Vn^T in the Vn slot, <dS', S> and
    //    each row's (Kd dS') . Vn in the B slot; the steps below read them.
    const float *Vg = p.Vnw + ch.ci * kC * DV;
    float accKdS[2][TV], accDK[2][TK];
    zero(accKdS);
    zero(accDK);
    if (p.img) {  // dk's share formed by the products kernel (every term but the unit-norm adjoint)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) accDK[i][j] = p.Bw[ch.ci * DK * DV + (ty + 32 * i) * DK + tx + 16 * j];
        if (tid < kThr / 32) red[tid] = tid == 0 ? p.Bw[ch.ci * DK * DV + 8192] : 0.f;
    } else {
        for (int h = 0; h < NH; ++h) {
            stage_rows<64, DV>(Hs, LV, dSg + (size_t)64 * h * DV);
            __syncthreads();
            mm<kThr, 2, TV>(accKdS, Ks + 64 * h, LK, 1, Hs, LV, 1, 64);
            float tz[2][4];
            zero(tz);
            mm_nt<kThr, 2, 4>(tz, Vns, LV, Hs, LV, DV);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float s = expf(gl - gam[ty + 32 * i]);
#pragma unroll
                for (int j = 0; j < 4; ++j) accDK[i][4 * h + j] += s * tz[i][j];
            }
            __syncthreads();
        }
        // <dS', S>
        float s = 0.f;
#pragma unroll 8
        for (int e = tid; e < DK * DV; e += kThr) s += dSg[e] * Sg[e];
        s = warp_sum(s);
        if ((tid & 31) == 0) red[tid >> 5] = s;
    }
    if (p.img) {  // (Kd dS') . Vn of each row from the products kernel
        if (tx == 0) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int b = ty + 32 * i;
                const float w = p.Bw[ch.ci * DK * DV + 8256 + b];
                rowg[b] -= w;
                lastg[b] = w;
            }
        }
    } else {  // K dS' -> Kd dS', and the decay gradients of the state's update
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float s = expf(gl - gam[ty + 32 * i]);
#pragma unroll
            for (int j = 0; j < TV; ++j) accKdS[i][j] *= s;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int b = ty + 32 * i;
            float w = 0.f;
#pragma unroll
            for (int j = 0; j < TV; ++j) w += accKdS[i][j] * Vns[b * LV + tx + 16 * j];
            w = row_sum16(w);
            if (tx == 0) {
                rowg[b] -= w;
                lastg[b] = w;
            }
        }
    }

    // 2. P^ (formed by the WY kernel) into Xa, T into Xb
    {
        const float *Pg = p.Pw + ch.ci * kC * kC, *Tg = p.Tw + ch.ci * kC * kC;
        stage_rows<kC, kC>(Xa, LC, Pg);
        if (p.img)
            stage_rows<64, DV>(Hs, LV, Sg);  // dR, from the products kernel
        else
            stage_rows<kC, kC>(Xb, LC, Tg);
    }
    __syncthreads();

    T *dvp = (T *)p.dv + ch.hrow * DV;
    if (p.img) {  // dv = beta dR
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TV; ++j) {
                const int m = ty + 32 * i, n = tx + 16 * j;
                if (m < nrows) st_f(dvp + (size_t)m * DV + n, bet[m] * Hs[m * LV + n]);
            }
    } else {
        // 3. dVn = Kd dS' + P^^T dO into Hs
        mm<kThr, 2, TV>(accKdS, Xa, 1, LC, dOs, LV, 1, kC);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TV; ++j) Hs[(ty + 32 * i) * LV + tx + 16 * j] = accKdS[i][j];
        __syncthreads();

        // 4. dR = T^T dVn into Hs; dv = beta dR
        float acc[2][TV];
        zero(acc);
        mm<kThr, 2, TV>(acc, Xb, 1, LC, Hs, LV, 1, kC);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TV; ++j) {
                const int m = ty + 32 * i, n = tx + 16 * j;
                Hs[m * LV + n] = acc[i][j];
                if (m < nrows) st_f(dvp + (size_t)m * DV + n, bet[m] * acc[i][j]);
            }
        __syncthreads();
    }

    // 5. DOV = dO Vn^T: the output's decay gradients, and P~ into Xa
    {
        float acc[2][4];
        zero(acc);
        if (p.img) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[i][j] = ty + 32 * i < ntok ? Vg[4096 + (ty + 32 * i) * kC + tx + 16 * j] : 0.f;
        } else {
            mm_nt<kThr, 2, 4>(acc, dOs, LV, Vns, LV, DV);
        }
        float col[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int qi = ty + 32 * i, rho = qi * r + r - 1;
            const bool qv = qi < ntok;
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int b = tx + 16 * j;
                const float pm = Xa[qi * LC + b] * acc[i][j];
                rs += pm;
                col[j] += pm;
                Xa[qi * LC + b] = (qv && b <= rho) ? p.scale * expf(gam[rho] - gam[b]) * acc[i][j] : 0.f;
            }
            rs = row_sum16(rs);
            if (tx == 0 && qv) qg[qi] += rs;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) colg[ty * kC + tx + 16 * j] -= col[j];
    }

    // 6. dA = -dR Vn^T below the diagonal, with K K^T: dbeta, decay gradients, L into Xb
    {
        float ta[2][4], tk[2][4];
        zero(ta);
        if (p.img) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) ta[i][j] = Vg[(ty + 32 * i) * kC + tx + 16 * j];
        } else {
            mm_nt<kThr, 2, 4>(ta, Hs, LV, Vns, LV, DV);
        }
        {  // K K^T, formed by the WY kernel
            const float *KKg = p.KKw + ch.ci * kC * kC;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) tk[i][j] = KKg[(ty + 32 * i) * kC + tx + 16 * j];
        }
        float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int b = ty + 32 * i;
            float rb = 0.f, rg = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = tx + 16 * j;
                float l = 0.f;
                if (c < b) {
                    const float E = expf(gam[b] - gam[c]), dA = -ta[i][j];
                    rb += dA * E * tk[i][j];
                    const float av = dA * bet[b] * E * tk[i][j];
                    rg += av;
                    cs[j] += av;
                    l = dA * bet[b] * E;
                }
                Xb[b * LC + c] = l;
            }
            rb = row_sum16(rb);
            rg = row_sum16(rg);
            if (tx == 0) {
                dbet[b] += rb;
                rowg[b] += rg;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) colg[ty * kC + tx + 16 * j] -= cs[j];
    }
    __syncthreads();

    // 7. dk += P~^T Q + (L + L^T) K;  dq = P~ K  (X1 = P~^T Q + L^T K, X2 = L K and
    //    P~ K from the products kernel with the tensor-core chains)
    float accDQ[2][TK];
    zero(accDQ);
    if (p.img) {  // P~ K from the products kernel (the dk terms are in its share already)
        const float *DQ = p.Ww + ch.ci * kC * DK;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                const int m = ty + 32 * i, n = tx + 16 * j;
                accDQ[i][j] = m < ntok ? DQ[m * DK + n] : 0.f;
            }
    } else {
        mm<kThr, 2, TK>(accDK, Xa, 1, LC, Qs, LK, 1, kC);
        mm<kThr, 2, TK>(accDK, Xb, LC, 1, Ks, LK, 1, kC);
        mm<kThr, 2, TK>(accDK, Xb, 1, LC, Ks, LK, 1, kC);
        mm<kThr, 2, TK>(accDQ, Xa, LC, 1, Ks, LK, 1, kC);
    }
    __syncthreads();

    // 8. through the state entering the chunk (staged in 64-row blocks of Dk in Vns):
    //    dq += diag(scale e^{gamma_rho}) dO S^T and dk -= diag(beta e^gamma) dR S^T.  The
    //    same two products give the dots the decay and beta gradients need:
    //    (S^T q_i).do_i = q_i.(S do_i) and (S^T k_b).dR_b = k_b.(S dR_b).
    float rq[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
    for (int h = 0; h < NH; ++h) {
        if (!p.img) stage_rows<64, DV>(Vns, LV, Sg + (size_t)64 * h * DV);
        __syncthreads();
        float t1[2][4], t2[2][4];
        zero(t1);
        zero(t2);
        if (p.img) {  // t1 = dO S^T from the products kernel (t2's terms are folded in there)
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int m = ty + 32 * i, c = 64 * h + tx + 16 * j;
                    t1[i][j] = m < ntok ? dSg[8192 + m * DK + c] : 0.f;
                }
        } else {
            mm_nt<kThr, 2, 4>(t1, dOs, LV, Vns, LV, DV);
            mm_nt<kThr, 2, 4>(t2, Hs, LV, Vns, LV, DV);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int m = ty + 32 * i;
            const float sq = m < ntok ? p.scale * eg[m * r + r - 1] : 0.f;
            const float sk = bet[m] * eg[m];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 64 * h + tx + 16 * j;
                accDQ[i][4 * h + j] += sq * t1[i][j];
                accDK[i][4 * h + j] -= sk * t2[i][j];
                rq[i] += Qs[m * LK + c] * t1[i][j];
                rk[i] += Ks[m * LK + c] * t2[i][j];
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int b = ty + 32 * i;
        float rv = 0.f;  // dR_b . v_b
#pragma unroll
        for (int j = 0; j < TV; ++j) {
            const int n = tx + 16 * j;
            rv += Hs[b * LV + n] * (b < nrows ? ld_f(vp + (size_t)b * DV + n) : 0.f);
        }
        rv = row_sum16(rv);
        const float sq = row_sum16(rq[i]), skr = row_sum16(rk[i]);
        const float skd = p.img ? p.Bw[ch.ci * DK * DV + 8320 + b] : skr;  // k_b . t2_b
        if (tx == 0) {
            dbet[b] += rv - eg[b] * skd;
            rowg[b] -= bet[b] * eg[b] * skd;
            if (b < ntok) qg[b] += p.scale * eg[b * r + r - 1] * sq;
        }
    }
    __syncthreads();

    // 9. dgamma in a fixed order, dg its reverse cumulative sum; dbeta
    if (tid < kC) {
        const int a = tid;
        float x = rowg[a];
        for (int y = 0; y < 32; ++y) x += colg[y * kC + a];
        if ((a + 1) % r == 0 && (a + 1) / r - 1 < ntok) x += qg[(a + 1) / r - 1];
        if (a == kC - 1) {
            float d = 0.f;
            for (int w = 0; w < kThr / 32; ++w) d += red[w];
            x += expf(gl) * d;
            for (int b = 0; b < kC; ++b) x += lastg[b];
        }
        gam[a] = x;  // gamma itself is no longer needed
    }
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int a = kC - 1; a >= 0; --a) {
            s += gam[a];
            gam[a] = s;
        }
    }
    __syncthreads();
    if (tid < nrows) p.dbeta[ch.hrow + tid] = dbet[tid];
    if (tid < ntok) p.dg[ch.htok + tid] = gam[tid * r];

    // 10. dk, dq through the unit-norm map when asked
    T *dkp = (T *)p.dk + ch.hrow * DK;
    T *dqp = (T *)p.dq + ch.htok * DK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int m = ty + 32 * i;
        float dk_dot = 0.f, dq_dot = 0.f;
#pragma unroll
        for (int j = 0; j < TK; ++j) {
            dk_dot += Ks[m * LK + tx + 16 * j] * accDK[i][j];
            dq_dot += Qs[m * LK + tx + 16 * j] * accDQ[i][j];
        }
        dk_dot = row_sum16(dk_dot);
        dq_dot = row_sum16(dq_dot);
#pragma unroll
        for (int j = 0; j < TK; ++j) {
            const int n = tx + 16 * j;
            float xk = accDK[i][j], xq = accDQ[i][j];
            if (p.l2) {
                const float rk = nk[m], rq = nq[m];
                xk = rk < 1e-12f ? xk * 1e12f : (xk - Ks[m * LK + n] * dk_dot) / rk;
                xq = rq < 1e-12f ? xq * 1e12f : (xq - Qs[m * LK + n] * dq_dot) / rq;
            }
            if (m < nrows) st_f(dkp + (size_t)m * DK + n, xk);
            if (m < ntok) st_f(dqp + (size_t)m * DK + n, xq);
        }
    }
}

constexpr size_t wy_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)3 * kC * (DK + 4) + 2 * kC * (DV + 1) + 2 * kC * LC + kC * kC / 4 + 4 * kC);
}
constexpr size_t grad_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)2 * kC * (DK + 1) + 3 * kC * (DV + 4) + 2 * kC * LC + 9 * kC + 32 * kC + 16);
}

// Workspace floats per (head, chunk).
size_t per_chunk_floats(int Dk, int Dv) {
    return 3 * (size_t)kC * kC + 2 * (size_t)kC * Dk + 2 * (size_t)kC * Dv + 3 * (size_t)Dk * Dv + kC;
}

template <typename T, int DK, int DV>
int run(const ChunkBwdArgs &a, cudaStream_t st) {
    const int BH = a.B * a.H, Ct = kC / a.r, NT = (a.T + Ct - 1) / Ct;
    const size_t nc = (size_t)BH * NT;
    float *w = static_cast<float *>(a.ws);
    BwdParams p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.beta = a.beta;
    p.dout = a.dout;
    p.g = a.g;
    p.s0 = a.s0;
    p.dsf = a.dsf;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.dbeta = a.dbeta;
    p.dg = a.dg;
    p.ds0 = a.ds0;
    p.Tw = w;
    p.Ww = p.Tw + nc * kC * kC;
    p.Uw = p.Ww + nc * kC * DK;
    p.Kdw = p.Uw + nc * kC * DV;
    p.Bw = p.Kdw + nc * kC * DK;
    p.Sw = p.Bw + nc * DK * DV;
    p.dSw = p.Sw + nc * DK * DV;
    p.Vnw = p.dSw + nc * DK * DV;
    p.Gw = p.Vnw + nc * kC * DV;
    p.Pw = p.Gw + nc * kC;
    p.KKw = p.Pw + nc * kC * kC;
    p.T = a.T;
    p.r = a.r;
    p.Ct = Ct;
    p.NT = NT;
    p.scale = a.scale;
    p.l2 = (a.flags & GDN_QK_L2NORM) ? 1 : 0;

    constexpr size_t s1 = wy_smem(DK, DV), s2 = wy_chain_smem<DK, kSlice>(), s3 = grad_smem(DK, DV);
    if (cudaFuncSetAttribute(bwd_wy_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(wy_chain_kernel<DK, DV, kSlice>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2) !=
            cudaSuccess ||
        cudaFuncSetAttribute(bwd_grad_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3) !=
            cudaSuccess)
        return GDN_ERR_CUDA;
    // the chains on tcgen05 for bf16 at Dk = Dv = 128 (W and Kd then travel as operand images)
    const bool tc_chain = std::is_same<T, __nv_bfloat16>::value && DK == 128 && DV == 128 &&
                          !(a.flags & GDN_PATH_SIMT) && sm100_family();
    p.img = tc_chain ? 1 : 0;
    if (tc_chain && 64 % a.r == 0 && a.r <= 8) {  // the WY factors on tcgen05 as well
        WyTcArgs ta{};
        ta.q = static_cast<const unsigned short *>(a.q);
        ta.k = static_cast<const unsigned short *>(a.k);
        ta.v = static_cast<const unsigned short *>(a.v);
        ta.beta = static_cast<const unsigned short *>(a.beta);
        ta.dout = static_cast<const unsigned short *>(a.dout);
        ta.g = a.g;
        ta.mask = nullptr;
        ta.Tw = p.Tw;
        ta.Ww = p.Ww;
        ta.Uw = p.Uw;
        ta.Kdw = p.Kdw;
        ta.Bw = p.Bw;
        ta.Pw = p.Pw;
        ta.KKw = p.KKw;
        ta.Gw = p.Gw;
        ta.BH = BH;
        ta.T = a.T;
        ta.r = a.r;
        ta.Ct = Ct;
        ta.NT = NT;
        ta.l2 = p.l2;
        ta.masked = 0;
        ta.bwd = 1;
        ta.scale = a.scale;
        const int rc = launch_wy_tc(ta, st);
        if (rc != GDN_OK) return rc;
    } else {
        bwd_wy_kernel<T, DK, DV><<<dim3((unsigned)NT, (unsigned)BH), kThr, s1, st>>>(p);
        note_launch();
    }
    if (tc_chain) {
        WyChainTcArgs ca{};
        ca.s0 = p.s0;
        ca.dsf = p.dsf;
        ca.ds0 = p.ds0;
        ca.Sw = p.Sw;
        ca.dSw = p.dSw;
        ca.Vnw = p.Vnw;
        ca.Wimg = reinterpret_cast<const unsigned char *>(p.Ww);
        ca.Kdimg = reinterpret_cast<const unsigned char *>(p.Kdw);
        ca.Uw = p.Uw;
        ca.Bw = p.Bw;
        ca.Gw = p.Gw;
        ca.Yw = p.Bw;  // Y = Kd dS' for the gradient kernel
        ca.BH = BH;
        ca.NT = NT;
        ca.roles = 2;
        int rc = launch_wy_chain_tc(ca, st);
        if (rc != GDN_OK) return rc;
        ChunkProductsTcArgs sa{};
        sa.Sw = p.Sw;
        sa.Vnw = p.Vnw;
        sa.dSw = p.dSw;
        sa.Bw = p.Bw;
        sa.Uw = p.Uw;
        sa.Ww = p.Ww;
        sa.Pw = p.Pw;
        sa.Tw = p.Tw;
        sa.Gw = p.Gw;
        sa.q = static_cast<const unsigned short *>(a.q);
        sa.k = static_cast<const unsigned short *>(a.k);
        sa.beta = static_cast<const unsigned short *>(a.beta);
        sa.dout = static_cast<const unsigned short *>(a.dout);
        sa.r = a.r;
        sa.l2 = p.l2;
        sa.scale = a.scale;
        sa.BH = BH;
        sa.NT = NT;
        sa.T = a.T;
        sa.Ct = Ct;
        rc = launch_chunk_products_tc(sa, st);
        if (rc != GDN_OK) return rc;
    } else {
        WyChainParams cp{p.s0, p.dsf, nullptr, p.ds0, p.Sw, p.dSw, p.Ww, p.Kdw, p.Uw, p.Vnw, p.Bw, p.Gw, NT};
        wy_chain_kernel<DK, DV, kSlice><<<dim3((unsigned)(DV / kSlice), (unsigned)BH, 2), kChainThr, s2, st>>>(cp);
        note_launch();
    }
    bwd_grad_kernel<T, DK, DV><<<dim3((unsigned)NT, (unsigned)BH), kThr, s3, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int run_t(const ChunkBwdArgs &a, cudaStream_t st) {
    if (a.Dk == 128 && a.Dv == 128) return run<T, 128, 128>(a, st);
    if (a.Dk == 128 && a.Dv == 64) return run<T, 128, 64>(a, st);
    if (a.Dk == 64 && a.Dv == 128) return run<T, 64, 128>(a, st);
    if (a.Dk == 64 && a.Dv == 64) return run<T, 64, 64>(a, st);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace

size_t chunk_bwd_workspace_bytes(const ChunkBwdArgs &a) {
    if (a.r < 1 || a.r > 8 || a.T <= 0) return 0;
    const int Ct = kC / a.r, NT = (a.T + Ct - 1) / Ct;
    return sizeof(float) * (size_t)a.B * a.H * NT * per_chunk_floats(a.Dk, a.Dv);
}

int launch_chunk_bwd(const ChunkBwdArgs &a, cudaStream_t stream) {
    return a.dtype == GDN_BF16 ? run_t<__nv_bfloat16>(a, stream) : run_t<float>(a, stream);
}

}  // namespace gdn
