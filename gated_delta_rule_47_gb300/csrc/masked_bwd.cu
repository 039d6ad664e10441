// masked_bwd.cu -- backward of the block-masked DeltaProduct forward
// (gated_deltaproduct test.py: `gated_chunk_delta_rule_bwd_kernel_dhu`,
// `gated_chunk_delta_rule_bwd_kernel_dqkw` and `gated_bwd_prepare_wy_repr_kernel`
// for the mask_ij variant): the chunk-local kernels on the CUDA cores in fp32,
// the chains on tcgen05 for bf16 at D = 128 (wy_chain_tc.cu).
//
// The sub-rows a = (t, i) of a 64-row chunk (64 / r tokens) carry the read key
// kr_a = k_t masked slice-wise by mask[i][:] and the write key kw_a = slice i
// of k_t; v, beta and the decay are the token's.  The chunk backward of
// chunk_bwd.cu carries over with the two keys apart (A = beta E o Kr Kw^T on
// the sub-rows of earlier tokens, W = T diag(beta e^gamma) Kr, the state and
// the outputs written and read through Kw):
//   dVn = Kd dS' + P^^T dO,  dR = T^T dVn        (Kd = diag(e^{gl-gamma}) Kw)
//   dKr = L Kw - diag(beta e^gamma) dR S^T        (L = dA o beta E, dA = -dR Vn^T)
//   dKw = L^T Kr + P~^T Q + diag(e^{gl-gamma}) Vn dS'^T
//   dq  = P~ Kw + diag(scale e^{gamma}) dO S^T
// and the token's gradients gather its sub-rows': dv_t = beta_t sum_i dR_(t,i),
// dbeta_t = sum_i dbeta_(t,i), and slice j of dk_t = slice j of
// (dKw_(t,j) + sum_i mask[i][j] dKr_(t,i)).  Each row accumulates its part
// D_a = mask[i][j(c)] dKr_a[c] + [j(c) = i] dKw_a[c] as it goes, and the
// token sums its rows at the end.  Three launches, as the chunk backward:
// mbwd_wy_kernel (T, W, U, Kd, gamma and the chunk's term B of the state
// gradient), the two chains (wy_chain_tc_kernel for bf16 at Dk = Dv = 128,
// with W and Kd handed over as operand images; wy_chain_kernel otherwise),
// mbwd_grad_kernel.
#include <cuda_bf16.h>

#include <type_traits>

#include "gdn_internal.h"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"
#include "wy_chain.cuh"

namespace gdn {
namespace {

using namespace tile;
constexpr int LC = kC + 1;
constexpr int kSlice = 64;

struct MbParams {
    const void *q, *k, *v, *beta, *dout;
    const float *g, *mask, *s0, *dsf;
    void *dq, *dk, *dv;
    float *dbeta, *dg, *ds0;
    // as the chunk backward's workspace (P^ and Kr Kw^T in the last two)
    float *Tw, *Ww, *Uw, *Kdw, *Bw, *Sw, *dSw, *Vnw, *Gw, *Pw, *KKw;
    int T, r, lr, lsl, Ct, NT;                              // lr = log2 r, lsl = log2 (Dk / r)
    float scale;
    int l2;
    int img;  // W and Kd stored as the tensor-core chain's bf16 hi | lo images, not in fp32
};

struct MbChunk {
    int ntok, nrows;
    size_t htok, ci;
};

__device__ __forceinline__ MbChunk mbchunk(const MbParams &p) {
    MbChunk ch;
    const int c = blockIdx.x, bh = blockIdx.y, t0 = c * p.Ct;
    ch.ntok = min(p.Ct, p.T - t0);
    ch.nrows = ch.ntok * p.r;
    ch.htok = (size_t)bh * p.T + t0;
    ch.ci = (size_t)bh * p.NT + c;
    return ch;
}

// The sub-rows' keys formed from the token keys Kt [tokens][ld]: row a,
// column c.  WRITE = false: kr (slice j of the token key times mask[i][j]);
// true: kw (slice i of the token key, zero elsewhere).
template <bool WRITE>
struct SubKey {
    const float *Kt, *msk;
    int ld, r, lr, lsl;
    __device__ __forceinline__ float operator()(int a, int c) const {
        const int i = a & (r - 1), j = c >> lsl;
        const float x = Kt[(a >> lr) * ld + c];
        return WRITE ? (j == i ? x : 0.f) : x * msk[i * r + j];
    }
};
// A key operand used transposed or with a column offset: (x, y) -> key(y, x + off).
template <class K>
struct Tr {
    K key;
    int off;
    __device__ __forceinline__ float operator()(int x, int y) const { return key(y, x + off); }
};
template <class K>
struct Off {
    K key;
    int off;
    __device__ __forceinline__ float operator()(int a, int c) const { return key(a, c + off); }
};
// A plain shared-memory operand: (m, k) -> X[m am + k ak].
struct Sm {
    const float *X;
    int am, ak;
    __device__ __forceinline__ float operator()(int m, int k) const { return X[m * am + k * ak]; }
};

// ============================================================ 1. WY factors
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) mbwd_wy_kernel(MbParams p) {
    extern __shared__ float sm[];
    // the key tiles are read by mm_nt (row strides 4 mod 32 words)
    constexpr int LK = DK + 4, LV = DV + 1, LX = (DK > DV ? DK : DV) + 4;
    float *Kt = sm;               // [64][LX] token keys, then W
    float *Kr = Kt + kC * LX;     // [64][LX] read keys, then -P^^T dO
    float *Kw = Kr + kC * LX;     // [64][LK] write keys
    float *Qs = Kw + kC * LK;     // [64][LK]
    float *Vs = Qs + kC * LK;     // [64][LV] sub-rows' values, then dO (queries)
    float *Xa = Vs + kC * LV, *Xb = Xa + kC * LC, *X4 = Xb + kC * LC;
    float *gam = X4 + kC * kC / 4, *eg = gam + kC, *bet = eg + kC, *nrm = bet + kC, *msk = nrm + kC;
    const MbChunk ch = mbchunk(p);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, r = p.r;

    // token keys into Kt with the row stride LX (loaded with the stride LK first)
    load_rows<T, DK, LK>(Kw, (const T *)p.k + ch.htok * DK, ch.ntok, p.l2 != 0, nrm);
    load_rows<T, DK, LK>(Qs, (const T *)p.q + ch.htok * DK, ch.ntok, p.l2 != 0, nrm);
    staged<kC * DV / kThr>(
        [&](int e) {
            const int a = e / DV;
            return a < ch.nrows ? ld_f((const T *)p.v + (ch.htok + (a >> p.lr)) * DV + e % DV) : 0.f;
        },
        [&](int e, float x) { Vs[(e / DV) * LV + e % DV] = x; });
    if (tid < kC) bet[tid] = tid < ch.nrows ? ld_f((const T *)p.beta + ch.htok + (tid >> p.lr)) : 0.f;
    if (tid < r * r) msk[tid] = p.mask[tid];
    if (tid < 32) {  // gamma per sub-row: the token's g enters on its first sub-row
        const int a0 = tid, a1 = tid + 32;
        float x0 = (a0 < ch.nrows && (a0 & (r - 1)) == 0) ? p.g[ch.htok + (a0 >> p.lr)] : 0.f;
        float x1 = (a1 < ch.nrows && (a1 & (r - 1)) == 0) ? p.g[ch.htok + (a1 >> p.lr)] : 0.f;
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
    for (int e = tid; e < kC * DK; e += kThr) Kt[(e / DK) * LX + e % DK] = Kw[(e / DK) * LK + e % DK];
    __syncthreads();
    for (int e = tid; e < kC * DK; e += kThr) {
        const int a = e / DK, c = e % DK, i = a & (r - 1), j = c >> p.lsl;
        const float x = Kt[(a >> p.lr) * LX + c];
        Kr[a * LX + c] = x * msk[i * r + j];
        Kw[a * LK + c] = j == i ? x : 0.f;
    }
    __syncthreads();
    {  // A over the sub-rows of earlier tokens
        float acc[2][4];
        zero(acc);
        mm_nt<kThr, 2, 4>(acc, Kr, LX, Kw, LK, DK);
        float *KKg = p.KKw + ch.ci * kC * kC;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int a = ty + 32 * i, b = tx + 16 * j;
                KKg[a * kC + b] = acc[i][j];
                Xa[a * LC + b] = (b >> p.lr) < (a >> p.lr) ? bet[a] * expf(gam[a] - gam[b]) * acc[i][j] : 0.f;
            }
    }
    __syncthreads();
    unit_lower_inverse<kC, kThr>(Xa, Xb, X4, LC);  // Xb = T
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
    float accW[2][DK / 16];
    zero(accW);
    mm<kThr, 2, DK / 16>(accW, Xa, LC, 1, Kr, LX, 1, kC);
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
    __syncthreads();  // Kt, Vs and Xa free
    {
        float *Wg = p.Ww + ch.ci * kC * DK;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < DK / 16; ++j) {
                const int m = ty + 32 * i, n = tx + 16 * j;
                if (!p.img) Wg[m * DK + n] = accW[i][j];
                Kt[m * LX + n] = accW[i][j];  // W
            }
        const float gl = gam[kC - 1];
        float *Kdg = p.Kdw + ch.ci * kC * DK;
        if (!p.img)
            for (int e = tid; e < kC * DK; e += kThr) Kdg[e] = expf(gl - gam[e / DK]) * Kw[(e / DK) * LK + e % DK];
        if (tid < kC) p.Gw[ch.ci * kC + tid] = gam[tid];
    }
    load_rows<T, DV>(Vs, (const T *)p.dout + ch.htok * DV, ch.ntok, false, nullptr);  // dO by query
    {  // P^ = scale e^{gamma_t - gamma_b} q_t . kw_b over the sub-rows of tokens up to t
        float acc[2][4];
        zero(acc);
        mm_nt<kThr, 2, 4>(acc, Qs, LK, Kw, LK, DK);
        float *Pg = p.Pw + ch.ci * kC * kC;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = ty + 32 * i, b = tx + 16 * j;
                const float x =
                    (t < ch.ntok && (b >> p.lr) <= t) ? p.scale * expf(gam[t * r] - gam[b]) * acc[i][j] : 0.f;
                Xa[t * LC + b] = x;
                Pg[t * kC + b] = x;
            }
    }
    __syncthreads();
    if constexpr (DK == 128) {
        if (p.img) {  // W (in Kt) and Kd = diag(e^{gl - gamma}) Kw as the chain's operand images
            const float gl = gam[kC - 1];
            write_chain_image<kThr>(reinterpret_cast<unsigned char *>(p.Ww + ch.ci * kC * DK), Kt, LX,
                                    [](int) { return 1.f; });
            write_chain_image<kThr>(reinterpret_cast<unsigned char *>(p.Kdw + ch.ci * kC * DK), Kw, LK,
                                    [&](int m) { return expf(gl - gam[m]); });
        }
    }
    {  // Kr = -P^^T dO; dO rows scaled by scale e^{gamma_t}
        float acc[2][DV / 16];
        zero(acc);
        mm<kThr, 2, DV / 16>(acc, Xa, 1, LC, Vs, LV, 1, kC);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) Kr[(ty + 32 * i) * LX + tx + 16 * j] = -acc[i][j];
        for (int e = tid; e < kC * DV; e += kThr) {
            const int t = e / DV, n = e % DV;
            if (t < ch.ntok) Vs[t * LV + n] *= p.scale * eg[t * r];
        }
    }
    __syncthreads();
    {  // B = Q^T (scaled dO) - W^T P^^T dO
        float acc[DK / 32][DV / 16];
        zero(acc);
        mm<kThr, DK / 32, DV / 16>(acc, Qs, 1, LK, Vs, LV, 1, kC);
        mm<kThr, DK / 32, DV / 16>(acc, Kt, 1, LX, Kr, LX, 1, kC);
        float *Bg = p.Bw + ch.ci * DK * DV;
#pragma unroll
        for (int i = 0; i < DK / 32; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) Bg[(ty + 32 * i) * DV + tx + 16 * j] = acc[i][j];
    }
}

// ===================================================== 3. the input gradients
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) mbwd_grad_kernel(MbParams p) {
    extern __shared__ float sm[];
    // the value-side tiles are read by mm_nt (row strides 4 mod 32 words)
    constexpr int LK = DK + 1, LV = DV + 4, TK = DK / 16, TV = DV / 16, NH = DK / 64;
    constexpr int LX = (DK > DV ? DK : DV) + 4;
    float *Kt = sm, *Qs = Kt + kC * LK, *Vns = Qs + kC * LK, *dOs = Vns + kC * LX, *Hs = dOs + kC * LV;
    float *Xa = Hs + kC * LV, *Xb = Xa + kC * LC;
    float *gam = Xb + kC * LC, *eg = gam + kC, *bet = eg + kC, *nk = bet + kC, *nq = nk + kC;
    // owner-written slots, summed in a fixed order (as in the chunk backward)
    float *rowg = nq + kC, *dbet = rowg + kC, *qg = dbet + kC, *lastg = qg + kC, *colg = lastg + kC;
    float *red = colg + 32 * kC, *msk = red + 16;
    const MbChunk ch = mbchunk(p);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, r = p.r, ntok = ch.ntok, nrows = ch.nrows;
    const int lr = p.lr, lsl = p.lsl;
    const T *vp = (const T *)p.v + ch.htok * DV;
    const float *Sg = p.Sw + ch.ci * DK * DV, *dSg = p.dSw + ch.ci * DK * DV;

    load_rows<T, DK>(Kt, (const T *)p.k + ch.htok * DK, ntok, p.l2 != 0, nk);
    load_rows<T, DK>(Qs, (const T *)p.q + ch.htok * DK, ntok, p.l2 != 0, nq);
    if (!p.img) {  // with the tensor-core products, dO and Vn enter only through them
        load_rows<T, DV, LV>(dOs, (const T *)p.dout + ch.htok * DV, ntok, false, nullptr);
        stage_rows<kC, DV>(Vns, LX, p.Vnw + ch.ci * kC * DV);
    }
    const float *Vg = p.Vnw + ch.ci * kC * DV;
    if (tid < kC) {
        gam[tid] = p.Gw[ch.ci * kC + tid];
        eg[tid] = expf(gam[tid]);
        bet[tid] = tid < nrows ? ld_f((const T *)p.beta + ch.htok + (tid >> lr)) : 0.f;
        rowg[tid] = 0.f;
        dbet[tid] = 0.f;
        qg[tid] = 0.f;
    }
    if (tid < r * r) msk[tid] = p.mask[tid];
    for (int e = tid; e < 32 * kC; e += kThr) colg[e] = 0.f;
    __syncthreads();
    const float gl = gam[kC - 1];
    const SubKey<false> KR{Kt, msk, LK, r, lr, lsl};
    const SubKey<true> KW{Kt, msk, LK, r, lr, lsl};
    // weights of a row's read- and write-key gradients in its share of dk
    auto wr = [&](int a, int c) { return msk[(a & (r - 1)) * r + (c >> lsl)]; };
    auto ww = [&](int a, int c) { return (c >> lsl) == (a & (r - 1)) ? 1.f : 0.f; };

    // 1. through the state leaving the chunk: Kd dS' (from the tensor-core chain,
    //    which forms it, when the chain ran there), and Vn dS'^T (write keys)
    float accKdS[2][TV], accD[2][TK];
    zero(accKdS);
    zero(accD);
    if (p.img) {  // from the products kernel (layout with ChunkProductsTcArgs): the rows' dk shares, <dS', S>
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) accD[i][j] = p.Bw[ch.ci * DK * DV + (ty + 32 * i) * DK + tx + 16 * j];
        if (tid < kThr / 32) red[tid] = tid == 0 ? p.Bw[ch.ci * DK * DV + 8192] : 0.f;
    } else {
        for (int h = 0; h < NH; ++h) {
            stage_rows<64, DV>(Hs, LV, dSg + (size_t)64 * h * DV);
            __syncthreads();
            mm_f<kThr, 2, TV>(accKdS, Off<SubKey<true>>{KW, 64 * h}, Sm{Hs, LV, 1}, 64);
            float tz[2][4];
            zero(tz);
            mm_nt<kThr, 2, 4>(tz, Vns, LX, Hs, LV, DV);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int a = ty + 32 * i;
                const float s = expf(gl - gam[a]);
#pragma unroll
                for (int j = 0; j < 4; ++j) accD[i][4 * h + j] += ww(a, 64 * h + tx + 16 * j) * s * tz[i][j];
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
    } else {  // Kw dS' -> Kd dS', and the decay gradients of the state's update
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
            for (int j = 0; j < TV; ++j) w += accKdS[i][j] * Vns[b * LX + tx + 16 * j];
            w = row_sum16(w);
            if (tx == 0) {
                rowg[b] -= w;
                lastg[b] = w;
            }
        }
    }
    // 2. P^ (formed by the WY kernel) into Xa, T into Xb (dR from the products kernel into Hs)
    {
        const float *Pg = p.Pw + ch.ci * kC * kC, *Tg = p.Tw + ch.ci * kC * kC;
        stage_rows<kC, kC>(Xa, LC, Pg);
        if (p.img)
            stage_rows<64, DV>(Hs, LV, Sg);
        else
            stage_rows<kC, kC>(Xb, LC, Tg);
    }
    __syncthreads();
    if (!p.img) {
        // 3. dVn = Kd dS' + P^^T dO into Hs
        mm<kThr, 2, TV>(accKdS, Xa, 1, LC, dOs, LV, 1, kC);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TV; ++j) Hs[(ty + 32 * i) * LV + tx + 16 * j] = accKdS[i][j];
        __syncthreads();
        // 4. dR = T^T dVn into Hs
        float acc[2][TV];
        zero(acc);
        mm<kThr, 2, TV>(acc, Xb, 1, LC, Hs, LV, 1, kC);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TV; ++j) Hs[(ty + 32 * i) * LV + tx + 16 * j] = acc[i][j];
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
            mm_nt<kThr, 2, 4>(acc, dOs, LV, Vns, LX, DV);
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
    // 6. dA = -dR Vn^T on the sub-rows of earlier tokens, with Kr Kw^T: dbeta,
    //    decay gradients, L into Xb
    {
        float ta[2][4], tk[2][4];
        zero(ta);
        if (p.img) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) ta[i][j] = Vg[(ty + 32 * i) * kC + tx + 16 * j];
        } else {
            mm_nt<kThr, 2, 4>(ta, Hs, LV, Vns, LX, DV);
        }
        {  // Kr Kw^T, formed by the WY kernel
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
                if ((c >> lr) < (b >> lr)) {
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
    // 7. dKw += P~^T Q + L^T Kr, dKr += L Kw (weighted into D); dq = P~ Kw  (X1 =
    //    P~^T Q + L^T Kr, X2 = L Kw and P~ Kw from the products kernel with the
    //    tensor-core chains)
    float accDQ[2][TK];
    zero(accDQ);
    if (p.img) {  // P~ Kw from the products kernel (the dk terms are in its shares already)
        const float *DQ = p.Ww + ch.ci * kC * DK;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                const int a = ty + 32 * i, c = tx + 16 * j;
                accDQ[i][j] = a < ntok ? DQ[a * DK + c] : 0.f;
            }
    } else {
        float t1[2][TK];
        zero(t1);
        mm<kThr, 2, TK>(t1, Xa, 1, LC, Qs, LK, 1, kC);
        mm_f<kThr, 2, TK>(t1, Sm{Xb, 1, LC}, KR, kC);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) accD[i][j] += ww(ty + 32 * i, tx + 16 * j) * t1[i][j];
        zero(t1);
        mm_f<kThr, 2, TK>(t1, Sm{Xb, LC, 1}, KW, kC);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) accD[i][j] += wr(ty + 32 * i, tx + 16 * j) * t1[i][j];
        mm_f<kThr, 2, TK>(accDQ, Sm{Xa, LC, 1}, KW, kC);
    }
    __syncthreads();
    // 8. through the state entering the chunk (staged in 64-row blocks of Dk in Vns):
    //    dq += diag(scale e^{gamma}) dO S^T and dKr -= diag(beta e^gamma) dR S^T; the same
    //    products give (S^T q_t).do_t = q_t.(S do_t) and (S^T kr_b).dR_b = kr_b.(S dR_b).
    float rq[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
    for (int h = 0; h < NH; ++h) {
        if (!p.img) stage_rows<64, DV>(Vns, LX, Sg + (size_t)64 * h * DV);
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
            mm_nt<kThr, 2, 4>(t1, dOs, LV, Vns, LX, DV);
            mm_nt<kThr, 2, 4>(t2, Hs, LV, Vns, LX, DV);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int m = ty + 32 * i;
            const float sq = m < ntok ? p.scale * eg[m * r] : 0.f;
            const float sk = bet[m] * eg[m];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 64 * h + tx + 16 * j;
                accDQ[i][4 * h + j] += sq * t1[i][j];
                accD[i][4 * h + j] -= wr(m, c) * sk * t2[i][j];
                rq[i] += Qs[m * LK + c] * t1[i][j];
                rk[i] += KR(m, c) * t2[i][j];
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int b = ty + 32 * i;
        float rv = 0.f;  // dR_b . v_(token of b)
#pragma unroll
        for (int j = 0; j < TV; ++j) {
            const int n = tx + 16 * j;
            rv += Hs[b * LV + n] * (b < nrows ? ld_f(vp + (size_t)(b >> lr) * DV + n) : 0.f);
        }
        rv = row_sum16(rv);
        const float sq = row_sum16(rq[i]), skr = row_sum16(rk[i]);
        const float skd = p.img ? p.Bw[ch.ci * DK * DV + 8320 + b] : skr;  // kr_b . t2_b
        if (tx == 0) {
            dbet[b] += rv - eg[b] * skd;
            rowg[b] -= bet[b] * eg[b] * skd;
            if (b < ntok) qg[b] += p.scale * eg[b * r] * sq;
        }
    }
    __syncthreads();

    // 9. dgamma in a fixed order, dg its reverse cumulative sum; dbeta and dv by token
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
        gam[a] = x;
    }
    // the rows' shares of dk into Vns
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < TK; ++j) Vns[(ty + 32 * i) * LX + tx + 16 * j] = accD[i][j];
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int a = kC - 1; a >= 0; --a) {
            s += gam[a];
            gam[a] = s;
        }
    }
    __syncthreads();
    if (tid < ntok) {
        float s = 0.f;
        for (int i = 0; i < r; ++i) s += dbet[tid * r + i];
        p.dbeta[ch.htok + tid] = s;
        p.dg[ch.htok + tid] = gam[tid * r];
    }
    // 10. by token (one warp each): dv, and dk through the unit-norm map
    {
        const int warp = tid >> 5, lane = tid & 31;
        T *dkp = (T *)p.dk + ch.htok * DK;
        T *dvp = (T *)p.dv + ch.htok * DV;
        for (int t = warp; t < ntok; t += kThr / 32) {
            for (int c = lane; c < DV; c += 32) {
                float s = 0.f;
                for (int i = 0; i < r; ++i) s += Hs[(t * r + i) * LV + c];
                st_f(dvp + (size_t)t * DV + c, bet[t * r] * s);
            }
            float x[DK / 32];
            float dot = 0.f;
#pragma unroll
            for (int u = 0; u < DK / 32; ++u) {
                const int c = lane + 32 * u;
                float s = 0.f;
                for (int i = 0; i < r; ++i) s += Vns[(t * r + i) * LX + c];
                x[u] = s;
                dot += Kt[t * LK + c] * s;
            }
            dot = warp_sum(dot);
#pragma unroll
            for (int u = 0; u < DK / 32; ++u) {
                const int c = lane + 32 * u;
                float xk = x[u];
                if (p.l2) xk = nk[t] < 1e-12f ? xk * 1e12f : (xk - Kt[t * LK + c] * dot) / nk[t];
                st_f(dkp + (size_t)t * DK + c, xk);
            }
        }
    }
    // dq through the unit-norm map
    T *dqp = (T *)p.dq + ch.htok * DK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int m = ty + 32 * i;
        float qd = 0.f;
#pragma unroll
        for (int j = 0; j < TK; ++j) qd += Qs[m * LK + tx + 16 * j] * accDQ[i][j];
        qd = row_sum16(qd);
#pragma unroll
        for (int j = 0; j < TK; ++j) {
            const int n = tx + 16 * j;
            float xq = accDQ[i][j];
            if (p.l2) xq = nq[m] < 1e-12f ? xq * 1e12f : (xq - Qs[m * LK + n] * qd) / nq[m];
            if (m < ntok) st_f(dqp + (size_t)m * DK + n, xq);
        }
    }
}

constexpr size_t mwy_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)2 * kC * ((DK > DV ? DK : DV) + 4) + 2 * kC * (DK + 4) + kC * (DV + 1) +
                            2 * kC * LC + kC * kC / 4 + 4 * kC + 64);
}
constexpr size_t mgrad_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)2 * kC * (DK + 1) + kC * ((DK > DV ? DK : DV) + 4) + 2 * kC * (DV + 4) +
                            2 * kC * LC + 9 * kC + 32 * kC + 16 + 64);
}

size_t per_chunk_floats(int Dk, int Dv) {
    return 3 * (size_t)kC * kC + 2 * (size_t)kC * Dk + 2 * (size_t)kC * Dv + 3 * (size_t)Dk * Dv + kC;
}

int ilog2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

template <typename T, int DK, int DV>
int run(const MaskedBwdArgs &a, cudaStream_t st) {
    const int BH = a.B * a.H, Ct = kC / a.r, NT = (a.T + Ct - 1) / Ct;
    const size_t nc = (size_t)BH * NT;
    float *w = static_cast<float *>(a.ws);
    MbParams p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.beta = a.beta;
    p.dout = a.dout;
    p.g = a.g;
    p.mask = a.mask;
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
    p.lr = ilog2(a.r);
    p.lsl = ilog2(DK / a.r);
    p.Ct = Ct;
    p.NT = NT;
    p.scale = a.scale;
    p.l2 = (a.flags & GDN_QK_L2NORM) ? 1 : 0;
    constexpr size_t s1 = mwy_smem(DK, DV), s2 = wy_chain_smem<DK, kSlice>(), s3 = mgrad_smem(DK, DV);
    if (cudaFuncSetAttribute(mbwd_wy_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(wy_chain_kernel<DK, DV, kSlice>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s2) != cudaSuccess ||
        cudaFuncSetAttribute(mbwd_grad_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3) !=
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
        ta.mask = a.mask;
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
        ta.masked = 1;
        ta.bwd = 1;
        ta.scale = a.scale;
        const int rc = launch_wy_tc(ta, st);
        if (rc != GDN_OK) return rc;
    } else {
        mbwd_wy_kernel<T, DK, DV><<<dim3((unsigned)NT, (unsigned)BH), kThr, s1, st>>>(p);
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
        sa.dout = static_cast<const unsigned short *>(a.dout);
        sa.BH = BH;
        sa.NT = NT;
        sa.T = a.T;
        sa.Ct = p.Ct;
        sa.Uw = p.Uw;
        sa.Ww = p.Ww;
        sa.Pw = p.Pw;
        sa.Tw = p.Tw;
        sa.Gw = p.Gw;
        sa.q = static_cast<const unsigned short *>(a.q);
        sa.k = static_cast<const unsigned short *>(a.k);
        sa.beta = static_cast<const unsigned short *>(a.beta);
        sa.mask = a.mask;
        sa.r = a.r;
        sa.masked = 1;
        sa.l2 = p.l2;
        sa.scale = a.scale;
        rc = launch_chunk_products_tc(sa, st);
        if (rc != GDN_OK) return rc;
    } else {
        WyChainParams cp{p.s0, p.dsf, nullptr, p.ds0, p.Sw, p.dSw, p.Ww, p.Kdw, p.Uw, p.Vnw, p.Bw, p.Gw, NT};
        wy_chain_kernel<DK, DV, kSlice><<<dim3((unsigned)(DV / kSlice), (unsigned)BH, 2), kChainThr, s2, st>>>(cp);
        note_launch();
    }
    mbwd_grad_kernel<T, DK, DV><<<dim3((unsigned)NT, (unsigned)BH), kThr, s3, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int run_t(const MaskedBwdArgs &a, cudaStream_t st) {
    if (a.Dk == 128 && a.Dv == 128) return run<T, 128, 128>(a, st);
    if (a.Dk == 128 && a.Dv == 64) return run<T, 128, 64>(a, st);
    if (a.Dk == 64 && a.Dv == 128) return run<T, 64, 128>(a, st);
    if (a.Dk == 64 && a.Dv == 64) return run<T, 64, 64>(a, st);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace

size_t masked_bwd_workspace_bytes(const MaskedBwdArgs &a) {
    if (a.r < 1 || a.r > 8 || kC % a.r != 0 || a.T <= 0) return 0;
    const int Ct = kC / a.r, NT = (a.T + Ct - 1) / Ct;
    return sizeof(float) * (size_t)a.B * a.H * NT * per_chunk_floats(a.Dk, a.Dv);
}

int launch_masked_bwd(const MaskedBwdArgs &a, cudaStream_t stream) {
    if (a.r < 1 || a.r > 8 || kC % a.r != 0 || a.Dk % a.r != 0) return GDN_ERR_UNSUPPORTED;
    return a.dtype == GDN_BF16 ? run_t<__nv_bfloat16>(a, stream) : run_t<float>(a, stream);
}

}  // namespace gdn
