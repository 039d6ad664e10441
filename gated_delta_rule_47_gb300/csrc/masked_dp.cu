// masked_dp.cu -- block-masked DeltaProduct forward, the chunk-local kernels on
// the CUDA cores in fp32 (gated_deltaproduct test.py: the mask_ij coupling of
// `gated_chunk_scaled_dot_kkt_fwd_kernel` and `gated_fwd_recompute_w_u_kernel`,
// the per-slice state update of `gated_chunk_delta_rule_fwd_kernel_h`, and the
// sum over r of `gated_chunk_fwd_o_fn`).
//
// The key dimension is cut into r slices of Dk/r.  Token t has r sub-rows
// (t, i): sub-row i predicts from the token's decayed state with the read key
// kr_(t,i) = k_t masked slice-wise by mask[i][:] (slice j scaled by
// mask[i][j]), and writes the state's slice-i rows with the write key
// kw_(t,i) = slice i of k_t (zero elsewhere); all sub-rows of a token act on
// the same state and share v_t and beta_t.  In the WY form over the chunk's
// sub-rows a = (t, i), with gamma the cumulative log-decay (one value per
// token) and S the state entering the chunk:
//   A[a][b] = beta_a e^{gamma_a - gamma_b} kr_a . kw_b   for token(b) < token(a)
//   T = (I + A)^-1,  W = T diag(beta e^gamma) Kr,  U = T diag(beta) V
//   Vn = U - W S,    S <- e^{gamma_last} S + Kw^T diag(e^{gamma_last - gamma}) Vn
//   o_t = scale (e^{gamma_t} S^T q_t + sum_{token(b) <= t} e^{gamma_t - gamma_b} (q_t . kw_b) vn_b)
// Three launches on 64-row chunks (64 / r tokens; r divides 64):
//   1. mdp_wy_kernel (one CTA per chunk): the keys, A, T, W, U,
//      Kd = diag(e^{gamma_last - gamma}) Kw, and the output factors
//      P[t][b] = scale e^{gamma_t - gamma_b} q_t . kw_b (token(b) <= t).
//   2. the state chain: the state entering each chunk and Vn, and the final
//      state; wy_chain_tc_kernel (tcgen05, one CTA per head) for bf16 at
//      Dk = Dv = 128, with W and Kd handed over as operand images, else
//      wy_chain_kernel (CUDA cores, fp32, 32 value columns per CTA).
//   3. mdp_out_kernel (one CTA per chunk): o = diag(scale e^gamma) Q S + P Vn.
// Tokens past the end of the sequence have k = v = beta = 0 and g = 0, so
// they change nothing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "gdn_internal.h"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"
#include "wy_chain.cuh"

namespace gdn {
namespace {

using namespace tile;
constexpr int LC = kC + 1;
constexpr int kMaxR = 8;
constexpr int kMSlice = 32;  // value columns per chain CTA

struct MdpParams {
    const void *q, *k, *v, *beta;
    const float *g, *mask;
    void *o;
    // workspace, per (head, chunk): W, Kd [64][Dk]; U, Vn [64][Dv]; S [Dk][Dv];
    // P [64][64]; gamma [64]
    float *Ww, *Kdw, *Uw, *Vnw, *Sw, *Pw, *Gw;
    int T, r, Ct, NT;
    float scale;
    int l2;
    int img;  // W and Kd stored as the tensor-core chain's bf16 hi | lo images, not in fp32
};

struct MChunk {
    int ntok, nrows;
    size_t htok, ci;
};

__device__ __forceinline__ MChunk mchunk(const MdpParams &p) {
    MChunk ch;
    const int c = blockIdx.x, bh = blockIdx.y, t0 = c * p.Ct;
    ch.ntok = min(p.Ct, p.T - t0);
    ch.nrows = ch.ntok * p.r;
    ch.htok = (size_t)bh * p.T + t0;
    ch.ci = (size_t)bh * p.NT + c;
    return ch;
}

// ============================================================ 1. WY factors
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) mdp_wy_kernel(MdpParams p) {
    extern __shared__ float sm[];
    constexpr int LK = DK + 4, LV = DV + 1;  // the key tiles are read by mm_nt (row stride 4 mod 32 words)
    float *Kt = sm;                // [64][LK] token keys (unit when asked)
    float *Kr = Kt + kC * LK;      // [64][LK] read keys of the sub-rows
    float *Kw = Kr + kC * LK;      // [64][LK] write keys of the sub-rows
    float *Qs = Kw + kC * LK;      // [64][LK] queries
    float *Vs = Qs + kC * LK;      // [64][LV] values of the sub-rows
    float *Xa = Vs + kC * LV, *Xb = Xa + kC * LC, *X4 = Xb + kC * LC;
    float *gam = X4 + kC * kC / 4, *eg = gam + kC, *bet = eg + kC, *nrm = bet + kC, *msk = nrm + kC;
    const MChunk ch = mchunk(p);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, r = p.r, sl = DK / r;

    load_rows<T, DK, LK>(Kt, (const T *)p.k + ch.htok * DK, ch.ntok, p.l2 != 0, nrm);
    load_rows<T, DK, LK>(Qs, (const T *)p.q + ch.htok * DK, ch.ntok, p.l2 != 0, nrm);
    staged<kC * DV / kThr>(
        [&](int e) {
            const int a = e / DV;
            return a < ch.nrows ? ld_f((const T *)p.v + (ch.htok + a / r) * DV + e % DV) : 0.f;
        },
        [&](int e, float x) { Vs[(e / DV) * LV + e % DV] = x; });
    if (tid < kC) bet[tid] = tid < ch.nrows ? ld_f((const T *)p.beta + ch.htok + tid / r) : 0.f;
    if (tid < r * r) msk[tid] = p.mask[tid];
    if (tid < 32) {  // gamma per sub-row: the token's g enters on its first sub-row
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
    // the sub-rows' read and write keys
    for (int e = tid; e < kC * DK; e += kThr) {
        const int a = e / DK, c = e % DK, i = a % r, j = c / sl;
        const float x = Kt[(a / r) * LK + c];
        Kr[a * LK + c] = x * msk[i * r + j];
        Kw[a * LK + c] = j == i ? x : 0.f;
    }
    __syncthreads();
    // A over the sub-rows of earlier tokens
    {
        float acc[2][4];
        zero(acc);
        mm_nt<kThr, 2, 4>(acc, Kr, LK, Kw, LK, DK);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int a = ty + 32 * i, b = tx + 16 * j;
                Xa[a * LC + b] = b / r < a / r ? bet[a] * expf(gam[a] - gam[b]) * acc[i][j] : 0.f;
            }
    }
    __syncthreads();
    unit_lower_inverse<kC, kThr>(Xa, Xb, X4, LC);  // Xb = T
    for (int e = tid; e < kC * kC; e += kThr) {
        const int m = e / kC, b = e % kC;
        const float t = Xb[m * LC + b];
        Xa[m * LC + b] = t * bet[b] * eg[b];
        Xb[m * LC + b] = t * bet[b];
    }
    __syncthreads();
    {
        float acc[2][DK / 16];
        zero(acc);
        mm<kThr, 2, DK / 16>(acc, Xa, LC, 1, Kr, LK, 1, kC);
        float *Wg = p.Ww + ch.ci * kC * DK;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < DK / 16; ++j) {
                if (p.img)
                    Kt[(ty + 32 * i) * LK + tx + 16 * j] = acc[i][j];  // the token keys are no longer needed
                else
                    Wg[(ty + 32 * i) * DK + tx + 16 * j] = acc[i][j];
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
        if (!p.img)
            for (int e = tid; e < kC * DK; e += kThr) Kdg[e] = expf(gl - gam[e / DK]) * Kw[(e / DK) * LK + e % DK];
        if (tid < kC) p.Gw[ch.ci * kC + tid] = gam[tid];
    }
    // the output factors P[t][b] over the sub-rows of tokens up to t
    {
        float acc[2][4];
        zero(acc);
        mm_nt<kThr, 2, 4>(acc, Qs, LK, Kw, LK, DK);
        float *Pg = p.Pw + ch.ci * kC * kC;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = ty + 32 * i, b = tx + 16 * j;
                Pg[t * kC + b] = (t < ch.ntok && b / r <= t) ? p.scale * expf(gam[t * r] - gam[b]) * acc[i][j] : 0.f;
            }
    }
    if constexpr (DK == 128) {
        if (p.img) {  // W (in Kt) and Kd = diag(e^{gl - gamma}) Kw as the chain's operand images
            __syncthreads();
            const float gl = gam[kC - 1];
            write_chain_image<kThr>(reinterpret_cast<unsigned char *>(p.Ww + ch.ci * kC * DK), Kt, LK,
                                    [](int) { return 1.f; });
            write_chain_image<kThr>(reinterpret_cast<unsigned char *>(p.Kdw + ch.ci * kC * DK), Kw, LK,
                                    [&](int m) { return expf(gl - gam[m]); });
        }
    }
}

// ============================================================== 3. outputs
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr, 1) mdp_out_kernel(MdpParams p) {
    extern __shared__ float sm[];
    // both products read their operands along k with 16-byte loads (mm_nt), so
    // Vn and the blocks of S are staged transposed; row strides 4 mod 32 words
    constexpr int LK = DK + 4, LT = kC + 4, NH = DK / 64;
    float *Qs = sm;              // [64][LK]
    float *VnT = Qs + kC * LK;   // [DV][LT] Vn transposed
    float *HsT = VnT + DV * LT;  // [DV][LT] a 64-row block of S, transposed
    float *Ps = HsT + DV * LT;   // [64][LT]
    float *gam = Ps + kC * LT, *nrm = gam + kC;
    const MChunk ch = mchunk(p);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, r = p.r;
    const float *Sg = p.Sw + ch.ci * DK * DV;

    load_rows<T, DK, LK>(Qs, (const T *)p.q + ch.htok * DK, ch.ntok, p.l2 != 0, nrm);
    const float *Vg = p.Vnw + ch.ci * kC * DV;
    staged<kC * DV / kThr>([&](int e) { return Vg[e]; }, [&](int e, float x) { VnT[(e % DV) * LT + e / DV] = x; });
    stage_rows<kC, kC>(Ps, LT, p.Pw + ch.ci * kC * kC);
    if (tid < kC) gam[tid] = p.Gw[ch.ci * kC + tid];
    float accQS[2][DV / 16], accPV[2][DV / 16];
    zero(accQS);
    zero(accPV);
    for (int h = 0; h < NH; ++h) {
        __syncthreads();
        const float *Sb = Sg + (size_t)64 * h * DV;
        staged<64 * DV / kThr>([&](int e) { return Sb[e]; }, [&](int e, float x) { HsT[(e % DV) * LT + e / DV] = x; });
        __syncthreads();
        mm_nt<kThr, 2, DV / 16>(accQS, Qs + 64 * h, LK, HsT, LT, 64);
    }
    mm_nt<kThr, 2, DV / 16>(accPV, Ps, LT, VnT, LT, kC);
    T *op = (T *)p.o + ch.htok * DV;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = ty + 32 * i;
        if (t < ch.ntok) {
            const float qs = p.scale * expf(gam[t * r]);
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) st_f(op + (size_t)t * DV + tx + 16 * j, qs * accQS[i][j] + accPV[i][j]);
        }
    }
}

constexpr size_t wy_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)4 * kC * (DK + 4) + kC * (DV + 1) + 2 * kC * LC + kC * kC / 4 + 4 * kC + 64);
}
constexpr size_t out_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)kC * (DK + 4) + 2 * (size_t)DV * (kC + 4) + kC * (kC + 4) + 2 * kC);
}

size_t per_chunk_floats(int Dk, int Dv) {
    return 2 * (size_t)kC * Dk + 2 * (size_t)kC * Dv + (size_t)Dk * Dv + (size_t)kC * kC + kC;
}

template <typename T, int DK, int DV>
int run(const MaskedDpArgs &a, cudaStream_t st) {
    const int BH = a.B * a.H, Ct = kC / a.r, NT = (a.T + Ct - 1) / Ct;
    const size_t nc = (size_t)BH * NT;
    float *w = static_cast<float *>(a.ws);
    MdpParams p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.beta = a.beta;
    p.g = a.g;
    p.mask = a.mask;
    p.o = a.o;
    p.Ww = w;
    p.Kdw = p.Ww + nc * kC * DK;
    p.Uw = p.Kdw + nc * kC * DK;
    p.Vnw = p.Uw + nc * kC * DV;
    p.Sw = p.Vnw + nc * kC * DV;
    p.Pw = p.Sw + nc * DK * DV;
    p.Gw = p.Pw + nc * kC * kC;
    p.T = a.T;
    p.r = a.r;
    p.Ct = Ct;
    p.NT = NT;
    p.scale = a.scale;
    p.l2 = (a.flags & GDN_QK_L2NORM) ? 1 : 0;
    constexpr size_t s1 = wy_smem(DK, DV), s2 = wy_chain_smem<DK, kMSlice>(), s3 = out_smem(DK, DV);
    if (cudaFuncSetAttribute(mdp_wy_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(wy_chain_kernel<DK, DV, kMSlice>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s2) != cudaSuccess ||
        cudaFuncSetAttribute(mdp_out_kernel<T, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3) !=
            cudaSuccess)
        return GDN_ERR_CUDA;
    // the state chain on tcgen05 for bf16 at Dk = Dv = 128 (W and Kd then travel as operand images)
    const bool tc_chain = std::is_same<T, __nv_bfloat16>::value && DK == 128 && DV == 128 &&
                          !(a.flags & GDN_PATH_SIMT) && sm100_family();
    p.img = tc_chain ? 1 : 0;
    // with the tensor-core chain the chunk-local kernels run on tcgen05 too
    WyTcArgs ta{};
    if (tc_chain) {
        ta.q = static_cast<const unsigned short *>(a.q);
        ta.k = static_cast<const unsigned short *>(a.k);
        ta.v = static_cast<const unsigned short *>(a.v);
        ta.beta = static_cast<const unsigned short *>(a.beta);
        ta.g = a.g;
        ta.mask = a.mask;
        ta.o = static_cast<unsigned short *>(a.o);
        ta.Ww = p.Ww;
        ta.Kdw = p.Kdw;
        ta.Uw = p.Uw;
        ta.Vnw = p.Vnw;
        ta.Sw = p.Sw;
        ta.Pw = p.Pw;
        ta.Gw = p.Gw;
        ta.BH = BH;
        ta.T = a.T;
        ta.r = a.r;
        ta.Ct = Ct;
        ta.NT = NT;
        ta.l2 = p.l2;
        ta.scale = a.scale;
        ta.masked = 1;
        const int rc = launch_wy_tc(ta, st);
        if (rc != GDN_OK) return rc;
    } else {
        mdp_wy_kernel<T, DK, DV><<<dim3((unsigned)NT, (unsigned)BH), kThr, s1, st>>>(p);
        note_launch();
    }
    if (tc_chain) {
        WyChainTcArgs ca{};
        ca.s0 = a.s0;
        ca.sf = a.sf;
        ca.Sw = p.Sw;
        ca.Vnw = p.Vnw;
        ca.Wimg = reinterpret_cast<const unsigned char *>(p.Ww);
        ca.Kdimg = reinterpret_cast<const unsigned char *>(p.Kdw);
        ca.Uw = p.Uw;
        ca.Gw = p.Gw;
        ca.BH = BH;
        ca.NT = NT;
        ca.roles = 1;
        const int rc = launch_wy_chain_tc(ca, st);
        if (rc != GDN_OK) return rc;
    } else {
        WyChainParams cp{a.s0, nullptr, a.sf, nullptr, p.Sw, nullptr, p.Ww, p.Kdw, p.Uw, p.Vnw, nullptr, p.Gw, NT};
        wy_chain_kernel<DK, DV, kMSlice><<<dim3((unsigned)(DV / kMSlice), (unsigned)BH, 1), kChainThr, s2, st>>>(cp);
        note_launch();
    }
    if (tc_chain) return launch_masked_out_tc(ta, st);
    mdp_out_kernel<T, DK, DV><<<dim3((unsigned)NT, (unsigned)BH), kThr, s3, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int run_t(const MaskedDpArgs &a, cudaStream_t st) {
    if (a.Dk == 128 && a.Dv == 128) return run<T, 128, 128>(a, st);
    if (a.Dk == 128 && a.Dv == 64) return run<T, 128, 64>(a, st);
    if (a.Dk == 64 && a.Dv == 128) return run<T, 64, 128>(a, st);
    if (a.Dk == 64 && a.Dv == 64) return run<T, 64, 64>(a, st);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace

size_t masked_dp_workspace_bytes(const MaskedDpArgs &a) {
    if (a.r < 1 || a.r > kMaxR || kC % a.r != 0 || a.T <= 0) return 0;
    const int Ct = kC / a.r, NT = (a.T + Ct - 1) / Ct;
    return sizeof(float) * (size_t)a.B * a.H * NT * per_chunk_floats(a.Dk, a.Dv);
}

int launch_masked_dp(const MaskedDpArgs &a, cudaStream_t stream) {
    if (a.r > kMaxR || kC % a.r != 0) return GDN_ERR_UNSUPPORTED;
    if (a.dtype == GDN_F32) return run_t<float>(a, stream);
    if (a.dtype == GDN_BF16) return run_t<__nv_bfloat16>(a, stream);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
