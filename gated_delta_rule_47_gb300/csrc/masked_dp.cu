// masked_dp.cu -- block-masked DeltaProduct forward on the CUDA cores, fp32
// arithmetic (gated_deltaproduct test.py: the mask_ij coupling of
// `gated_chunk_scaled_dot_kkt_fwd_kernel` and `gated_fwd_recompute_w_u_kernel`,
// the per-slice state update of `gated_chunk_delta_rule_fwd_kernel_h`, and the
// sum over r of `gated_chunk_fwd_o_fn`).
//
// The key dimension is cut into r slices of dk = Dk/r.  Token t has r sub-rows
// (t, i): sub-row i predicts from the token's decayed state with the read key
// k_t masked slice-wise by mask[i][:], and writes the state's slice-i rows with
// the write key k_t,(i); all sub-rows of a token act on the same state.  Per
// chunk of CQ tokens (rows rho = (t, i), C = CQ r), from state S:
//   G_t       = within-chunk cumulative log-decay
//   A[(t,i),(s,j)] = beta_t e^{G_t - G_s} mask[i][j] (k_t,(j) . k_s,(j)),  s < t
//   R[(t,i)]  = beta_t (v_t - e^{G_t} sum_j mask[i][j] S_(j)^T k_t,(j))
//   Delta     = (I + A)^-1 R
//   o_t       = scale (e^{G_t} S^T q_t + sum_{s<=t, j} e^{G_t-G_s} (q_t,(j) . k_s,(j)) Delta_(s,j))
//   S_(j)    <- e^{G_last} S_(j) + sum_s e^{G_last - G_s} k_s,(j) Delta_(s,j)^T
// One CTA per (batch*head, 64-wide value tile), the fp32 state tile resident in
// shared memory.  Tokens past the end of the sequence have k = v = beta = 0 and
// g = 0, so they change nothing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "tri_inverse.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kBV = 64;
constexpr int kMaxR = 8;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

struct MdpParams {
    const void *q, *k, *v, *beta;
    const float *g, *mask, *s0;
    void *o;
    float *sf;
    int T, r, Dv;
    float scale;
    unsigned flags;
};

template <int DK, int C>
struct MdpSmem {
    static constexpr int KP = DK + 1, VP = kBV + 1, CP = C + 1;
    // Ks, Qs [C][KP]; Vs [C][VP]; Ss [DK][VP]; As, Ts, Ps [C][CP]; Rs, Ds [C][VP];
    // gam, bet, eS [C]; mask [kMaxR * kMaxR]
    static constexpr int floats =
        2 * C * KP + C * VP + DK * VP + 3 * C * CP + 2 * C * VP + 3 * C + kMaxR * kMaxR + C * C / 4;
    static constexpr size_t bytes = sizeof(float) * floats;
};

__device__ __forceinline__ void warp_cumsum64(float *x, int n, int lane) {
    float a = lane < n ? x[lane] : 0.f;
    float b = lane + 32 < n ? x[lane + 32] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float ya = __shfl_up_sync(0xffffffffu, a, off);
        const float yb = __shfl_up_sync(0xffffffffu, b, off);
        if (lane >= off) {
            a += ya;
            b += yb;
        }
    }
    b += __shfl_sync(0xffffffffu, a, 31);
    __syncwarp();
    if (lane < n) x[lane] = a;
    if (lane + 32 < n) x[lane + 32] = b;
}

template <int DK>
__device__ void unit_rows(float *X, int stride, int nrows, int warp, int lane, int nwarps) {
    for (int t = warp; t < nrows; t += nwarps) {
        float s = 0.f;
        for (int d = lane; d < DK; d += 32) s += X[t * stride + d] * X[t * stride + d];
#pragma unroll
        for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float inv = 1.f / fmaxf(sqrtf(s), 1e-12f);
        for (int d = lane; d < DK; d += 32) X[t * stride + d] *= inv;
    }
}

template <typename Tin, int DK, int C>
__global__ void __launch_bounds__(kThreads) masked_dp_kernel(MdpParams p) {
    using L = MdpSmem<DK, C>;
    constexpr int KP = L::KP, VP = L::VP, CP = L::CP;
    extern __shared__ float smem[];
    float *Ks = smem;            // [CQ][KP] token keys
    float *Qs = Ks + C * KP;     // [CQ][KP] token queries
    float *Vs = Qs + C * KP;     // [CQ][VP] token values (value tile)
    float *Ss = Vs + C * VP;     // [DK][VP] state tile
    float *As = Ss + DK * VP;    // [C][CP]  A over sub-rows
    float *Ts = As + C * CP;     // [C][CP]  (I + A)^-1
    float *Ps = Ts + C * CP;     // [CQ][CP] decay-masked slice-wise q.k scores, s <= t
    float *Rs = Ps + C * CP;     // [C][VP]  R
    float *Ds = Rs + C * VP;     // [C][VP]  per-slice predictions, then Delta
    float *gam = Ds + C * VP;    // [CQ]
    float *bet = gam + C;        // [CQ]
    float *eS = bet + C;         // [CQ] exp(gam_last - gam_s)
    float *msk = eS + C;         // [r][r]
    float *Xs = msk + kMaxR * kMaxR;  // [C*C/4] scratch of the blocked inverse

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vt = blockIdx.x;
    const size_t head = blockIdx.y;
    const int r = p.r, Dv = p.Dv, T = p.T;
    const int CQ = C / r;  // tokens per chunk
    const int dk = DK / r;

    const Tin *kp = static_cast<const Tin *>(p.k) + head * (size_t)T * DK;
    const Tin *qp = static_cast<const Tin *>(p.q) + head * (size_t)T * DK;
    const Tin *vp = static_cast<const Tin *>(p.v) + head * (size_t)T * Dv + vt * kBV;
    const Tin *bp = static_cast<const Tin *>(p.beta) + head * (size_t)T;
    const float *gp = p.g + head * (size_t)T;
    Tin *op = static_cast<Tin *>(p.o) + head * (size_t)T * Dv + vt * kBV;

    for (int i = tid; i < DK * kBV; i += kThreads) {
        const int d = i / kBV, j = i % kBV;
        Ss[d * VP + j] = p.s0 ? p.s0[(head * DK + d) * Dv + vt * kBV + j] : 0.f;
    }
    if (tid < r * r) msk[tid] = p.mask[tid];

    for (long c0 = 0; c0 < T; c0 += CQ) {
        const int LQ = (int)min((long)CQ, (long)T - c0);  // valid tokens
        __syncthreads();
        for (int i = tid; i < CQ * DK; i += kThreads) {
            const int t = i / DK, d = i % DK;
            Ks[t * KP + d] = t < LQ ? to_f32(kp[(c0 + t) * DK + d]) : 0.f;
            Qs[t * KP + d] = t < LQ ? to_f32(qp[(c0 + t) * DK + d]) : 0.f;
        }
        for (int i = tid; i < CQ * kBV; i += kThreads) {
            const int t = i / kBV, j = i % kBV;
            Vs[t * VP + j] = t < LQ ? to_f32(vp[(c0 + t) * Dv + j]) : 0.f;
        }
        if (tid < C) {
            const bool ok = tid < LQ;
            bet[tid] = ok ? to_f32(bp[c0 + tid]) : 0.f;
            gam[tid] = ok ? gp[c0 + tid] : 0.f;
        }
        __syncthreads();
        if (p.flags & GDN_QK_L2NORM) {
            unit_rows<DK>(Ks, KP, LQ, warp, lane, kThreads / 32);
            unit_rows<DK>(Qs, KP, LQ, warp, lane, kThreads / 32);
        }
        if (warp == 0) warp_cumsum64(gam, CQ, lane);
        __syncthreads();
        const float glast = gam[CQ - 1];
        if (tid < CQ) eS[tid] = expf(glast - gam[tid]);

        // A over sub-rows, and the slice-wise query-key scores
        for (int e = tid; e < C * C; e += kThreads) {
            const int rho = e / C, rho2 = e % C;
            const int t = rho / r, i = rho % r, s = rho2 / r, j = rho2 % r;
            float a = 0.f;
            if (s < t) {
                float acc = 0.f;
                for (int d = j * dk; d < (j + 1) * dk; ++d) acc += Ks[t * KP + d] * Ks[s * KP + d];
                a = bet[t] * expf(gam[t] - gam[s]) * msk[i * r + j] * acc;
            }
            As[rho * CP + rho2] = a;
            if (rho < CQ) {  // query row t = rho against sub-row (s, j)
                float pv = 0.f;
                if (s <= rho) {
                    float acc = 0.f;
                    for (int d = j * dk; d < (j + 1) * dk; ++d) acc += Qs[rho * KP + d] * Ks[s * KP + d];
                    pv = expf(gam[rho] - gam[s]) * acc;
                }
                Ps[rho * CP + rho2] = pv;
            }
        }
        // per-slice predictions Z[(t,j)] = S_(j)^T k_t,(j) into Ds
        for (int e = tid; e < C * kBV; e += kThreads) {
            const int rho = e / kBV, c = e % kBV;
            const int t = rho / r, j = rho % r;
            float acc = 0.f;
            for (int d = j * dk; d < (j + 1) * dk; ++d) acc += Ks[t * KP + d] * Ss[d * VP + c];
            Ds[rho * VP + c] = acc;
        }
        __syncthreads();
        // R[(t,i)] = beta_t (v_t - e^{G_t} sum_j mask[i][j] Z[(t,j)])
        for (int e = tid; e < C * kBV; e += kThreads) {
            const int rho = e / kBV, c = e % kBV;
            const int t = rho / r, i = rho % r;
            float pr = 0.f;
            for (int j = 0; j < r; ++j) pr += msk[i * r + j] * Ds[(t * r + j) * VP + c];
            Rs[rho * VP + c] = bet[t] * (Vs[t * VP + c] - expf(gam[t]) * pr);
        }
        // (I + A)^-1: 16 x 16 diagonal blocks, then the 16- and 32-level merges
        unit_lower_inverse<C, kThreads>(As, Ts, Xs, CP);
        // Delta = (I + A)^-1 R
        for (int e = tid; e < C * kBV; e += kThreads) {
            const int rho = e / kBV, c = e % kBV;
            float acc = 0.f;
            for (int s = 0; s <= rho; ++s) acc += Ts[rho * CP + s] * Rs[s * VP + c];
            Ds[rho * VP + c] = acc;
        }
        __syncthreads();
        // outputs of the chunk's tokens (the state before this chunk's update)
        for (int e = tid; e < LQ * kBV; e += kThreads) {
            const int t = e / kBV, c = e % kBV;
            float inter = 0.f;
            for (int d = 0; d < DK; ++d) inter += Qs[t * KP + d] * Ss[d * VP + c];
            float intra = 0.f;
            for (int rho2 = 0; rho2 < (t + 1) * r; ++rho2) intra += Ps[t * CP + rho2] * Ds[rho2 * VP + c];
            from_f32(op + (c0 + t) * Dv + c, p.scale * (expf(gam[t]) * inter + intra));
        }
        __syncthreads();
        // state update: slice j rows take the sub-rows (s, j)
        const float dl = expf(glast);
        for (int e = tid; e < DK * kBV; e += kThreads) {
            const int d = e / kBV, c = e % kBV;
            const int j = d / dk;
            float acc = 0.f;
            for (int s = 0; s < CQ; ++s) acc += Ks[s * KP + d] * eS[s] * Ds[(s * r + j) * VP + c];
            Ss[d * VP + c] = dl * Ss[d * VP + c] + acc;
        }
    }
    __syncthreads();
    if (p.sf) {
        for (int i = tid; i < DK * kBV; i += kThreads) {
            const int d = i / kBV, j = i % kBV;
            p.sf[(head * DK + d) * Dv + vt * kBV + j] = Ss[d * VP + j];
        }
    }
}

template <typename Tin, int DK, int C>
int launch_one(const MaskedDpArgs &a, cudaStream_t stream) {
    auto kern = masked_dp_kernel<Tin, DK, C>;
    constexpr size_t smem = MdpSmem<DK, C>::bytes;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    MdpParams p{a.q, a.k, a.v, a.beta, a.g, a.mask, a.s0, a.o, a.sf, a.T, a.r, a.Dv, a.scale, a.flags};
    dim3 grid(a.Dv / kBV, a.B * a.H);
    kern<<<grid, kThreads, smem, stream>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename Tin, int DK>
int launch_chunk(const MaskedDpArgs &a, cudaStream_t stream) {
    switch (a.chunk) {
        case 16: return launch_one<Tin, DK, 16>(a, stream);
        case 32: return launch_one<Tin, DK, 32>(a, stream);
        case 64: return launch_one<Tin, DK, 64>(a, stream);
        default: return GDN_ERR_UNSUPPORTED;
    }
}

template <typename Tin>
int launch_dk(const MaskedDpArgs &a, cudaStream_t stream) {
    switch (a.Dk) {
        case 64: return launch_chunk<Tin, 64>(a, stream);
        case 128: return launch_chunk<Tin, 128>(a, stream);
        default: return GDN_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_masked_dp(const MaskedDpArgs &a, cudaStream_t stream) {
    if (a.Dv % kBV != 0 || a.r > kMaxR) return GDN_ERR_UNSUPPORTED;
    if (a.dtype == GDN_F32) return launch_dk<float>(a, stream);
    if (a.dtype == GDN_BF16) return launch_dk<__nv_bfloat16>(a, stream);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
