// scan_simt.cu -- chunkwise GDN / DeltaProduct forward on the CUDA cores, in
// fp32 arithmetic.  This is the path for fp32 tensors (tensor-core kinds with
// fp32 operands would round to tf32) and for shapes the tcgen05 path does not
// take.  One CTA per (batch*head, 64-wide value tile); the chunks of a head are
// processed in order with the fp32 state tile resident in shared memory.
//
// Per chunk of C rows starting from state S (gated_deltaproduct test.py, the
// KK^T, triangular solve, w/u recompute, state-scan and output kernels):
//   gam_t = sum_{i<=t} g_i within the chunk
//   A[t][s] = beta_t exp(gam_t - gam_s) (k_t . k_s)           for s < t
//   R[t]    = beta_t (v_t - exp(gam_t) S^T k_t)
//   Delta   = (I + A)^-1 R          (= u - w S in the WY form)
//   o_t     = scale (exp(gam_t) S^T q_t + sum_{s<=t} exp(gam_t-gam_s)(q_t.k_s) Delta_s)
//   S      <- exp(gam_last) S + sum_s exp(gam_last - gam_s) k_s Delta_s^T
// Rows past the end of the sequence are zero (k, v, beta) with g = 0, so they
// change nothing.  For DeltaProduct the decay g_t sits on row (t, 0) and the
// query q_t is read at row (t, r-1); a chunk holds floor(C/r) whole tokens.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kBV = 64;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

struct SimtParams {
    const void *q, *k, *v, *beta;
    const float *g, *s0;
    void *o;
    float *sf;
    int T, r, Dv;
    float scale;
    unsigned flags;
};

template <int DK, int C>
struct SimtSmem {
    // the key and query tiles have a row stride of DK + 4 (4 mod 32 words), so
    // that the K K^T and Q K^T products read them with 16-byte loads
    static constexpr int KP = DK + 4, VP = kBV + 1, CP = C + 1;
    static constexpr int floats = 2 * C * KP + C * VP + DK * VP + 3 * C * CP + 2 * C * VP + 3 * C + C * C / 4;
    static constexpr size_t bytes = sizeof(float) * floats;
};

// Inclusive prefix sum of x[0..n) (n <= 64) by one warp.
__device__ __forceinline__ void warp_cumsum64(float *x, int n, int lane) {
    float a = lane < n ? x[lane] : 0.f;
    float b = lane + 32 < n ? x[lane + 32] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float ya = __shfl_up_sync(0xffffffffu, a, off);
        float yb = __shfl_up_sync(0xffffffffu, b, off);
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

// Scale rows [0, nrows) of a [.][stride] fp32 tile to unit L2 norm over DK.
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
__global__ void __launch_bounds__(kThreads, 1) scan_simt_kernel(SimtParams p) {
    using L = SimtSmem<DK, C>;
    constexpr int KP = L::KP, VP = L::VP, CP = L::CP;
    constexpr int TC = C / 16;   // 16-row blocks of a chunk a thread covers (rows ty + 16 i)
    constexpr int TD = DK / 16;  // 16-row blocks of the state
    extern __shared__ __align__(16) float smem[];
    float *Ks = smem;            // [C][KP]   keys of the chunk
    float *Qs = Ks + C * KP;     // [C][KP]   queries (C/r rows used)
    float *Vs = Qs + C * KP;     // [C][VP]   value tile
    float *Ss = Vs + C * VP;     // [DK][VP]  fp32 state tile
    float *As = Ss + DK * VP;    // [C][CP]   A (strictly lower)
    float *Ts = As + C * CP;     // [C][CP]   (I + A)^-1 (zero above the diagonal)
    float *Ps = Ts + C * CP;     // [C][CP]   decay-masked q.k, s <= t
    float *Rs = Ps + C * CP;     // [C][VP]   R
    float *Ds = Rs + C * VP;     // [C][VP]   Delta
    float *gam = Ds + C * VP;    // [C]
    float *bet = gam + C;        // [C]
    float *eS = bet + C;         // [C] exp(gam_last - gam_s)
    float *Xs = eS + C;          // [C*C/4] scratch of the blocked inverse

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, tx = tid & 15, ty = tid >> 4;
    const int vt = blockIdx.x;
    const size_t head = blockIdx.y;
    const int r = p.r, Dv = p.Dv, T = p.T;
    const int CQ = C / r;    // whole tokens per chunk
    const int Ce = CQ * r;   // rows per chunk (<= C; the rest of the tile is padding)
    const long rows = (long)T * r;

    const Tin *kp = static_cast<const Tin *>(p.k) + head * rows * DK;
    const Tin *vp = static_cast<const Tin *>(p.v) + head * rows * Dv + vt * kBV;
    const Tin *qp = static_cast<const Tin *>(p.q) + head * (size_t)T * DK;
    const Tin *bp = static_cast<const Tin *>(p.beta) + head * rows;
    const float *gp = p.g + head * (size_t)T;
    Tin *op = static_cast<Tin *>(p.o) + head * (size_t)T * Dv + vt * kBV;

    for (int i = tid; i < DK * kBV; i += kThreads) {
        const int d = i / kBV, j = i % kBV;
        Ss[d * VP + j] = p.s0 ? p.s0[(head * DK + d) * Dv + vt * kBV + j] : 0.f;
    }
    // the inverse writes only the lower triangle of T; its product reads all of it
    for (int i = tid; i < C * CP; i += kThreads) Ts[i] = 0.f;

    for (long c0 = 0; c0 < rows; c0 += Ce) {
        const int Lr = (int)min((long)Ce, rows - c0);  // valid rows (a multiple of r)
        const int LQ = Lr / r;                         // valid query rows
        const long tok0 = c0 / r;
        __syncthreads();
        for (int i = tid; i < C * DK; i += kThreads) {
            const int t = i / DK, d = i % DK;
            Ks[t * KP + d] = t < Lr ? to_f32(kp[(c0 + t) * DK + d]) : 0.f;
            Qs[t * KP + d] = t < LQ ? to_f32(qp[(tok0 + t) * DK + d]) : 0.f;
        }
        for (int i = tid; i < C * kBV; i += kThreads) {
            const int t = i / kBV, j = i % kBV;
            Vs[t * VP + j] = t < Lr ? to_f32(vp[(c0 + t) * Dv + j]) : 0.f;
        }
        if (tid < C) {
            const bool ok = tid < Lr;
            bet[tid] = ok ? to_f32(bp[c0 + tid]) : 0.f;
            gam[tid] = (ok && (c0 + tid) % r == 0) ? gp[(c0 + tid) / r] : 0.f;
        }
        __syncthreads();
        if (p.flags & GDN_QK_L2NORM) {
            unit_rows<DK>(Ks, KP, Lr, warp, lane, kThreads / 32);
            unit_rows<DK>(Qs, KP, LQ, warp, lane, kThreads / 32);
        }
        if (warp == 0) warp_cumsum64(gam, C, lane);
        __syncthreads();
        const float glast = gam[C - 1];
        if (tid < C) eS[tid] = expf(glast - gam[tid]);

        // A (strictly lower) and the decay-masked query-key scores, from the
        // block products K K^T and Q K^T
        {
            float acc[TC][TC];
            tile::zero(acc);
            tile::mm_nt<kThreads, TC, TC>(acc, Ks, KP, Ks, KP, DK);
#pragma unroll
            for (int i = 0; i < TC; ++i)
#pragma unroll
                for (int j = 0; j < TC; ++j) {
                    const int t = ty + 16 * i, s = tx + 16 * j;
                    As[t * CP + s] = s < t ? bet[t] * expf(gam[t] - gam[s]) * acc[i][j] : 0.f;
                }
            tile::zero(acc);
            tile::mm_nt<kThreads, TC, TC>(acc, Qs, KP, Ks, KP, DK);
#pragma unroll
            for (int i = 0; i < TC; ++i)
#pragma unroll
                for (int j = 0; j < TC; ++j) {
                    const int t = ty + 16 * i, s = tx + 16 * j, row = t * r + r - 1;
                    Ps[t * CP + s] = (t < CQ && s <= row) ? expf(gam[row] - gam[s]) * acc[i][j] : 0.f;
                }
        }
        // R = diag(beta) (V - diag(exp(gam)) K S)
        {
            float acc[TC][4];
            tile::zero(acc);
            tile::mm<kThreads, TC, 4>(acc, Ks, KP, 1, Ss, VP, 1, DK);
#pragma unroll
            for (int i = 0; i < TC; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = ty + 16 * i, c = tx + 16 * j;
                    Rs[t * VP + c] = bet[t] * (Vs[t * VP + c] - expf(gam[t]) * acc[i][j]);
                }
        }
        __syncthreads();
        // (I + A)^-1: 16 x 16 diagonal blocks, then the 16- and 32-level merges
        unit_lower_inverse<C, kThreads>(As, Ts, Xs, CP);
        // Delta = (I + A)^-1 R
        {
            float acc[TC][4];
            tile::zero(acc);
            tile::mm<kThreads, TC, 4>(acc, Ts, CP, 1, Rs, VP, 1, C);
#pragma unroll
            for (int i = 0; i < TC; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) Ds[(ty + 16 * i) * VP + tx + 16 * j] = acc[i][j];
        }
        __syncthreads();
        // Outputs of the chunk's tokens (read the state before this chunk's update).
        {
            float inter[TC][4], intra[TC][4];
            tile::zero(inter);
            tile::zero(intra);
            tile::mm<kThreads, TC, 4>(inter, Qs, KP, 1, Ss, VP, 1, DK);
            tile::mm<kThreads, TC, 4>(intra, Ps, CP, 1, Ds, VP, 1, C);
#pragma unroll
            for (int i = 0; i < TC; ++i) {
                const int t = ty + 16 * i;
                if (t < LQ) {
                    const float eg = expf(gam[t * r + r - 1]);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        from_f32(op + (tok0 + t) * Dv + tx + 16 * j, p.scale * (eg * inter[i][j] + intra[i][j]));
                }
            }
        }
        __syncthreads();
        // State update S <- exp(gam_last) S + K^T diag(exp(gam_last - gam)) Delta
        for (int i = tid; i < C * kBV; i += kThreads) Ds[(i / kBV) * VP + i % kBV] *= eS[i / kBV];
        __syncthreads();
        {
            const float dl = expf(glast);
            float acc[TD][4];
            tile::zero(acc);
            tile::mm<kThreads, TD, 4>(acc, Ks, 1, KP, Ds, VP, 1, C);
#pragma unroll
            for (int i = 0; i < TD; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int d = ty + 16 * i, c = tx + 16 * j;
                    Ss[d * VP + c] = dl * Ss[d * VP + c] + acc[i][j];
                }
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
int launch_one(const ScanArgs &a, cudaStream_t stream) {
    auto kern = scan_simt_kernel<Tin, DK, C>;
    constexpr size_t smem = SimtSmem<DK, C>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    SimtParams p{a.q, a.k, a.v, a.beta, a.g, a.s0, a.o, a.sf, a.T, a.r, a.Dv, a.scale, a.flags};
    dim3 grid(a.Dv / kBV, a.B * a.H);
    kern<<<grid, kThreads, smem, stream>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename Tin, int DK>
int launch_chunk(const ScanArgs &a, cudaStream_t stream) {
    switch (a.chunk) {
        case 16: return launch_one<Tin, DK, 16>(a, stream);
        case 32: return launch_one<Tin, DK, 32>(a, stream);
        case 64: return launch_one<Tin, DK, 64>(a, stream);
        default: return GDN_ERR_UNSUPPORTED;
    }
}

template <typename Tin>
int launch_dk(const ScanArgs &a, cudaStream_t stream) {
    switch (a.Dk) {
        case 64: return launch_chunk<Tin, 64>(a, stream);
        case 128: return launch_chunk<Tin, 128>(a, stream);
        default: return GDN_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_scan_simt(const ScanArgs &a, cudaStream_t stream) {
    if (a.Dv % kBV != 0) return GDN_ERR_UNSUPPORTED;
    if (a.dtype == GDN_F32) return launch_dk<float>(a, stream);
    if (a.dtype == GDN_BF16) return launch_dk<__nv_bfloat16>(a, stream);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
