// wy_chain.cuh -- the sequential part of the chunkwise WY form on the CUDA
// cores (fp32), for kernels that have formed each chunk's factors in a
// parallel pass: per head, with W, U, Kd = diag(e^{gamma_last - gamma}) K_write
// and gamma of every 64-row chunk in global memory,
//   forward:  Vn = U - W S  (kept),  S <- e^{gamma_last} S + Kd^T Vn
//   reverse:  dS <- e^{gamma_last} dS - W^T (Kd dS) + B_c
// keeping the state entering each chunk (forward) and the gradient of the
// state leaving it (reverse).  The value columns of both chains are
// independent, so each CTA holds SLICE columns of one head's state.
#pragma once

#include "simt_tile.cuh"
#include "tc_util.cuh"

namespace gdn {
namespace {

constexpr int kChainThr = 256;  // threads of a chain CTA

struct WyChainParams {
    const float *s0, *dsf;  // [BH][Dk][Dv] or null (zero)
    float *sf, *ds0;        // [BH][Dk][Dv] or null (not wanted): final state, initial state's gradient
    // per (head, chunk): S entering and dS' leaving [Dk][Dv], W and Kd [64][Dk], U and Vn
    // [64][Dv], B [Dk][Dv], gamma [64]
    float *Sw, *dSw, *Ww, *Kdw, *Uw, *Vnw, *Bw, *Gw;
    int NT;  // chunks per head
};

// Rows 0..63 of an fp32 tile of 128 columns (row m at src + m * ld, scaled by
// rs(m)) as the tensor-core chain's bf16 hi | lo operand image (32 KB):
// element (m, c) in the 8 KB block c / 64, at row m and 16-byte chunk
// (c % 64) / 8 of the 128-byte row, the chunk index XORed with m % 8 (the
// 128-byte swizzle); hi at +0, lo = x - hi at +16 KB.  The same bytes serve
// the chain's MMAs as a K-major (rows) and as an MN-major (columns) operand.
template <int NTHR, typename RowScale>
__device__ __forceinline__ void write_chain_image(unsigned char *img, const float *src, int ld, RowScale rs) {
    for (int e = threadIdx.x; e < tile::kC * 16; e += NTHR) {
        const int m = e >> 4, c8 = (e & 15) * 8;
        const float f = rs(m);
        uint32_t h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = f * src[m * ld + c8 + 2 * i], x1 = f * src[m * ld + c8 + 2 * i + 1];
            h[i] = tc::pack_bf16(x0, x1);
            l[i] = tc::pack_bf16(x0 - __uint_as_float(h[i] << 16), x1 - __uint_as_float(h[i] & 0xffff0000u));
        }
        const uint32_t off = (uint32_t)(c8 >> 6) * 8192u + tc::sw128_offset((uint32_t)m, (uint32_t)(c8 & 63));
        *reinterpret_cast<uint4 *>(img + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(img + 16384 + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

template <int DK, int SLICE>
constexpr size_t wy_chain_smem() {
    return sizeof(float) * ((size_t)DK * (SLICE + 1) + tile::kC * (DK + 4) + tile::kC * (SLICE + 4));
}

// blockIdx.x: SLICE-column slice of the value dimension; blockIdx.y: head;
// blockIdx.z: 0 = forward state chain, 1 = reverse gradient chain.
template <int DK, int DV, int SLICE>
__global__ void __launch_bounds__(kChainThr) wy_chain_kernel(WyChainParams p) {
    using namespace tile;
    extern __shared__ __align__(16) float sm[];
    // St rows are odd-strided (conflict-free both ways); Wt and Ut rows are
    // 16-byte aligned for the asynchronous copies that stage them
    constexpr int LS = SLICE + 1, LW = DK + 4, LU = SLICE + 4;
    constexpr int TI = DK / 16, TJ = SLICE / 16;
    float *St = sm;             // [DK][LS]  state (or gradient) slice
    float *Wt = St + DK * LS;   // [kC][LW]  W or Kd of the chunk
    float *Ut = Wt + kC * LW;   // [kC][LU]  U / Vn or Kd dS'
    const int col0 = blockIdx.x * SLICE, bh = blockIdx.y, role = blockIdx.z;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int NT = p.NT;

    const float *init = role == 0 ? p.s0 : p.dsf;
    for (int e = tid; e < DK * SLICE; e += kChainThr) {
        const int m = e / SLICE, n = e % SLICE;
        St[m * LS + n] = init ? init[((size_t)bh * DK + m) * DV + col0 + n] : 0.f;
    }
    __syncthreads();
    for (int s = 0; s < NT; ++s) {
        const int c = role == 0 ? s : NT - 1 - s;
        const size_t ci = (size_t)bh * NT + c;
        const float el = expf(p.Gw[ci * kC + kC - 1]);
        const float *Wg = p.Ww + ci * kC * DK, *Kdg = p.Kdw + ci * kC * DK;
        const float *first = role == 0 ? Wg : Kdg, *second = role == 0 ? Kdg : Wg;
        for (int e = tid; e < kC * DK / 4; e += kChainThr) {
            const int m = e / (DK / 4), c4 = 4 * (e % (DK / 4));
            cp_async16(Wt + m * LW + c4, first + (size_t)m * DK + c4);
        }
        if (role == 0) {
            const float *Ug = p.Uw + ci * kC * DV;
            for (int e = tid; e < kC * SLICE / 4; e += kChainThr) {
                const int m = e / (SLICE / 4), c4 = 4 * (e % (SLICE / 4));
                cp_async16(Ut + m * LU + c4, Ug + (size_t)m * DV + col0 + c4);
            }
        }
        // the reverse chain's B slice, loaded now and used at the end of the step
        float bpre[TI][TJ];
        if (role == 1) {
            const float *Bg = p.Bw + ci * DK * DV;
#pragma unroll
            for (int i = 0; i < TI; ++i)
#pragma unroll
                for (int j = 0; j < TJ; ++j) bpre[i][j] = Bg[(size_t)(ty + 16 * i) * DV + col0 + tx + 16 * j];
        }
        float *snap = (role == 0 ? p.Sw : p.dSw) + ci * DK * DV;
        for (int e = tid; e < DK * SLICE; e += kChainThr) {
            const int m = e / SLICE, n = e % SLICE;
            snap[(size_t)m * DV + col0 + n] = St[m * LS + n];
        }
        cp_async_wait_all();
        __syncthreads();
        // role 0: Vn = U - W S;  role 1: Y = Kd dS'
        {
            float acc[4][TJ];
            zero(acc);
            mm<kChainThr, 4, TJ>(acc, Wt, LW, 1, St, LS, 1, DK);
            float *Vng = p.Vnw + ci * kC * DV;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < TJ; ++j) {
                    const int m = ty + 16 * i, n = tx + 16 * j;
                    if (role == 0) {
                        const float vn = Ut[m * LU + n] - acc[i][j];
                        Vng[(size_t)m * DV + col0 + n] = vn;
                        Ut[m * LU + n] = vn;
                    } else {
                        Ut[m * LU + n] = acc[i][j];
                    }
                }
        }
        __syncthreads();
        for (int e = tid; e < kC * DK / 4; e += kChainThr) {
            const int m = e / (DK / 4), c4 = 4 * (e % (DK / 4));
            cp_async16(Wt + m * LW + c4, second + (size_t)m * DK + c4);
        }
        cp_async_wait_all();
        __syncthreads();
        // role 0: S = e^{gl} S + Kd^T Vn;  role 1: dS = e^{gl} dS' - W^T Y + B
        {
            float acc[TI][TJ];
            zero(acc);
            mm<kChainThr, TI, TJ>(acc, Wt, 1, LW, Ut, LU, 1, kC);
#pragma unroll
            for (int i = 0; i < TI; ++i)
#pragma unroll
                for (int j = 0; j < TJ; ++j) {
                    const int m = ty + 16 * i, n = tx + 16 * j;
                    const float old = St[m * LS + n];
                    St[m * LS + n] = role == 0 ? el * old + acc[i][j] : el * old - acc[i][j] + bpre[i][j];
                }
        }
        __syncthreads();
    }
    float *out = role == 0 ? p.sf : p.ds0;
    if (out) {
        for (int e = tid; e < DK * SLICE; e += kChainThr) {
            const int m = e / SLICE, n = e % SLICE;
            out[((size_t)bh * DK + m) * DV + col0 + n] = St[m * LS + n];
        }
    }
}

}  // namespace
}  // namespace gdn
