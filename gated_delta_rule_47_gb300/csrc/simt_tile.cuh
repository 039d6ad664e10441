// simt_tile.cuh -- CUDA-core building blocks of the backward kernels: fp32
// tiles of 64 rows in shared memory (leading dimension = columns + 1, odd, so
// that rows and columns are both read without bank conflicts; columns + 4 for
// tiles that mm_nt reads with 16-byte loads), register-tiled block products
// over them, and row / warp reductions.
#pragma once

#include <cuda_bf16.h>

namespace gdn {
namespace tile {

constexpr int kC = 64;     // rows of a tile (a chunk of tokens or sub-steps)
constexpr int kThr = 512;  // threads of a per-tile CTA

__device__ __forceinline__ float ld_f(const float *p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// acc[i][j] += sum_{k < K} A(m_i, k) B(k, n_j) with m_i = ty + (NTHR/16) i and
// n_j = tx + 16 j (tx = thread % 16, ty = thread / 16), A(m, k) = A[m am + k ak]
// and B(k, n) = B[k bk + n bn] in shared memory.  Tiles with an odd leading
// dimension keep both orientations free of bank conflicts.
template <int NTHR, int TI, int TJ>
__device__ __forceinline__ void mm(float (&acc)[TI][TJ], const float *A, int am, int ak, const float *B, int bk,
                                   int bn, int K) {
    constexpr int RS = NTHR / 16;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const float *a0 = A + ty * am;
    const float *b0 = B + tx * bn;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float a[TI], b[TJ];
#pragma unroll
        for (int i = 0; i < TI; ++i) a[i] = a0[RS * i * am + k * ak];
#pragma unroll
        for (int j = 0; j < TJ; ++j) b[j] = b0[k * bk + 16 * j * bn];
#pragma unroll
        for (int i = 0; i < TI; ++i)
#pragma unroll
            for (int j = 0; j < TJ; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

// As mm for operands that are both contiguous in k: A(m, k) = A[m lda + k] and
// B(k, n) = B[n ldb + k], read four k at a time with 16-byte loads.  A and B
// 16-byte aligned, lda and ldb multiples of 4 (a row stride of 4 mod 32 words
// keeps the loads free of bank conflicts: the 16 rows a warp reads then cover
// every bank twice), K a multiple of 4.  Each accumulator sums over k in
// increasing order, as mm does, so the two give the same bits.
template <int NTHR, int TI, int TJ>
__device__ __forceinline__ void mm_nt(float (&acc)[TI][TJ], const float *A, int lda, const float *B, int ldb, int K) {
    constexpr int RS = NTHR / 16;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const float *a0 = A + ty * lda;
    const float *b0 = B + tx * ldb;
#pragma unroll 1
    for (int k = 0; k < K; k += 4) {
        float4 a[TI], b[TJ];
#pragma unroll
        for (int i = 0; i < TI; ++i) a[i] = *reinterpret_cast<const float4 *>(a0 + RS * i * lda + k);
#pragma unroll
        for (int j = 0; j < TJ; ++j) b[j] = *reinterpret_cast<const float4 *>(b0 + 16 * j * ldb + k);
#pragma unroll
        for (int i = 0; i < TI; ++i)
#pragma unroll
            for (int j = 0; j < TJ; ++j) {
                acc[i][j] = fmaf(a[i].x, b[j].x, acc[i][j]);
                acc[i][j] = fmaf(a[i].y, b[j].y, acc[i][j]);
                acc[i][j] = fmaf(a[i].z, b[j].z, acc[i][j]);
                acc[i][j] = fmaf(a[i].w, b[j].w, acc[i][j]);
            }
    }
}

// As mm, with the operands given by accessors fa(m, k) and fb(k, n) (for
// operands formed on the fly from others).
template <int NTHR, int TI, int TJ, class FA, class FB>
__device__ __forceinline__ void mm_f(float (&acc)[TI][TJ], const FA &fa, const FB &fb, int K) {
    constexpr int RS = NTHR / 16;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float a[TI], b[TJ];
#pragma unroll
        for (int i = 0; i < TI; ++i) a[i] = fa(ty + RS * i, k);
#pragma unroll
        for (int j = 0; j < TJ; ++j) b[j] = fb(k, tx + 16 * j);
#pragma unroll
        for (int i = 0; i < TI; ++i)
#pragma unroll
            for (int j = 0; j < TJ; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

template <int TI, int TJ>
__device__ __forceinline__ void zero(float (&a)[TI][TJ]) {
#pragma unroll
    for (int i = 0; i < TI; ++i)
#pragma unroll
        for (int j = 0; j < TJ; ++j) a[i][j] = 0.f;
}

// 16-byte asynchronous copy global -> shared (both addresses 16-byte
// aligned), completed by cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void *sdst, const void *gsrc) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(sdst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Sum over the 16 lanes that hold one row of a tile (lanes differing in bits 0..3).
__device__ __forceinline__ float row_sum16(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Element u of this thread's share of a kThr-strided pass, e = thread + u kThr
// for u < N: all N values are loaded (load(e)) before any is stored
// (store(e, x)), so that a pass over global memory waits for one round trip,
// not N.
template <int N, class Load, class Store>
__device__ __forceinline__ void staged(const Load &load, const Store &store) {
    float x[N];
#pragma unroll
    for (int u = 0; u < N; ++u) x[u] = load((int)threadIdx.x + u * kThr);
#pragma unroll
    for (int u = 0; u < N; ++u) store((int)threadIdx.x + u * kThr, x[u]);
}

// dst[(e / C) ld + e % C] = src[e] for the R x C row-major values of src (R C a
// multiple of kThr), every load in flight before the stores.
template <int R, int C, typename T>
__device__ __forceinline__ void stage_rows(float *dst, int ld, const T *src) {
    static_assert(R * C % kThr == 0, "whole passes");
    staged<R * C / kThr>([&](int e) { return ld_f(src + e); },
                         [&](int e, float x) { dst[(e / C) * ld + e % C] = x; });
}

// dst[a][0..D) (leading dimension LD, D + 1 unless given) = row a of src for
// a < nvalid, else 0, for the 64 rows of a chunk (each warp loads all its rows
// before it stores any).  With norm, each row is divided by max(|row|, 1e-12)
// and its plain norm kept in nrm[a].
template <typename T, int D, int LD = D + 1>
__device__ void load_rows(float *dst, const T *src, int nvalid, bool norm, float *nrm) {
    constexpr int NW = kThr / 32, NR = kC / NW;  // warps, rows per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float x[NR][D / 32];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int a = warp + NW * j;
#pragma unroll
        for (int u = 0; u < D / 32; ++u) x[j][u] = a < nvalid ? ld_f(src + (size_t)a * D + lane + 32 * u) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int a = warp + NW * j;
        if (norm) {
            float ss = 0.f;
#pragma unroll
            for (int u = 0; u < D / 32; ++u) ss += x[j][u] * x[j][u];
            ss = warp_sum(ss);
            const float n = sqrtf(ss);
            const float inv = 1.f / fmaxf(n, 1e-12f);
#pragma unroll
            for (int u = 0; u < D / 32; ++u) x[j][u] *= inv;
            if (lane == 0) nrm[a] = n;
        }
#pragma unroll
        for (int u = 0; u < D / 32; ++u) dst[a * LD + lane + 32 * u] = x[j][u];
    }
}

}  // namespace tile
}  // namespace gdn
