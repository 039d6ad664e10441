// tri_inverse.cuh -- (I + A)^-1 for a strictly lower-triangular C x C fp32
// matrix A in shared memory, C in {16, 32, 64}, by the whole CTA: the 16 x 16
// diagonal blocks by forward substitution (one column per thread), then the
// block merges T_ij = -T_ii A_ij T_jj at the 16 and 32 levels as small
// matrix products spread over all threads (gated_deltaproduct test.py:
// `solve_tril_16x16_kernel` and the 16 -> 32 -> 64 merge kernels compute the
// same blocked inverse).  Only the lower triangle of T (columns <= row) is
// written; the products read only entries known to be nonzero, so nothing
// has to be cleared between calls.
#pragma once

namespace gdn {

// A, T: [C][stride] fp32; X: scratch of at least C*C/4 floats.  Must be called
// by all NT threads of the CTA; ends with the CTA synchronised.
template <int C, int NT>
__device__ __forceinline__ void unit_lower_inverse(const float *A, float *T, float *X, int stride) {
    static_assert(C == 16 || C == 32 || C == 64, "chunk of 16, 32 or 64 rows");
    const int tid = threadIdx.x;
    // 1. diagonal 16 x 16 blocks: thread (block b, column c)
    if (tid < C) {
        const int b = tid >> 4, c = tid & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float v = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < i; ++k) v -= A[(o + i) * stride + o + k] * x[k];
            x[i] = v;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i >= c) T[(o + i) * stride + o + c] = x[i];
    }
    __syncthreads();
    // 2. merges of block pairs at level L (16, then 32): for each pair p, with
    //    top-left corner (o, o), X = A[o+L.., o..] T[o.., o..] (the L x L
    //    block below the top diagonal block) and T[o+L.., o..] = -T_bot X
#pragma unroll
    for (int L = 16; L < C; L *= 2) {
        const int pairs = C / (2 * L), n = pairs * L * L;
        for (int e = tid; e < n; e += NT) {
            const int p = e / (L * L), i = (e / L) % L, j = e % L, o = 2 * L * p;
            float acc = 0.f;
            for (int k = j; k < L; ++k) acc += A[(o + L + i) * stride + o + k] * T[(o + k) * stride + o + j];
            X[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < n; e += NT) {
            const int p = e / (L * L), i = (e / L) % L, j = e % L, o = 2 * L * p;
            float acc = 0.f;
            for (int k = 0; k <= i; ++k) acc += T[(o + L + i) * stride + o + L + k] * X[p * L * L + k * L + j];
            T[(o + L + i) * stride + o + j] = -acc;
        }
        __syncthreads();
    }
}

// As unit_lower_inverse for C = 64 (NT >= 256 threads, the merges on the
// first 256), for tiles whose rows are 16-byte aligned (A and T 16-byte
// aligned, stride a multiple of 4): T is cleared first, so that the merges can
// run over whole blocks, and each merge thread keeps a column of a 2- or
// 4-row tile in registers, reading the left factor's rows four k at a time
// with 16-byte loads (one broadcast wavefront each) and the right factor's
// column once per k.  X: scratch of 1024 floats (16-byte aligned).  Ends with
// the CTA synchronised.
template <int NT>
__device__ __forceinline__ void unit_lower_inverse64_v4(const float *A, float *T, float *X, int stride) {
    static_assert(NT >= 256 && NT % 32 == 0, "the merges' tiles take 256 threads");
    const int tid = threadIdx.x;
    const bool act = tid < 256;
    for (int e = tid; e < 64 * stride / 4; e += NT) reinterpret_cast<float4 *>(T)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    // 1. diagonal 16 x 16 blocks: thread (block b, column c)
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float v = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < i; ++k) v -= A[(o + i) * stride + o + k] * x[k];
            x[i] = v;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i >= c) T[(o + i) * stride + o + c] = x[i];
    }
    __syncthreads();
    // 2. the 16-level merges, pairs p at (o, o) = (32 p, 32 p): Y = A[o+16.., o..] T[o.., o..],
    //    then T[o+16.., o..] = -T[o+16.., o+16..] Y.  Thread: pair tid / 128, rows 2 ((tid / 16) % 8) + {0, 1},
    //    column tid % 16.
    {
        const int pp = (tid >> 7) & 1, i0 = 2 * ((tid >> 4) & 7), j = tid & 15, o = 32 * pp;
        if (act) {
            float y[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                float4 a[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) a[r] = *reinterpret_cast<const float4 *>(A + (o + 16 + i0 + r) * stride + o + k);
                const float t0 = T[(o + k) * stride + o + j], t1 = T[(o + k + 1) * stride + o + j];
                const float t2 = T[(o + k + 2) * stride + o + j], t3 = T[(o + k + 3) * stride + o + j];
#pragma unroll
                for (int r = 0; r < 2; ++r) y[r] += a[r].x * t0 + a[r].y * t1 + a[r].z * t2 + a[r].w * t3;
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) X[pp * 256 + (i0 + r) * 16 + j] = y[r];
        }
        __syncthreads();
        if (act) {
            float z[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                float4 a[2];
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    a[r] = *reinterpret_cast<const float4 *>(T + (o + 16 + i0 + r) * stride + o + 16 + k);
                const float *Y = X + pp * 256 + k * 16 + j;
#pragma unroll
                for (int r = 0; r < 2; ++r) z[r] += a[r].x * Y[0] + a[r].y * Y[16] + a[r].z * Y[32] + a[r].w * Y[48];
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) T[(o + 16 + i0 + r) * stride + o + j] = -z[r];
        }
        __syncthreads();
    }
    // 3. the 32-level merge: Y = A[32.., 0..] T[0.., 0..], T[32.., 0..] = -T[32.., 32..] Y.
    //    Thread: rows 4 (tid / 32) + {0..3}, column tid % 32.
    {
        const int i0 = 4 * ((tid >> 5) & 7), j = tid & 31;
        if (act) {
            float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int k = 0; k < 32; k += 4) {
                float4 a[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4 *>(A + (32 + i0 + r) * stride + k);
                const float t0 = T[k * stride + j], t1 = T[(k + 1) * stride + j];
                const float t2 = T[(k + 2) * stride + j], t3 = T[(k + 3) * stride + j];
#pragma unroll
                for (int r = 0; r < 4; ++r) y[r] += a[r].x * t0 + a[r].y * t1 + a[r].z * t2 + a[r].w * t3;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) X[(i0 + r) * 32 + j] = y[r];
        }
        __syncthreads();
        if (act) {
            float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int k = 0; k < 32; k += 4) {
                float4 a[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    a[r] = *reinterpret_cast<const float4 *>(T + (32 + i0 + r) * stride + 32 + k);
                const float *Y = X + k * 32 + j;
#pragma unroll
                for (int r = 0; r < 4; ++r) z[r] += a[r].x * Y[0] + a[r].y * Y[32] + a[r].z * Y[64] + a[r].w * Y[96];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) T[(32 + i0 + r) * stride + j] = -z[r];
        }
        __syncthreads();
    }
}

}  // namespace gdn
