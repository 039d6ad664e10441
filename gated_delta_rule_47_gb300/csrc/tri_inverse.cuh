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

}  // namespace gdn
