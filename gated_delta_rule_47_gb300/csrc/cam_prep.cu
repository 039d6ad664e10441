// cam_prep.cu -- fused camera-branch prep (fused_cam_gdn.py, `_cam_prep_kernel`
// and `_torch_cam_prep_reference`), one pass over q, k and v.
//
// The pages run a separate full-C RMS reduction first and then one 1-warp
// program per (b, n, h).  Here a token is handled whole, so the two full-C
// sums of squares never leave the chip, and the three outputs are written in
// the head-major [B,H,N,D] layout the scan reads.  Two kernels:
//
//  - cam_prep_stream_kernel (bf16, C <= 2048, rotary tables given): one
//    persistent CTA per SM walks stages of 8 consecutive tokens; a producer
//    warp bulk-copies each stage's q, k, v rows, projections and rotary rows
//    into one of two shared-memory buffers while 16 compute warps, two per
//    token (each with half of the token's heads), work on the other buffer.
//  - cam_prep_kernel (everything else: fp32 tensors, or angles formed in the
//    kernel): one warp per token holds the token's rows in registers from
//    16-byte loads, 8 tokens per CTA, the rotary rows of the 8 positions
//    staged once in shared memory.
//
// The backward has the same split: cam_prep_bwd_stream_kernel (bf16, C <=
// 2048, rotary tables given; persistent CTAs fed by bulk copies, four warps
// per token) and cam_prep_bwd_kernel (one CTA per token) for the rest.
//
// The path is HBM-bound: 3 reads + 3 writes of C elements per token (the
// backward: 5 reads + 3 writes).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"
#include "tc_util.cuh"

namespace gdn {
namespace {

__device__ unsigned int g_cam_error = 0;  // set when a bounded wait of the streamed kernel runs out

constexpr int kTokPerCta = 8;  // one warp per token
constexpr int kMaxDh = 128;    // D/2 <= 128

struct CamParams {
    const void *q_raw, *k_raw, *v_raw;
    const float *q_norm_w, *k_norm_w, *proj_q, *proj_kv, *rope_cos, *rope_sin;
    double log2_base;  // log2(rope_base) in double: a float one would shift angles at large positions
    void *q_out, *k_out, *v_out;
    float *k_pre_sq, *k_post_sq;
    int B, N, H, D;
    float k_scale, eps;
};

// Eight consecutive elements as fp32.
struct F8 {
    float x[8];
};

__device__ __forceinline__ F8 load8(const float *p) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    F8 r = {{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
    return r;
}

// Eight consecutive raw elements as loaded (bf16: one 16-byte word; fp32: two),
// kept packed in registers until they are used.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = __ldg(reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ F8 unpack() const {
        F8 r;
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            r.x[2 * i] = __uint_as_float(w[i] << 16);
            r.x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
        return r;
    }
};
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p) {
        a = __ldg(reinterpret_cast<const float4 *>(p));
        b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ F8 unpack() const {
        F8 r = {{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
        return r;
    }
};

__device__ __forceinline__ void store8(__nv_bfloat16 *p, const F8 &v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v.x[2 * i], v.x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void store8(float *p, const F8 &v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v.x[0], v.x[1], v.x[2], v.x[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v.x[4], v.x[5], v.x[6], v.x[7]);
}

// NPL = 8-element groups per lane (C = H*D <= 256*NPL).
template <typename T, int NPL>
__global__ void __launch_bounds__(32 * kTokPerCta, 2) cam_prep_kernel(CamParams p) {
    __shared__ float s_cos[kTokPerCta][kMaxDh];
    __shared__ float s_sin[kTokPerCta][kMaxDh];
    __shared__ float s_pre[kTokPerCta][64];
    __shared__ float s_post[kTokPerCta][64];

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int H = p.H, D = p.D, N = p.N;
    const int C = H * D, Dh = D / 2, G8 = C / 8;
    const long tok_base = (long)blockIdx.x * kTokPerCta;
    const long BN = (long)p.B * N;

    // Rotary tables of the CTA's positions.
    for (int i = threadIdx.x; i < kTokPerCta * Dh; i += blockDim.x) {
        const int tt = i / Dh, d = i % Dh;
        const long tok = tok_base + tt;
        if (tok >= BN) continue;
        const int n = (int)(tok % N);
        float c, s;
        if (p.rope_cos) {
            c = p.rope_cos[(size_t)n * Dh + d];
            s = p.rope_sin[(size_t)n * Dh + d];
        } else {
            // th = n * base^(-2i/Dh), i = d/2; the product and its reduction
            // modulo 2*pi are done in double so large positions keep precision.
            const int i2 = d >> 1;
            const double inv_freq = exp2(p.log2_base * (-2.0 * i2 / (double)Dh));
            double th = (double)n * inv_freq;
            const double two_pi = 6.283185307179586476925286766559;
            th -= two_pi * rint(th / two_pi);
            float sv, cv;
            sincosf((float)th, &sv, &cv);
            c = cv;
            s = (d & 1) ? sv : -sv;
        }
        s_cos[tt][d] = c;
        s_sin[tt][d] = s;
    }
    __syncthreads();

    const long tok = tok_base + w;
    const bool active = tok < BN;
    if (active) {
        const int b = (int)(tok / N), n = (int)(tok % N);
        const T *qr = static_cast<const T *>(p.q_raw) + (size_t)tok * C;
        const T *kr = static_cast<const T *>(p.k_raw) + (size_t)tok * C;
        const T *vr = static_cast<const T *>(p.v_raw) + (size_t)tok * C;
        Raw8<T> xq[NPL], xk[NPL], xv[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int gi = lane + 32 * i;
            if (gi < G8) {
                xq[i].load(qr + gi * 8);
                xk[i].load(kr + gi * 8);
                xv[i].load(vr + gi * 8);
            }
        }
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if (lane + 32 * i < G8) {
                const F8 a = xq[i].unpack(), b = xk[i].unpack();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sq += a.x[e] * a.x[e];
                    sk += b.x[e] * b.x[e];
                }
            }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
        }
        const float iq = rsqrtf(sq / (float)C + p.eps);
        const float ik = rsqrtf(sk / (float)C + p.eps);

        float Pq[16], Pk[16];
        const float4 *pq4 = reinterpret_cast<const float4 *>(p.proj_q + (size_t)tok * 16);
        const float4 *pk4 = reinterpret_cast<const float4 *>(p.proj_kv + (size_t)tok * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 a = __ldg(pq4 + i), c = __ldg(pk4 + i);
            Pq[4 * i] = a.x; Pq[4 * i + 1] = a.y; Pq[4 * i + 2] = a.z; Pq[4 * i + 3] = a.w;
            Pk[4 * i] = c.x; Pk[4 * i + 1] = c.y; Pk[4 * i + 2] = c.z; Pk[4 * i + 3] = c.w;
        }

        const int lanes_per_head = D / 8;  // divides 32
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int gi = lane + 32 * i;
            const bool ok = gi < G8;
            const int e0 = gi * 8;
            const int h = e0 / D, d0 = e0 % D;
            F8 q = xq[i].unpack(), k = xk[i].unpack(), v = xv[i].unpack();
            float pre = 0.f, post = 0.f;
            if (ok) {
                F8 wq, wk;
                if (p.q_norm_w) wq = load8(p.q_norm_w + e0);
                else for (int e = 0; e < 8; ++e) wq.x[e] = 1.f;
                if (p.k_norm_w) wk = load8(p.k_norm_w + e0);
                else for (int e = 0; e < 8; ++e) wk.x[e] = 1.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    q.x[e] = fmaxf(q.x[e] * iq * wq.x[e], 0.f);
                    k.x[e] = fmaxf(k.x[e] * ik * wk.x[e], 0.f) * p.k_scale;
                    pre += k.x[e] * k.x[e];
                }
                F8 oq, ok8, ov;
                if (d0 < Dh) {
#pragma unroll
                    for (int gsub = 0; gsub < 2; ++gsub) {
#pragma unroll
                        for (int a = 0; a < 4; ++a) {
                            float s0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                s0 += Pq[a * 4 + c] * q.x[4 * gsub + c];
                                s1 += Pk[a * 4 + c] * k.x[4 * gsub + c];
                                s2 += Pk[a * 4 + c] * v.x[4 * gsub + c];
                            }
                            oq.x[4 * gsub + a] = s0;
                            ok8.x[4 * gsub + a] = s1;
                            ov.x[4 * gsub + a] = s2;
                        }
                    }
                } else {
                    const int dr = d0 - Dh;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float c = s_cos[w][dr + e], s = s_sin[w][dr + e];
                        oq.x[e] = q.x[e] * c + q.x[e ^ 1] * s;
                        ok8.x[e] = k.x[e] * c + k.x[e ^ 1] * s;
                        ov.x[e] = v.x[e] * c + v.x[e ^ 1] * s;
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) post += ok8.x[e] * ok8.x[e];
                const size_t ob = (((size_t)b * H + h) * N + n) * D + d0;
                store8(static_cast<T *>(p.q_out) + ob, oq);
                store8(static_cast<T *>(p.k_out) + ob, ok8);
                store8(static_cast<T *>(p.v_out) + ob, ov);
            }
            // per-head sums over the lanes_per_head lanes that hold head h
            for (int off = lanes_per_head >> 1; off; off >>= 1) {
                pre += __shfl_xor_sync(0xffffffffu, pre, off);
                post += __shfl_xor_sync(0xffffffffu, post, off);
            }
            if (ok && (lane % lanes_per_head) == 0 && h < 64) {
                s_pre[w][h] = pre;
                s_post[w][h] = post;
            }
        }
    }
    __syncthreads();
    // Norm statistics: for each head, the CTA's consecutive tokens are
    // consecutive in [B,H,N]; write them run by run.
    if (p.k_pre_sq || p.k_post_sq) {
        for (int i = threadIdx.x; i < H * kTokPerCta; i += blockDim.x) {
            const int h = i / kTokPerCta, tt = i % kTokPerCta;
            const long t2 = tok_base + tt;
            if (t2 >= BN || h >= 64) continue;
            const int b = (int)(t2 / N), n = (int)(t2 % N);
            const size_t si = ((size_t)b * H + h) * N + n;
            if (p.k_pre_sq) p.k_pre_sq[si] = s_pre[tt][h];
            if (p.k_post_sq) p.k_post_sq[si] = s_post[tt][h];
        }
    }
}

// ------------------------------------------------------------------ streamed
// The same per-token computation for bf16 rows of C = H*D <= 2048 elements
// with rotary tables given, fed by the bulk-copy engine: one persistent CTA
// per SM walks stages of 8 consecutive tokens.  A producer warp copies each
// stage's q, k, v rows (3 x C x 2 bytes per token), the two 4x4 projections
// and the rotary rows into one of two shared-memory buffers; 16 compute warps
// (two per token, each with half the row's heads) read them from there, so
// the next stage's loads are in flight while the current one is computed.
// Measured on the B2 N32760 H16 D128 camera workload: 4.31 TB/s against
// 3.36 TB/s for the one-warp-per-token kernel above.  Every wait is bounded.
constexpr int kStageTok = 8;
constexpr int kMaxC = 2048;
constexpr uint32_t kRowBytes = kMaxC * 2;                                  // one q/k/v row
constexpr uint32_t kTokBytes = 3 * kRowBytes + 2 * 64 + 2 * kMaxDh * 4;    // rows, projections, rotary
constexpr uint32_t kStageBytes = kStageTok * kTokBytes;
constexpr uint32_t kStreamSmem = 2 * kStageBytes + 64 + 2 * 2 * kStageTok * 2 * 4 + 1024;
constexpr unsigned long long kCamTimeoutNs = 1000000000ull;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

// Bounded wait; on expiry records the error and returns false.
__device__ __forceinline__ bool cam_wait(uint64_t *bar, uint32_t parity) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::global_timer_ns();
    while (!tc::mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (tc::global_timer_ns() - t0 > kCamTimeoutNs) {
            atomicOr(&g_cam_error, 1u);
            return false;
        }
    }
    return true;
}

template <int NPL>
__global__ void __launch_bounds__(32 * (2 * kStageTok + 1), 1) cam_prep_stream_kernel(CamParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((128u - (tc::smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + 2 * kStageBytes);  // [2]
    uint64_t *empty = full + 2;                                          // [2]
    float *part = reinterpret_cast<float *>(empty + 2);                  // [2 stages][2 * kStageTok][2] partial sums
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int H = p.H, D = p.D, N = p.N;
    const int C = H * D, Dh = D / 2, G8 = C / 8;
    const uint32_t row_bytes = (uint32_t)C * 2;
    const long BN = (long)p.B * N;
    const long nstages = (BN + kStageTok - 1) / kStageTok;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 2 * kStageTok);
        }
        tc::fence_mbar_init();
    }
    __syncthreads();
    // per-token layout inside a stage buffer: q | k | v rows, proj_q, proj_kv, cos, sin
    auto tok_base = [&](int buf, int t) -> uint8_t * { return sm + buf * kStageBytes + t * kTokBytes; };

    if (w == 2 * kStageTok) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint32_t pbytes = 64, tbytes = (uint32_t)Dh * 4;
            int j = 0;
            for (long st = blockIdx.x; st < nstages; st += gridDim.x, ++j) {
                const int buf = j & 1;
                if (j >= 2 && !cam_wait(&empty[buf], ((j - 2) >> 1) & 1)) break;
                const long t0 = st * kStageTok;
                const int nt = (int)min((long)kStageTok, BN - t0);
                tc::mbar_arrive_expect_tx(&full[buf], (uint32_t)nt * (3 * row_bytes + 2 * pbytes + 2 * tbytes));
                for (int t = 0; t < nt; ++t) {
                    const long tok = t0 + t;
                    const int n = (int)(tok % N);
                    uint8_t *tb = tok_base(buf, t);
                    const uint32_t d = tc::smem_u32(tb);
                    const size_t ro = (size_t)tok * C;
                    bulk_g2s(d, static_cast<const __nv_bfloat16 *>(p.q_raw) + ro, row_bytes, &full[buf]);
                    bulk_g2s(d + kRowBytes, static_cast<const __nv_bfloat16 *>(p.k_raw) + ro, row_bytes, &full[buf]);
                    bulk_g2s(d + 2 * kRowBytes, static_cast<const __nv_bfloat16 *>(p.v_raw) + ro, row_bytes, &full[buf]);
                    bulk_g2s(d + 3 * kRowBytes, p.proj_q + (size_t)tok * 16, pbytes, &full[buf]);
                    bulk_g2s(d + 3 * kRowBytes + 64, p.proj_kv + (size_t)tok * 16, pbytes, &full[buf]);
                    bulk_g2s(d + 3 * kRowBytes + 128, p.rope_cos + (size_t)n * Dh, tbytes, &full[buf]);
                    bulk_g2s(d + 3 * kRowBytes + 128 + kMaxDh * 4, p.rope_sin + (size_t)n * Dh, tbytes, &full[buf]);
                }
            }
            // the last stage's copies land before the CTA leaves
            const int jn = j;
            for (int q = (jn >= 2 ? jn - 2 : 0); q < jn; ++q) cam_wait(&empty[q & 1], (q >> 1) & 1);
        }
        return;
    }
    // -------------------------------------------------------------- compute
    // warps 2t and 2t+1 share token t of a stage: each takes every other
    // 32-group block of the row (whole heads), and they add their sums of
    // squares through shared memory
    const int tw = w >> 1, hf = w & 1;
    int j = 0;
    const int lanes_per_head = D / 8;              // a power of two that divides 32
    const int lph_shift = __ffs(lanes_per_head) - 1;
    const size_t ND = (size_t)N * D;
    for (long st = blockIdx.x; st < nstages; st += gridDim.x, ++j) {
        const int buf = j & 1;
        if (!cam_wait(&full[buf], (j >> 1) & 1)) break;
        const long tok = st * kStageTok + tw;
        if (tok < BN) {
            const int b = (int)(tok / N), n = (int)(tok % N);
            const size_t obase = (size_t)b * H * ND + (size_t)n * D;  // head 0, dim 0 of this token's outputs
            const uint8_t *tb = tok_base(buf, tw);
            const __nv_bfloat16 *sq_ = reinterpret_cast<const __nv_bfloat16 *>(tb);
            const __nv_bfloat16 *sk_ = reinterpret_cast<const __nv_bfloat16 *>(tb + kRowBytes);
            const __nv_bfloat16 *sv_ = reinterpret_cast<const __nv_bfloat16 *>(tb + 2 * kRowBytes);
            const float *Pq = reinterpret_cast<const float *>(tb + 3 * kRowBytes);
            const float *Pk = Pq + 16;
            const float *cs = reinterpret_cast<const float *>(tb + 3 * kRowBytes + 128);
            const float *sn = cs + kMaxDh;
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int i = 0; i < NPL / 2; ++i) {
                const int gi = lane + 32 * (2 * i + hf);
                if (gi < G8) {
                    Raw8<__nv_bfloat16> a, c;
                    a.u = *reinterpret_cast<const uint4 *>(sq_ + gi * 8);
                    c.u = *reinterpret_cast<const uint4 *>(sk_ + gi * 8);
                    const F8 x = a.unpack(), y = c.unpack();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sq += x.x[e] * x.x[e];
                        sk += y.x[e] * y.x[e];
                    }
                }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
            }
            float *pp = part + (buf * 2 * kStageTok + w) * 2;
            if (lane == 0) {
                pp[0] = sq;
                pp[1] = sk;
            }
            asm volatile("bar.sync %0, 64;" ::"r"(1 + tw) : "memory");  // the token's two warps
            const float *po = part + (buf * 2 * kStageTok + (w ^ 1)) * 2;
            sq += po[0];
            sk += po[1];
            const float iq = rsqrtf(sq / (float)C + p.eps);
            const float ik = rsqrtf(sk / (float)C + p.eps);
#pragma unroll
            for (int i = 0; i < NPL / 2; ++i) {
                const int gi = lane + 32 * (2 * i + hf);
                const bool ok = gi < G8;
                const int e0 = gi * 8;
                const int h = gi >> lph_shift, d0 = (gi & (lanes_per_head - 1)) << 3;
                float pre = 0.f, post = 0.f;
                if (ok) {
                    Raw8<__nv_bfloat16> a, c, e;
                    a.u = *reinterpret_cast<const uint4 *>(sq_ + e0);
                    c.u = *reinterpret_cast<const uint4 *>(sk_ + e0);
                    e.u = *reinterpret_cast<const uint4 *>(sv_ + e0);
                    F8 q = a.unpack(), k = c.unpack(), v = e.unpack();
                    F8 wq, wk;
                    if (p.q_norm_w) wq = load8(p.q_norm_w + e0);
                    else for (int t = 0; t < 8; ++t) wq.x[t] = 1.f;
                    if (p.k_norm_w) wk = load8(p.k_norm_w + e0);
                    else for (int t = 0; t < 8; ++t) wk.x[t] = 1.f;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        q.x[t] = fmaxf(q.x[t] * iq * wq.x[t], 0.f);
                        k.x[t] = fmaxf(k.x[t] * ik * wk.x[t], 0.f) * p.k_scale;
                        pre += k.x[t] * k.x[t];
                    }
                    F8 oq, ok8, ov;
                    if (d0 < Dh) {
#pragma unroll
                        for (int gsub = 0; gsub < 2; ++gsub) {
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                float s0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
                                for (int cc = 0; cc < 4; ++cc) {
                                    s0 += Pq[r * 4 + cc] * q.x[4 * gsub + cc];
                                    s1 += Pk[r * 4 + cc] * k.x[4 * gsub + cc];
                                    s2 += Pk[r * 4 + cc] * v.x[4 * gsub + cc];
                                }
                                oq.x[4 * gsub + r] = s0;
                                ok8.x[4 * gsub + r] = s1;
                                ov.x[4 * gsub + r] = s2;
                            }
                        }
                    } else {
                        // dr is a multiple of 8 and Dh of 4: 16-byte aligned rows
                        const int dr = d0 - Dh;
                        const float4 c0 = *reinterpret_cast<const float4 *>(cs + dr);
                        const float4 c1 = *reinterpret_cast<const float4 *>(cs + dr + 4);
                        const float4 s0 = *reinterpret_cast<const float4 *>(sn + dr);
                        const float4 s1 = *reinterpret_cast<const float4 *>(sn + dr + 4);
                        const float cva[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        const float sva[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const float cv = cva[t], sv = sva[t];
                            oq.x[t] = q.x[t] * cv + q.x[t ^ 1] * sv;
                            ok8.x[t] = k.x[t] * cv + k.x[t ^ 1] * sv;
                            ov.x[t] = v.x[t] * cv + v.x[t ^ 1] * sv;
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 8; ++t) post += ok8.x[t] * ok8.x[t];
                    const size_t ob = obase + (size_t)h * ND + d0;
                    store8(static_cast<__nv_bfloat16 *>(p.q_out) + ob, oq);
                    store8(static_cast<__nv_bfloat16 *>(p.k_out) + ob, ok8);
                    store8(static_cast<__nv_bfloat16 *>(p.v_out) + ob, ov);
                }
                for (int off = lanes_per_head >> 1; off; off >>= 1) {
                    pre += __shfl_xor_sync(0xffffffffu, pre, off);
                    post += __shfl_xor_sync(0xffffffffu, post, off);
                }
                if (ok && (lane & (lanes_per_head - 1)) == 0) {
                    const size_t si = ((size_t)b * H + h) * N + n;
                    if (p.k_pre_sq) p.k_pre_sq[si] = pre;
                    if (p.k_post_sq) p.k_post_sq[si] = post;
                }
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[buf]);  // this warp is done with the stage buffer
    }
}

template <int NPL>
int launch_stream(const CamParams &p, long BN, cudaStream_t stream) {
    auto kern = cam_prep_stream_kernel<NPL>;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem) != cudaSuccess)
        return GDN_ERR_CUDA;
    const long nstages = (BN + kStageTok - 1) / kStageTok;
    const unsigned grid = (unsigned)(nstages < sms ? nstages : sms);
    kern<<<grid, 32 * (2 * kStageTok + 1), kStreamSmem, stream>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int launch_t(const CamArgs &a, cudaStream_t stream) {
    CamParams p{a.q_raw, a.k_raw, a.v_raw, a.q_norm_w, a.k_norm_w, a.proj_q, a.proj_kv,
                a.rope_cos, a.rope_sin, log2((double)a.rope_base), a.q_out, a.k_out, a.v_out,
                a.k_pre_sq, a.k_post_sq, a.B, a.N, a.H, a.D, a.k_scale, a.eps};
    const long BN = (long)a.B * a.N;
    if (sizeof(T) == 2 && a.rope_cos != nullptr && a.H * a.D <= kMaxC && (a.D / 2) % 4 == 0) {
        // rows, projections and rotary rows start on 16-byte boundaries (the
        // API checks the bases; C*2 and D/2*4 are multiples of 16 here)
        const int npl = (a.H * a.D / 8 + 31) / 32;
        if (npl <= 2) return launch_stream<2>(p, BN, stream);
        if (npl <= 4) return launch_stream<4>(p, BN, stream);
        return launch_stream<8>(p, BN, stream);
    }
    const unsigned grid = (unsigned)((BN + kTokPerCta - 1) / kTokPerCta);
    const int C = a.H * a.D;
    const int npl = (C / 8 + 31) / 32;
    if (npl <= 1) cam_prep_kernel<T, 1><<<grid, 32 * kTokPerCta, 0, stream>>>(p);
    else if (npl <= 2) cam_prep_kernel<T, 2><<<grid, 32 * kTokPerCta, 0, stream>>>(p);
    else if (npl <= 4) cam_prep_kernel<T, 4><<<grid, 32 * kTokPerCta, 0, stream>>>(p);
    else if (npl <= 8) cam_prep_kernel<T, 8><<<grid, 32 * kTokPerCta, 0, stream>>>(p);
    else if (npl <= 16) cam_prep_kernel<T, 16><<<grid, 32 * kTokPerCta, 0, stream>>>(p);
    else return GDN_ERR_UNSUPPORTED;
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

int cam_prep_read_clear_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_cam_error, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_cam_error, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
    return v ? GDN_ERR_TIMEOUT : GDN_OK;
}

namespace {

// Backward of the camera prep (fused_cam_gdn.py, `_cam_prep_bwd_kernel`,
// continued through the full-C RMSNorm, which the page leaves to torch).  The
// streamed kernel further below takes bf16 rows of C <= 2048 with rotary
// tables; this one takes the rest.  One CTA per token, thread i taking
// channels 8i .. 8i+7 (head c / D, dims c % D):
// the forward values it needs are recomputed, the rotation and projection are
// transposed, the ||k||^2 terms, K-scale and ReLU mask are applied, and the
// RMSNorm backward dx_j = r w_j dxhat_j - (r^3 / C) x_j sum_c w_c x_c dxhat_c
// takes one block reduction.  All arithmetic in fp32.
struct CamBwdParams {
    const void *q_raw, *k_raw;
    const float *q_norm_w, *k_norm_w, *proj_q, *proj_kv, *rope_cos, *rope_sin;
    double log2_base;
    const void *dq_out, *dk_out, *dv_out;
    const float *dpre, *dpost;
    void *dq_raw, *dk_raw, *dv_raw;
    int B, N, H, D;
    float k_scale, eps;
};

template <typename T>
__device__ __forceinline__ void ld8(const T *p, float (&x)[8]);
template <>
__device__ __forceinline__ void ld8<float>(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
__device__ __forceinline__ void ld8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}
__device__ __forceinline__ void st8(float *p, const float (&x)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
__device__ __forceinline__ void st8(__nv_bfloat16 *p, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Sum of a and b over the CTA (at most 16 warps).
__device__ __forceinline__ float2 block_sum2(float a, float b, float2 *red) {
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();  // red may still be read from a previous call
    if ((threadIdx.x & 31) == 0) red[w] = make_float2(a, b);
    __syncthreads();
    float2 t = make_float2(0.f, 0.f);
    for (int i = 0; i < nw; ++i) {
        t.x += red[i].x;
        t.y += red[i].y;
    }
    return t;
}

template <typename T>
__global__ void __launch_bounds__(512) cam_prep_bwd_kernel(CamBwdParams p) {
    __shared__ float2 red[16];
    const long long bn = blockIdx.x;
    const int b = (int)(bn / p.N), n = (int)(bn % p.N);
    const int C = p.H * p.D, Dh = p.D / 2;
    const int c0 = 8 * threadIdx.x;
    const bool act = c0 < C;
    const int h = act ? c0 / p.D : 0, d0 = act ? c0 % p.D : 0;
    // the token's streamed loads are all issued before the first block
    // reduction, so that the CTA waits for one memory round trip
    float q[8] = {0}, k[8] = {0}, dy[3][8];
    float gpre = 0.f, gpost = 0.f;
    const size_t ob = (((size_t)b * p.H + h) * p.N + n) * p.D + d0;
    if (act) {
        ld8(static_cast<const T *>(p.q_raw) + bn * C + c0, q);
        ld8(static_cast<const T *>(p.k_raw) + bn * C + c0, k);
        ld8(static_cast<const T *>(p.dq_out) + ob, dy[0]);
        ld8(static_cast<const T *>(p.dk_out) + ob, dy[1]);
        ld8(static_cast<const T *>(p.dv_out) + ob, dy[2]);
        const size_t si = ((size_t)b * p.H + h) * p.N + n;
        gpre = p.dpre ? p.dpre[si] : 0.f;
        gpost = p.dpost ? p.dpost[si] : 0.f;
    }
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        sq += q[e] * q[e];
        sk += k[e] * k[e];
    }
    const float2 ss = block_sum2(sq, sk, red);
    const float iq = rsqrtf(ss.x / C + p.eps), ik = rsqrtf(ss.y / C + p.eps);
    float wq[8], wk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        wq[e] = (act && p.q_norm_w) ? p.q_norm_w[c0 + e] : 1.f;
        wk[e] = (act && p.k_norm_w) ? p.k_norm_w[c0 + e] : 1.f;
    }
    float dxq[8] = {0}, dxk[8] = {0}, dav[8] = {0};
    if (act) {
        float P[2][16];  // the token's projections (the same for every thread: cached loads)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            P[0][e] = p.proj_q[bn * 16 + e];
            P[1][e] = p.proj_kv[bn * 16 + e];
        }
        // rotation of the four pairs of these dims (when in the last D/2)
        float cs[8], sn[8];
        if (d0 >= Dh) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = d0 - Dh + e;
                if (p.rope_cos) {
                    cs[e] = p.rope_cos[(size_t)n * Dh + d];
                    sn[e] = p.rope_sin[(size_t)n * Dh + d];
                } else {
                    const double inv_freq = exp2(p.log2_base * (-2.0 * (d >> 1) / (double)Dh));
                    double th = (double)n * inv_freq;
                    const double two_pi = 6.283185307179586476925286766559;
                    th -= two_pi * rint(th / two_pi);
                    float sv, cv;
                    sincosf((float)th, &sv, &cv);
                    cs[e] = cv;
                    sn[e] = (d & 1) ? sv : -sv;
                }
            }
        }
        float xq[8], xk[8], ak[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            xq[e] = q[e] * iq * wq[e];
            xk[e] = k[e] * ik * wk[e];
            ak[e] = fmaxf(xk[e], 0.f) * p.k_scale;
        }
        // k_out of these dims (for the ||k_out||^2 term)
        float ko[8];
        if (d0 < Dh) {
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    ko[4 * g + i] = P[1][4 * i] * ak[4 * g] + P[1][4 * i + 1] * ak[4 * g + 1] +
                                    P[1][4 * i + 2] * ak[4 * g + 2] + P[1][4 * i + 3] * ak[4 * g + 3];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) ko[e] = ak[e] * cs[e] + ak[e ^ 1] * sn[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) dy[1][e] += 2.f * ko[e] * gpost;
        float da[3][8];
#pragma unroll
        for (int tt = 0; tt < 3; ++tt) {
            const float *PP = P[tt == 0 ? 0 : 1];
            if (d0 < Dh) {
#pragma unroll
                for (int g = 0; g < 2; ++g)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        da[tt][4 * g + j] = PP[j] * dy[tt][4 * g] + PP[4 + j] * dy[tt][4 * g + 1] +
                                            PP[8 + j] * dy[tt][4 * g + 2] + PP[12 + j] * dy[tt][4 * g + 3];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) da[tt][e] = dy[tt][e] * cs[e] + dy[tt][e ^ 1] * sn[e ^ 1];
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            dxq[e] = xq[e] > 0.f ? da[0][e] : 0.f;
            dxk[e] = xk[e] > 0.f ? p.k_scale * (da[1][e] + 2.f * ak[e] * gpre) : 0.f;
            dav[e] = da[2][e];
        }
    }
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        tq += wq[e] * q[e] * dxq[e];
        tk += wk[e] * k[e] * dxk[e];
    }
    const float2 ts = block_sum2(tq, tk, red);
    if (act) {
        float oq[8], okk[8];
        const float cq3 = iq * iq * iq / C * ts.x, ck3 = ik * ik * ik / C * ts.y;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            oq[e] = iq * wq[e] * dxq[e] - cq3 * q[e];
            okk[e] = ik * wk[e] * dxk[e] - ck3 * k[e];
        }
        st8(static_cast<T *>(p.dq_raw) + bn * C + c0, oq);
        st8(static_cast<T *>(p.dk_raw) + bn * C + c0, okk);
        st8(static_cast<T *>(p.dv_raw) + bn * C + c0, dav);
    }
}

// ------------------------------------------------------------------ streamed backward
// The same backward for bf16 rows of C = H*D <= 2048 elements with rotary
// tables given, fed by the bulk-copy engine as in the streamed forward: one
// persistent CTA per SM walks stages of kBTok consecutive positions of one
// batch row.  A producer warp copies each stage's raw q and k rows, the three
// output gradients (head-major, so one copy per gradient and head holds the
// stage's kBTok rows of D), the projections and the rotary rows into one of
// kBBuf shared-memory buffers; 12 compute warps, four per token (each a
// quarter of the token's 8-channel groups), form the gradients from there
// while the next stages' copies are in flight.  Thirteen warps leave each
// thread 128 registers, which the token's values need without spilling.  The two full-C sums each token needs
// (the RMS factors, then the RMSNorm backward's dot products) meet through
// shared memory under a named barrier of the token's four warps.
constexpr int kBTok = 3;
constexpr int kBBuf = 3;                                     // stage buffers
constexpr uint32_t kBRows = kBTok * kMaxC * 2;              // kBTok bf16 rows of C (12 KB)
constexpr uint32_t kBQ = 0, kBK = kBRows, kBG = 2 * kBRows;  // q rows | k rows | dq, dk, dv blocks
constexpr uint32_t kBPJ = 5 * kBRows;                        // proj_q [kBTok][16] | proj_kv [kBTok][16]
constexpr uint32_t kBRT = kBPJ + 2 * kBTok * 64;             // cos [kBTok][Dh] | sin [kBTok][Dh]
constexpr uint32_t kBStage = kBRT + 2 * kBTok * kMaxDh * 4;
constexpr int kBWarps = 4 * kBTok;                           // compute warps
constexpr uint32_t kBSmem = kBBuf * kBStage + 16 * kBBuf + 2 * kBWarps * 2 * 4 + 128;
static_assert(kBStage % 128 == 0, "stage buffers keep 128-byte alignment");

__device__ __forceinline__ F8 unpack_bf16x8(uint4 u) {
    F8 r;
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r.x[2 * i] = __uint_as_float(w4[i] << 16);
        r.x[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
    }
    return r;
}

// NPL = 8-element groups per lane (C <= 1024 * NPL); DT = the head size D when
// it is fixed at compile time (its divisions become shifts), else 0.
template <int NPL, int DT>
__global__ void __launch_bounds__(32 * (kBWarps + 1), 1) cam_prep_bwd_stream_kernel(CamBwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((128u - (tc::smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kBBuf * kBStage);  // [kBBuf]
    uint64_t *empty = full + kBBuf;                                       // [kBBuf]
    float *part = reinterpret_cast<float *>(empty + kBBuf);               // [2 sums][kBWarps][2] per-warp partials
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int H = p.H, D = DT ? DT : p.D, N = p.N;
    const int C = H * D, Dh = D / 2, G8 = C / 8;
    const int spb = (N + kBTok - 1) / kBTok;  // stages per batch row
    const long nst = (long)p.B * spb;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kBBuf; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], kBWarps);
        }
        tc::fence_mbar_init();
    }
    __syncthreads();

    if (w == kBWarps) {
        // ---------------------------------------------------------- producer
        // lane 0 arms the stage's barrier, then the 32 lanes share its copies
        int j = 0;
        for (long st = blockIdx.x; st < nst; st += gridDim.x, ++j) {
            const int buf = j % kBBuf;
            int ok = 1;
            if (lane == 0 && j >= kBBuf) ok = cam_wait(&empty[buf], ((j - kBBuf) / kBBuf) & 1) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const int b = (int)(st / spb), n0 = (int)(st % spb) * kBTok;
            const int nt = min(kBTok, N - n0);
            const uint32_t rowb = (uint32_t)nt * C * 2, grb = (uint32_t)nt * D * 2;
            const uint32_t pjb = (uint32_t)nt * 64, rtb = (uint32_t)nt * Dh * 4;
            if (lane == 0) tc::mbar_arrive_expect_tx(&full[buf], 2 * rowb + 3u * H * grb + 2 * pjb + 2 * rtb);
            __syncwarp();
            const uint32_t sb = tc::smem_u32(sm + buf * kBStage);
            const size_t bn0 = (size_t)b * N + n0;
            for (int i = lane; i < 3 * H + 6; i += 32) {
                if (i < 3 * H) {
                    const int g = i / H, h = i % H;
                    const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(
                        g == 0 ? p.dq_out : (g == 1 ? p.dk_out : p.dv_out));
                    bulk_g2s(sb + kBG + g * kBRows + (uint32_t)h * (kBTok * D * 2),
                             src + (((size_t)b * H + h) * N + n0) * D, grb, &full[buf]);
                } else if (i == 3 * H) {
                    bulk_g2s(sb + kBQ, static_cast<const __nv_bfloat16 *>(p.q_raw) + bn0 * C, rowb, &full[buf]);
                } else if (i == 3 * H + 1) {
                    bulk_g2s(sb + kBK, static_cast<const __nv_bfloat16 *>(p.k_raw) + bn0 * C, rowb, &full[buf]);
                } else if (i == 3 * H + 2) {
                    bulk_g2s(sb + kBPJ, p.proj_q + bn0 * 16, pjb, &full[buf]);
                } else if (i == 3 * H + 3) {
                    bulk_g2s(sb + kBPJ + kBTok * 64, p.proj_kv + bn0 * 16, pjb, &full[buf]);
                } else if (i == 3 * H + 4) {
                    bulk_g2s(sb + kBRT, p.rope_cos + (size_t)n0 * Dh, rtb, &full[buf]);
                } else {
                    bulk_g2s(sb + kBRT + kBTok * kMaxDh * 4, p.rope_sin + (size_t)n0 * Dh, rtb, &full[buf]);
                }
            }
        }
        // the last stages' copies land before the CTA leaves
        if (lane == 0)
            for (int q = (j >= kBBuf ? j - kBBuf : 0); q < j; ++q) cam_wait(&empty[q % kBBuf], (q / kBBuf) & 1);
        return;
    }
    // -------------------------------------------------------------- compute
    const int tw = w >> 2, qw = w & 3;  // token of the stage, quarter of its groups
    int j = 0;
    for (long st = blockIdx.x; st < nst; st += gridDim.x, ++j) {
        const int buf = j % kBBuf;
        if (!cam_wait(&full[buf], (j / kBBuf) & 1)) break;
        const int b = (int)(st / spb), n = (int)(st % spb) * kBTok + tw;
        if (n < N) {
            const size_t bn = (size_t)b * N + n;
            const uint8_t *sb = sm + buf * kBStage;
            const __nv_bfloat16 *sq_ = reinterpret_cast<const __nv_bfloat16 *>(sb + kBQ) + (size_t)tw * C;
            const __nv_bfloat16 *sk_ = reinterpret_cast<const __nv_bfloat16 *>(sb + kBK) + (size_t)tw * C;
            const float *Pq = reinterpret_cast<const float *>(sb + kBPJ) + tw * 16;
            const float *Pk = reinterpret_cast<const float *>(sb + kBPJ + kBTok * 64) + tw * 16;
            const float *cs = reinterpret_cast<const float *>(sb + kBRT) + tw * Dh;
            const float *sn = reinterpret_cast<const float *>(sb + kBRT + kBTok * kMaxDh * 4) + tw * Dh;
            // the token's RMS factors
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int gi = lane + 32 * (4 * i + qw);
                if (gi < G8) {
                    const F8 x = unpack_bf16x8(*reinterpret_cast<const uint4 *>(sq_ + gi * 8));
                    const F8 y = unpack_bf16x8(*reinterpret_cast<const uint4 *>(sk_ + gi * 8));
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sq += x.x[e] * x.x[e];
                        sk += y.x[e] * y.x[e];
                    }
                }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
            }
            if (lane == 0) {
                part[2 * w] = sq;
                part[2 * w + 1] = sk;
            }
            asm volatile("bar.sync %0, 128;" ::"r"(1 + tw) : "memory");  // the token's four warps
            sq = sk = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                sq += part[2 * (4 * tw + r)];
                sk += part[2 * (4 * tw + r) + 1];
            }
            const float iq = rsqrtf(sq / (float)C + p.eps), ik = rsqrtf(sk / (float)C + p.eps);
            // gradients of the normalised rows; dv goes out at once
            float dxq[NPL][8], dxk[NPL][8];
            float tq = 0.f, tk = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int gi = lane + 32 * (4 * i + qw);
#pragma unroll
                for (int e = 0; e < 8; ++e) dxq[i][e] = dxk[i][e] = 0.f;
                if (gi >= G8) continue;
                const int c0 = gi * 8, h = c0 / D, d0 = c0 % D;
                const F8 q = unpack_bf16x8(*reinterpret_cast<const uint4 *>(sq_ + c0));
                const F8 k = unpack_bf16x8(*reinterpret_cast<const uint4 *>(sk_ + c0));
                F8 wq, wk;
                if (p.q_norm_w) wq = load8(p.q_norm_w + c0);
                else for (int e = 0; e < 8; ++e) wq.x[e] = 1.f;
                if (p.k_norm_w) wk = load8(p.k_norm_w + c0);
                else for (int e = 0; e < 8; ++e) wk.x[e] = 1.f;
                const uint8_t *gr = sb + kBG + (uint32_t)h * (kBTok * D * 2) + (uint32_t)(tw * D + d0) * 2;
                F8 dy[3];
#pragma unroll
                for (int g = 0; g < 3; ++g) dy[g] = unpack_bf16x8(*reinterpret_cast<const uint4 *>(gr + g * kBRows));
                const size_t si = ((size_t)b * H + h) * N + n;
                const float gpre = p.dpre ? p.dpre[si] : 0.f, gpost = p.dpost ? p.dpost[si] : 0.f;
                float xq[8], xk[8], ak[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    xq[e] = q.x[e] * iq * wq.x[e];
                    xk[e] = k.x[e] * ik * wk.x[e];
                    ak[e] = fmaxf(xk[e], 0.f) * p.k_scale;
                }
                float cva[8], sva[8];
                if (d0 >= Dh) {
                    const int dr = d0 - Dh;  // a multiple of 8: 16-byte aligned rows
                    const float4 c0v = *reinterpret_cast<const float4 *>(cs + dr);
                    const float4 c1v = *reinterpret_cast<const float4 *>(cs + dr + 4);
                    const float4 s0v = *reinterpret_cast<const float4 *>(sn + dr);
                    const float4 s1v = *reinterpret_cast<const float4 *>(sn + dr + 4);
                    cva[0] = c0v.x; cva[1] = c0v.y; cva[2] = c0v.z; cva[3] = c0v.w;
                    cva[4] = c1v.x; cva[5] = c1v.y; cva[6] = c1v.z; cva[7] = c1v.w;
                    sva[0] = s0v.x; sva[1] = s0v.y; sva[2] = s0v.z; sva[3] = s0v.w;
                    sva[4] = s1v.x; sva[5] = s1v.y; sva[6] = s1v.z; sva[7] = s1v.w;
                }
                // k_out of these dims, for the ||k_out||^2 term
                float ko[8];
                if (d0 < Dh) {
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            ko[4 * gg + r] = Pk[4 * r] * ak[4 * gg] + Pk[4 * r + 1] * ak[4 * gg + 1] +
                                             Pk[4 * r + 2] * ak[4 * gg + 2] + Pk[4 * r + 3] * ak[4 * gg + 3];
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) ko[e] = ak[e] * cva[e] + ak[e ^ 1] * sva[e];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) dy[1].x[e] += 2.f * ko[e] * gpost;
                // transposed projection (first D/2 dims) or rotation (last D/2)
                F8 da[3];
#pragma unroll
                for (int g = 0; g < 3; ++g) {
                    const float *PP = g == 0 ? Pq : Pk;
                    if (d0 < Dh) {
#pragma unroll
                        for (int gg = 0; gg < 2; ++gg)
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                da[g].x[4 * gg + c] = PP[c] * dy[g].x[4 * gg] + PP[4 + c] * dy[g].x[4 * gg + 1] +
                                                      PP[8 + c] * dy[g].x[4 * gg + 2] + PP[12 + c] * dy[g].x[4 * gg + 3];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) da[g].x[e] = dy[g].x[e] * cva[e] + dy[g].x[e ^ 1] * sva[e ^ 1];
                    }
                }
                store8(static_cast<__nv_bfloat16 *>(p.dv_raw) + bn * C + c0, da[2]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    dxq[i][e] = xq[e] > 0.f ? da[0].x[e] : 0.f;
                    dxk[i][e] = xk[e] > 0.f ? p.k_scale * (da[1].x[e] + 2.f * ak[e] * gpre) : 0.f;
                    tq += wq.x[e] * q.x[e] * dxq[i][e];
                    tk += wk.x[e] * k.x[e] * dxk[i][e];
                }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                tq += __shfl_xor_sync(0xffffffffu, tq, off);
                tk += __shfl_xor_sync(0xffffffffu, tk, off);
            }
            if (lane == 0) {
                part[2 * kBWarps + 2 * w] = tq;
                part[2 * kBWarps + 2 * w + 1] = tk;
            }
            asm volatile("bar.sync %0, 128;" ::"r"(1 + tw) : "memory");
            tq = tk = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                tq += part[2 * kBWarps + 2 * (4 * tw + r)];
                tk += part[2 * kBWarps + 2 * (4 * tw + r) + 1];
            }
            // RMSNorm backward: dx = r w dxhat - (r^3 / C) x sum_c w_c x_c dxhat_c
            const float cq3 = iq * iq * iq / C * tq, ck3 = ik * ik * ik / C * tk;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int gi = lane + 32 * (4 * i + qw);
                if (gi >= G8) continue;
                const int c0 = gi * 8;
                const F8 q = unpack_bf16x8(*reinterpret_cast<const uint4 *>(sq_ + c0));
                const F8 k = unpack_bf16x8(*reinterpret_cast<const uint4 *>(sk_ + c0));
                F8 wq, wk, oq, okk;
                if (p.q_norm_w) wq = load8(p.q_norm_w + c0);
                else for (int e = 0; e < 8; ++e) wq.x[e] = 1.f;
                if (p.k_norm_w) wk = load8(p.k_norm_w + c0);
                else for (int e = 0; e < 8; ++e) wk.x[e] = 1.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    oq.x[e] = iq * wq.x[e] * dxq[i][e] - cq3 * q.x[e];
                    okk.x[e] = ik * wk.x[e] * dxk[i][e] - ck3 * k.x[e];
                }
                store8(static_cast<__nv_bfloat16 *>(p.dq_raw) + bn * C + c0, oq);
                store8(static_cast<__nv_bfloat16 *>(p.dk_raw) + bn * C + c0, okk);
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[buf]);  // this warp is done with the stage buffer
    }
}

template <int NPL, int DT>
int launch_bwd_stream(const CamBwdParams &p, cudaStream_t stream) {
    auto kern = cam_prep_bwd_stream_kernel<NPL, DT>;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBSmem) != cudaSuccess)
        return GDN_ERR_CUDA;
    const long nst = (long)p.B * ((p.N + kBTok - 1) / kBTok);
    const unsigned grid = (unsigned)(nst < sms ? nst : sms);
    kern<<<grid, 32 * (kBWarps + 1), kBSmem, stream>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

int launch_cam_prep_bwd(const CamBwdArgs &a, cudaStream_t stream) {
    CamBwdParams p{a.q_raw, a.k_raw, a.q_norm_w, a.k_norm_w, a.proj_q, a.proj_kv, a.rope_cos, a.rope_sin,
                   log2((double)a.rope_base), a.dq_out, a.dk_out, a.dv_out, a.dpre, a.dpost, a.dq_raw, a.dk_raw,
                   a.dv_raw, a.B, a.N, a.H, a.D, a.k_scale, a.eps};
    const int C = a.H * a.D;
    if (a.dtype == GDN_BF16 && a.rope_cos && C <= kMaxC && a.D / 2 <= kMaxDh)
        return a.D == 128 ? (C <= 1024 ? launch_bwd_stream<1, 128>(p, stream) : launch_bwd_stream<2, 128>(p, stream))
                          : (C <= 1024 ? launch_bwd_stream<1, 0>(p, stream) : launch_bwd_stream<2, 0>(p, stream));
    const int threads = ((C / 8 + 31) / 32) * 32;
    const long long tokens = (long long)a.B * a.N;
    if (a.dtype == GDN_BF16)
        cam_prep_bwd_kernel<__nv_bfloat16><<<(unsigned)tokens, threads, 0, stream>>>(p);
    else
        cam_prep_bwd_kernel<float><<<(unsigned)tokens, threads, 0, stream>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int launch_cam_prep(const CamArgs &a, cudaStream_t stream) {
    if (a.dtype == GDN_BF16) return launch_t<__nv_bfloat16>(a, stream);
    if (a.dtype == GDN_F32) return launch_t<float>(a, stream);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
