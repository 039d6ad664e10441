// cam_scan.cu -- frame-level camera scan (fused_cam_gdn.py, `_cam_scan_kernel`,
// `_torch_cam_scan_single_chunk`, `_torch_cam_scan_reference`), forward and
// reverse.  The tokens of each (batch, head) form F frames of S tokens; per
// frame the state is decayed once by the frame's factor d_f, every token of the
// frame predicts from that same state, all S corrections enter at once, and
// the frame's tokens read the state after the update:
//
//     S_f = d_f S_{f-1} + K_f^T diag(beta_f) (V_f - K_f d_f S_{f-1})
//         = d_f (S_{f-1} - G_f S_{f-1}) + H_f,      o_s = scale S_f^T q_s,
//     G_f = K_f^T diag(beta_f) K_f,   H_f = K_f^T diag(beta_f) V_f.
//
// G_f and H_f do not depend on the state, so the tensor-core path (bf16,
// Dk = Dv = 128) runs three launches:
//
//   cam_gram_kernel   one (head, frame) item at a time per CTA: streams the
//                     frame's K and V through TMA in 64-token tiles, scales a
//                     copy of K by beta (and the unit-norm factors) on the CUDA
//                     cores, and accumulates [G | H] = (beta K)^T [K | V] in TMEM
//                     with tcgen05 (M = 128, N = 256); writes G as a bf16 MMA
//                     operand image and H^T in fp32 to the workspace.
//   cam_chain_kernel  one CTA per head: the 128 x 128 fp32 state lives in TMEM;
//                     per frame one MMA S += (-G_f) bf16(S), then S <- d_f S + H_f
//                     in fp32, and bf16(S_f) goes out as the output's operand.
//   cam_out_kernel    (head, frame, 128-token tile) items: O = scale Q S_f by
//                     tcgen05, rows scaled by 1/||q|| when asked.
//
// Keeping S in fp32 and rounding only G S's operands to bf16 keeps the chain's
// error at the bf16 level of the correction term, not of the state.  The
// reverse mode runs the same chain from the last frame to the first, frame f
// reading the state built from frames f+1 .. F-1 (the last frame reads zero).
// Every other shape and dtype takes cam_scan_simt_kernel, which runs the frame
// loop as written on the CUDA cores in fp32.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "gdn_internal.h"
#include "tc_util.cuh"

namespace gdn {
namespace {
using namespace tc;

__device__ unsigned int g_cs_error = 0;  // set when a bounded wait of these kernels gives up
constexpr unsigned long long kWaitNs = 1000000000ull;

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, unsigned code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile unsigned *>(&g_cs_error) != 0u) return false;
        if (global_timer_ns() - t0 > kWaitNs) {
            atomicOr(&g_cs_error, code);
            return false;
        }
    }
}

// A wait's outcome made uniform across the warp, so that the warp's
// .sync.aligned tcgen05 loads that follow are reached by all of its lanes.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok) != 0; }

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)(32 * (warp & 3)) << 16; }

__device__ __forceinline__ float bf16_bits_to_float(unsigned short b) { return __uint_as_float((uint32_t)b << 16); }

// ============================================================== gram kernel
constexpr int kGramThreads = 704;       // warp 0 TMA, warp 1 MMA, warps 2..17 A copies, warps 18..21 epilogue
constexpr int kGramWorkers = 512;       // A-copy threads: 8 per token row of a 64-row tile, 16 dims each
constexpr int kGramStages = 4;          // K | V tiles in flight
constexpr uint32_t GR_STAGE = 32768;    // K (16 KB) | V (16 KB)
constexpr uint32_t GR_K = 0, GR_V = 16384;
constexpr uint32_t GR_A = kGramStages * GR_STAGE;  // two A buffers (16 KB each)
constexpr uint32_t GR_T64 = GR_A + 2 * 16384;      // fused prep: cos / sin (t w_i), t < 64, i < 32
constexpr uint32_t GR_BASE = GR_T64 + 16384;       // fused prep: per stage cos / sin (n0 w_i) of the tile's first token
constexpr uint32_t GR_BAR = GR_BASE + kGramStages * 256;
enum { GB_FULL = 0, GB_EMPTY = 4, GB_AREADY = 8, GB_AEMPTY = 10, GB_ACCF = 12, GB_ACCE = 14, GB_DRAIN = 16, GB_NUM = 17 };
constexpr uint32_t GR_SMEM = GR_BAR + 8 * GB_NUM + 16 + 1024;
constexpr uint32_t kImgBytes = 32768;                 // a 128 x 128 bf16 operand image
constexpr uint32_t kHtFloats = 128 * 128;
constexpr size_t kPerFrame = 2 * (size_t)kImgBytes + sizeof(float) * kHtFloats;  // G image | S image | H^T
static_assert(GR_SMEM <= 232448, "gram kernel fits the shared memory of one CTA");

// The camera prep applied to raw rows at load (fused_cam_gdn.py,
// `_cam_prep_kernel`): per-token inverse RMS over all heads (from the
// pre-pass), per-channel norm weight, ReLU and K-scale (k only), the token's
// 4 x 4 projection on the first 64 dims and the interleaved rotation on the
// last 64 by th_i = n base^(-2i/64).  The rotation of token n = n0 + t is that
// of n0, formed per tile in double precision and reduced modulo 2 pi, composed
// with that of t < 64, formed once per CTA: cos(th) = cos(n0 w) cos(t w) -
// sin(n0 w) sin(t w), and so on.
struct PrepParams {
    const float *inv_rms;             // [B*N][2]: q, k
    const float *wq, *wk;             // [H*128] or null (ones)
    const float *proj_q, *proj_kv;    // [B*N][4][4]
    double log2_base;                 // log2 of the rotary base
    float k_scale;
    int H;
};

struct GramParams {
    const unsigned short *beta;  // bf16 bits [BH][N]
    uint8_t *gimg;               // [BH*F][32 KB]
    float *ht;                   // [BH*F][128][128]: H^T
    int BH, F, S, N;
    unsigned flags;
    PrepParams pp;               // used when the kernel fuses the prep
};

__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8]) {
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w4[e] << 16);
        x[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

// cos / sin of th_i = t w_i for t < 64, i < 32, by the threads of a group.
__device__ __forceinline__ void fill_t64(float *t64, double log2_base, int tid, int nthreads) {
    for (int e = tid; e < 64 * 32; e += nthreads) {
        const int t = e >> 5, i = e & 31;
        const float w = (float)exp2(-log2_base * (2.0 * i / 64.0));
        float sv, cv;
        sincosf((float)t * w, &sv, &cv);
        t64[e] = cv;
        t64[2048 + e] = sv;
    }
}

// cos / sin of th_i = n0 w_i for the 32 frequencies, lane i, the angle formed
// and reduced modulo 2 pi in double so that large positions keep precision.
__device__ __forceinline__ void base_angle(int n0, double log2_base, int i, float *dst) {
    const double w = exp2(-log2_base * (2.0 * i / 64.0));
    const double two_pi = 6.283185307179586476925286766559;
    double th = (double)n0 * w;
    th -= two_pi * rint(th / two_pi);
    float sv, cv;
    sincosf((float)th, &sv, &cv);
    dst[i] = cv;
    dst[32 + i] = sv;
}

// Eight consecutive dims d0 .. d0+7 of one head row after the prep: x * rms * w,
// then ReLU and `post` when `relu`, then the projection (d0 < 64: two groups
// of four, out_i = sum_j P[i][j] x_j) or the rotation of row t of the tile
// (d0 >= 64: pairs (2p, 2p+1), y_2p = x_2p cos - x_2p+1 sin,
// y_2p+1 = x_2p sin + x_2p+1 cos with th of frequency p).
__device__ __forceinline__ void prep8(float (&x)[8], int d0, float rms, const float *w, bool relu, float post,
                                      const float *P, const float *t64, int t, const float *base) {
    if (w) {  // the head's norm weights (the same for every token: cached after the first tile)
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(w + d0));
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(w + d0) + 1);
        const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= rms * ww[e];
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= rms;
    }
    if (relu) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = fmaxf(x[e], 0.f) * post;
    }
    if (d0 < 64) {
        float y[8];
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                y[4 * g + i] = P[4 * i] * x[4 * g] + P[4 * i + 1] * x[4 * g + 1] + P[4 * i + 2] * x[4 * g + 2] +
                               P[4 * i + 3] * x[4 * g + 3];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = y[e];
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int f = ((d0 - 64) >> 1) + q;  // frequency of pair q
            const float ct = t64[t * 32 + f], st = t64[2048 + t * 32 + f];
            const float cb = base[f], sb = base[32 + f];
            const float c = cb * ct - sb * st, sn = sb * ct + cb * st;
            const float a = x[2 * q], b = x[2 * q + 1];
            x[2 * q] = a * c - b * sn;
            x[2 * q + 1] = a * sn + b * c;
        }
    }
}

template <bool PREP>
__global__ void __launch_bounds__(kGramThreads, 1)
    cam_gram_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, GramParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + GR_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + GR_BAR + 8 * GB_NUM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool l2n = (p.flags & GDN_QK_L2NORM) != 0;
    const int nt = (p.S + 63) / 64;
    const int items = p.BH * p.F;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGramStages; ++s) {
            mbar_init(&bars[GB_FULL + s], 1);
            mbar_init(&bars[GB_EMPTY + s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars[GB_AREADY + a], kGramWorkers);
            mbar_init(&bars[GB_AEMPTY + a], 1);
            mbar_init(&bars[GB_ACCF + a], 1);
            mbar_init(&bars[GB_ACCE + a], 128);
        }
        mbar_init(&bars[GB_DRAIN], 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32 * 2) {
        prefetch_tensormap(&mK);
        prefetch_tensormap(&mV);
    }
    if (PREP && warp >= 2 && warp < 18) fill_t64(reinterpret_cast<float *>(sm + GR_T64), p.pp.log2_base,
                                                threadIdx.x - 64, kGramWorkers);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // Tiles of 64 tokens; a tile that runs past its frame's last token is
        // clipped there by the frame-shaped map (zeros, no memory traffic).
        // With the fused prep the warp's lanes also form the tile's base
        // rotation before the tile is armed.
        int j = 0, armed[kGramStages] = {0, 0, 0, 0};
        bool ok = true;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            const int bh = it / p.F, f = it % p.F;
            for (int i = 0; i < nt; ++i, ++j) {
                const int s = j % kGramStages;
                bool w = true;
                if (lane == 0 && j >= kGramStages) w = wait_phase(&bars[GB_EMPTY + s], ((j / kGramStages) - 1) & 1, 1u);
                if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
                if (PREP) base_angle(f * p.S + 64 * i, p.pp.log2_base, lane,
                                     reinterpret_cast<float *>(sm + GR_BASE + s * 256));
                __syncwarp();
                if (lane == 0) {
                    uint8_t *st = sm + s * GR_STAGE;
                    // fused prep: raw rows [B][N][H*128], head h's 128 columns
                    const int x0 = PREP ? 128 * (bh % p.pp.H) : 0, outer = PREP ? bh / p.pp.H : bh;
                    mbar_arrive_expect_tx(&bars[GB_FULL + s], 32768);
                    tma_load_4d(st + GR_K, &mK, &bars[GB_FULL + s], x0, 64 * i, f, outer);
                    tma_load_4d(st + GR_K + 8192, &mK, &bars[GB_FULL + s], x0 + 64, 64 * i, f, outer);
                    tma_load_4d(st + GR_V, &mV, &bars[GB_FULL + s], x0, 64 * i, f, outer);
                    tma_load_4d(st + GR_V + 8192, &mV, &bars[GB_FULL + s], x0 + 64, 64 * i, f, outer);
                }
                armed[s]++;
            }
        }
        if (lane == 0)
            for (int s = 0; s < kGramStages; ++s)
                if (armed[s]) mbar_wait(&bars[GB_FULL + s], (armed[s] - 1) & 1, 200000000ull);
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // [G | H] += A^T [K | V]: the K and V atoms sit at a uniform 8 KB stride,
        // so one N = 256 operand covers both
        if (lane == 0) {
            const uint32_t id256 = idesc_bf16(128, 256, true, true);
            int j = 0, acc = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++acc) {
                const int a = acc & 1;
                if (acc >= 2 && !wait_phase(&bars[GB_ACCE + a], ((acc >> 1) - 1) & 1, 2u)) break;
                const uint32_t d = tmem + 256u * a;
                for (int i = 0; i < nt; ++i, ++j) {
                    const int s = j % kGramStages, x = j & 1;
                    if (!wait_phase(&bars[GB_FULL + s], (j / kGramStages) & 1, 2u) ||
                        !wait_phase(&bars[GB_AREADY + x], (j >> 1) & 1, 2u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t st = sbase + s * GR_STAGE, ab = sbase + GR_A + x * 16384;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ss(d, smem_desc(ab + ks * 2048, 8192, 1024),
                                    smem_desc(st + GR_K + ks * 2048, 8192, 1024), id256,
                                    (i > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&bars[GB_EMPTY + s]);
                    mma_commit(&bars[GB_AEMPTY + x]);
                }
                if (!ok) break;
                mma_commit(&bars[GB_ACCF + a]);
            }
            // every MMA issued here is complete before TMEM is released
            mma_commit(&bars[GB_DRAIN]);
            mbar_wait(&bars[GB_DRAIN], 0, 200000000ull);
        }
    } else if (warp < 18) {
        // ------------------------------------------------------ A copies
        // Each thread takes 16 columns (two 8-column chunks) of one token row.
        // With the fused prep it first preps its k and v values in place (the B
        // operand [K | V]).  A = beta n^2 k, with n = 1 / ||k|| for unit-norm
        // keys (else 1); then G = sum beta (n k)(n k)^T, and H = sum beta (n k)
        // v^T holds once each v row is scaled by ||k|| = 1 / n in place.
        const int wt = threadIdx.x - 64;  // 0..511
        const int r = wt >> 3, cq = wt & 7;
        const int atom = cq >> 2, c0 = 16 * (cq & 3);
        const float *t64 = reinterpret_cast<const float *>(sm + GR_T64);
        int j = 0;
        bool ok = true;
        // beta of this thread's row, loaded a tile ahead of its use (raw bits)
        auto beta_bits = [&](int it2, int i2) -> unsigned short {
            if (it2 >= items) return 0;
            const int t2 = 64 * i2 + r;
            return t2 < p.S ? p.beta[(size_t)(it2 / p.F) * p.N + (size_t)(it2 % p.F) * p.S + t2] : (unsigned short)0;
        };
        unsigned short beta_nx = beta_bits(blockIdx.x, 0);
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            const int bh = it / p.F, f = it % p.F;
            const float *wk = (PREP && p.pp.wk) ? p.pp.wk + 128 * (bh % p.pp.H) : nullptr;
            for (int i = 0; i < nt; ++i, ++j) {
                const int s = j % kGramStages, x = j & 1;
                const int t = 64 * i + r;  // token within the frame
                const bool valid = t < p.S;
                const unsigned short bcur = beta_nx;
                beta_nx = i + 1 < nt ? beta_bits(it, i + 1) : beta_bits(it + (int)gridDim.x, 0);
                const float beta = valid ? bf16_bits_to_float(bcur) : 0.f;
                // the prep's per-token values, loaded before the wait
                float P[16], rk = 0.f;
                if (PREP && valid) {
                    const size_t tok = (size_t)(bh / p.pp.H) * p.N + (size_t)f * p.S + t;
                    rk = p.pp.inv_rms[2 * tok + 1];
                    if (atom == 0) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 q4 = __ldg(reinterpret_cast<const float4 *>(p.pp.proj_kv + tok * 16) + e);
                            P[4 * e] = q4.x; P[4 * e + 1] = q4.y; P[4 * e + 2] = q4.z; P[4 * e + 3] = q4.w;
                        }
                    }
                }
                bool w = wait_phase(&bars[GB_FULL + s], (j / kGramStages) & 1, 4u);
                if (w && j >= 2) w = wait_phase(&bars[GB_AEMPTY + x], ((j >> 1) - 1) & 1, 4u);
                if (!warp_all(w)) {
                    ok = false;
                    break;
                }
                uint8_t *st = sm + s * GR_STAGE;
                uint8_t *ab = sm + GR_A + x * 16384;
                const float *base = reinterpret_cast<const float *>(sm + GR_BASE + s * 256);
                float xk[2][8], xv[2][8];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t off = atom * 8192 + sw128_offset(r, c0 + 8 * u);
                    unpack8(*reinterpret_cast<const uint4 *>(st + GR_K + off), xk[u]);
                    if (PREP || l2n) unpack8(*reinterpret_cast<const uint4 *>(st + GR_V + off), xv[u]);
                    if (PREP && valid) {
                        const int d0 = 64 * atom + c0 + 8 * u;
                        // k: norm, ReLU, K-scale; v: none of these
                        if (wk) {
                            const float4 w0 = __ldg(reinterpret_cast<const float4 *>(wk + d0));
                            const float4 w1 = __ldg(reinterpret_cast<const float4 *>(wk + d0) + 1);
                            const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) xk[u][e] = fmaxf(xk[u][e] * rk * ww[e], 0.f) * p.pp.k_scale;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) xk[u][e] = fmaxf(xk[u][e] * rk, 0.f) * p.pp.k_scale;
                        }
                        float yk[8], yv[8];
                        if (d0 < 64) {
#pragma unroll
                            for (int g = 0; g < 2; ++g)
#pragma unroll
                                for (int ii = 0; ii < 4; ++ii) {
                                    yk[4 * g + ii] = P[4 * ii] * xk[u][4 * g] + P[4 * ii + 1] * xk[u][4 * g + 1] +
                                                     P[4 * ii + 2] * xk[u][4 * g + 2] + P[4 * ii + 3] * xk[u][4 * g + 3];
                                    yv[4 * g + ii] = P[4 * ii] * xv[u][4 * g] + P[4 * ii + 1] * xv[u][4 * g + 1] +
                                                     P[4 * ii + 2] * xv[u][4 * g + 2] + P[4 * ii + 3] * xv[u][4 * g + 3];
                                }
                        } else {
                            // one rotation per pair for both k and v
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int fq = ((d0 - 64) >> 1) + q;
                                const float ct = t64[r * 32 + fq], stt = t64[2048 + r * 32 + fq];
                                const float cb = base[fq], sb = base[32 + fq];
                                const float c = cb * ct - sb * stt, sn = sb * ct + cb * stt;
                                yk[2 * q] = xk[u][2 * q] * c - xk[u][2 * q + 1] * sn;
                                yk[2 * q + 1] = xk[u][2 * q] * sn + xk[u][2 * q + 1] * c;
                                yv[2 * q] = xv[u][2 * q] * c - xv[u][2 * q + 1] * sn;
                                yv[2 * q + 1] = xv[u][2 * q] * sn + xv[u][2 * q + 1] * c;
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            xk[u][e] = yk[e];
                            xv[u][e] = yv[e];
                        }
                    }
                }
                float nrm = 1.f;
                if (l2n) {
                    float ss = 0.f;
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss += xk[u][e] * xk[u][e];
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                    nrm = rsqrtf(fmaxf(ss, 1e-24f));  // 1 / max(||k||, 1e-12)
                }
                const float c1 = beta * nrm * nrm, vs = 1.f / nrm;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t off = atom * 8192 + sw128_offset(r, c0 + 8 * u);
                    float a8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) a8[e] = c1 * xk[u][e];
                    *reinterpret_cast<uint4 *>(ab + off) = pack8(a8);
                    if (PREP) *reinterpret_cast<uint4 *>(st + GR_K + off) = pack8(xk[u]);
                    if (PREP || l2n) {
                        if (l2n) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) xv[u][e] *= vs;
                        }
                        *reinterpret_cast<uint4 *>(st + GR_V + off) = pack8(xv[u]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&bars[GB_AREADY + x]);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        // thread dk: row dk of G (bf16 operand image) and of H (as H^T, fp32)
        const int dk = 32 * (warp & 3) + lane;
        const uint32_t lb = lane_base(warp);
        int acc = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x, ++acc) {
            const int bh = it / p.F, f = it % p.F;
            const int a = acc & 1;
            if (!warp_all(wait_phase(&bars[GB_ACCF + a], (acc >> 1) & 1, 4u))) break;
            tc_fence_after_sync();
            const size_t fi = (size_t)bh * p.F + f;
            uint8_t *gimg = p.gimg + fi * kImgBytes;
            float *ht = p.ht + fi * kHtFloats;
#pragma unroll 1
            for (int c = 0; c < 128; c += 16) {
                uint32_t g[16], h[16];
                tmem_ld16(tmem + lb + 256u * a + c, g);
                tmem_ld16(tmem + lb + 256u * a + 128u + c, h);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) pk[e] = pack_bf16(__uint_as_float(g[2 * e]), __uint_as_float(g[2 * e + 1]));
                uint8_t *blk = gimg + (c >> 6) * 16384;
                *reinterpret_cast<uint4 *>(blk + sw128_offset(dk, c & 63)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(blk + sw128_offset(dk, (c & 63) + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
#pragma unroll
                for (int e = 0; e < 16; ++e) ht[(size_t)(c + e) * 128 + dk] = __uint_as_float(h[e]);
            }
            tc_fence_before_sync();
            mbar_arrive(&bars[GB_ACCE + a]);
        }
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ============================================================= chain kernel
constexpr int kChainThreads = 256;  // thread (dk, half): TMEM lane dk, state columns 64 half .. 64 half + 63
constexpr uint32_t CH_G = 0;        // two G images (32 KB each)
constexpr uint32_t CH_H = 65536;    // two H^T blocks (64 KB each)
constexpr uint32_t CH_S = 196608;   // bf16(S) as the MMA's B operand (32 KB), also the image sent out
constexpr uint32_t CH_BAR = CH_S + kImgBytes;
constexpr uint32_t CH_SMEM = CH_BAR + 64 + 1024;
static_assert(CH_SMEM <= 232448, "chain kernel fits the shared memory of one CTA");

struct ChainParams {
    const uint8_t *gimg;
    const float *ht;
    uint8_t *simg;       // [BH*F][32 KB]: bf16(S_f) read by the output kernel
    const float *decay;  // [BH][F]
    const float *s0;
    float *sf;
    int BH, F;
    int reverse;
};

// One row of bf16(S) into a 128 x 128 MN-major operand image (two 64-column
// atoms of 128 rows x 128 bytes, 128-byte swizzle): row dk, columns c .. c+15.
__device__ __forceinline__ void put_img_row16(uint8_t *img, int dk, int c, const uint32_t (&pk)[8]) {
    uint8_t *blk = img + (c >> 6) * 16384;
    *reinterpret_cast<uint4 *>(blk + sw128_offset(dk, c & 63)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4 *>(blk + sw128_offset(dk, (c & 63) + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

__global__ void __launch_bounds__(kChainThreads, 1) cam_chain_kernel(ChainParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + CH_BAR);  // LOAD0, LOAD1, MMA, DRAIN
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + CH_BAR + 32);
    const int warp = threadIdx.x >> 5;
    const int dk = 32 * (warp & 3) + (threadIdx.x & 31);
    const int c0 = 64 * (warp >> 2);  // this thread's 64 state columns
    const int bh = blockIdx.x;
    const int F = p.F;
    const int nsteps = p.reverse ? F - 1 : F;
    const size_t fbase = (size_t)bh * F;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tl = tmem + lane_base(warp);
    const uint32_t sbase = smem_u32(sm);
    int armed[2] = {0, 0};  // thread 0: loads issued into each buffer
    auto kv_frame = [&](int st) { return p.reverse ? F - 1 - st : st; };
    auto load = [&](int st) {  // G and H^T of step st into buffer st & 1
        const int b = st & 1;
        armed[b]++;
        const size_t fi = fbase + kv_frame(st);
        mbar_arrive_expect_tx(&bars[b], kImgBytes + 4 * kHtFloats);
        bulk_load_global(sm + CH_G + b * kImgBytes, p.gimg + fi * kImgBytes, kImgBytes, &bars[b]);
        bulk_load_global(sm + CH_H + b * 65536, p.ht + fi * kHtFloats, 32768, &bars[b]);
        bulk_load_global(sm + CH_H + b * 65536 + 32768, p.ht + fi * kHtFloats + 8192, 32768, &bars[b]);
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < 2 && st < nsteps; ++st) load(st);
    }
    // initial state (forward) or zero, and bf16(S) for the first product
    {
        const float *s0 = (p.s0 && !p.reverse) ? p.s0 + (size_t)bh * 16384 : nullptr;
#pragma unroll 1
        for (int c = c0; c < c0 + 64; c += 16) {
            uint32_t v[16], pk[8];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(s0 ? s0[dk * 128 + c + e] : 0.f);
            tmem_st16(tl + c, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            put_img_row16(sm + CH_S, dk, c, pk);
        }
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && p.reverse) {
        // the last frame reads the zero state
        bulk_store_global(p.simg + (fbase + F - 1) * kImgBytes, sm + CH_S, kImgBytes);
        tma_store_commit();
    }
    bool ok = true;
    float d_next = nsteps > 0 ? p.decay[fbase + kv_frame(0)] : 0.f;
    for (int st = 0; st < nsteps; ++st) {
        const int b = st & 1;
        const int kf = kv_frame(st);
        const int of = p.reverse ? kf - 1 : kf;  // frame whose queries read the new state
        const float d = d_next;  // read one step ahead, off the chain's path
        if (st + 1 < nsteps) d_next = p.decay[fbase + kv_frame(st + 1)];
        if (threadIdx.x == 0) {
            if (wait_phase(&bars[b], (st >> 1) & 1, 8u)) {
                tc_fence_after_sync();
                const uint32_t idm = idesc_bf16(128, 128, false, true, true);
                const uint32_t g = sbase + CH_G + b * kImgBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ss(tmem, smem_desc(g + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                smem_desc(sbase + CH_S + ks * 2048, 16384, 1024), idm, 1u);
                mma_commit(&bars[2]);
            }
            tma_store_wait_read<0>();  // the previous state image has left CH_S
        }
        // every thread waits for the product S - G bf16(S) (the bounded wait
        // also ends once thread 0 has reported an expired load)
        if (!__syncthreads_and(wait_phase(&bars[2], st & 1, 8u) ? 1 : 0)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const float *ht = reinterpret_cast<const float *>(sm + CH_H + b * 65536);
#pragma unroll 1
        for (int c = c0; c < c0 + 64; c += 32) {
            uint32_t v[2][16];
            tmem_ld16(tl + c, v[0]);
            tmem_ld16(tl + c + 16, v[1]);
            tmem_wait_ld();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    v[hh][e] = __float_as_uint(fmaf(d, __uint_as_float(v[hh][e]), ht[(c + 16 * hh + e) * 128 + dk]));
                tmem_st16(tl + c + 16 * hh, v[hh]);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    pk[e] = pack_bf16(__uint_as_float(v[hh][2 * e]), __uint_as_float(v[hh][2 * e + 1]));
                put_img_row16(sm + CH_S, dk, c + 16 * hh, pk);
            }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();  // buffer b and the old bf16(S) consumed; the new bf16(S) is complete
        if (threadIdx.x == 0) {
            bulk_store_global(p.simg + (fbase + of) * kImgBytes, sm + CH_S, kImgBytes);
            tma_store_commit();
            if (st + 2 < nsteps) load(st + 2);
        }
    }
    if (ok && p.sf && !p.reverse) {
        tc_fence_after_sync();
        float *sf = p.sf + (size_t)bh * 16384;
#pragma unroll 1
        for (int c = c0; c < c0 + 64; c += 16) {
            uint32_t v[16];
            tmem_ld16(tl + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) sf[dk * 128 + c + e] = __uint_as_float(v[e]);
        }
    }
    if (threadIdx.x == 0) {
        // drain: every MMA issued, every load armed and every image sent out
        // completes before the CTA releases TMEM and its shared memory
        mma_commit(&bars[3]);
        mbar_wait(&bars[3], 0, 200000000ull);
        for (int b = 0; b < 2; ++b)
            if (armed[b]) mbar_wait(&bars[b], (armed[b] - 1) & 1, 200000000ull);
        tma_store_wait_all<0>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// =============================================================== out kernel
constexpr int kOutThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kOutStages = 3;
constexpr uint32_t OU_Q = 0;                        // Q tiles: [128 rows][128] as 2 K-blocks (32 KB)
constexpr uint32_t OU_S = kOutStages * 32768;       // two bf16(S_f) images
constexpr uint32_t OU_O = OU_S + 2 * kImgBytes;     // two output staging tiles (TMA store boxes)
constexpr uint32_t OU_BAR = OU_O + 2 * 32768;
enum { OB_QFULL = 0, OB_QEMPTY = 3, OB_SFULL = 6, OB_SEMPTY = 8, OB_OFULL = 10, OB_OEMPTY = 12, OB_DRAIN = 14,
       OB_QPREP = 15, OB_NUM = 18 };
constexpr uint32_t OU_QN = OU_BAR + 256;            // [stage][128] inverse norms of the prepped q rows
// fused prep: the second staging slot holds cos / sin (t w_i), t < 64, and the
// per-stage base rotations of the tile's two 64-row halves
constexpr uint32_t OU_T64 = OU_O + 32768;
constexpr uint32_t OU_QBASE = OU_T64 + 16384;
constexpr uint32_t OU_SMEM = OU_QN + kOutStages * 128 * 4 + 1024;
static_assert(8 * OB_NUM + 16 <= 256, "output kernel barriers fit their slot");
static_assert(OU_SMEM <= 232448, "output kernel fits the shared memory of one CTA");
constexpr int kOutThreadsPrep = 448;  // + warps 6..13, which apply the prep to each Q tile (two threads a row)

struct OutParams {
    const uint8_t *simg;
    int BH, F, S, nt;  // nt: 128-token tiles per frame
    long long items;
    float scale;
    unsigned flags;
    int N;
    PrepParams pp;     // used when the kernel fuses the prep
};

__device__ __forceinline__ void named_sync_epi() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Named barrier over the 128 epilogue threads that also ANDs a flag across
// them, so that they all take the same branch after a bounded wait.
__device__ __forceinline__ bool epi_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

template <bool PREP>
__global__ void __launch_bounds__(PREP ? kOutThreadsPrep : kOutThreads, 1)
    cam_out_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mO, OutParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OU_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OU_BAR + 8 * OB_NUM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool l2n = (p.flags & GDN_QK_L2NORM) != 0;
    const long long i0 = p.items * blockIdx.x / gridDim.x, i1 = p.items * (blockIdx.x + 1) / gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kOutStages; ++s) {
            mbar_init(&bars[OB_QFULL + s], 1);
            mbar_init(&bars[OB_QEMPTY + s], l2n ? 129u : 1u);  // the MMA, and the row norms when asked
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[OB_SFULL + b], 1);
            mbar_init(&bars[OB_SEMPTY + b], 1);
            mbar_init(&bars[OB_OFULL + b], 1);
            mbar_init(&bars[OB_OEMPTY + b], 128);
        }
        mbar_init(&bars[OB_DRAIN], 1);
        for (int s = 0; s < kOutStages; ++s) mbar_init(&bars[OB_QPREP + s], 256);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&mQ);
        prefetch_tensormap(&mO);
    }
    if (PREP && warp >= 6) fill_t64(reinterpret_cast<float *>(sm + OU_T64), p.pp.log2_base, threadIdx.x - 192, 256);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t sbase = smem_u32(sm);
    auto frame_of = [&](long long it) { return it / p.nt; };  // item -> bh * F + f

    if (warp == 0) {
        // the whole warp walks the items: lane 0 issues the copies; with the
        // fused prep every lane also forms one frequency of the tile's base
        // rotations before the tile is armed
        int armed[kOutStages] = {0, 0, 0}, sarmed[2] = {0, 0};
        long long prev = -1;
        int sidx = -1;
        for (long long it = i0; it < i1; ++it) {
            const int j = (int)(it - i0), s = j % kOutStages;
            const long long fi = frame_of(it);
            const int i = (int)(it % p.nt);
            const int bh = (int)(fi / p.F), f = (int)(fi % p.F);
            bool w = true;
            if (fi != prev) {
                ++sidx;
                const int sb = sidx & 1;
                if (lane == 0) {
                    if (sidx >= 2) w = wait_phase(&bars[OB_SEMPTY + sb], ((sidx >> 1) - 1) & 1, 16u);
                    if (w) {
                        mbar_arrive_expect_tx(&bars[OB_SFULL + sb], kImgBytes);
                        bulk_load_global(sm + OU_S + sb * kImgBytes, p.simg + (size_t)fi * kImgBytes, kImgBytes,
                                         &bars[OB_SFULL + sb]);
                    }
                }
                sarmed[sb]++;
                prev = fi;
            }
            if (lane == 0 && w && j >= kOutStages) w = wait_phase(&bars[OB_QEMPTY + s], ((j / kOutStages) - 1) & 1, 16u);
            if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) break;
            if (PREP) {
                float *qb = reinterpret_cast<float *>(sm + OU_QBASE + s * 512);
                base_angle(f * p.S + 128 * i, p.pp.log2_base, lane, qb);
                base_angle(f * p.S + 128 * i + 64, p.pp.log2_base, lane, qb + 64);
            }
            __syncwarp();
            if (lane == 0) {
                const int x0 = PREP ? 128 * (bh % p.pp.H) : 0, outer = PREP ? bh / p.pp.H : bh;
                mbar_arrive_expect_tx(&bars[OB_QFULL + s], 32768);
                tma_load_4d(sm + OU_Q + s * 32768, &mQ, &bars[OB_QFULL + s], x0, 128 * i, f, outer);
                tma_load_4d(sm + OU_Q + s * 32768 + 16384, &mQ, &bars[OB_QFULL + s], x0 + 64, 128 * i, f, outer);
            }
            armed[s]++;
        }
        if (lane == 0) {
            for (int s = 0; s < kOutStages; ++s)
                if (armed[s]) mbar_wait(&bars[OB_QFULL + s], (armed[s] - 1) & 1, 200000000ull);
            for (int b = 0; b < 2; ++b)
                if (sarmed[b]) mbar_wait(&bars[OB_SFULL + b], (sarmed[b] - 1) & 1, 200000000ull);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t ido = idesc_bf16(128, 128, false, true);
            long long prev = -1;
            int sidx = -1;
            for (long long it = i0; it < i1; ++it) {
                const int j = (int)(it - i0), s = j % kOutStages, a = j & 1;
                const long long fi = frame_of(it);
                if (fi != prev) {
                    ++sidx;
                    prev = fi;
                    if (!wait_phase(&bars[OB_SFULL + (sidx & 1)], (sidx >> 1) & 1, 32u)) break;
                }
                if (j >= 2 && !wait_phase(&bars[OB_OEMPTY + a], ((j >> 1) - 1) & 1, 32u)) break;
                if (!wait_phase(&bars[(PREP ? OB_QPREP : OB_QFULL) + s], (j / kOutStages) & 1, 32u)) break;
                tc_fence_after_sync();
                const uint32_t q = sbase + OU_Q + s * 32768, sb = sbase + OU_S + (sidx & 1) * kImgBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ss(tmem + 128u * a, smem_desc(q + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                smem_desc(sb + ks * 2048, 16384, 1024), ido, ks > 0 ? 1u : 0u);
                mma_commit(&bars[OB_QEMPTY + s]);
                mma_commit(&bars[OB_OFULL + a]);
                if (it + 1 >= i1 || frame_of(it + 1) != fi) mma_commit(&bars[OB_SEMPTY + (sidx & 1)]);
            }
            mma_commit(&bars[OB_DRAIN]);
            mbar_wait(&bars[OB_DRAIN], 0, 200000000ull);
        }
    } else if (warp >= 6) {
        // (fused prep only) warps 6..13: the prep of each Q tile in place, two
        // threads a row (dims 0..63, the projection, and 64..127, the
        // rotation), and the row's inverse norm for the unit-norm flag
        const int pt = threadIdx.x - 192;  // 0..255
        const int row = pt >> 1, half = pt & 1;
        const PrepParams &pp = p.pp;
        float *qn = reinterpret_cast<float *>(sm + OU_QN);
        const float *t64 = reinterpret_cast<const float *>(sm + OU_T64);
        for (long long it = i0; it < i1; ++it) {
            const int j = (int)(it - i0), s = j % kOutStages;
            const long long fi = frame_of(it);
            const int i = (int)(it % p.nt);
            const int bh = (int)(fi / p.F), f = (int)(fi % p.F);
            const int t = 128 * i + row;
            // the token's values, loaded before the wait
            const int h = bh % pp.H, b = bh / pp.H, n = f * p.S + t;
            const size_t tok = (size_t)b * p.N + n;
            float rq = 0.f, P[16];
            if (t < p.S) {
                rq = pp.inv_rms[2 * tok];
                if (half == 0) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 q4 = __ldg(reinterpret_cast<const float4 *>(pp.proj_q + tok * 16) + e);
                        P[4 * e] = q4.x; P[4 * e + 1] = q4.y; P[4 * e + 2] = q4.z; P[4 * e + 3] = q4.w;
                    }
                }
            }
            if (!wait_phase(&bars[OB_QFULL + s], (j / kOutStages) & 1, 64u)) break;
            uint8_t *qt = sm + OU_Q + s * 32768;
            float ssq = 0.f;
            if (t < p.S) {
                const float *base = reinterpret_cast<const float *>(sm + OU_QBASE + s * 512) + 64 * (row >> 6);
                const float *wq = pp.wq ? pp.wq + 128 * h : nullptr;
#pragma unroll 2
                for (int u = 0; u < 8; ++u) {
                    const uint32_t off = half * 16384 + sw128_offset(row, 8 * u);
                    float x8[8];
                    unpack8(*reinterpret_cast<const uint4 *>(qt + off), x8);
                    prep8(x8, 64 * half + 8 * u, rq, wq, true, 1.f, P, t64, row & 63, base);
                    const uint4 pk = pack8(x8);
                    *reinterpret_cast<uint4 *>(qt + off) = pk;
                    float y8[8];
                    unpack8(pk, y8);  // the norm of the operand the MMA sees
#pragma unroll
                    for (int e = 0; e < 8; ++e) ssq += y8[e] * y8[e];
                }
            }
            ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
            if (half == 0) qn[s * 128 + row] = rsqrtf(fmaxf(ssq, 1e-24f));
            fence_proxy_async_smem();
            mbar_arrive(&bars[OB_QPREP + s]);
        }
    } else {
        // epilogue: thread = token row of the tile (TMEM lane); the tile goes
        // through a 128-byte-swizzled staging buffer and leaves as two TMA
        // stores, clipped at the frame's last row by the frame-shaped map
        const int row = 32 * (warp & 3) + lane;
        const bool storer = threadIdx.x == 64;
        for (long long it = i0; it < i1; ++it) {
            const int j = (int)(it - i0), s = j % kOutStages, a = j & 1, x = PREP ? 0 : (j & 1);
            const long long fi = frame_of(it);
            const int i = (int)(it % p.nt);
            const int bh = (int)(fi / p.F), f = (int)(fi % p.F);
            float m = p.scale;
            bool w = true;
            if (l2n && PREP) {
                w = wait_phase(&bars[OB_QPREP + s], (j / kOutStages) & 1, 64u);
                if (w) {
                    m *= reinterpret_cast<const float *>(sm + OU_QN)[s * 128 + row];
                    mbar_arrive(&bars[OB_QEMPTY + s]);
                }
            } else if (l2n) {
                w = wait_phase(&bars[OB_QFULL + s], (j / kOutStages) & 1, 64u);
                if (w) {
                    const uint8_t *qt = sm + OU_Q + s * 32768;
                    float ss = 0.f;
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint4 xq = *reinterpret_cast<const uint4 *>(qt + kb * 16384 + sw128_offset(row, 8 * u));
                            const uint32_t w4[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                                ss += lo * lo + hi * hi;
                            }
                        }
                    m *= rsqrtf(fmaxf(ss, 1e-24f));
                    mbar_arrive(&bars[OB_QEMPTY + s]);
                }
            }
            if (w) w = wait_phase(&bars[OB_OFULL + a], (j >> 1) & 1, 64u);
            // the staging buffer (item j-2's, or with the fused prep, which keeps
            // one buffer, item j-1's) has been read out
            if (storer) {
                if (PREP)
                    tma_store_wait_read<0>();
                else
                    tma_store_wait_read<1>();
            }
            if (!epi_all(w)) break;
            tc_fence_after_sync();
            uint8_t *stg = sm + OU_O + x * 32768;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                uint32_t v0[16], v1[16];
                tmem_ld16(tmem + lane_base(warp) + 128u * a + c, v0);
                tmem_ld16(tmem + lane_base(warp) + 128u * a + c + 16, v1);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    pk[e] = pack_bf16(m * __uint_as_float(v0[2 * e]), m * __uint_as_float(v0[2 * e + 1]));
                    pk[8 + e] = pack_bf16(m * __uint_as_float(v1[2 * e]), m * __uint_as_float(v1[2 * e + 1]));
                }
                uint8_t *half = stg + (c >> 6) * 16384;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4 *>(half + sw128_offset(row, (c & 63) + 8 * u)) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
            tc_fence_before_sync();
            mbar_arrive(&bars[OB_OEMPTY + a]);
            fence_proxy_async_smem();
            named_sync_epi();
            if (storer) {
                tma_store_4d(&mO, stg, 0, 128 * i, f, bh);
                tma_store_4d(&mO, stg + 16384, 64, 128 * i, f, bh);
                tma_store_commit();
            }
        }
        if (storer) tma_store_wait_all<0>();
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// ========================================================= RMS pre-pass
// Per token of the raw [B*N][C] q and k rows: 1 / sqrt(sum x^2 / C + eps), the
// full-C RMSNorm factor every head of the token shares (fused_cam_gdn.py,
// `_precompute_cam_inv_rms`).  One warp per token, 16-byte loads.
__global__ void __launch_bounds__(256) cam_rms_kernel(const __nv_bfloat16 *q, const __nv_bfloat16 *k, float *out,
                                                      long long BN, int C, float eps) {
    const long long tok = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= BN) return;
    const uint4 *qr = reinterpret_cast<const uint4 *>(q + tok * C);
    const uint4 *kr = reinterpret_cast<const uint4 *>(k + tok * C);
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < C / 8; c += 32) {
        float x[8], y[8];
        unpack8(__ldg(qr + c), x);
        unpack8(__ldg(kr + c), y);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            sq += x[e] * x[e];
            sk += y[e] * y[e];
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
    }
    if (lane == 0) {
        out[2 * tok] = rsqrtf(sq / C + eps);
        out[2 * tok + 1] = rsqrtf(sk / C + eps);
    }
}

// ============================================================== SIMT kernel
// One CTA per (head, 32-column slice of the value dim); the slice of the fp32
// state sits in shared memory.  Per frame: P = K S for 32-token tiles, the
// corrections beta (v - d P) summed into registers as K^T (.), then
// S <- d S + sum, then the frame's outputs from the new state.  All fp32.
constexpr int kSimtThreads = 256;
constexpr int kTile = 32;

template <typename T>
__device__ __forceinline__ float ldf(const T *p, size_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
template <typename T>
__device__ __forceinline__ void stf(T *p, size_t i, float v);
template <>
__device__ __forceinline__ void stf<float>(float *p, size_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

struct SimtParams {
    const void *q, *k, *v, *beta;
    const float *decay, *s0;
    void *o;
    float *sf;
    int F, S, N, Dk, Dv;
    float scale;
    unsigned flags;
};

template <typename T>
__global__ void __launch_bounds__(kSimtThreads) cam_scan_simt_kernel(SimtParams p) {
    __shared__ float sS[128][33];     // state slice [dk][j]
    __shared__ float sX[kTile][129];  // K (or Q) tile [token][dk]
    __shared__ float sV[kTile][33];   // V slice tile, then the corrections
    __shared__ float sB[kTile];       // beta (0 past the frame), then the query scales
    const int bh = blockIdx.x, j0 = blockIdx.y * 32;
    const int tid = threadIdx.x, Dk = p.Dk, Dv = p.Dv;
    const bool l2n = (p.flags & GDN_QK_L2NORM) != 0, rev = (p.flags & GDN_CAM_REVERSE) != 0;
    const T *q = static_cast<const T *>(p.q) + (size_t)bh * p.N * Dk;
    const T *k = static_cast<const T *>(p.k) + (size_t)bh * p.N * Dk;
    const T *v = static_cast<const T *>(p.v) + (size_t)bh * p.N * Dv;
    const T *beta = static_cast<const T *>(p.beta) + (size_t)bh * p.N;
    T *o = static_cast<T *>(p.o) + (size_t)bh * p.N * Dv;
    for (int e = tid; e < Dk * 32; e += kSimtThreads) {
        const int i = e >> 5, jj = e & 31;
        sS[i][jj] = (p.s0 && !rev) ? p.s0[((size_t)bh * Dk + i) * Dv + j0 + jj] : 0.f;
    }
    __syncthreads();
    // thread -> (row group, column) for the tile products: column jj = tid & 31,
    // rows r8 = tid >> 5 .. step 8
    const int jj = tid & 31, r8 = tid >> 5;
    // load a [kTile][Dk] tile of x (K or Q) rows t0.. into sX, optionally unit rows
    auto load_rows = [&](const T *x, long t0, int nrow) {
        for (int e = tid; e < kTile * Dk; e += kSimtThreads) {
            const int t = e / Dk, i = e % Dk;
            sX[t][i] = t < nrow ? ldf(x, (size_t)(t0 + t) * Dk + i) : 0.f;
        }
        __syncthreads();
        if (l2n) {
            // one warp per 4 rows: sum of squares, then scale
            const int w = tid >> 5, ln = tid & 31;
            for (int t = w; t < kTile; t += kSimtThreads / 32) {
                float ss = 0.f;
                for (int i = ln; i < Dk; i += 32) ss += sX[t][i] * sX[t][i];
#pragma unroll
                for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float n = 1.f / fmaxf(sqrtf(ss), 1e-12f);
                for (int i = ln; i < Dk; i += 32) sX[t][i] *= n;
            }
            __syncthreads();
        }
    };
    for (int itf = 0; itf < p.F; ++itf) {
        const int qf = rev ? p.F - 1 - itf : itf;
        const int kf = rev ? p.F - itf : itf;
        if (!rev || itf > 0) {
            const float d = p.decay[(size_t)bh * p.F + kf];
            // dS[i][jj] for rows i = r8 + 8 m, accumulated over the frame
            float acc[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = 0.f;
            for (int t0 = 0; t0 < p.S; t0 += kTile) {
                const int nrow = min(kTile, p.S - t0);
                const long g0 = (long)kf * p.S + t0;
                load_rows(k, g0, nrow);
                for (int e = tid; e < kTile * 32; e += kSimtThreads) {
                    const int t = e >> 5, c = e & 31;
                    sV[t][c] = t < nrow ? ldf(v, (size_t)(g0 + t) * Dv + j0 + c) : 0.f;
                }
                if (tid < kTile) sB[tid] = tid < nrow ? ldf(beta, (size_t)(g0 + tid)) : 0.f;
                __syncthreads();
                // corrections c[t][jj] = beta_t (v - d (K S))[t][jj], rows t = r8 + 8 m
                float cr[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = r8 + 8 * m;
                    float pr = 0.f;
                    for (int i = 0; i < Dk; ++i) pr = fmaf(sX[t][i], sS[i][jj], pr);
                    cr[m] = sB[t] * (sV[t][jj] - d * pr);
                }
                __syncthreads();
#pragma unroll
                for (int m = 0; m < 4; ++m) sV[r8 + 8 * m][jj] = cr[m];
                __syncthreads();
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int i = r8 + 8 * m;
                    if (i < Dk) {
                        float s = acc[m];
                        for (int t = 0; t < kTile; ++t) s = fmaf(sX[t][i], sV[t][jj], s);
                        acc[m] = s;
                    }
                }
                __syncthreads();
            }
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int i = r8 + 8 * m;
                if (i < Dk) sS[i][jj] = fmaf(d, sS[i][jj], acc[m]);
            }
            __syncthreads();
        }
        // outputs of frame qf from the state as it now stands
        for (int t0 = 0; p.o && t0 < p.S; t0 += kTile) {
            const int nrow = min(kTile, p.S - t0);
            const long g0 = (long)qf * p.S + t0;
            load_rows(q, g0, nrow);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int t = r8 + 8 * m;
                float pr = 0.f;
                for (int i = 0; i < Dk; ++i) pr = fmaf(sX[t][i], sS[i][jj], pr);
                if (t < nrow) stf(o, (size_t)(g0 + t) * Dv + j0 + jj, p.scale * pr);
            }
            __syncthreads();
        }
    }
    if (p.sf && !rev)
        for (int e = tid; e < Dk * 32; e += kSimtThreads) {
            const int i = e >> 5, c = e & 31;
            p.sf[((size_t)bh * Dk + i) * Dv + j0 + c] = sS[i][c];
        }
}


// ================================================================ host side
int launch_tc(const CamScanArgs &a, cudaStream_t stream) {
    const int BH = a.B * a.H, N = a.F * a.S;
    CUtensorMap mK, mV, mQ, mO;
    if (!make_bf16_frame_map(&mK, a.k, BH, a.F, a.S, 64, 64) || !make_bf16_frame_map(&mV, a.v, BH, a.F, a.S, 64, 64) ||
        !make_bf16_frame_map(&mQ, a.q, BH, a.F, a.S, 64, 128) || !make_bf16_frame_map(&mO, a.o, BH, a.F, a.S, 64, 128))
        return GDN_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    const size_t frames = (size_t)BH * a.F;
    uint8_t *gimg = ws;
    uint8_t *simg = ws + frames * kImgBytes;
    float *ht = reinterpret_cast<float *>(ws + 2 * frames * kImgBytes);
    const int sms = device_sm_count();
    if (sms <= 0) return GDN_ERR_CUDA;
    const bool rev = (a.flags & GDN_CAM_REVERSE) != 0;

    // 1. G and H^T of every (head, frame); in reverse mode frame 0 is never
    //    taken in, but computing it keeps the item map simple
    if (cudaFuncSetAttribute(cam_gram_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GR_SMEM) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    GramParams gp{static_cast<const unsigned short *>(a.beta), gimg, ht, BH, a.F, a.S, N, a.flags, PrepParams{}};
    const int g_grid = (int)std::min<size_t>(frames, (size_t)sms);
    cam_gram_kernel<false><<<g_grid, kGramThreads, GR_SMEM, stream>>>(mK, mV, gp);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;

    // 2. the state chain, one CTA per head
    if (cudaFuncSetAttribute(cam_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CH_SMEM) != cudaSuccess)
        return GDN_ERR_CUDA;
    ChainParams cp{gimg, ht, simg, a.decay, a.s0, a.sf, BH, a.F, rev ? 1 : 0};
    cam_chain_kernel<<<BH, kChainThreads, CH_SMEM, stream>>>(cp);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;

    // 3. outputs
    if (cudaFuncSetAttribute(cam_out_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)OU_SMEM) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    const int nt = (a.S + 127) / 128;
    OutParams op{simg, BH, a.F, a.S, nt, (long long)frames * nt, a.scale, a.flags, N, PrepParams{}};
    const int o_grid = (int)std::min<long long>(op.items, (long long)sms);
    cam_out_kernel<false><<<o_grid, kOutThreads, OU_SMEM, stream>>>(mQ, mO, op);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Prep fused into the frame scan: the RMS pre-pass, then the three frame-scan
// launches reading the raw rows through maps over [B][N][H*128], the gram
// kernel applying the prep to K and V and the output kernel to Q at load.
int launch_fused(const CamFusedArgs &a, cudaStream_t stream) {
    const int BH = a.B * a.H, N = a.F * a.S, C = a.H * 128;
    CUtensorMap mK, mV, mQ, mO;
    // raw rows as [B][F][S][C]: a 128-column box at column 128 h is head h's row slice
    if (!make_bf16_frame_map_wide(&mK, a.k_raw, a.B, a.F, a.S, C, 64, 64) ||
        !make_bf16_frame_map_wide(&mV, a.v_raw, a.B, a.F, a.S, C, 64, 64) ||
        !make_bf16_frame_map_wide(&mQ, a.q_raw, a.B, a.F, a.S, C, 64, 128) ||
        !make_bf16_frame_map(&mO, a.o, BH, a.F, a.S, 64, 128))
        return GDN_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    const size_t frames = (size_t)BH * a.F;
    uint8_t *gimg = ws;
    uint8_t *simg = ws + frames * kImgBytes;
    float *ht = reinterpret_cast<float *>(ws + 2 * frames * kImgBytes);
    float *inv_rms = reinterpret_cast<float *>(ws + frames * kPerFrame);
    const int sms = device_sm_count();
    if (sms <= 0) return GDN_ERR_CUDA;
    const long long BN = (long long)a.B * N;
    cam_rms_kernel<<<(unsigned)((BN + 7) / 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(a.q_raw),
                                                                 static_cast<const __nv_bfloat16 *>(a.k_raw), inv_rms,
                                                                 BN, C, a.eps);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    const PrepParams pp{inv_rms, a.q_norm_w, a.k_norm_w, a.proj_q, a.proj_kv, log2((double)a.rope_base), a.k_scale,
                        a.H};
    if (cudaFuncSetAttribute(cam_gram_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GR_SMEM) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    GramParams gp{static_cast<const unsigned short *>(a.beta), gimg, ht, BH, a.F, a.S, N, a.flags, pp};
    cam_gram_kernel<true><<<(int)std::min<size_t>(frames, (size_t)sms), kGramThreads, GR_SMEM, stream>>>(mK, mV, gp);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(cam_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CH_SMEM) != cudaSuccess)
        return GDN_ERR_CUDA;
    const bool rev = (a.flags & GDN_CAM_REVERSE) != 0;
    ChainParams cp{gimg, ht, simg, a.decay, a.s0, a.sf, BH, a.F, rev ? 1 : 0};
    cam_chain_kernel<<<BH, kChainThreads, CH_SMEM, stream>>>(cp);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(cam_out_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)OU_SMEM) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    const int nt = (a.S + 127) / 128;
    OutParams op{simg, BH, a.F, a.S, nt, (long long)frames * nt, a.scale, a.flags, N, pp};
    cam_out_kernel<true><<<(int)std::min<long long>(op.items, (long long)sms), kOutThreadsPrep, OU_SMEM, stream>>>(
        mQ, mO, op);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int launch_simt(const CamScanArgs &a, cudaStream_t stream) {
    SimtParams sp{a.q, a.k, a.v, a.beta, a.decay, a.s0, a.o, a.sf, a.F, a.S, a.F * a.S, a.Dk, a.Dv, a.scale, a.flags};
    dim3 grid((unsigned)(a.B * a.H), (unsigned)(a.Dv / 32));
    cam_scan_simt_kernel<T><<<grid, kSimtThreads, 0, stream>>>(sp);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}


}  // namespace


bool cam_scan_tc_supported(const CamScanArgs &a) {
    if (a.flags & GDN_PATH_SIMT) return false;
    if (a.dtype != GDN_BF16 || a.Dk != 128 || a.Dv != 128) return false;
    if ((long long)a.F * a.S >= (1LL << 31)) return false;
    return sm100_family();
}

size_t cam_scan_workspace_bytes(const CamScanArgs &a) {
    return cam_scan_tc_supported(a) ? (size_t)a.B * a.H * a.F * kPerFrame : 0;
}

int launch_cam_scan(const CamScanArgs &a, cudaStream_t stream) {
    if (cam_scan_tc_supported(a)) return launch_tc(a, stream);
    if (a.dtype == GDN_BF16) return launch_simt<__nv_bfloat16>(a, stream);
    return launch_simt<float>(a, stream);
}

size_t cam_fused_workspace_bytes(const CamFusedArgs &a) {
    return (size_t)a.B * a.H * a.F * kPerFrame + (size_t)a.B * a.F * a.S * 2 * sizeof(float);
}

int launch_cam_fused(const CamFusedArgs &a, cudaStream_t stream) {
    if (!sm100_family()) return GDN_ERR_UNSUPPORTED;
    return launch_fused(a, stream);
}

int cam_scan_read_clear_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_cs_error, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_cs_error, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
    return v ? GDN_ERR_TIMEOUT : GDN_OK;
}

}  // namespace gdn
