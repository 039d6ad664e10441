// scan_tc.cu -- fused chunkwise GDN / DeltaProduct forward on the tcgen05
// tensor cores (bf16 tensors, Dk = Dv = 128, 64-row chunks, fp32 state).
//
// One CTA per (batch, head) walks the chunks in order.  Everything is held
// value-dimension-major so that every MMA has M = 128 (the value dim dv):
//
//   KQ   = [K; Q] K^T            128x64   rows 0..63 K K^T, rows 64.. Q K^T
//   A[t][s] = beta_t exp(g_t - g_s) (k_t . k_s), s < t     (CUDA cores)
//   T    = (I + A)^-1                                      (CUDA cores, blocked)
//   W^T  = K^T (T diag(beta e^g))^T                        tcgen05
//   U^T  = V^T (T diag(beta))^T                            tcgen05
//   Vn^T = U^T - S^T W^T            (v_new of the WY form) tcgen05, negated A
//   O^T  = S^T Qg^T + Vn^T P^T      Qg = diag(e^g) Q,  P[t][s] = e^{g_t-g_s} q_t.k_s, s <= t
//   S^T <- e^{g_last} S^T + (Vn^T diag(e^{g_last - g_s})) K
//
// with g the within-chunk cumulative log-decay (gated_deltaproduct test.py:
// `gated_chunk_scaled_dot_kkt_fwd_kernel`, `solve_tril_16x16_kernel` and the
// merge kernels, `gated_fwd_recompute_w_u_kernel`, `preprocess_qkw`,
// `gated_chunk_delta_rule_fwd_kernel_h`, `gated_chunk_linear_attn_fwd_kernel_o`).
// The pages run these as separate launches with HBM round trips; here the
// state S^T stays in tensor memory in fp32 for the whole sequence and only
// q, k, v, beta, g are read and o written.
//
// Warp roles (384 threads):
//   warp 0        TMA producer: K, Q (two stages) and V tiles.
//   warp 1        MMA issuer; owns the 512-column TMEM allocation.
//   warps 4..7    scan epilogue (SE): S^T -> bf16 operand, state decay,
//                 Vn^T -> bf16 operands, output tile -> TMA store.
//   warps 8..11   WY producer: cumulative decay, A, blocked (I+A)^-1, the
//                 scaled T tiles, P, Qg, and W^T -> bf16 operand.
// Every wait on an mbarrier is bounded in wall time; on expiry the CTA sets
// an error word, stops issuing work, drains what is in flight, frees TMEM
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "gdn_internal.h"
#include "tc_util.cuh"

namespace gdn {

namespace {
__device__ unsigned int g_tc_error = 0;
unsigned long long g_timeout_ns = 1000000000ull;  // host copy of the wait limit
}  // namespace

namespace {
using namespace tc;

constexpr int kThreads = 384;
constexpr int kAS = 68;  // fp32 row stride of the A / T tiles

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ0 = 0;        // [K rows 0..63 | Q rows 64..] x 2 K-blocks, 32 KB
constexpr uint32_t OFF_KQ1 = 32768;
constexpr uint32_t OFF_V = 65536;      // V tile [64 s][128 dv], 2 MN-atoms, 16 KB
constexpr uint32_t OFF_AF = 81920;     // A fp32 [64][68]; later Tw (+0) and Tu (+8192), bf16
constexpr uint32_t OFF_TF = 99328;     // T fp32 [64][68]
constexpr uint32_t OFF_P0 = 116736;    // P bf16 [NQ t][64 s] K-major, 8 KB each
constexpr uint32_t OFF_P1 = 124928;
constexpr uint32_t OFF_WT = 133120;    // W^T bf16 [128 d][64 t] MN-major, 16 KB
constexpr uint32_t OFF_ST = 149504;    // S^T bf16 [128 dv][128 dk] K-major, 32 KB
constexpr uint32_t OFF_VN = 182272;    // Vn^T bf16 [128 dv][64 s] K-major, 16 KB
constexpr uint32_t OFF_VS = 198656;    // decayed Vn^T, 16 KB; also the output staging tile
constexpr uint32_t OFF_MISC = 215040;  // 2 x Misc
constexpr uint32_t OFF_SEF = 219136;   // SE: exp(g_last - g_s) n_s, 64 floats
constexpr uint32_t OFF_X = 219392;     // inverse scratch, 32x32 fp32
constexpr uint32_t OFF_BAR = 223488;   // mbarriers
constexpr uint32_t OFF_FLAGS = 223744; // TMEM base, abort flag
constexpr uint32_t kSmemBytes = OFF_FLAGS + 64 + 1024;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_VN0 = 128, TM_VN1 = 192, TM_O0 = 256, TM_KQ = 320, TM_W = 384, TM_O1 = 448;

enum Bar {
    B_FULL0, B_FULL1, B_VFULL, B_KQ_DONE, B_KQ_FREE, B_WY_READY, B_WU_DONE, B_WT_READY, B_S_READY,
    B_VN_DONE, B_VN_READY, B_UPD_DONE, B_STG_FREE0, B_STG_FREE1, B_MISC0, B_MISC1, B_DRAIN, B_NUM
};

struct Misc {
    float beta[64];  // beta of each row (0 past the end)
    float gam[64];   // within-chunk cumulative log-decay
    float n[64];     // 1/||k_s|| with GDN_QK_L2NORM, else 1
    float m[64];     // 1/||q_t|| with GDN_QK_L2NORM, else 1
    float wsc[64];   // beta_s exp(gam_s) n_s
    float pad[192];
};
static_assert(sizeof(Misc) == 2048, "Misc layout");

struct TcParams {
    const __nv_bfloat16 *beta;
    const float *g;
    const float *s0;
    float *sf;
    int T, rows, NT;
    float scale;
    unsigned flags;
    unsigned long long timeout_ns;
};

constexpr unsigned long long kCleanupNs = 200000000ull;  // 0.2 s for draining on the way out


// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, unsigned long long timeout_ns,
                                         volatile int *abort_flag, unsigned code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicOr(&g_tc_error, code);
            return false;
        }
    }
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier over a warp group that also ORs a failure bit across it, so
// that every member takes the same branch after a bounded wait.
__device__ __forceinline__ bool group_all(bool ok, int id, int n) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.eq.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(n)
        : "memory");
    return r == 0;
}

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return (uint32_t)(32 * (warp & 3)) << 16; }

__device__ __forceinline__ void ld64(uint32_t taddr, float (&x)[64]) {
    uint32_t r[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        tmem_ld16(taddr + 16 * j, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) x[16 * j + i] = __uint_as_float(r[i]);
    }
}

// Writes 64 fp32 values as one bf16 row of a 128-byte-swizzled tile.
__device__ __forceinline__ void store_row_sw128(uint8_t *tile, int row, const float (&x)[64]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint4 v;
        v.x = pack_bf16(x[8 * ch + 0], x[8 * ch + 1]);
        v.y = pack_bf16(x[8 * ch + 2], x[8 * ch + 3]);
        v.z = pack_bf16(x[8 * ch + 4], x[8 * ch + 5]);
        v.w = pack_bf16(x[8 * ch + 6], x[8 * ch + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, 8 * ch)) = v;
    }
}

// =========================================================================== kernel
template <int R>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_tc_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
                  const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO, TcParams p) {
    constexpr int NQ = 64 / R;  // query rows (tokens) per chunk
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_FLAGS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_FLAGS + 4);
    Misc *misc = reinterpret_cast<Misc *>(sm + OFF_MISC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int NT = p.NT;
    const unsigned long long tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        const uint32_t counts[B_NUM] = {1, 1, 1, 1, 1, 1, 1, 1, 128, 1, 128, 1, 1, 1, 1, 1, 1};
        for (int i = 0; i < B_NUM; ++i) mbar_init(&bars[i], counts[i]);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&mK);
        prefetch_tensormap(&mQ);
        prefetch_tensormap(&mV);
        prefetch_tensormap(&mO);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int armed_full[2] = {0, 0}, armed_v = 0;
            for (int c = 0; c < NT; ++c) {
                const int s = c & 1;
                if (c >= 2 && !wait_bar(&bars[B_STG_FREE0 + s], ((c - 2) >> 1) & 1, tmo, abort_flag, 1u)) break;
                uint8_t *kq = sm + (s ? OFF_KQ1 : OFF_KQ0);
                mbar_arrive_expect_tx(&bars[B_FULL0 + s], 2 * 8192 + 2 * NQ * 128);
                tma_load_3d(kq, &mK, &bars[B_FULL0 + s], 0, c * 64, bh);
                tma_load_3d(kq + 16384, &mK, &bars[B_FULL0 + s], 64, c * 64, bh);
                tma_load_3d(kq + 8192, &mQ, &bars[B_FULL0 + s], 0, c * NQ, bh);
                tma_load_3d(kq + 24576, &mQ, &bars[B_FULL0 + s], 64, c * NQ, bh);
                armed_full[s]++;
                if (c >= 1 && !wait_bar(&bars[B_WU_DONE], (c - 1) & 1, tmo, abort_flag, 1u)) break;
                mbar_arrive_expect_tx(&bars[B_VFULL], 16384);
                tma_load_3d(sm + OFF_V, &mV, &bars[B_VFULL], 0, c * 64, bh);
                tma_load_3d(sm + OFF_V + 8192, &mV, &bars[B_VFULL], 64, c * 64, bh);
                armed_v++;
            }
            // every armed load lands before the CTA may exit
            for (int s = 0; s < 2; ++s)
                if (armed_full[s]) mbar_wait(&bars[B_FULL0 + s], (armed_full[s] - 1) & 1, kCleanupNs);
            if (armed_v) mbar_wait(&bars[B_VFULL], (armed_v - 1) & 1, kCleanupNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idKQ = idesc_bf16(128, 64, false, false);
            const uint32_t idWU = idesc_bf16(128, 64, true, false);
            const uint32_t idVN = idesc_bf16(128, 64, false, true, true);
            const uint32_t idO = idesc_bf16(128, NQ, false, false);
            const uint32_t idUP = idesc_bf16(128, 128, false, true);
            const uint32_t sbase = smem_u32(sm);
            auto issue_kq = [&](int c) -> bool {
                const int s = c & 1;
                if (!wait_bar(&bars[B_FULL0 + s], (c >> 1) & 1, tmo, abort_flag, 2u)) return false;
                if (c >= 1 && !wait_bar(&bars[B_KQ_FREE], (c - 1) & 1, tmo, abort_flag, 2u)) return false;
                tc_fence_after_sync();
                const uint32_t kq = sbase + (s ? OFF_KQ1 : OFF_KQ0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a = kq + (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16_ss(tmem + TM_KQ, smem_desc(a, 16, 1024), smem_desc(a, 16, 1024), idKQ, ks > 0);
                }
                mma_commit(&bars[B_KQ_DONE]);
                return true;
            };
            bool ok = NT > 0 ? issue_kq(0) : true;
            for (int c = 0; c < NT && ok; ++c) {
                const int s = c & 1;
                const uint32_t kq = sbase + (s ? OFF_KQ1 : OFF_KQ0);
                const uint32_t tvn = tmem + ((c & 1) ? TM_VN1 : TM_VN0);
                const uint32_t tO = tmem + ((c & 1) ? TM_O1 : TM_O0);
                // W^T and U^T of chunk c
                if (!wait_bar(&bars[B_WY_READY], c & 1, tmo, abort_flag, 2u)) break;
                if (!wait_bar(&bars[B_VFULL], c & 1, tmo, abort_flag, 2u)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(kq + ks * 2048, 16384, 1024);
                    const uint64_t b = smem_desc(sbase + OFF_AF + ks * 32, 16, 1024);
                    mma_bf16_ss(tmem + TM_W, a, b, idWU, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_V + ks * 2048, 8192, 1024);
                    const uint64_t b = smem_desc(sbase + OFF_AF + 8192 + ks * 32, 16, 1024);
                    mma_bf16_ss(tvn, a, b, idWU, ks > 0);
                }
                mma_commit(&bars[B_WU_DONE]);
                // K K^T / Q K^T of the next chunk, so the WY warps can start on it
                if (c + 1 < NT && !issue_kq(c + 1)) break;
                // Vn^T = U^T - S^T W^T ;  O^T = S^T Qg^T
                if (!wait_bar(&bars[B_WT_READY], c & 1, tmo, abort_flag, 2u)) break;
                if (!wait_bar(&bars[B_S_READY], c & 1, tmo, abort_flag, 2u)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_ST + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc(sbase + OFF_WT + ks * 2048, 8192, 1024);
                    mma_bf16_ss(tvn, a, b, idVN, 1u);
                }
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_ST + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc(kq + 8192 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    mma_bf16_ss(tO, a, b, idO, ks > 0);
                }
                mma_commit(&bars[B_VN_DONE]);
                // O^T += Vn^T P^T ;  S^T += (decayed Vn^T) K
                if (!wait_bar(&bars[B_VN_READY], c & 1, tmo, abort_flag, 2u)) break;
                tc_fence_after_sync();
                const uint32_t pt = sbase + ((c & 1) ? OFF_P1 : OFF_P0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_VN + ks * 32, 16, 1024);
                    const uint64_t b = smem_desc(pt + ks * 32, 16, 1024);
                    mma_bf16_ss(tO, a, b, idO, 1u);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_VS + ks * 32, 16, 1024);
                    const uint64_t b = smem_desc(kq + ks * 2048, 16384, 1024);
                    mma_bf16_ss(tmem + TM_S, a, b, idUP, 1u);
                }
                mma_commit(&bars[B_UPD_DONE]);
                mma_commit(&bars[B_STG_FREE0 + s]);
            }
            // every issued MMA completes before TMEM is released
            mma_commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0, kCleanupNs);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ scan epilogue
        const int st = threadIdx.x - 128;  // value index dv = TMEM lane
        const uint32_t lb = tmem_lane_base(warp);
        float *sef = reinterpret_cast<float *>(sm + OFF_SEF);
        uint8_t *ostage = sm + OFF_VS;
        // initial state into TMEM: S^T[dv][dk] = S0[dk][dv]
        {
            const float *s0 = p.s0 ? p.s0 + (size_t)bh * 128 * 128 : nullptr;
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(s0 ? s0[(16 * j + i) * 128 + st] : 0.f);
                tmem_st16(tmem + lb + TM_S + 16 * j, r);
            }
            tmem_wait_st();
        }
        auto out_epilogue = [&](int cc) {
            const uint32_t tO = tmem + lb + ((cc & 1) ? TM_O1 : TM_O0);
#pragma unroll 1
            for (int j = 0; j < NQ / 16; ++j) {
                uint32_t r[16];
                tmem_ld16(tO + 16 * j, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(p.scale * __uint_as_float(r[i]));
                    *reinterpret_cast<__nv_bfloat16 *>(ostage + (16 * j + i) * 256 + st * 2) = h;
                }
            }
            tc_fence_before_sync();
            fence_proxy_async_smem();
            named_bar(2, 128);
            if (st == 0) {
                tma_store_3d(&mO, ostage, 0, cc * NQ, bh);
                tma_store_commit();
            }
        };
        bool ok = true;
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1;
            Misc *ms = misc + s;
            bool w = wait_bar(&bars[B_MISC0 + s], (c >> 1) & 1, tmo, abort_flag, 4u);
            if (w && c >= 1) w = wait_bar(&bars[B_UPD_DONE], (c - 1) & 1, tmo, abort_flag, 4u);
            if (!group_all(w, 2, 128)) { ok = false; break; }
            tc_fence_after_sync();
            const float glast = ms->gam[63];
            if (st < 64) sef[st] = __expf(glast - ms->gam[st]) * ms->n[st];
            // state: S^T -> bf16 operand, then S^T <- exp(g_last) S^T in TMEM
            const float el = __expf(glast);
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                uint32_t r[16];
                tmem_ld16(tmem + lb + TM_S + 16 * j, r);
                tmem_wait_ld();
                uint8_t *blk = sm + OFF_ST + (j >> 2) * 16384;
                const int col = (16 * j) & 63;
                uint4 v0, v1;
                v0.x = pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1]));
                v0.y = pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3]));
                v0.z = pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5]));
                v0.w = pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7]));
                v1.x = pack_bf16(__uint_as_float(r[8]), __uint_as_float(r[9]));
                v1.y = pack_bf16(__uint_as_float(r[10]), __uint_as_float(r[11]));
                v1.z = pack_bf16(__uint_as_float(r[12]), __uint_as_float(r[13]));
                v1.w = pack_bf16(__uint_as_float(r[14]), __uint_as_float(r[15]));
                *reinterpret_cast<uint4 *>(blk + sw128_offset(st, col)) = v0;
                *reinterpret_cast<uint4 *>(blk + sw128_offset(st, col + 8)) = v1;
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(el * __uint_as_float(r[i]));
                tmem_st16(tmem + lb + TM_S + 16 * j, r);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_S_READY]);
            // output of the previous chunk (its MMAs completed with UPD_DONE)
            if (c >= 1) out_epilogue(c - 1);
            // Vn^T of this chunk -> two bf16 operands
            const bool wv = wait_bar(&bars[B_VN_DONE], c & 1, tmo, abort_flag, 4u);
            if (st == 0) tma_store_wait_read<0>();
            if (!group_all(wv, 2, 128)) { ok = false; break; }  // staging tile free, sef visible
            tc_fence_after_sync();
            float x[64];
            ld64(tmem + lb + ((c & 1) ? TM_VN1 : TM_VN0), x);
            store_row_sw128(sm + OFF_VN, st, x);
#pragma unroll
            for (int i = 0; i < 64; ++i) x[i] *= sef[i];
            store_row_sw128(sm + OFF_VS, st, x);
            tc_fence_before_sync();
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_VN_READY]);
        }
        bool fin = ok && NT > 0 && wait_bar(&bars[B_UPD_DONE], (NT - 1) & 1, tmo, abort_flag, 4u);
        if (st == 0) tma_store_wait_read<0>();
        if (group_all(fin, 2, 128)) {
            tc_fence_after_sync();
            out_epilogue(NT - 1);
            if (p.sf) {
                float *sf = p.sf + (size_t)bh * 128 * 128;
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lb + TM_S + 16 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) sf[(16 * j + i) * 128 + st] = __uint_as_float(r[i]);
                }
            }
        }
        if (st == 0) tma_store_wait_all<0>();
    } else if (warp >= 8) {
        // ------------------------------------------------------------ WY producer
        const int wt = threadIdx.x - 256;  // 0..127
        const int wq = wt >> 5;
        const uint32_t lb = tmem_lane_base(warp);
        float *AF = reinterpret_cast<float *>(sm + OFF_AF);
        float *TF = reinterpret_cast<float *>(sm + OFF_TF);
        float *XS = reinterpret_cast<float *>(sm + OFF_X);
        const bool l2n = (p.flags & GDN_QK_L2NORM) != 0;
        const __nv_bfloat16 *betap = p.beta + (size_t)bh * p.rows;
        const float *gp = p.g + (size_t)bh * p.T;
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1;
            Misc *ms = misc + s;
            uint8_t *kq = sm + (s ? OFF_KQ1 : OFF_KQ0);
            uint8_t *ptile = sm + ((c & 1) ? OFF_P1 : OFF_P0);
            // 1. beta and g of the chunk's rows
            if (wt < 64) {
                const int row = c * 64 + wt;
                ms->beta[wt] = row < p.rows ? __bfloat162float(betap[row]) : 0.f;
            } else {
                const int t = wt - 64, row = c * 64 + t;
                ms->gam[t] = (row < p.rows && row % R == 0) ? gp[row / R] : 0.f;
            }
            named_bar(1, 128);
            if (wq == 0) {
                float a = ms->gam[lane], b = ms->gam[lane + 32];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float ya = __shfl_up_sync(0xffffffffu, a, off);
                    const float yb = __shfl_up_sync(0xffffffffu, b, off);
                    if (lane >= off) { a += ya; b += yb; }
                }
                b += __shfl_sync(0xffffffffu, a, 31);
                ms->gam[lane] = a;
                ms->gam[lane + 32] = b;
            }
            const bool wk = wait_bar(&bars[B_KQ_DONE], c & 1, tmo, abort_flag, 8u);
            if (!group_all(wk, 1, 128)) break;  // also makes gam visible
            tc_fence_after_sync();
            // 2. rows of K K^T (warps 0,1) and Q K^T (warps 2,3)
            float x[64];
            ld64(tmem + lb + TM_KQ, x);
            if (wq < 2) {
                float diag = 0.f;
#pragma unroll
                for (int i = 0; i < 64; ++i) diag = (i == wt) ? x[i] : diag;
                ms->n[wt] = l2n ? rsqrtf(fmaxf(diag, 1e-24f)) : 1.f;
            } else {
                const int t = wt - 64;
                float mq = 1.f;
                if (l2n && t < NQ) {
                    float ss = 0.f;
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        const uint4 *row = reinterpret_cast<const uint4 *>(kq + 8192 + blk * 16384 + t * 128);
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint4 u = row[ch];
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                                ss += lo * lo + hi * hi;
                            }
                        }
                    }
                    mq = rsqrtf(fmaxf(ss, 1e-24f));
                }
                ms->m[t] = mq;
            }
            tc_fence_before_sync();
            named_bar(1, 128);  // n, m visible; TMEM rows read
            if (wt == 0) mbar_arrive(&bars[B_KQ_FREE]);
            if (wt < 64) {
                const float bn = ms->beta[wt] * ms->n[wt];
                const float gt = ms->gam[wt];
                ms->wsc[wt] = ms->beta[wt] * __expf(gt) * ms->n[wt];
#pragma unroll
                for (int sidx = 0; sidx < 64; ++sidx) {
                    float a = 0.f;
                    if (sidx < wt) a = bn * __expf(gt - ms->gam[sidx]) * ms->n[sidx] * x[sidx];
                    AF[wt * kAS + sidx] = a;
                }
            } else {
                const int t = wt - 64;
                if (t < NQ) {
                    const int row = t * R + R - 1;
                    const float gr = ms->gam[row];
                    const float mq = ms->m[t];
#pragma unroll
                    for (int sidx = 0; sidx < 64; ++sidx)
                        x[sidx] = (sidx <= row) ? __expf(gr - ms->gam[sidx]) * mq * ms->n[sidx] * x[sidx] : 0.f;
                    store_row_sw128(ptile, t, x);
                    // Qg row: q_t exp(g_row) / ||q_t||
                    const float qs = __expf(gr) * mq;
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        uint4 *rowp = reinterpret_cast<uint4 *>(kq + 8192 + blk * 16384 + t * 128);
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            uint4 u = rowp[ch];
                            uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(w4[e] << 16) * qs;
                                const float hi = __uint_as_float(w4[e] & 0xffff0000u) * qs;
                                w4[e] = pack_bf16(lo, hi);
                            }
                            rowp[ch] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
            }
            named_bar(1, 128);  // A complete
            if (wt == 0) mbar_arrive(&bars[B_MISC0 + s]);
            // 3. T = (I + A)^-1, blocked: 16x16 diagonal blocks by substitution,
            //    then the 16- and 32-level off-diagonal merges T21 = -T22 A21 T11.
            if (wt < 64) {
                const int b = wt >> 4, cc = wt & 15;
                float xs[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc = (i == cc) ? 1.f : 0.f;
#pragma unroll
                    for (int j = 0; j < i; ++j) acc -= AF[(16 * b + i) * kAS + 16 * b + j] * xs[j];
                    xs[i] = acc;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) TF[(16 * b + i) * kAS + 16 * b + cc] = xs[i];
            } else {
                // zero the blocks above the diagonal
                for (int e = wt - 64; e < 6 * 256; e += 64) {
                    const int blk = e >> 8, rr = (e >> 4) & 15, cl = e & 15;
                    const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                    const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                    TF[(16 * bi + rr) * kAS + 16 * bj + cl] = 0.f;
                }
            }
            named_bar(1, 128);
            // 16-level merges inside each 32 half: blocks (1,0) and (3,2)
            {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = wt + 128 * k;           // 0..511
                    const int h = e >> 8, rr = (e >> 4) & 15, cl = e & 15;
                    const int i0 = 32 * h + 16, j0 = 32 * h;  // block (i0, j0)
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc += AF[(i0 + rr) * kAS + j0 + m] * TF[(j0 + m) * kAS + j0 + cl];
                    XS[e] = acc;
                }
                named_bar(1, 128);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = wt + 128 * k;
                    const int h = e >> 8, rr = (e >> 4) & 15, cl = e & 15;
                    const int i0 = 32 * h + 16, j0 = 32 * h;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc += TF[(i0 + rr) * kAS + i0 + m] * XS[(h << 8) + m * 16 + cl];
                    TF[(i0 + rr) * kAS + j0 + cl] = -acc;
                }
                named_bar(1, 128);
            }
            // 32-level merge: rows 32..63, cols 0..31
            {
                const int cl = wt & 31, r0 = wt >> 5;  // rows r0 + 4k
                float acc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll 4
                for (int m = 0; m < 32; m += 4) {
                    const float t0 = TF[(m + 0) * kAS + cl], t1 = TF[(m + 1) * kAS + cl];
                    const float t2 = TF[(m + 2) * kAS + cl], t3 = TF[(m + 3) * kAS + cl];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&AF[(32 + r0 + 4 * k) * kAS + m]);
                        acc[k] += a4.x * t0 + a4.y * t1 + a4.z * t2 + a4.w * t3;
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) XS[(r0 + 4 * k) * 32 + cl] = acc[k];
                named_bar(1, 128);
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll 4
                for (int m = 0; m < 32; m += 4) {
                    const float x0 = XS[(m + 0) * 32 + cl], x1 = XS[(m + 1) * 32 + cl];
                    const float x2 = XS[(m + 2) * 32 + cl], x3 = XS[(m + 3) * 32 + cl];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(&TF[(32 + r0 + 4 * k) * kAS + 32 + m]);
                        acc[k] += t4.x * x0 + t4.y * x1 + t4.z * x2 + t4.w * x3;
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) TF[(32 + r0 + 4 * k) * kAS + cl] = -acc[k];
                named_bar(1, 128);
            }
            // 4. Tw = T diag(beta e^g n), Tu = T diag(beta) as bf16 K-major tiles
            {
                const int t = wt & 63;
                const bool isw = wt < 64;
                float row[64];
#pragma unroll
                for (int sidx = 0; sidx < 64; sidx += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(&TF[t * kAS + sidx]);
                    row[sidx] = t4.x; row[sidx + 1] = t4.y; row[sidx + 2] = t4.z; row[sidx + 3] = t4.w;
                }
#pragma unroll
                for (int sidx = 0; sidx < 64; ++sidx) row[sidx] *= isw ? ms->wsc[sidx] : ms->beta[sidx];
                store_row_sw128(sm + OFF_AF + (isw ? 0 : 8192), t, row);
            }
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (wt == 0) mbar_arrive(&bars[B_WY_READY]);
            // 5. W^T -> bf16 MN-major operand (thread = key dim d)
            bool ww = wait_bar(&bars[B_WU_DONE], c & 1, tmo, abort_flag, 8u);
            if (ww && c >= 1) ww = wait_bar(&bars[B_VN_DONE], (c - 1) & 1, tmo, abort_flag, 8u);
            if (!group_all(ww, 1, 128)) break;
            tc_fence_after_sync();
            ld64(tmem + lb + TM_W, x);
            store_row_sw128(sm + OFF_WT, wt, x);
            tc_fence_before_sync();
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (wt == 0) mbar_arrive(&bars[B_WT_READY]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ====================================================================== host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over a [heads][rows][128] bf16 tensor with a {box0, box1, 1} box.
bool make_map(CUtensorMap *m, const void *base, int heads, long rows, int box0, int box1, bool swizzle) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {256, (cuuint64_t)rows * 256};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool device_is_sm100_family() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10;
}

template <int R>
int launch_r(const ScanArgs &a, cudaStream_t stream) {
    constexpr int NQ = 64 / R;
    const long rows = (long)a.T * R;
    const int BH = a.B * a.H;
    CUtensorMap mK, mQ, mV, mO;
    if (!make_map(&mK, a.k, BH, rows, 64, 64, true) || !make_map(&mQ, a.q, BH, a.T, 64, NQ, true) ||
        !make_map(&mV, a.v, BH, rows, 64, 64, true) || !make_map(&mO, a.o, BH, a.T, 128, NQ, false))
        return GDN_ERR_CUDA;
    TcParams p;
    p.beta = static_cast<const __nv_bfloat16 *>(a.beta);
    p.g = a.g;
    p.s0 = a.s0;
    p.sf = a.sf;
    p.T = a.T;
    p.rows = (int)rows;
    p.NT = (int)((rows + 63) / 64);
    p.scale = a.scale;
    p.flags = a.flags;
    p.timeout_ns = g_timeout_ns;
    auto kern = gdn_tc_kernel<R>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<BH, kThreads, kSmemBytes, stream>>>(mK, mQ, mV, mO, p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool scan_tc_supported(const ScanArgs &a) {
    if (a.flags & GDN_PATH_SIMT) return false;
    if (a.dtype != GDN_BF16 || a.Dk != 128 || a.Dv != 128 || a.chunk != 64) return false;
    if (a.r != 1 && a.r != 2 && a.r != 4) return false;
    if ((long long)a.T * a.r > (1LL << 30)) return false;
    static int sm100 = -1;
    if (sm100 < 0) sm100 = device_is_sm100_family() ? 1 : 0;
    return sm100 == 1;
}

size_t scan_tc_workspace_bytes(const ScanArgs &) { return 0; }

int launch_scan_tc(const ScanArgs &a, cudaStream_t stream) {
    switch (a.r) {
        case 1: return launch_r<1>(a, stream);
        case 2: return launch_r<2>(a, stream);
        case 4: return launch_r<4>(a, stream);
        default: return GDN_ERR_UNSUPPORTED;
    }
}

int scan_tc_read_clear_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
    return v ? GDN_ERR_TIMEOUT : GDN_OK;
}

int scan_tc_set_wait_limit(unsigned long long us) {
    g_timeout_ns = us == 0 ? 1000000000ull : us * 1000ull;
    return GDN_OK;
}

}  // namespace gdn
