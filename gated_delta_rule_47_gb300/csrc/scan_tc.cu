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
// Warp roles (512 threads):
//   warp 0        TMA producer: K, Q (two stages) and V tiles.
//   warp 1        MMA issuer; owns the 512-column TMEM allocation.
//   warps 4..7    scan epilogue (SE): S^T -> bf16 operand, state decay,
//                 Vn^T -> bf16 operands, output tile -> TMA store.
//   warps 8..15   WY producer: cumulative decay, A, blocked (I+A)^-1 in
//                 place, the scaled T tiles, P, Qg, and W^T -> bf16 operand.
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

// Optional timeline instrumentation (compiled in only with -DGDN_TRACE): the
// first CTA records clock64() at fixed points of each role, per chunk.
#ifdef GDN_TRACE
__device__ unsigned long long *g_trace = nullptr;
#define GDN_TR(c, ev)                                                          \
    do {                                                                       \
        if (blockIdx.x == 0 && g_trace != nullptr && (c) < 1024)               \
            g_trace[(size_t)(c) * 32 + (ev)] = clock64();                      \
    } while (0)
#else
#define GDN_TR(c, ev) \
    do {              \
    } while (0)
#endif

namespace {
using namespace tc;

constexpr int kThreads = 512;
constexpr int kAS = 68;  // fp32 row stride of the A / T tiles

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ0 = 0;        // [K rows 0..63 | Q rows 64..] x 2 K-blocks, 32 KB
constexpr uint32_t OFF_KQ1 = 32768;
constexpr uint32_t OFF_V = 65536;      // V tile [64 s][128 dv], 2 MN-atoms, 16 KB
constexpr uint32_t OFF_AF = 81920;     // A fp32 [64][68], inverted in place into T
constexpr uint32_t OFF_TWU = 99328;    // Tw (+0) and Tu (+8192), bf16 [64 t][64 s] K-major
constexpr uint32_t OFF_P0 = 116736;    // P bf16 [NQ t][64 s] K-major, 8 KB each
constexpr uint32_t OFF_P1 = 124928;
constexpr uint32_t OFF_WT = 133120;    // W^T bf16 [128 d][64 t] MN-major, 16 KB
constexpr uint32_t OFF_ST = 149504;    // S^T bf16 [128 dv][128 dk] K-major, 32 KB
constexpr uint32_t OFF_VN = 182272;    // Vn^T bf16 [128 dv][64 s] K-major, 16 KB
constexpr uint32_t OFF_VS = 198656;    // decayed Vn^T, 16 KB; also the output staging tile
constexpr uint32_t OFF_MISC = 215040;  // 2 x Misc
constexpr uint32_t OFF_X = 221184;     // inverse scratch, 32x32 fp32
constexpr uint32_t OFF_BAR = 225280;   // mbarriers
constexpr uint32_t OFF_FLAGS = 225536; // TMEM base, abort flag
constexpr uint32_t kSmemBytes = OFF_FLAGS + 64 + 1024;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_VN0 = 128, TM_VN1 = 192, TM_O0 = 256, TM_KQ = 320, TM_W = 384, TM_O1 = 448;

enum Bar {
    B_FULL0, B_FULL1, B_VFULL, B_KQ_DONE, B_KQ_FREE, B_WY_READY, B_WU_DONE, B_WT_READY, B_S_READY,
    B_VN_DONE, B_VN_READY, B_UPD_DONE, B_STG_FREE0, B_STG_FREE1, B_MISC0, B_MISC1, B_DRAIN, B_NUM
};

// Per-chunk vectors written by the WY warps (two copies, by chunk parity).
struct Misc {
    float beta[64];   // beta of each row (0 past the end)
    float gam[64];    // within-chunk cumulative log-decay
    float n[64];      // 1/||k_s|| with GDN_QK_L2NORM, else 1
    float m[64];      // 1/||q_t|| with GDN_QK_L2NORM, else 1
    float wsc[64];    // beta_s exp(gam_s) n_s          (columns of Tw)
    float bn[64];     // exp(gam_0 - gam_s) n_s         (column factor of A and P)
    float ea[64];     // exp(gam_t - gam_0)             (row factor of A and P)
    float sef[64];    // exp(gam_last - gam_s) n_s      (columns of the decayed Vn^T)
    float qp[2][64];  // partial q_t^2 sums over the two key-dim halves
    float el;         // exp(gam_last)
    int safe;         // 1 if |gam_t - gam_0| <= 80 for all rows (factorised exponentials)
    float pad[126];
};
static_assert(sizeof(Misc) == 3072, "Misc layout");

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
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
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
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
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
                GDN_TR(c, 0);
                uint8_t *kq = sm + (s ? OFF_KQ1 : OFF_KQ0);
                mbar_arrive_expect_tx(&bars[B_FULL0 + s], 2 * 8192 + 2 * NQ * 128);
                tma_load_3d(kq, &mK, &bars[B_FULL0 + s], 0, c * 64, bh);
                tma_load_3d(kq + 16384, &mK, &bars[B_FULL0 + s], 64, c * 64, bh);
                tma_load_3d(kq + 8192, &mQ, &bars[B_FULL0 + s], 0, c * NQ, bh);
                tma_load_3d(kq + 24576, &mQ, &bars[B_FULL0 + s], 64, c * NQ, bh);
                armed_full[s]++;
                if (c >= 1 && !wait_bar(&bars[B_WU_DONE], (c - 1) & 1, tmo, abort_flag, 1u)) break;
                GDN_TR(c, 1);
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
                GDN_TR(c, 2);
                if (!wait_bar(&bars[B_VFULL], c & 1, tmo, abort_flag, 2u)) break;
                GDN_TR(c, 3);
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(kq + ks * 2048, 16384, 1024);
                    const uint64_t b = smem_desc(sbase + OFF_TWU + ks * 32, 16, 1024);
                    mma_bf16_ss(tmem + TM_W, a, b, idWU, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_V + ks * 2048, 8192, 1024);
                    const uint64_t b = smem_desc(sbase + OFF_TWU + 8192 + ks * 32, 16, 1024);
                    mma_bf16_ss(tvn, a, b, idWU, ks > 0);
                }
                mma_commit(&bars[B_WU_DONE]);
                // K K^T / Q K^T of the next chunk, so the WY warps can start on it
                if (c + 1 < NT && !issue_kq(c + 1)) break;
                GDN_TR(c, 4);
                // Vn^T = U^T - S^T W^T ;  O^T = S^T Qg^T
                if (!wait_bar(&bars[B_WT_READY], c & 1, tmo, abort_flag, 2u)) break;
                GDN_TR(c, 5);
                if (!wait_bar(&bars[B_S_READY], c & 1, tmo, abort_flag, 2u)) break;
                GDN_TR(c, 6);
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_ST + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc(sbase + OFF_WT + ks * 2048, 8192, 1024);
                    mma_bf16_ss(tvn, a, b, idVN, 1u);
                }
                mma_commit(&bars[B_VN_DONE]);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_ST + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc(kq + 8192 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    mma_bf16_ss(tO, a, b, idO, ks > 0);
                }
                // O^T += Vn^T P^T ;  S^T += (decayed Vn^T) K
                if (!wait_bar(&bars[B_VN_READY], c & 1, tmo, abort_flag, 2u)) break;
                GDN_TR(c, 7);
                tc_fence_after_sync();
                const uint32_t pt = sbase + ((c & 1) ? OFF_P1 : OFF_P0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_VS + ks * 32, 16, 1024);
                    const uint64_t b = smem_desc(kq + ks * 2048, 16384, 1024);
                    mma_bf16_ss(tmem + TM_S, a, b, idUP, 1u);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = smem_desc(sbase + OFF_VN + ks * 32, 16, 1024);
                    const uint64_t b = smem_desc(pt + ks * 32, 16, 1024);
                    mma_bf16_ss(tO, a, b, idO, 1u);
                }
                mma_commit(&bars[B_UPD_DONE]);
                mma_commit(&bars[B_STG_FREE0 + s]);
                GDN_TR(c, 8);
            }
            // every issued MMA completes before TMEM is released
            mma_commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0, kCleanupNs);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ scan epilogue
        const int st = threadIdx.x - 128;  // value index dv = TMEM lane
        const uint32_t lb = tmem_lane_base(warp);
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
            for (int j = 0; j < NQ / 32 + (NQ == 16); ++j) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tO + 32 * j, r0);
                if (NQ >= 32) tmem_ld16(tO + 32 * j + 16, r1);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    *reinterpret_cast<__nv_bfloat16 *>(ostage + (32 * j + i) * 256 + st * 2) =
                        __float2bfloat16_rn(p.scale * __uint_as_float(r0[i]));
                    if (NQ >= 32)
                        *reinterpret_cast<__nv_bfloat16 *>(ostage + (32 * j + 16 + i) * 256 + st * 2) =
                            __float2bfloat16_rn(p.scale * __uint_as_float(r1[i]));
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
            if (st == 0) GDN_TR(c, 9);
            tc_fence_after_sync();
            // state: S^T -> bf16 operand, then S^T <- exp(g_last) S^T in TMEM
            const float el = ms->el;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tmem + lb + TM_S + 32 * j, r0);
                tmem_ld16(tmem + lb + TM_S + 32 * j + 16, r1);
                tmem_wait_ld();
                uint8_t *blk = sm + OFF_ST + (j >> 1) * 16384;
                const int col = (32 * j) & 63;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint32_t *r = k ? r1 : r0;
                    uint4 v0, v1;
                    v0.x = pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1]));
                    v0.y = pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3]));
                    v0.z = pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5]));
                    v0.w = pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7]));
                    v1.x = pack_bf16(__uint_as_float(r[8]), __uint_as_float(r[9]));
                    v1.y = pack_bf16(__uint_as_float(r[10]), __uint_as_float(r[11]));
                    v1.z = pack_bf16(__uint_as_float(r[12]), __uint_as_float(r[13]));
                    v1.w = pack_bf16(__uint_as_float(r[14]), __uint_as_float(r[15]));
                    *reinterpret_cast<uint4 *>(blk + sw128_offset(st, col + 16 * k)) = v0;
                    *reinterpret_cast<uint4 *>(blk + sw128_offset(st, col + 16 * k + 8)) = v1;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    r0[i] = __float_as_uint(el * __uint_as_float(r0[i]));
                    r1[i] = __float_as_uint(el * __uint_as_float(r1[i]));
                }
                tmem_st16(tmem + lb + TM_S + 32 * j, r0);
                tmem_st16(tmem + lb + TM_S + 32 * j + 16, r1);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_S_READY]);
            if (st == 0) GDN_TR(c, 10);
            // output of the previous chunk (its MMAs completed with UPD_DONE)
            if (c >= 1) out_epilogue(c - 1);
            if (st == 0) GDN_TR(c, 11);
            // Vn^T of this chunk -> two bf16 operands
            const bool wv = wait_bar(&bars[B_VN_DONE], c & 1, tmo, abort_flag, 4u);
            if (st == 0) tma_store_wait_read<0>();
            if (!group_all(wv, 2, 128)) { ok = false; break; }  // staging tile free
            if (st == 0) GDN_TR(c, 12);
            tc_fence_after_sync();
            float x[64];
            {
                const uint32_t tv = tmem + lb + ((c & 1) ? TM_VN1 : TM_VN0);
                uint32_t r[4][16];
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld16(tv + 16 * j, r[j]);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[16 * j + i] = __uint_as_float(r[j][i]);
            }
            store_row_sw128(sm + OFF_VN, st, x);
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(&ms->sef[i]);
                x[i] *= f.x;
                x[i + 1] *= f.y;
                x[i + 2] *= f.z;
                x[i + 3] *= f.w;
            }
            store_row_sw128(sm + OFF_VS, st, x);
            tc_fence_before_sync();
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_VN_READY]);
            if (st == 0) GDN_TR(c, 13);
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
        // 8 warps.  Warp w reads TMEM lane quarter (w & 3) and works on column
        // half h = (w - 8) / 4 of the 64-wide chunk tiles.
        const int wt = threadIdx.x - 256;  // 0..255
        const int q = warp & 3;
        const int h = (warp - 8) >> 2;
        const uint32_t lb = tmem_lane_base(warp);
        float *AF = reinterpret_cast<float *>(sm + OFF_AF);
        float *XS = reinterpret_cast<float *>(sm + OFF_X);
        uint8_t *twu = sm + OFF_TWU;
        const bool l2n = (p.flags & GDN_QK_L2NORM) != 0;
        const __nv_bfloat16 *betap = p.beta + (size_t)bh * p.rows;
        const float *gp = p.g + (size_t)bh * p.T;
        // beta / g of a chunk, fetched one chunk ahead into a register
        auto prefetch = [&](int cc) -> float {
            if (wt < 64) {
                const int row = cc * 64 + wt;
                return row < p.rows ? __bfloat162float(betap[row]) : 0.f;
            }
            if (wt < 128) {
                const int row = cc * 64 + wt - 64;
                return (row < p.rows && row % R == 0) ? gp[row / R] : 0.f;
            }
            return 0.f;
        };
        float pf = NT > 0 ? prefetch(0) : 0.f;
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1;
            Misc *ms = misc + s;
            uint8_t *kq = sm + (s ? OFF_KQ1 : OFF_KQ0);
            uint8_t *ptile = sm + ((c & 1) ? OFF_P1 : OFF_P0);
            if (wt == 0) GDN_TR(c, 14);
            // 1. beta and g of the chunk's rows; cumulative decay
            if (wt < 64) ms->beta[wt] = pf;
            else if (wt < 128) ms->gam[wt - 64] = pf;
            if (c + 1 < NT) pf = prefetch(c + 1);
            named_bar(1, 256);
            if (wt < 32) {
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
                const float g0 = __shfl_sync(0xffffffffu, a, 0);
                float dev = fmaxf(fabsf(a - g0), fabsf(b - g0));
#pragma unroll
                for (int off = 16; off; off >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, off));
                if (lane == 31) {
                    ms->safe = dev <= 80.f ? 1 : 0;
                    ms->el = __expf(b);
                }
            }
            const bool wk = wait_bar(&bars[B_KQ_DONE], c & 1, tmo, abort_flag, 8u);
            if (!group_all(wk, 1, 256)) break;  // also publishes gam
            if (wt == 0) GDN_TR(c, 15);
            tc_fence_after_sync();
            // 2. this thread's 32 columns of its K K^T (q < 2) or Q K^T (q >= 2) row
            float x[32];
            {
                uint32_t r0[16], r1[16];
                tmem_ld16(tmem + lb + TM_KQ + 32 * h, r0);
                tmem_ld16(tmem + lb + TM_KQ + 32 * h + 16, r1);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    x[i] = __uint_as_float(r0[i]);
                    x[16 + i] = __uint_as_float(r1[i]);
                }
            }
            const int t = 32 * (q & 1) + lane;  // row of K K^T, or query row of Q K^T
            if (q < 2) {
                if (h == (q & 1)) {
                    float diag = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) diag = (i == lane) ? x[i] : diag;
                    ms->n[t] = l2n ? rsqrtf(fmaxf(diag, 1e-24f)) : 1.f;
                }
            } else if (l2n) {
                float ss = 0.f;
                const uint4 *rowp = reinterpret_cast<const uint4 *>(kq + 8192 + h * 16384 + t * 128);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 u = rowp[ch];
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                        ss += lo * lo + hi * hi;
                    }
                }
                ms->qp[h][t] = ss;
            }
            tc_fence_before_sync();
            named_bar(1, 256);  // n and partial q norms visible; TMEM rows read
            if (wt == 0) mbar_arrive(&bars[B_KQ_FREE]);
            if (wt == 0) GDN_TR(c, 16);
            // per-row / per-column factors of the chunk
            if (wt < 64) {
                const float g0 = ms->gam[0], gi = ms->gam[wt], gl = ms->gam[63];
                const float ni = ms->n[wt];
                ms->m[wt] = l2n ? rsqrtf(fmaxf(ms->qp[0][wt] + ms->qp[1][wt], 1e-24f)) : 1.f;
                ms->wsc[wt] = ms->beta[wt] * __expf(gi) * ni;
                ms->bn[wt] = __expf(g0 - gi) * ni;
                ms->ea[wt] = __expf(gi - g0);
                ms->sef[wt] = __expf(gl - gi) * ni;
            }
            named_bar(1, 256);
            if (wt == 0) mbar_arrive(&bars[B_MISC0 + s]);
            // 3. A rows (q < 2), P rows and scaled query rows (q >= 2)
            const bool safe = ms->safe != 0;
            if (q < 2) {
                const float gt = ms->gam[t];
                const float rowb = ms->beta[t] * ms->n[t];
                float av[32];
                if (safe) {
                    const float rowf = rowb * ms->ea[t];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 bn4 = *reinterpret_cast<const float4 *>(&ms->bn[32 * h + 4 * j]);
                        av[4 * j] = rowf * bn4.x * x[4 * j];
                        av[4 * j + 1] = rowf * bn4.y * x[4 * j + 1];
                        av[4 * j + 2] = rowf * bn4.z * x[4 * j + 2];
                        av[4 * j + 3] = rowf * bn4.w * x[4 * j + 3];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        av[i] = rowb * __expf(gt - ms->gam[32 * h + i]) * ms->n[32 * h + i] * x[i];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int s0 = 32 * h + 4 * j;
                    *reinterpret_cast<float4 *>(&AF[t * kAS + s0]) =
                        make_float4(s0 < t ? av[4 * j] : 0.f, s0 + 1 < t ? av[4 * j + 1] : 0.f,
                                    s0 + 2 < t ? av[4 * j + 2] : 0.f, s0 + 3 < t ? av[4 * j + 3] : 0.f);
                }
            } else if (t < NQ) {
                const int row = t * R + R - 1;
                const float gr = ms->gam[row];
                const float mt = ms->m[t];
                float pv[32];
                if (safe) {
                    const float rowf = mt * ms->ea[row];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 bn4 = *reinterpret_cast<const float4 *>(&ms->bn[32 * h + 4 * j]);
                        pv[4 * j] = rowf * bn4.x * x[4 * j];
                        pv[4 * j + 1] = rowf * bn4.y * x[4 * j + 1];
                        pv[4 * j + 2] = rowf * bn4.z * x[4 * j + 2];
                        pv[4 * j + 3] = rowf * bn4.w * x[4 * j + 3];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        pv[i] = mt * __expf(gr - ms->gam[32 * h + i]) * ms->n[32 * h + i] * x[i];
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s0 = 32 * h + 2 * j;
                    pk[j] = pack_bf16(s0 <= row ? pv[2 * j] : 0.f, s0 + 1 <= row ? pv[2 * j + 1] : 0.f);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4 *>(ptile + sw128_offset(t, 32 * h + 8 * j)) =
                        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                // Qg row t, key-dim half h: q_t exp(g_row) / ||q_t||
                const float qs = __expf(gr) * mt;
                uint4 *rowp = reinterpret_cast<uint4 *>(kq + 8192 + h * 16384 + t * 128);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 u = rowp[ch];
                    uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w4[e] = pack_bf16(__uint_as_float(w4[e] << 16) * qs, __uint_as_float(w4[e] & 0xffff0000u) * qs);
                    rowp[ch] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
            named_bar(1, 256);  // A complete
            if (wt == 0) GDN_TR(c, 17);
            // 4. T = (I + A)^-1 in place over A: 16x16 diagonal blocks by
            //    substitution, then the merges T_ij = -T_ii A_ij T_jj (16 level)
            //    and T_bl = -T_bot A_bl T_top (32 level).
            float xs[16];
            const int db = wt >> 4, dc = wt & 15;
            if (wt < 64) {
                float pp[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pp[i] = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    xs[j] = ((j == dc) ? 1.f : 0.f) - pp[j];
#pragma unroll
                    for (int i = j + 1; i < 16; ++i) pp[i] += AF[(16 * db + i) * kAS + 16 * db + j] * xs[j];
                }
            }
            if (wt == 0) GDN_TR(c, 22);
            named_bar(1, 256);
            if (wt < 64) {
#pragma unroll
                for (int i = 0; i < 16; ++i) AF[(16 * db + i) * kAS + 16 * db + dc] = xs[i];
            }
            named_bar(1, 256);
            {
                float acc[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = wt + 256 * k;
                    const int hh = e >> 8, rr = (e >> 4) & 15, cl = e & 15;
                    const int i0 = 32 * hh + 16, j0 = 32 * hh;
                    float a = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) a += AF[(i0 + rr) * kAS + j0 + m] * AF[(j0 + m) * kAS + j0 + cl];
                    acc[k] = a;
                }
                XS[wt] = acc[0];
                XS[wt + 256] = acc[1];
                if (wt == 0) GDN_TR(c, 23);
                named_bar(1, 256);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = wt + 256 * k;
                    const int hh = e >> 8, rr = (e >> 4) & 15, cl = e & 15;
                    const int i0 = 32 * hh + 16;
                    float a = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) a += AF[(i0 + rr) * kAS + i0 + m] * XS[(hh << 8) + m * 16 + cl];
                    acc[k] = a;
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = wt + 256 * k;
                    const int hh = e >> 8, rr = (e >> 4) & 15, cl = e & 15;
                    AF[(32 * hh + 16 + rr) * kAS + 32 * hh + cl] = -acc[k];
                }
                named_bar(1, 256);
            }
            {
                const int cl = wt & 31, r0 = wt >> 5;  // rows r0 + 8k, k < 4
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < 32; m += 4) {
                    const float t0 = AF[(m + 0) * kAS + cl], t1 = AF[(m + 1) * kAS + cl];
                    const float t2 = AF[(m + 2) * kAS + cl], t3 = AF[(m + 3) * kAS + cl];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&AF[(32 + r0 + 8 * k) * kAS + m]);
                        acc[k] += a4.x * t0 + a4.y * t1 + a4.z * t2 + a4.w * t3;
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) XS[(r0 + 8 * k) * 32 + cl] = acc[k];
                if (wt == 0) GDN_TR(c, 24);
                named_bar(1, 256);
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = 0.f;
#pragma unroll
                for (int m = 0; m < 32; m += 4) {
                    const float x0 = XS[(m + 0) * 32 + cl], x1 = XS[(m + 1) * 32 + cl];
                    const float x2 = XS[(m + 2) * 32 + cl], x3 = XS[(m + 3) * 32 + cl];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(&AF[(32 + r0 + 8 * k) * kAS + 32 + m]);
                        acc[k] += t4.x * x0 + t4.y * x1 + t4.z * x2 + t4.w * x3;
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) AF[(32 + r0 + 8 * k) * kAS + cl] = -acc[k];
                named_bar(1, 256);
            }
            if (wt == 0) GDN_TR(c, 18);
            // 5. Tw = T diag(beta e^g n), Tu = T diag(beta) as bf16 K-major tiles
            {
                const int tr = wt & 63, which = (wt >> 6) & 1, hf = wt >> 7;
                const float *sc = which ? ms->beta : ms->wsc;
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int s0 = 32 * hf + 4 * j;
                    const float4 t4 = *reinterpret_cast<const float4 *>(&AF[tr * kAS + s0]);
                    const float4 f4 = *reinterpret_cast<const float4 *>(&sc[s0]);
                    pk[2 * j] = pack_bf16(t4.x * f4.x, t4.y * f4.y);
                    pk[2 * j + 1] = pack_bf16(t4.z * f4.z, t4.w * f4.w);
                }
                uint8_t *tile = twu + which * 8192;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4 *>(tile + sw128_offset(tr, 32 * hf + 8 * j)) =
                        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            fence_proxy_async_smem();
            named_bar(1, 256);
            if (wt == 0) mbar_arrive(&bars[B_WY_READY]);
            if (wt == 0) GDN_TR(c, 19);
            // 6. W^T -> bf16 MN-major operand (row = key index d)
            bool ww = wait_bar(&bars[B_WU_DONE], c & 1, tmo, abort_flag, 8u);
            if (ww && c >= 1) ww = wait_bar(&bars[B_VN_DONE], (c - 1) & 1, tmo, abort_flag, 8u);
            if (!group_all(ww, 1, 256)) break;
            if (wt == 0) GDN_TR(c, 20);
            tc_fence_after_sync();
            {
                uint32_t r0[16], r1[16];
                tmem_ld16(tmem + lb + TM_W + 32 * h, r0);
                tmem_ld16(tmem + lb + TM_W + 32 * h + 16, r1);
                tmem_wait_ld();
                const int d = 32 * q + lane;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t *r = j ? r1 : r0;
                    uint4 v0, v1;
                    v0.x = pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1]));
                    v0.y = pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3]));
                    v0.z = pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5]));
                    v0.w = pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7]));
                    v1.x = pack_bf16(__uint_as_float(r[8]), __uint_as_float(r[9]));
                    v1.y = pack_bf16(__uint_as_float(r[10]), __uint_as_float(r[11]));
                    v1.z = pack_bf16(__uint_as_float(r[12]), __uint_as_float(r[13]));
                    v1.w = pack_bf16(__uint_as_float(r[14]), __uint_as_float(r[15]));
                    *reinterpret_cast<uint4 *>(sm + OFF_WT + sw128_offset(d, 32 * h + 16 * j)) = v0;
                    *reinterpret_cast<uint4 *>(sm + OFF_WT + sw128_offset(d, 32 * h + 16 * j + 8)) = v1;
                }
            }
            tc_fence_before_sync();
            fence_proxy_async_smem();
            named_bar(1, 256);
            if (wt == 0) mbar_arrive(&bars[B_WT_READY]);
            if (wt == 0) GDN_TR(c, 21);
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

#ifdef GDN_TRACE
extern "C" int gdn_trace_set(void *buf) {
    return cudaMemcpyToSymbol(g_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
#endif

int scan_tc_set_wait_limit(unsigned long long us) {
    g_timeout_ns = us == 0 ? 1000000000ull : us * 1000ull;
    return GDN_OK;
}

}  // namespace gdn
