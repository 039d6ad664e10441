// scan_tc.cu -- fused chunkwise GDN / DeltaProduct forward on the tcgen05
// tensor cores (bf16 tensors, Dk = Dv = 128, 64-row chunks, fp32 state).
//
// Every product is held value-dimension-major so that every scan MMA has
// M = 128 (the value dim dv).  Per chunk, with g the within-chunk cumulative
// log-decay (gated_deltaproduct test.py: `gated_chunk_scaled_dot_kkt_fwd_kernel`,
// `solve_tril_16x16_kernel` and the merge kernels, `gated_fwd_recompute_w_u_kernel`,
// `preprocess_qkw`, `gated_chunk_delta_rule_fwd_kernel_h`,
// `gated_chunk_linear_attn_fwd_kernel_o`):
//
//   KQ   = [K; Q] K^T                   rows 0..63 K K^T, rows 64.. Q K^T
//   A[t][s] = beta_t exp(g_t - g_s) (k_t . k_s), s < t      (CUDA cores)
//   T    = (I + A)^-1     16x16 diagonal blocks and 16-level merges on the CUDA
//                         cores, the 32-level merge on the tensor cores (bf16
//                         hi/lo products)
//   W^T  = K^T (T diag(beta e^g))^T,  U^T = V^T (T diag(beta))^T
//   Vn^T = U^T - S^T W^T                (v_new of the WY form, negated-A MMA)
//   O^T  = diag-scaled S^T Q^T + Vn^T P^T,  P[t][s] = e^{g_t-g_s} q_t.k_s (s <= t)
//   S^T <- e^{g_last} S^T + (Vn^T diag(e^{g_last - g_s})) K
//
// The pages run these as separate launches with HBM round trips.  Here one
// launch holds two kinds of CTA, one per SM:
//
//   "WY" CTAs   compute the chunk-local products, which need no state: two
//               independent 8-warp pipelines per CTA take (chunk, head) items
//               (K K^T / Q K^T by MMA, A, the blocked inverse, Tw/Tu, P) and
//               ship Tw, Tu, P and the per-row factors to the head's scan CTA.
//   scan CTAs   (one per head) run the sequential part: the fp32 state S^T lives
//               in tensor memory for the whole sequence; a TMA warp streams K,
//               Q, V; one thread issues the chain's MMAs and another W^T =
//               K^T Tw^T; 8 epilogue warps turn S^T and Vn^T into bf16
//               operands; 4 aux warps convert W^T and write the output rows of
//               the previous chunk.
//
// Two ways to ship.  Ring mode (the default for up to min(80, SMs/2) heads):
// one cooperative grid of all the scan CTAs and as many WY CTAs as SMs remain
// (up to 1.5 per head); an item goes through slot c % 8 of its head's ring in
// the workspace, with a tag published after it and a count of the chunks taken
// out published back.  Cluster mode (more heads, or a forced shape): clusters
// of hc scan CTAs and nwy WY CTAs, an item going straight into the scan CTA's
// shared memory with cp.async.bulk over the cluster (DSMEM).
//
// Only q, k, v, beta, g are read from HBM and o written (the ring stays in L2).
// Every wait is bounded in wall time; on expiry the CTA sets an error word,
// stops issuing work, drains what is in flight, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gdn_internal.h"
#include "tc_util.cuh"

namespace gdn {

namespace {
__device__ unsigned int g_tc_error = 0;
unsigned long long g_timeout_ns = 1000000000ull;  // host copy of the wait limit
int g_force_hc = 0, g_force_nwy = 0;               // cluster shape override (0: automatic)
}  // namespace

// Optional timeline instrumentation (compiled in only with -DGDN_TRACE): the
// first cluster records clock64() at fixed points of each role, per chunk of
// its first head (tr_on is true in the roles and items that belong to it).
#ifdef GDN_TRACE
__device__ unsigned long long *g_trace = nullptr;
#define GDN_TR(c, ev)                                                          \
    do {                                                                       \
        if (tr_on && tr_buf != nullptr && (c) < 1024)                          \
            tr_buf[(size_t)(c) * 64 + (ev)] = clock64();                       \
    } while (0)
#else
#define GDN_TR(c, ev) \
    do {              \
    } while (0)
#endif

namespace {
using namespace tc;

constexpr int kThreads = 512;  // 16 warps: 4 per SM sub-partition, up to 128 registers a thread
constexpr int kAS = 68;        // fp32 row stride of the A / T tiles

// ---------------------------------------------------------------- scan CTA map
constexpr uint32_t S_K0 = 0, S_K1 = 16384;      // K tile [64][128] as 2 MN-atoms
constexpr uint32_t S_Q0 = 32768, S_Q1 = 49152;  // Q tile [NQ][128] as 2 K-blocks
constexpr uint32_t S_V = 65536;                 // V tile [64][128] as 2 MN-atoms
constexpr uint32_t S_RECV0 = 81920;             // receive slots (one per chunk parity)
constexpr uint32_t RS = 25600;                  // slot: Tw | Tu | P | vectors
constexpr uint32_t R_TW = 0, R_TU = 8192, R_P = 16384, R_VEC = 24576;
constexpr uint32_t S_WT = S_RECV0 + 2 * RS;     // W^T bf16 [128 d][64 t] MN-major
constexpr uint32_t S_ST = S_WT + 16384;         // S^T bf16 [128 dv][128 dk] K-major
constexpr uint32_t S_VN = S_ST + 32768;         // Vn^T bf16 [128 dv][64 s]
constexpr uint32_t S_VS = S_VN + 16384;         // decayed Vn^T
constexpr uint32_t S_QS = S_VS + 16384;         // per-query output scales, 2 x 64 floats (aux warps)
constexpr uint32_t S_BAR = S_QS + 512;
constexpr uint32_t S_FLAGS = S_BAR + 256;
constexpr uint32_t S_END = S_FLAGS + 64;

// ------------------------------------------------------------------ WY CTA map
constexpr uint32_t GS = 107520;  // bytes per WY pipeline
constexpr uint32_t G_KQ = 0;        // [K rows 0..63 | Q rows 64..] x 2 K-blocks
constexpr uint32_t G_TWU = 32768;   // Tw (+0), Tu (+8192): bf16 [64 t][64 s] K-major
constexpr uint32_t G_PV = 49152;    // two buffers (+9216) of P bf16 [NQ][64] K-major (8 KB) + vectors (1 KB)
constexpr uint32_t G_AF = 73728;    // A fp32 [64][68], inverted in place
constexpr uint32_t G_X = 91136;     // inverse scratch: 32x32 fp32, row stride kXS (36) words
constexpr int kXS = 36;             // makes the column-strided stores of X conflict-free
constexpr uint32_t G_MISC = 96256;  // Misc
static_assert(G_X + 32 * kXS * 4 <= G_MISC, "inverse scratch fits");
// Operands of the tensor-core 32-level merge of the inverse, bf16 hi / lo halves
// (4 KB each, 128-byte rows).  The K-major M = 64 operands hold rows 32..63
// only: their descriptors start 4 KB lower, inside this pipeline's region, and
// rows 0..31 of the products are not used.  A2 and B1 borrow the Tw / Tu tile,
// B2 the A1 tile.
constexpr uint32_t G_A1 = 99328;   // A[32..63][0..31]            K-major, rows 32..63 (hi | lo)
constexpr uint32_t G_A2 = 32768;   // T_bot = T[32..63][32..63]   K-major, rows 32..63 (hi | lo)
constexpr uint32_t G_B1 = 40960;   // T_top = T[0..31][0..31]     MN-major, 32 k-rows (hi | lo)
constexpr uint32_t G_B2 = G_A1;    // Y = A_bl T_top              MN-major, 32 k-rows (hi | lo)
static_assert(G_MISC + sizeof(float) * 768 <= G_A1 && G_A1 + 8192 <= GS, "WY map");
constexpr uint32_t W_BAR = 2 * GS;
constexpr uint32_t W_FLAGS = W_BAR + 256;
constexpr uint32_t W_END = W_FLAGS + 64;

constexpr uint32_t kSmemBytes = (S_END > W_END ? S_END : W_END) + 1024;

// vectors shipped per chunk (floats): exp(g_last - g_s) n_s, output scale of
// each query row, exp(g_last)
constexpr uint32_t V_SEF = 0, V_QS = 64, V_EL = 128;
// bytes shipped per chunk: Tw | Tu (16 KB), then P (8 KB region) | vectors (1 KB)
constexpr uint32_t kShipBytes = 16384 + 8192 + 1024;
constexpr int kRing = 8;           // ring slots per head in ring mode
constexpr int kMaxRingHeads = 80;  // heads a ring-mode launch serves at most
static_assert(R_TU == R_TW + 8192 && R_VEC == R_P + 8192, "receive slot layout matches the two shipped blocks");

// scan TMEM columns
constexpr uint32_t TM_S = 0, TM_VN = 128, TM_W = 192, TM_O10 = 256, TM_O11 = 320, TM_O20 = 384, TM_O21 = 448;

enum ScanBar {
    SB_FULLKQ0, SB_FULLKQ1, SB_VFULL, SB_S_READY, SB_VN_DONE, SB_VN_READY, SB_UPD_DONE,
    SB_SLOT_DONE0, SB_SLOT_DONE1, SB_RECV0, SB_RECV1, SB_W_DONE, SB_WT_READY,
    SB_DRAIN, SB_WDRAIN, SB_OFREE0, SB_OFREE1, SB_VN2_READY, SB_NUM
};
// Per WY pipeline: FULL, KQ_DONE, DRAIN, then RECV_FREE for each (scan CTA of
// the cluster, receive slot) the pipeline may ship to.
constexpr int kMaxHc = 4;  // heads per cluster at most
enum WyBar { WB_FULL, WB_KQ_DONE, WB_DRAIN, WB_INV, WB_RECV_FREE0, WB_PER_GROUP = WB_RECV_FREE0 + 2 * kMaxHc };
static_assert(2 * WB_PER_GROUP <= 32, "WY barriers fit their 256 bytes");

// Per-chunk vectors of one WY pipeline.
struct Misc {
    alignas(16) unsigned long long tag[2];  // ring mode: the ready tag being published
    float beta[64];   // beta of each row (0 past the end)
    float gam[64];    // within-chunk cumulative log-decay
    float n[64];      // 1/||k_s|| with GDN_QK_L2NORM, else 1
    float m[64];      // 1/||q_t|| with GDN_QK_L2NORM, else 1
    float wsc[64];    // beta_s exp(gam_s) n_s          (columns of Tw)
    float bn[64];     // exp(gam_0 - gam_s) n_s         (column factor of A and P)
    float ea[64];     // exp(gam_t - gam_0)             (row factor of A and P)
    float qp[2][64];  // partial q_t^2 sums over the two key-dim halves
    int safe;         // 1 if |gam_t - gam_0| <= 80 for all rows (factorised exponentials)
    unsigned ccache[80];  // ring mode: chunks each head's scan CTA was last seen to have taken out
    float pad[107];
};
static_assert(sizeof(Misc) == 3072, "Misc layout");

struct TcParams {
    const __nv_bfloat16 *beta;
    const float *g;
    const float *s0;
    float *sf;
    __nv_bfloat16 *o;
    int T, rows, NT;
    int BH;   // heads (batch x head)
    int hc;   // scan CTAs (heads) per cluster, ranks 0 .. hc-1
    int nwy;  // WY CTAs per cluster, ranks hc .. hc+nwy-1
    float scale;
    unsigned flags;
    unsigned long long timeout_ns;
    // Ring mode (flat != 0): one grid of BH scan CTAs and nwy WY CTAs, all
    // resident (a cooperative launch); chunk c of head h travels through slot
    // c % kRing of the head's ring in global memory instead of a cluster copy.
    int flat;
    uint8_t *ring;                // [BH][kRing] slots of kShipBytes
    unsigned long long *ready;    // [BH][kRing] x 16 B: epoch << 32 | (chunk + 1) of the slot's contents
    unsigned long long *cons;     // [BH]: epoch << 32 | chunks the scan CTA has taken out of its ring
    unsigned epoch;               // tag of this launch, never 0
};

constexpr unsigned long long kCleanupNs = 200000000ull;  // 0.2 s for draining on the way out

// Bounded wait that also gives up as soon as another role of this CTA has
// aborted.  cluster = true acquires at cluster scope (phases completed by the
// other CTA).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, unsigned long long timeout_ns,
                                         volatile int *abort_flag, unsigned code, bool cluster = false) {
    if (cluster ? mbar_try_wait_cluster(bar, parity, 0u) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (cluster ? mbar_try_wait_cluster(bar, parity, 20000u) : mbar_try_wait_sleep(bar, parity, 20000u))
            return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicOr(&g_tc_error, code);
            return false;
        }
    }
}

// Bounded wait, like wait_bar, until *flag (written by another CTA with a
// release store) holds this launch's epoch in its high word and at least
// `need` in its low word.  Gives up early once any CTA has reported an error.
__device__ __forceinline__ bool wait_tag(const unsigned long long *flag, unsigned epoch, unsigned need,
                                         unsigned long long timeout_ns, volatile int *abort_flag, unsigned code,
                                         unsigned *seen = nullptr) {
    unsigned long long v = ld_acquire_gpu(flag);
    if ((unsigned)(v >> 32) == epoch && (unsigned)v >= need) {
        if (seen) *seen = (unsigned)v;
        return true;
    }
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(100);
        v = ld_acquire_gpu(flag);
        if ((unsigned)(v >> 32) == epoch && (unsigned)v >= need) {
            if (seen) *seen = (unsigned)v;
            return true;
        }
        if (*abort_flag || *reinterpret_cast<volatile unsigned *>(&g_tc_error) != 0u) {
            *abort_flag = 1;
            return false;
        }
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

// 16 fp32 values as bf16 into two 16-byte chunks of a 128-byte-swizzled row.
__device__ __forceinline__ void store16_sw128(uint8_t *tile, int row, int col, const uint32_t (&r)[16],
                                              float mul = 1.f) {
    uint4 v0, v1;
    v0.x = pack_bf16(mul * __uint_as_float(r[0]), mul * __uint_as_float(r[1]));
    v0.y = pack_bf16(mul * __uint_as_float(r[2]), mul * __uint_as_float(r[3]));
    v0.z = pack_bf16(mul * __uint_as_float(r[4]), mul * __uint_as_float(r[5]));
    v0.w = pack_bf16(mul * __uint_as_float(r[6]), mul * __uint_as_float(r[7]));
    v1.x = pack_bf16(mul * __uint_as_float(r[8]), mul * __uint_as_float(r[9]));
    v1.y = pack_bf16(mul * __uint_as_float(r[10]), mul * __uint_as_float(r[11]));
    v1.z = pack_bf16(mul * __uint_as_float(r[12]), mul * __uint_as_float(r[13]));
    v1.w = pack_bf16(mul * __uint_as_float(r[14]), mul * __uint_as_float(r[15]));
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, col)) = v0;
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, col + 8)) = v1;
}

// =========================================================================== kernel
template <int R>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_tc_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
                  const __grid_constant__ CUtensorMap mV, TcParams p) {
    constexpr int NQ = 64 / R;  // query rows (tokens) per chunk
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
    // A cluster holds hc scan CTAs (one head each, ranks 0..hc-1) and nwy WY CTAs
    // whose 2*nwy pipelines take the cluster's (head, chunk) items round-robin.
    // In ring mode the whole grid plays the part of one cluster: hc = BH scan
    // CTAs, then nwy WY CTAs, ranked by block index.
    const bool flat = p.flat != 0;
    const uint32_t rank = flat ? blockIdx.x : cluster_ctarank();
    const int hc = p.hc, nwy = p.nwy;
    const int h0 = (int)(blockIdx.x / (unsigned)(hc + nwy)) * hc;  // first head of the cluster
    const int hce = min(hc, p.BH - h0);                             // heads it holds
    const bool is_scan = (int)rank < hc;
    bool tr_on = blockIdx.x < (unsigned)(hc + nwy) && rank == 0;
    (void)tr_on;
#ifdef GDN_TRACE
    unsigned long long *const tr_buf = g_trace;  // read once: a global load per event would skew the timeline
#endif
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + (is_scan ? S_BAR : W_BAR));
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + (is_scan ? S_FLAGS : W_FLAGS));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + (is_scan ? S_FLAGS : W_FLAGS) + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = h0 + (int)rank;  // the scan CTA's head
    const int NT = p.NT;
    const unsigned long long tmo = p.timeout_ns;
    const uint32_t ncols = is_scan ? 512u : 256u;

    if (threadIdx.x == 0) {
        if (is_scan) {
            for (int i = 0; i < SB_NUM; ++i)
                mbar_init(&bars[i], (i == SB_S_READY || i == SB_VN_READY || i == SB_VN2_READY)
                                        ? 256u
                                        : ((i == SB_WT_READY || i == SB_OFREE0 || i == SB_OFREE1) ? 128u : 1u));
        } else {
            for (int i = 0; i < 2 * WB_PER_GROUP; ++i) mbar_init(&bars[i], 1u);  // pipelines 2*(rank-hc) + 0, 1
        }
        if (!flat && is_scan && (int)rank < hce) {
            // the receive barriers expect their first shipments; later phases are
            // armed by the slot-release warp when it hands a slot back
            for (int b = 0; b < 2 && b < p.NT; ++b) mbar_arrive_expect_tx(&bars[SB_RECV0 + b], kShipBytes);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, ncols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32 * 3) {
        prefetch_tensormap(&mK);
        prefetch_tensormap(&mQ);
        prefetch_tensormap(&mV);
    }
    tc_fence_before_sync();
    if (flat)
        __syncthreads();
    else
        cluster_sync_all();  // every CTA's barriers exist before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t sbase = smem_u32(sm);

    if (is_scan) {
        // ================================================================= scan CTA
        // (a scan CTA past the last head only takes part in the cluster barriers)
        if ((int)rank >= hce) {
        } else if (warp == 0) {
            // ------------------------------------------------------ TMA producer
            if (lane == 0) {
                int armed[2] = {0, 0}, armed_v = 0;
                for (int c = 0; c < NT; ++c) {
                    const int b = c & 1;
                    // stage b held chunk c-2, whose MMAs all completed before its slot's release
                    if (c >= 2 && !wait_bar(&bars[SB_SLOT_DONE0 + b], ((c - 2) >> 1) & 1, tmo, abort_flag, 1u)) break;
                    uint8_t *kt = sm + (b ? S_K1 : S_K0);
                    uint8_t *qt = sm + (b ? S_Q1 : S_Q0);
                    mbar_arrive_expect_tx(&bars[SB_FULLKQ0 + b], 16384 + 2 * NQ * 128);
                    tma_load_3d(kt, &mK, &bars[SB_FULLKQ0 + b], 0, c * 64, bh);
                    tma_load_3d(kt + 8192, &mK, &bars[SB_FULLKQ0 + b], 64, c * 64, bh);
                    tma_load_3d(qt, &mQ, &bars[SB_FULLKQ0 + b], 0, c * NQ, bh);
                    tma_load_3d(qt + NQ * 128, &mQ, &bars[SB_FULLKQ0 + b], 64, c * NQ, bh);
                    armed[b]++;
                    // V(c-1) has been read once Vn(c-1), issued after U(c-1), is complete
                    if (c >= 1 && !wait_bar(&bars[SB_VN_DONE], (c - 1) & 1, tmo, abort_flag, 1u)) break;
                    mbar_arrive_expect_tx(&bars[SB_VFULL], 16384);
                    tma_load_3d(sm + S_V, &mV, &bars[SB_VFULL], 0, c * 64, bh);
                    tma_load_3d(sm + S_V + 8192, &mV, &bars[SB_VFULL], 64, c * 64, bh);
                    armed_v++;
                }
                for (int b = 0; b < 2; ++b)
                    if (armed[b]) mbar_wait(&bars[SB_FULLKQ0 + b], (armed[b] - 1) & 1, kCleanupNs);
                if (armed_v) mbar_wait(&bars[SB_VFULL], (armed_v - 1) & 1, kCleanupNs);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------ MMA issuer
            if (lane == 0) {
                const uint32_t idU = idesc_bf16(128, 64, true, false);
                const uint32_t idVN = idesc_bf16(128, 64, false, true, true);
                const uint32_t idO = idesc_bf16(128, NQ, false, false);
                const uint32_t idUP = idesc_bf16(128, 128, false, true);
                for (int c = 0; c < NT; ++c) {
                    const int b = c & 1;
                    const uint32_t recv = sbase + S_RECV0 + b * RS;
                    const uint32_t kt = sbase + (b ? S_K1 : S_K0);
                    const uint32_t qt = sbase + (b ? S_Q1 : S_Q0);
                    const uint32_t tvn = tmem + TM_VN;
                    // U^T = V^T Tu^T
                    if (!wait_bar(&bars[SB_RECV0 + b], (c >> 1) & 1, tmo, abort_flag, 2u)) break;
                    if (!wait_bar(&bars[SB_VFULL], c & 1, tmo, abort_flag, 2u)) break;
                    GDN_TR(c, 0);
                    tc_fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ss(tvn, smem_desc(sbase + S_V + ks * 2048, 8192, 1024),
                                    smem_desc(recv + R_TU + ks * 32, 16, 1024), idU, ks > 0);
                    // Vn^T = U^T - S^T W^T
                    if (!wait_bar(&bars[SB_WT_READY], c & 1, tmo, abort_flag, 2u)) break;
                    if (!wait_bar(&bars[SB_S_READY], c & 1, tmo, abort_flag, 2u)) break;
                    GDN_TR(c, 1);
                    tc_fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ss(tvn, smem_desc(sbase + S_ST + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                    smem_desc(sbase + S_WT + ks * 2048, 8192, 1024), idVN, 1u);
                    mma_commit(&bars[SB_VN_DONE]);
                    // O1^T = S^T Q^T (its TMEM columns free once chunk c-2's output is read)
                    if (!wait_bar(&bars[SB_FULLKQ0 + b], (c >> 1) & 1, tmo, abort_flag, 2u)) break;
                    if (c >= 2 && !wait_bar(&bars[SB_OFREE0 + b], ((c - 2) >> 1) & 1, tmo, abort_flag, 2u)) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ss(tmem + (b ? TM_O11 : TM_O10),
                                    smem_desc(sbase + S_ST + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                    smem_desc(qt + (ks >> 2) * (NQ * 128) + (ks & 3) * 32, 16, 1024), idO, ks > 0);
                    // S^T += (decayed Vn^T) K ;  O2^T = Vn^T P^T
                    if (!wait_bar(&bars[SB_VN_READY], c & 1, tmo, abort_flag, 2u)) break;
                    GDN_TR(c, 2);
                    tc_fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ss(tmem + TM_S, smem_desc(sbase + S_VS + ks * 32, 16, 1024),
                                    smem_desc(kt + ks * 2048, 8192, 1024), idUP, 1u);
                    // the state is ready before O2 runs (S_VN, which O2 reads, is only
                    // rewritten after the next VN_DONE, which completes after O2)
                    mma_commit(&bars[SB_UPD_DONE]);
                    if (!wait_bar(&bars[SB_VN2_READY], c & 1, tmo, abort_flag, 2u)) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ss(tmem + (b ? TM_O21 : TM_O20), smem_desc(sbase + S_VN + ks * 32, 16, 1024),
                                    smem_desc(recv + R_P + ks * 32, 16, 1024), idO, ks > 0);
                    mma_commit(&bars[SB_SLOT_DONE0 + b]);
                }
                mma_commit(&bars[SB_DRAIN]);
                mbar_wait(&bars[SB_DRAIN], 0, kCleanupNs);
            }
        } else if (warp == 2) {
            // ------------------------------------------------------ slot release
            // hands each receive slot back to the WY pipeline that fills it
            if (lane == 0 && flat) {
                // ring mode: fetch each chunk's Tw | Tu | P | vectors from the ring
                // once its WY pipeline has published it (checked ahead, while the
                // slot is still in use) and the receive slot is free, then report
                // the chunks taken out so that their ring slots can be refilled
                const unsigned long long tagc = (unsigned long long)p.epoch << 32;
                int armed[2] = {0, 0};
                int c = 0;
                for (; c < NT; ++c) {
                    const int b = c & 1;
                    const size_t slot = (size_t)bh * kRing + c % kRing;
                    GDN_TR(c, 11);
                    if (!wait_tag(p.ready + 2 * slot, p.epoch, (unsigned)(c + 1), tmo, abort_flag, 256u)) break;
                    GDN_TR(c, 12);
                    fence_proxy_async_global();
                    if (c >= 2 && !wait_bar(&bars[SB_SLOT_DONE0 + b], ((c - 2) >> 1) & 1, tmo, abort_flag, 16u)) break;
                    GDN_TR(c, 13);
                    mbar_arrive_expect_tx(&bars[SB_RECV0 + b], kShipBytes);
                    bulk_load_global(sm + S_RECV0 + b * RS, p.ring + slot * kShipBytes, kShipBytes, &bars[SB_RECV0 + b]);
                    armed[b]++;
                    if (c >= 2) st_release_gpu(p.cons + bh, tagc | (unsigned)(c - 1));  // chunks 0 .. c-2 are out
                }
                for (int b = 0; b < 2; ++b)
                    if (armed[b]) mbar_wait(&bars[SB_RECV0 + b], (armed[b] - 1) & 1, kCleanupNs);
                if (c == NT) {
                    // Every chunk of this head has been published and taken out, so
                    // nothing reads or writes its tags again in this launch: zero
                    // them, so that the next launch on this workspace starts from
                    // clean tags even when it carries the same epoch (a replayed
                    // CUDA graph freezes the epoch it was captured with).
                    for (int s = 0; s < kRing; ++s) p.ready[2 * ((size_t)bh * kRing + s)] = 0ull;
                    p.cons[bh] = 0ull;
                }
            } else if (lane == 0) {
                for (int c = 0; c < NT; ++c) {
                    const int b = c & 1;
                    if (!wait_bar(&bars[SB_SLOT_DONE0 + b], (c >> 1) & 1, tmo, abort_flag, 16u)) break;
                    if (c + 2 < NT) {
                        mbar_arrive_expect_tx(&bars[SB_RECV0 + b], kShipBytes);  // chunk c+2's shipment
                        // the pipeline that ships chunk c+2 of this head: item (c+2)*hce + rank
                        const int pp = ((c + 2) * hce + (int)rank) % (2 * nwy);
                        const uint32_t fb = sbase + W_BAR + 8 * (WB_PER_GROUP * (pp & 1) + WB_RECV_FREE0 + 2 * (int)rank + b);
                        mbar_arrive_remote(map_to_rank(fb, (uint32_t)(hc + (pp >> 1))));
                    }
                }
            }
        } else if (warp == 3) {
            // ------------------------------------------------------ W^T issuer
            // W^T = K^T Tw^T for each chunk as soon as its K and Tw are here, off
            // the state chain
            if (lane == 0) {
                const uint32_t idW = idesc_bf16(128, 64, true, false);
                for (int c = 0; c < NT; ++c) {
                    const int b = c & 1;
                    if (!wait_bar(&bars[SB_RECV0 + b], (c >> 1) & 1, tmo, abort_flag, 2u)) break;
                    if (!wait_bar(&bars[SB_FULLKQ0 + b], (c >> 1) & 1, tmo, abort_flag, 2u)) break;
                    if (c >= 1 && !wait_bar(&bars[SB_WT_READY], (c - 1) & 1, tmo, abort_flag, 2u)) break;
                    tc_fence_after_sync();
                    GDN_TR(c, 10);
                    const uint32_t kt = sbase + (b ? S_K1 : S_K0);
                    const uint32_t recv = sbase + S_RECV0 + b * RS;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ss(tmem + TM_W, smem_desc(kt + ks * 2048, 8192, 1024),
                                    smem_desc(recv + R_TW + ks * 32, 16, 1024), idW, ks > 0);
                    mma_commit(&bars[SB_W_DONE]);
                }
                mma_commit(&bars[SB_WDRAIN]);
                mbar_wait(&bars[SB_WDRAIN], 0, kCleanupNs);
            }
        } else if (warp >= 12 && warp < 16) {
            // ------------------------------------------------------ aux warps
            // W^T -> bf16 operand for each chunk, and the output rows of the
            // previous chunk, o_t = scale (qs_t O1_t + O2_t): each thread holds one
            // value index for all NQ queries, so a warp writes 64 contiguous bytes
            // of a row per store
            const int d = 32 * (warp & 3) + lane;  // TMEM lane: key index of W^T, value index of O^T
            const int ai = (warp - 12) * 32 + lane;
            const uint32_t lb = tmem_lane_base(warp);
            float *qsl = reinterpret_cast<float *>(sm + S_QS);
            auto out_tile = [&](int cc) {
                const int b = cc & 1;
                const uint32_t t1 = tmem + lb + (b ? TM_O11 : TM_O10);
                const uint32_t t2 = tmem + lb + (b ? TM_O21 : TM_O20);
                const float *qs = qsl + 64 * b;
                __nv_bfloat16 *orow = p.o + ((size_t)bh * p.T + (size_t)cc * NQ) * 128 + d;
                const int nrow = min(NQ, p.T - cc * NQ);
                static_assert(NQ >= 16, "at least one 16-column TMEM block per chunk");
                constexpr int NB = NQ >= 32 ? 2 : 1;  // 16-column blocks per TMEM wait
#pragma unroll
                for (int j0 = 0; j0 < NQ / 16; j0 += NB) {
                    uint32_t a[NB][16], e[NB][16];
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        tmem_ld16(t1 + 16 * (j0 + j), a[j]);
                        tmem_ld16(t2 + 16 * (j0 + j), e[j]);
                    }
                    tmem_wait_ld();
                    if (j0 + NB == NQ / 16) {
                        tc_fence_before_sync();
                        mbar_arrive(&bars[SB_OFREE0 + b]);  // O1/O2 columns of parity b may be overwritten
                    }
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int t = 16 * (j0 + j) + i;
                            const float o = p.scale * (qs[t] * __uint_as_float(a[j][i]) + __uint_as_float(e[j][i]));
                            if (t < nrow) orow[(size_t)t * 128] = __float2bfloat16_rn(o);
                        }
                    }
                }
            };
            bool ok = true;
            for (int c = 0; c < NT; ++c) {
                const int b = c & 1;
                bool w = wait_bar(&bars[SB_RECV0 + b], (c >> 1) & 1, tmo, abort_flag, 128u);
                if (w) w = wait_bar(&bars[SB_W_DONE], c & 1, tmo, abort_flag, 128u);
                if (w && c >= 1) w = wait_bar(&bars[SB_VN_DONE], (c - 1) & 1, tmo, abort_flag, 128u);
                if (!group_all(w, 4, 128)) { ok = false; break; }
                tc_fence_after_sync();
                // this chunk's per-query output scales, kept past the slot's release
                if (ai < NQ) qsl[64 * b + ai] = reinterpret_cast<const float *>(sm + S_RECV0 + b * RS + R_VEC)[V_QS + ai];
                uint32_t r[4][16];
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld16(tmem + lb + TM_W + 16 * j, r[j]);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) store16_sw128(sm + S_WT, d, 16 * j, r[j]);
                tc_fence_before_sync();
                fence_proxy_async_smem();
                mbar_arrive(&bars[SB_WT_READY]);
                if (ai == 0) GDN_TR(c, 7);
                if (c >= 1) {
                    // chunk c-1's MMAs (O1, O2) are complete with its slot's release
                    const bool wo = wait_bar(&bars[SB_SLOT_DONE0 + (b ^ 1)], ((c - 1) >> 1) & 1, tmo, abort_flag, 128u);
                    if (!group_all(wo, 4, 128)) { ok = false; break; }
                    tc_fence_after_sync();
                    if (ai == 0) GDN_TR(c, 8);
                    out_tile(c - 1);
                    if (ai == 0) GDN_TR(c, 9);
                }
            }
            if (ok && NT > 0) {
                const bool wo = wait_bar(&bars[SB_SLOT_DONE0 + ((NT - 1) & 1)], ((NT - 1) >> 1) & 1, tmo, abort_flag, 128u);
                if (group_all(wo, 4, 128)) {
                    tc_fence_after_sync();
                    out_tile(NT - 1);
                }
            }
        } else if (warp >= 4 && warp < 12) {
            // ------------------------------------------------------ scan epilogue
            const int sq = warp & 3, hh = (warp - 4) >> 2;
            const int dv = 32 * sq + lane;          // TMEM lane = value index
            const int si = (warp - 4) * 32 + lane;  // 0..255
            const uint32_t lb = tmem_lane_base(warp);
            {  // initial state: S^T[dv][dk] = S0[dk][dv], this thread's 64 columns
                const float *s0 = p.s0 ? p.s0 + (size_t)bh * 128 * 128 : nullptr;
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[16];
                    const int dk0 = 64 * hh + 16 * j;
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(s0 ? s0[(dk0 + i) * 128 + dv] : 0.f);
                    tmem_st16(tmem + lb + TM_S + dk0, r);
                }
                tmem_wait_st();
            }
            bool ok = true;
            for (int c = 0; c < NT; ++c) {
                const int b = c & 1;
                const float *vec = reinterpret_cast<const float *>(sm + S_RECV0 + b * RS + R_VEC);
                bool w = wait_bar(&bars[SB_RECV0 + b], (c >> 1) & 1, tmo, abort_flag, 4u);
                if (w && c >= 1) w = wait_bar(&bars[SB_UPD_DONE], (c - 1) & 1, tmo, abort_flag, 4u);
                if (!group_all(w, 3, 256)) { ok = false; break; }
                if (si == 0) GDN_TR(c, 3);
                tc_fence_after_sync();
                // state: S^T -> bf16 operand (K-block hh), signalled at once (Vn and
                // O1 read only the operand); then S^T <- exp(g_last) S^T in TMEM,
                // which only the state update (after VN_READY) needs
                const float el = vec[V_EL];
                {
                    uint32_t r[4][16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) tmem_ld16(tmem + lb + TM_S + 64 * hh + 16 * j, r[j]);
                    tmem_wait_ld();
                    uint8_t *blk = sm + S_ST + hh * 16384;
#pragma unroll
                    for (int j = 0; j < 4; ++j) store16_sw128(blk, dv, 16 * j, r[j]);
                    tc_fence_before_sync();
                    fence_proxy_async_smem();
                    mbar_arrive(&bars[SB_S_READY]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[j][i] = __float_as_uint(el * __uint_as_float(r[j][i]));
                        tmem_st16(tmem + lb + TM_S + 64 * hh + 16 * j, r[j]);
                    }
                }
                if (si == 0) GDN_TR(c, 4);
                // Vn^T -> bf16 operand and its decayed copy (columns 32hh..32hh+31)
                const bool wv = wait_bar(&bars[SB_VN_DONE], c & 1, tmo, abort_flag, 4u);
                if (!group_all(wv, 3, 256)) { ok = false; break; }
                if (si == 0) GDN_TR(c, 5);
                tc_fence_after_sync();
                {
                    const uint32_t tv = tmem + lb + TM_VN + 32 * hh;
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tv, r0);
                    tmem_ld16(tv + 16, r1);
                    tmem_wait_ld();
                    // the decayed copy first: the state update needs it (and the
                    // decayed state stored above); the plain copy is for O2 only
                    uint32_t e0[16], e1[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        e0[i] = __float_as_uint(vec[V_SEF + 32 * hh + i] * __uint_as_float(r0[i]));
                        e1[i] = __float_as_uint(vec[V_SEF + 32 * hh + 16 + i] * __uint_as_float(r1[i]));
                    }
                    store16_sw128(sm + S_VS, dv, 32 * hh, e0);
                    store16_sw128(sm + S_VS, dv, 32 * hh + 16, e1);
                    tmem_wait_st();
                    tc_fence_before_sync();
                    fence_proxy_async_smem();
                    mbar_arrive(&bars[SB_VN_READY]);
                    store16_sw128(sm + S_VN, dv, 32 * hh, r0);
                    store16_sw128(sm + S_VN, dv, 32 * hh + 16, r1);
                    fence_proxy_async_smem();
                    mbar_arrive(&bars[SB_VN2_READY]);
                }
                if (si == 0) GDN_TR(c, 6);
            }
            bool fin = ok && NT > 0 && wait_bar(&bars[SB_UPD_DONE], (NT - 1) & 1, tmo, abort_flag, 4u);
            if (group_all(fin, 3, 256)) {
                tc_fence_after_sync();
                if (p.sf) {
                    float *sf = p.sf + (size_t)bh * 128 * 128;
#pragma unroll 1
                    for (int j = 0; j < 4; ++j) {
                        uint32_t r[16];
                        const int dk0 = 64 * hh + 16 * j;
                        tmem_ld16(tmem + lb + TM_S + dk0, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) sf[(dk0 + i) * 128 + dv] = __uint_as_float(r[i]);
                    }
                }
            }
        }
    } else {
        // ================================================================== WY CTA
        {
            // ---------------------------------- WY pipeline g: warps 0..7 / 8..15.
            // Pipeline pidx = 2 (rank - hc) + g of the cluster (in ring mode, of
            // the grid) takes items pidx, pidx + 2 nwy, ...; item i is chunk
            // i / hce of head h0 + i % hce, shipped to that head's scan CTA.  One thread of warp 6
            // also loads K/Q with TMA and issues the K K^T / Q K^T MMA: the next
            // item's load starts as soon as this item's tile and TMEM rows have
            // been read, its MMA once this item's Tw / Tu are built.
            const int g = warp >> 3;
            const int wi = warp & 7;
            const int wt = wi * 32 + lane;  // 0..255
            const int q = warp & 3;         // TMEM lane quarter
            const int h = wi >> 2;          // column half of the 64-wide tiles
            const int bar_id = 1 + g;
            uint64_t *gb = bars + WB_PER_GROUP * g;
            uint8_t *gbase = sm + g * GS;
            uint8_t *kq = gbase + G_KQ;
            uint8_t *twu = gbase + G_TWU;
            float *AF = reinterpret_cast<float *>(gbase + G_AF);
            float *XS = reinterpret_cast<float *>(gbase + G_X);
            Misc *ms = reinterpret_cast<Misc *>(gbase + G_MISC);
            const uint32_t kqa = sbase + g * GS + G_KQ;
            const uint32_t idKQ = idesc_bf16(128, 64, false, false);
            const bool ctl = wt == 192;  // warp 6: not one of the diagonal-block warps
            const int nP = 2 * nwy, pidx = 2 * ((int)rank - hc) + g;  // pipelines of the cluster, this one
            const int nitems = NT * hce;
            int armed = 0, kq_issued = 0;  // control thread: TMA loads and KQ MMAs issued
            auto load_kq = [&](int item) {
                const int cc = item / hce, ibh = h0 + item % hce;
                mbar_arrive_expect_tx(&gb[WB_FULL], 16384 + 2 * NQ * 128);
                tma_load_3d(kq, &mK, &gb[WB_FULL], 0, cc * 64, ibh);
                tma_load_3d(kq + 16384, &mK, &gb[WB_FULL], 64, cc * 64, ibh);
                tma_load_3d(kq + 8192, &mQ, &gb[WB_FULL], 0, cc * NQ, ibh);
                tma_load_3d(kq + 16384 + 8192, &mQ, &gb[WB_FULL], 64, cc * NQ, ibh);
                armed++;
            };
            auto mma_kq = [&]() -> bool {
                if (!wait_bar(&gb[WB_FULL], kq_issued & 1, tmo, abort_flag, 32u)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a = kqa + (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16_ss(tmem + 128 * g, smem_desc(a, 16, 1024), smem_desc(a, 16, 1024), idKQ, ks > 0);
                }
                mma_commit(&gb[WB_KQ_DONE]);
                kq_issued++;
                return true;
            };
            bool kq_ok = true;  // control thread only
            if (ctl && pidx < nitems) {
                load_kq(pidx);
                kq_ok = mma_kq();
            }
            const uint32_t lb = tmem_lane_base(warp);
            const uint32_t tkq = tmem + 128 * g;
            const bool l2n = (p.flags & GDN_QK_L2NORM) != 0;
            // beta (warp 0) and g (warp 1) of rows lane and lane + 32 of a chunk are
            // loaded one chunk ahead; warp 1 turns g into the within-chunk
            // cumulative decay in registers at the end of the previous chunk, so
            // that the start of a chunk only stores them
            // The loads read clamped in-range addresses and nothing touches their
            // results until the values are used, so no thread waits on them here.
            float pf0 = 0.f, pf1 = 0.f;             // values of the current chunk
            uint32_t ld0 = 0, ld1 = 0;              // raw loads for the next chunk
            bool lv0 = false, lv1 = false;          // whether those rows exist
            auto prefetch = [&](int item) {
                const int cc = item / hce, ibh = h0 + item % hce;
                const unsigned short *betab = reinterpret_cast<const unsigned short *>(p.beta) + (size_t)ibh * p.rows;
                const uint32_t *gpb = reinterpret_cast<const uint32_t *>(p.g) + (size_t)ibh * p.T;
                const int r0 = cc * 64 + lane, r1 = r0 + 32;
                if (wi == 0) {
                    lv0 = r0 < p.rows;
                    lv1 = r1 < p.rows;
                    ld0 = betab[lv0 ? r0 : 0];
                    ld1 = betab[lv1 ? r1 : 0];
                } else if (wi == 1) {
                    lv0 = r0 < p.rows && r0 % R == 0;
                    lv1 = r1 < p.rows && r1 % R == 0;
                    ld0 = gpb[lv0 ? r0 / R : 0];
                    ld1 = gpb[lv1 ? r1 / R : 0];
                }
            };
            auto take = [&]() {  // the prefetched values, as floats
                if (wi == 0) {
                    pf0 = lv0 ? __uint_as_float(ld0 << 16) : 0.f;
                    pf1 = lv1 ? __uint_as_float(ld1 << 16) : 0.f;
                } else {
                    pf0 = lv0 ? __uint_as_float(ld0) : 0.f;
                    pf1 = lv1 ? __uint_as_float(ld1) : 0.f;
                }
            };
            int cs_safe = 1;
            float cs_el = 1.f;
            auto cumsum = [&]() {  // warp 1: g of rows lane / lane + 32 -> cumulative decay
                take();
                float a = pf0, b2 = pf1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float ya = __shfl_up_sync(0xffffffffu, a, off);
                    const float yb = __shfl_up_sync(0xffffffffu, b2, off);
                    if (lane >= off) { a += ya; b2 += yb; }
                }
                b2 += __shfl_sync(0xffffffffu, a, 31);
                const float g0 = __shfl_sync(0xffffffffu, a, 0);
                float dev = fmaxf(fabsf(a - g0), fabsf(b2 - g0));
#pragma unroll
                for (int off = 16; off; off >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, off));
                pf0 = a;
                pf1 = b2;
                cs_safe = dev <= 80.f ? 1 : 0;
                cs_el = __expf(b2);
            };
            if (pidx < nitems) {
                prefetch(pidx);
                if (wi == 0) take();
                if (wi == 1) cumsum();
            }
            uint32_t rf_par = 0;  // thread 0: parity of the next RECV_FREE phase, bit 2 * head + slot
            bool ship_ok = true;
            // The thread that ships: thread 0 into the cluster; in ring mode lane 0
            // of warp 5, which is idle while warps 0 and 1 form the chunk's factors
            // and publishes the previous shipment then.
            const bool shipper = flat ? wt == 160 : wt == 0;
            if (flat && shipper)
                for (int i = 0; i < kMaxRingHeads; ++i) ms->ccache[i] = 0u;
            int pend = -1, pend_tag = 0;  // ring mode, shipper: slot and tag still to publish
            // Publishing a slot: once its copies are complete, the ready tag goes
            // out as one more bulk copy (16 B from shared memory), which costs the
            // thread far less than a release store.
            auto publish = [&]() {
                if (pend >= 0) {
                    tma_store_wait_all<0>();  // the slot's bytes, and the previous tag, are written
                    ms->tag[0] = ((unsigned long long)p.epoch << 32) | (unsigned)pend_tag;
                    ms->tag[1] = 0ull;
                    fence_proxy_async_smem();
                    bulk_store_global(p.ready + 2 * pend, ms->tag, 16);
                    tma_store_commit();
                    pend = -1;
                }
            };
            for (int k = 0, it = pidx; it < nitems; ++k, it += nP) {
                const int c = it / hce, hh = it % hce;  // chunk c of the cluster's head hh
                const bool more = it + nP < nitems;     // this pipeline has a next item
                tr_on = blockIdx.x < (unsigned)(hc + nwy) && hh == 0;
                if (wt == 0) GDN_TR(c, 32 + 16 * g);
                // P and the vectors alternate between two buffers; the shipment of
                // chunk c-2 that last read this pair was waited for in chunk c-1
                uint8_t *ptile = gbase + G_PV + (k & 1) * 9216;
                float *vec = reinterpret_cast<float *>(ptile + 8192);
                // 1. beta, cumulative decay (published by the barrier below)
                if (wi == 0) {
                    if (k > 0) take();
                    ms->beta[lane] = pf0;
                    ms->beta[lane + 32] = pf1;
                } else if (wi == 1) {
                    ms->gam[lane] = pf0;
                    ms->gam[lane + 32] = pf1;
                    if (lane == 31) {
                        ms->safe = cs_safe;
                        vec[V_EL] = cs_el;
                    }
                }
                if (more) prefetch(it + nP);
                if (wt == 0) GDN_TR(c, 44 + 16 * g);
                const bool wk = wait_bar(&gb[WB_KQ_DONE], k & 1, tmo, abort_flag, 8u);
                if (wt == 0) GDN_TR(c, 45 + 16 * g);
                if (!group_all(wk && ship_ok && kq_ok, bar_id, 256)) break;  // also publishes beta, gam
                if (wt == 0) GDN_TR(c, 33 + 16 * g);
                tc_fence_after_sync();
                // 2. this thread's 32 columns of its K K^T (q < 2) or Q K^T (q >= 2) row
                float x[32];
                {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tkq + lb + 32 * h, r0);
                    tmem_ld16(tkq + lb + 32 * h + 16, r1);
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
                named_bar(bar_id, 256);  // n and partial q norms visible; K/Q tile and TMEM rows read
                if (ctl && kq_ok && more) load_kq(it + nP);
                if (wt == 0) GDN_TR(c, 34 + 16 * g);
                // per-row / per-column factors of the chunk
                if (wt < 64) {
                    const float g0 = ms->gam[0], gi = ms->gam[wt], gl = ms->gam[63];
                    const float ni = ms->n[wt];
                    const float mi = l2n ? rsqrtf(fmaxf(ms->qp[0][wt] + ms->qp[1][wt], 1e-24f)) : 1.f;
                    ms->m[wt] = mi;
                    ms->wsc[wt] = ms->beta[wt] * __expf(gi) * ni;
                    ms->bn[wt] = __expf(g0 - gi) * ni;
                    ms->ea[wt] = __expf(gi - g0);
                    vec[V_SEF + wt] = __expf(gl - gi) * ni;
                    vec[V_QS + wt] = wt < NQ ? __expf(ms->gam[wt * R + R - 1]) * mi : 0.f;
                } else if (flat && shipper) {
                    publish();  // the previous chunk's ring slot, while warps 0-1 form the factors
                }
                named_bar(bar_id, 256);
                if (wt == 0) GDN_TR(c, 35 + 16 * g);
                // 3. A rows (q < 2) and P rows (q >= 2)
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
                    if (t >= 32 && h == 0) {
                        // A[t][0..31] (all below the diagonal) as the merge's A1 operand
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const __nv_bfloat162 hv = __floats2bfloat162_rn(av[2 * i], av[2 * i + 1]);
                            const float2 hf2 = __bfloat1622float2(hv);
                            hi[i] = *reinterpret_cast<const uint32_t *>(&hv);
                            lo[i] = pack_bf16(av[2 * i] - hf2.x, av[2 * i + 1] - hf2.y);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            *reinterpret_cast<uint4 *>(gbase + G_A1 + sw128_offset(t - 32, 8 * j)) =
                                make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
                            *reinterpret_cast<uint4 *>(gbase + G_A1 + 4096 + sw128_offset(t - 32, 8 * j)) =
                                make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
                        }
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
                }
                named_bar(bar_id, 256);  // A complete
                if (wt == 0) GDN_TR(c, 36 + 16 * g);
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
                named_bar(bar_id, 256);
                if (wt == 0) GDN_TR(c, 37 + 16 * g);
                if (wt < 64) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) AF[(16 * db + i) * kAS + 16 * db + dc] = xs[i];
                }
                named_bar(bar_id, 256);
                {
                    // 16-level merges T_10 = -T_11 (A_10 T_00) (warps 0..3) and
                    // T_32 = -T_33 (A_32 T_22) (warps 4..7): rows rr and rr + 8 of the
                    // 16x16 block and column cl per thread, sharing each T / X load
                    const int hb = wi >> 2, rr = (wt >> 4) & 7, cl = wt & 15;
                    const int i0 = 32 * hb + 16, j0 = 32 * hb;
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const float tv = AF[(j0 + m) * kAS + j0 + cl];
                        a0 += AF[(i0 + rr) * kAS + j0 + m] * tv;
                        a1 += AF[(i0 + rr + 8) * kAS + j0 + m] * tv;
                    }
                    XS[(hb << 8) + rr * 16 + cl] = a0;
                    XS[(hb << 8) + (rr + 8) * 16 + cl] = a1;
                    named_bar(bar_id, 256);
                    float b0 = 0.f, b1 = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const float xv = XS[(hb << 8) + m * 16 + cl];
                        b0 += AF[(i0 + rr) * kAS + i0 + m] * xv;
                        b1 += AF[(i0 + rr + 8) * kAS + i0 + m] * xv;
                    }
                    AF[(i0 + rr) * kAS + j0 + cl] = -b0;
                    AF[(i0 + rr + 8) * kAS + j0 + cl] = -b1;
                    named_bar(bar_id, 256);
                }
                if (wt == 0) GDN_TR(c, 38 + 16 * g);
                // 32-level merge T_bl = -T_bot (A_bl T_top) on the tensor cores, each
                // product as hi*hi + hi*lo + lo*hi of bf16 halves (about 2^-16
                // relative), M = 64 with rows 32..63 used, into TMEM columns 64..127
                // of this pipeline.  First T_top and T_bot become operands (in the
                // Tw / Tu tile, which the previous shipment has left by then).
                {
                    const int which = wt >> 7, row = (wt >> 2) & 31, c8 = (wt & 3) * 8;
                    const float *src = &AF[(32 * which + row) * kAS + 32 * which + c8];
                    const float4 x0 = *reinterpret_cast<const float4 *>(src);
                    const float4 x1 = *reinterpret_cast<const float4 *>(src + 4);
                    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_bfloat162 hv = __floats2bfloat162_rn(xv[2 * i], xv[2 * i + 1]);
                        const float2 hf2 = __bfloat1622float2(hv);
                        hi[i] = *reinterpret_cast<const uint32_t *>(&hv);
                        lo[i] = pack_bf16(xv[2 * i] - hf2.x, xv[2 * i + 1] - hf2.y);
                    }
                    // T_top[row][c8..] is (k = row, n = c8..) of the MN-major B1; T_bot[row][c8..]
                    // is (m = 32 + row, k = c8..) of the K-major A2: the same offsets
                    uint8_t *opnd = gbase + (which ? G_A2 : G_B1);
                    if (shipper) tma_store_wait_read<0>();
                    named_bar(bar_id, 256);  // the previous shipment has left the Tw / Tu tile
                    *reinterpret_cast<uint4 *>(opnd + sw128_offset(row, c8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(opnd + 4096 + sw128_offset(row, c8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    fence_proxy_async_smem();
                    named_bar(bar_id, 256);
                }
                const uint32_t tinv = tmem + 128 * g + 64;
                const uint32_t gsb = sbase + g * GS;
                auto merge_mma = [&](uint32_t abase, uint32_t bbase) {
                    const uint32_t idM = idesc_bf16(64, 64, false, true);
                    int n = 0;
#pragma unroll
                    for (int hl = 0; hl < 3; ++hl) {
                        const uint32_t a = abase - 4096 + (hl == 2 ? 4096 : 0);  // hi, hi, lo (rows 32..63)
                        const uint32_t b = bbase + (hl == 1 ? 4096 : 0);         // hi, lo, hi
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            mma_bf16_ss(tinv, smem_desc(a + ks * 32, 16, 1024), smem_desc(b + ks * 2048, 8192, 1024),
                                        idM, (n++) > 0);
                    }
                    mma_commit(&gb[WB_INV]);
                };
                if (ctl) {
                    tc_fence_after_sync();
                    merge_mma(gsb + G_A1, gsb + G_B1);  // Y = A_bl T_top
                }
                // rows 32..63 of a product sit in TMEM lanes 64..79 and 96..111
                const bool rd = (wi == 2 || wi == 3) && lane < 16;
                const int mrow = 16 * (wi - 2) + lane;  // row of Y / T_bl within the bottom half
                bool ok_inv = true;
                if (wi == 2 || wi == 3) {
                    ok_inv = wait_bar(&gb[WB_INV], 0, tmo, abort_flag, 8u);
                    if (ok_inv) {
                        tc_fence_after_sync();
                        uint32_t r0[16], r1[16];
                        tmem_ld16(tinv + lb, r0);
                        tmem_ld16(tinv + lb + 16, r1);
                        tmem_wait_ld();
                        if (rd) {
                            // Y row mrow as row k = mrow of the MN-major B2 (hi, lo)
                            uint32_t hi[16], lo[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float y0 = __uint_as_float(i < 8 ? r0[2 * i] : r1[2 * i - 16]);
                                const float y1 = __uint_as_float(i < 8 ? r0[2 * i + 1] : r1[2 * i - 15]);
                                const __nv_bfloat162 hv = __floats2bfloat162_rn(y0, y1);
                                const float2 hf2 = __bfloat1622float2(hv);
                                hi[i] = *reinterpret_cast<const uint32_t *>(&hv);
                                lo[i] = pack_bf16(y0 - hf2.x, y1 - hf2.y);
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                *reinterpret_cast<uint4 *>(gbase + G_B2 + sw128_offset(mrow, 8 * j)) =
                                    make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
                                *reinterpret_cast<uint4 *>(gbase + G_B2 + 4096 + sw128_offset(mrow, 8 * j)) =
                                    make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
                            }
                        }
                        fence_proxy_async_smem();
                    }
                    tc_fence_before_sync();
                }
                if (!group_all(ok_inv, bar_id, 256)) break;
                if (ctl) {
                    tc_fence_after_sync();
                    merge_mma(gsb + G_A2, gsb + G_B2);  // T_bot Y
                }
                if (wi == 2 || wi == 3) {
                    ok_inv = wait_bar(&gb[WB_INV], 1, tmo, abort_flag, 8u);
                    if (ok_inv) {
                        tc_fence_after_sync();
                        uint32_t r0[16], r1[16];
                        tmem_ld16(tinv + lb, r0);
                        tmem_ld16(tinv + lb + 16, r1);
                        tmem_wait_ld();
                        if (rd) {
                            float *trow = &AF[(32 + mrow) * kAS];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                *reinterpret_cast<float4 *>(trow + 4 * j) =
                                    make_float4(-__uint_as_float(r0[4 * j]), -__uint_as_float(r0[4 * j + 1]),
                                                -__uint_as_float(r0[4 * j + 2]), -__uint_as_float(r0[4 * j + 3]));
                                *reinterpret_cast<float4 *>(trow + 16 + 4 * j) =
                                    make_float4(-__uint_as_float(r1[4 * j]), -__uint_as_float(r1[4 * j + 1]),
                                                -__uint_as_float(r1[4 * j + 2]), -__uint_as_float(r1[4 * j + 3]));
                            }
                        }
                    }
                    tc_fence_before_sync();
                }
                if (!group_all(ok_inv, bar_id, 256)) break;
                if (wt == 0) GDN_TR(c, 40 + 16 * g);
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
                named_bar(bar_id, 256);
                if (wt == 0) GDN_TR(c, 41 + 16 * g);
                // K K^T / Q K^T of the next chunk (its load has had the whole chunk)
                if (ctl && kq_ok && more) {
                    GDN_TR(c, 46 + 16 * g);
                    kq_ok = mma_kq();
                }
                if (wi == 1 && more) cumsum();
                // 6. ship Tw, Tu, P and the vectors into slot c & 1 of head hh's scan
                //    CTA (cluster rank hh), once that head's chunk c-2 has left it
                if (shipper && flat) {
                    // ring mode: into slot c % kRing of the head's ring, once its
                    // scan CTA has taken chunk c - kRing out of it (known without a
                    // global load while the last count seen suffices); the ready tag
                    // follows in the next chunk, when the copies are complete
                    const int ibh = h0 + hh;
                    const unsigned need = (unsigned)(c - kRing + 1);
                    if (c >= kRing && ms->ccache[ibh] < need) {
                        unsigned seen = 0;
                        ship_ok = wait_tag(p.cons + ibh, p.epoch, need, tmo, abort_flag, 512u, &seen);
                        if (ship_ok) ms->ccache[ibh] = seen;
                    }
                    GDN_TR(c, 47 + 16 * g);
                    if (ship_ok) {
                        fence_proxy_async_global();
                        const int slot = ibh * kRing + c % kRing;
                        uint8_t *dst = p.ring + (size_t)slot * kShipBytes;
                        bulk_store_global(dst, twu, 16384);
                        bulk_store_global(dst + 16384, ptile, 8192 + 1024);
                        tma_store_commit();
                        pend = slot;
                        pend_tag = c + 1;
                    }
                    GDN_TR(c, 42 + 16 * g);
                } else if (shipper) {  // cluster mode: thread 0
                    const int sl = c & 1, fbit = 2 * hh + sl;
                    if (c >= 2) {
                        ship_ok = wait_bar(&gb[WB_RECV_FREE0 + fbit], (rf_par >> fbit) & 1u, tmo, abort_flag, 64u, true);
                        rf_par ^= 1u << fbit;
                    }
                    GDN_TR(c, 47 + 16 * g);
                    if (ship_ok) {
                        // the scan CTA armed its receive barrier for these bytes
                        const uint32_t recv = sbase + S_RECV0 + sl * RS;
                        const uint32_t rb = map_to_rank(sbase + S_BAR + 8 * (SB_RECV0 + sl), (uint32_t)hh);
                        bulk_copy_to_peer(map_to_rank(recv + R_TW, (uint32_t)hh), twu, 16384, rb);
                        bulk_copy_to_peer(map_to_rank(recv + R_P, (uint32_t)hh), ptile, 8192 + 1024, rb);
                        tma_store_commit();
                    }
                    GDN_TR(c, 42 + 16 * g);
                }
            }
            if (shipper) {
                tma_store_wait_all<0>();
                if (flat) publish();
            }
            if (ctl) {
                mma_commit(&gb[WB_DRAIN]);
                mbar_wait(&gb[WB_DRAIN], 0, kCleanupNs);
                if (armed) mbar_wait(&gb[WB_FULL], (armed - 1) & 1, kCleanupNs);
            }
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    if (flat)
        __syncthreads();
    else
        cluster_sync_all();  // no CTA leaves while its peer may still touch its shared memory
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, ncols);
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

// Cluster shape for BH heads: hc heads (scan CTAs) and nwy WY CTAs per cluster,
// one CTA per SM.  Among the shapes whose clusters are all resident at once, the
// most WY pipelines per head (2 nwy / hc, counted up to 4, past which the state
// chain is the limit) wins; then two heads per cluster, then three, one, four
// (with two, a head's chunks alternate between two WY CTAs that also serve
// another head, which measured fastest: B4 H16 T4096 0.201 ms against 0.233 ms
// for one head per cluster on the same 128 SMs); then the fewest SMs.  With too
// many heads for one wave, one WY CTA per head.  Cached per head count and device.
template <int R>
bool pick_shape(int BH, int *hc_out, int *nwy_out) {
    static std::mutex mu;
    static int cache_dev[16], cache_bh[16], cache_hc[16], cache_nwy[16], cache_n = 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < cache_n; ++i)
        if (cache_dev[i] == dev && cache_bh[i] == BH) {
            *hc_out = cache_hc[i];
            *nwy_out = cache_nwy[i];
            return true;
        }
    static const int kPref[kMaxHc + 1] = {0, 2, 4, 3, 1};  // preference among equal pipeline counts
    int best_hc = 1, best_nwy = 1, best_q = -1, best_pref = -1, best_sms = 1 << 30;
    for (int hc = 1; hc <= kMaxHc; ++hc) {
        for (int nwy = 1; hc + nwy <= 16; ++nwy) {
            const int clusters = (BH + hc - 1) / hc, need = clusters * (hc + nwy);
            if (need > sms) continue;
            const int q = std::min(8 * nwy / hc, 16);  // 4x WY pipelines per head, capped at 4
            if (q < best_q) continue;
            if (q == best_q && (kPref[hc] < best_pref || (kPref[hc] == best_pref && need >= best_sms))) continue;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            cfg.gridDim = dim3((unsigned)need);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmemBytes;
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)(hc + nwy);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int resident = 0;
            if (cudaOccupancyMaxActiveClusters(&resident, gdn_tc_kernel<R>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                continue;
            }
            if (resident < clusters) continue;
            best_hc = hc;
            best_nwy = nwy;
            best_q = q;
            best_pref = kPref[hc];
            best_sms = need;
        }
    }
    if (cache_n < 16) {
        cache_dev[cache_n] = dev;
        cache_bh[cache_n] = BH;
        cache_hc[cache_n] = best_hc;
        cache_nwy[cache_n] = best_nwy;
        ++cache_n;
    }
    *hc_out = best_hc;
    *nwy_out = best_nwy;
    return true;
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

// Ring mode serves up to half as many heads as there are SMs: each head gets a
// scan CTA, and the other SMs, at least as many, run WY CTAs for all heads.
bool ring_fits(int BH, int sms) { return BH >= 1 && BH <= kMaxRingHeads && 2 * BH <= sms; }

constexpr size_t ring_bytes(int BH) {
    return (size_t)BH * kRing * kShipBytes + (size_t)BH * kRing * 16 + (size_t)BH * sizeof(unsigned long long);
}

// Scratch of the allocation-free entry point: the ring of up to kNoAllocHeads
// heads (13.1 MB on every GPU that loads the library, until the process
// exits).  It is zero when the module loads and is never cleared: each tag in
// it carries the launch that wrote it, so one call's leftovers are never read
// as another's.
constexpr int kNoAllocHeads = 64;
constexpr size_t kNoAllocBytes = ring_bytes(kNoAllocHeads);
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

std::atomic<unsigned> g_epoch{0};

// Launches the ring mode if it applies (no forced cluster shape, few enough
// heads, a 16-byte aligned workspace of ring_bytes); returns -1 if it does not.
template <int R>
int launch_ring(const ScanArgs &a, TcParams p, const CUtensorMap &mK, const CUtensorMap &mQ, const CUtensorMap &mV,
                cudaStream_t stream) {
    const int BH = p.BH, sms = sm_count();
    if (g_force_hc > 0 || !ring_fits(BH, sms) || a.ws == nullptr || a.ws_bytes < ring_bytes(BH) ||
        (reinterpret_cast<uintptr_t>(a.ws) & 15u) != 0)
        return -1;
    auto kern = gdn_tc_kernel<R>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    // WY CTAs: three pipelines per head (past which the state chain is the
    // limit), on the SMs the scan CTAs leave
    const int nwy = std::max(1, std::min(per_sm * sms - BH, (3 * BH + 1) / 2));
    if (per_sm < 1 || BH + nwy > per_sm * sms) return -1;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    p.flat = 1;
    p.hc = BH;
    p.nwy = nwy;
    p.ring = ws;
    p.ready = reinterpret_cast<unsigned long long *>(ws + (size_t)BH * kRing * kShipBytes);
    p.cons = p.ready + (size_t)BH * kRing * 2;
    unsigned e = ++g_epoch;
    if (e == 0) e = ++g_epoch;
    p.epoch = e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(BH + nwy));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeCooperative;  // scan and WY CTAs wait on one another
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mK, mQ, mV, p) != cudaSuccess) return GDN_ERR_CUDA;
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <int R>
int launch_r(const ScanArgs &a, cudaStream_t stream) {
    constexpr int NQ = 64 / R;
    const long rows = (long)a.T * R;
    const int BH = a.B * a.H;
    CUtensorMap mK, mQ, mV;
    if (!make_map(&mK, a.k, BH, rows, 64, 64, true) || !make_map(&mQ, a.q, BH, a.T, 64, NQ, true) ||
        !make_map(&mV, a.v, BH, rows, 64, 64, true))
        return GDN_ERR_CUDA;
    TcParams p;
    p.beta = static_cast<const __nv_bfloat16 *>(a.beta);
    p.g = a.g;
    p.s0 = a.s0;
    p.sf = a.sf;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.T = a.T;
    p.rows = (int)rows;
    p.NT = (int)((rows + 63) / 64);
    p.scale = a.scale;
    p.flags = a.flags;
    p.timeout_ns = g_timeout_ns;
    p.BH = BH;
    p.flat = 0;
    p.ring = nullptr;
    p.ready = p.cons = nullptr;
    p.epoch = 0;
    auto kern = gdn_tc_kernel<R>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return GDN_ERR_CUDA;
    const int rs = launch_ring<R>(a, p, mK, mQ, mV, stream);
    if (rs >= 0) return rs;
    int hc = 1, nwy = 1;
    if (g_force_hc > 0) {
        hc = g_force_hc;
        nwy = g_force_nwy;
    } else if (!pick_shape<R>(BH, &hc, &nwy)) {
        return GDN_ERR_CUDA;
    }
    p.BH = BH;
    p.hc = hc;
    p.nwy = nwy;
    const int clusters = (BH + hc - 1) / hc;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(clusters * (hc + nwy)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)(hc + nwy);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mK, mQ, mV, p) != cudaSuccess) return GDN_ERR_CUDA;
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool make_bf16_map(CUtensorMap *m, const void *base, int heads, long rows, int box0, int box1) {
    return make_map(m, base, heads, rows, box0, box1, true);
}

bool make_bf16_frame_map(CUtensorMap *m, const void *base, int heads, int frames, int frame_rows, int box0,
                         int box1) {
    return make_bf16_frame_map_wide(m, base, heads, frames, frame_rows, 128, box0, box1);
}

bool make_bf16_frame_map_wide(CUtensorMap *m, const void *base, int outer, int frames, int frame_rows, int cols,
                              int box0, int box1) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t rb = (cuuint64_t)cols * 2;  // bytes per row
    cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)frame_rows, (cuuint64_t)frames, (cuuint64_t)outer};
    cuuint64_t strides[3] = {rb, (cuuint64_t)frame_rows * rb, (cuuint64_t)frame_rows * frames * rb};
    cuuint32_t box[4] = {(cuuint32_t)box0, (cuuint32_t)box1, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool sm100_family() {
    static int sm100 = -1;
    if (sm100 < 0) sm100 = device_is_sm100_family() ? 1 : 0;
    return sm100 == 1;
}

int device_sm_count() { return sm_count(); }

bool scan_tc_supported(const ScanArgs &a) {
    if (a.flags & GDN_PATH_SIMT) return false;
    if (a.dtype != GDN_BF16 || a.Dk != 128 || a.Dv != 128 || a.chunk != 64) return false;
    if (a.r != 1 && a.r != 2 && a.r != 4) return false;
    if ((long long)a.T * a.r > (1LL << 30)) return false;
    return sm100_family();
}

size_t scan_tc_workspace_bytes(const ScanArgs &a) {
    const int BH = a.B * a.H;
    return ring_fits(BH, sm_count()) ? ring_bytes(BH) : 0;
}

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

int scan_tc_noalloc_scratch(void **ptr, size_t *bytes) {
    // the device address of g_noalloc_scratch, looked up once per device with
    // that device current (its host-side name is not a device address)
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GDN_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *ptr = addr[dev];
    *bytes = kNoAllocBytes;
    return GDN_OK;
}

int scan_tc_set_cluster_shape(int hc, int nwy) {
    if (hc == 0 && nwy == 0) {
        g_force_hc = g_force_nwy = 0;
        return GDN_OK;
    }
    if (hc < 1 || hc > kMaxHc || nwy < 1 || hc + nwy > 16) return GDN_ERR_INVALID_ARG;
    g_force_hc = hc;
    g_force_nwy = nwy;
    return GDN_OK;
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

unsigned long long wait_limit_ns() { return g_timeout_ns; }

}  // namespace gdn
