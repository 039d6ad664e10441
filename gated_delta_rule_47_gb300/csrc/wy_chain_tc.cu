// wy_chain_tc.cu -- the sequential state chains of the chunkwise WY form on
// tcgen05, for Dk = Dv = 128 and 64-row chunks (gated_deltaproduct test.py:
// the state loop of `gated_chunk_delta_rule_fwd_kernel_h` forward and of
// `gated_chunk_delta_rule_bwd_kernel_dhu` in reverse).  One CTA per head and
// chain:
//   forward:  Vn = U - W S,  S <- e^{gl} S + Kd^T Vn    (S entering each chunk and Vn kept)
//   reverse:  dS <- e^{gl} dS' - W^T (Kd dS') + B_c     (dS' leaving each chunk kept)
// The state lives in tensor memory as X^T (128 value lanes x 128 key columns,
// fp32).  Per chunk:
//   1. eight epilogue warps read X^T, write it out (the chunk's snapshot),
//      split it into bf16 hi + lo operand tiles in shared memory, and put
//      e^{gl} X^T (+ B_c^T on the reverse chain) back;
//   2. one thread issues Z^T = X^T M1^T (M1 = W forward, Kd reverse) as the
//      products hi.hi + hi.lo + lo.hi (24 MMAs, M = 128, N = 64);
//   3. the epilogue warps read Z^T, form Vn = U - Z (forward, written out) or
//      Y = Z (reverse), and split it into hi + lo operand tiles;
//   4. the thread issues X^T += Z'^T M2 (forward, M2 = Kd) or X^T -= Z'^T M2
//      (reverse, M2 = W), again as three products (12 MMAs, N = 128).
// The split products carry about 2^-16 relative error, against 2^-8 for a
// plain bf16 product.  W and Kd arrive as bf16 hi | lo operand images written
// by the WY kernels (wy_chain.cuh, write_chain_image), two 32 KB bulk copies
// per chunk, double-buffered.  Every wait is bounded; a CTA that gives up sets
// the error word, which gdn_get_device_error reads.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_internal.h"
#include "tc_util.cuh"
#include "tri_inverse.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kRows = 64;    // rows of a chunk
constexpr int kCThr = 384;   // warp 0 issues, warp 1 holds TMEM, warp 2 loads, warps 4..11 epilogue
constexpr uint32_t C_SLOT = 65536;         // one chunk's W hi | W lo | Kd hi | Kd lo, 16 KB each
constexpr uint32_t C_XOP = 2 * C_SLOT;     // X^T hi | lo: K-major [2 key blocks][128 value rows][128 B]
constexpr uint32_t C_ZOP = C_XOP + 65536;  // Z'^T hi | lo: K-major [128 value rows][128 B]
constexpr uint32_t C_BAR = C_ZOP + 32768;
enum { CB_FULL = 0, CB_FREE = 2, CB_XREADY = 4, CB_ZDONE, CB_ZREADY, CB_XDONE, CB_DRAIN, CB_NUM };
constexpr uint32_t C_TSLOT = C_BAR + 8 * CB_NUM;
constexpr uint32_t C_SMEM = C_TSLOT + 16 + 1024;  // + slack to align the base to 1024 bytes
static_assert(C_SMEM <= 232448, "chain kernel fits the shared memory of one CTA");
constexpr uint32_t TM_X = 0, TM_Z = 128, kTmemCols = 256;

__device__ unsigned int g_wyc_error = 0;  // set when a bounded wait of the chain kernel gives up
constexpr unsigned long long kWycDrainNs = 200000000ull;

// Waits for the phase of the given parity for at most limit ns; gives up at
// once when another CTA has set the error word.
__device__ __forceinline__ bool wyc_wait(uint64_t *bar, uint32_t parity, unsigned code, unsigned long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile unsigned *>(&g_wyc_error) != 0u) return false;
        if (global_timer_ns() - t0 > limit) {
            atomicOr(&g_wyc_error, code);
            return false;
        }
    }
}

// A wait's outcome made uniform across the warp, so that the warp's
// .sync.aligned TMEM accesses that follow are reached by all of its lanes.
__device__ __forceinline__ bool warp_ok(bool ok) { return __all_sync(0xffffffffu, ok) != 0; }

// x[0..7] as bf16 hi and lo = x - hi, 16 bytes each
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = pack_bf16(x[2 * i], x[2 * i + 1]);
        l[i] = pack_bf16(x[2 * i] - __uint_as_float(h[i] << 16), x[2 * i + 1] - __uint_as_float(h[i] & 0xffff0000u));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(kCThr, 1) wy_chain_tc_kernel(WyChainTcArgs p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C_TSLOT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, role = blockIdx.y, NT = p.NT;
    const size_t ci0 = (size_t)bh * NT;
    const unsigned long long tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < CB_NUM; ++i) mbar_init(&bars[i], (i == CB_XREADY || i == CB_ZREADY) ? 256u : 1u);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idZ = idesc_bf16(128, 64, false, false);
            const uint32_t idX = idesc_bf16(128, 128, false, true, role == 1);
            const uint32_t m1 = role == 0 ? 0u : 32768u, m2 = role == 0 ? 32768u : 0u;
            for (int s = 0; s < NT; ++s) {
                const int b = s & 1;
                const uint32_t slot = sb + (uint32_t)b * C_SLOT;
                if (!wyc_wait(&bars[CB_FULL + b], (s >> 1) & 1, 1u, tmo)) break;
                if (!wyc_wait(&bars[CB_XREADY], s & 1, 1u, tmo)) break;
                tc_fence_after_sync();
                // Z^T = X^T M1^T over the 128 keys: hi.hi, hi.lo, lo.hi
#pragma unroll
                for (int pr = 0; pr < 3; ++pr) {
                    const uint32_t xa = sb + C_XOP + (pr == 2 ? 32768u : 0u);
                    const uint32_t mb = slot + m1 + (pr == 1 ? 16384u : 0u);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ss(tmem + TM_Z, smem_desc(xa + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                    smem_desc(mb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), idZ,
                                    (pr | ks) != 0);
                }
                mma_commit(&bars[CB_ZDONE]);
                if (!wyc_wait(&bars[CB_ZREADY], s & 1, 1u, tmo)) break;
                tc_fence_after_sync();
                // X^T +/-= Z'^T M2 over the 64 rows
#pragma unroll
                for (int pr = 0; pr < 3; ++pr) {
                    const uint32_t za = sb + C_ZOP + (pr == 2 ? 16384u : 0u);
                    const uint32_t nb = slot + m2 + (pr == 1 ? 16384u : 0u);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ss(tmem + TM_X, smem_desc(za + ks * 32, 16, 1024), smem_desc(nb + ks * 2048, 8192, 1024),
                                    idX, 1u);
                }
                mma_commit(&bars[CB_XDONE]);
                mma_commit(&bars[CB_FREE + b]);
            }
            mma_commit(&bars[CB_DRAIN]);
            mbar_wait(&bars[CB_DRAIN], 0, kWycDrainNs);
        }
    } else if (warp == 2) {
        // ----------------------------------------- W and Kd images, bulk copies
        if (lane == 0) {
            int armed[2] = {0, 0};
            for (int s = 0; s < NT; ++s) {
                const int b = s & 1;
                // slot b held chunk s-2, whose MMAs are complete when CB_FREE + b completes
                if (s >= 2 && !wyc_wait(&bars[CB_FREE + b], ((s - 2) >> 1) & 1, 2u, tmo)) break;
                const size_t ci = ci0 + (size_t)(role == 0 ? s : NT - 1 - s);
                mbar_arrive_expect_tx(&bars[CB_FULL + b], 65536u);
                bulk_load_global(sm + b * C_SLOT, p.Wimg + ci * 32768, 32768u, &bars[CB_FULL + b]);
                bulk_load_global(sm + b * C_SLOT + 32768, p.Kdimg + ci * 32768, 32768u, &bars[CB_FULL + b]);
                armed[b]++;
            }
            for (int b = 0; b < 2; ++b)
                if (armed[b]) mbar_wait(&bars[CB_FULL + b], (armed[b] - 1) & 1, kWycDrainNs);
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------- epilogue
        // thread = value index dv (its TMEM lane); hh picks the half of the key
        // columns of X^T (and of the rows of Z^T) it handles
        const int q = warp & 3, hh = (warp - 4) >> 2;
        const int dv = 32 * q + lane;
        const uint32_t lb = (uint32_t)(32 * q) << 16;
        const float *init = role == 0 ? p.s0 : p.dsf;
        float *snap = role == 0 ? p.Sw : p.dSw;
        bool ok = true;
        for (int s = 0; s < NT; ++s) {
            const size_t ci = ci0 + (size_t)(role == 0 ? s : NT - 1 - s);
            const float el = expf(p.Gw[ci * kRows + kRows - 1]);
            // forward: U[t][dv] for the rows 32hh..32hh+31; reverse: B[dk][dv] for
            // the keys 64hh..64hh+63 (loaded ahead of the waits)
            float pre[64];
            if (role == 0) {
                const float *Ug = p.Uw + ci * (kRows * 128) + (size_t)(32 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 32; ++i) pre[i] = Ug[(size_t)i * 128];
            } else {
                const float *Bg = p.Bw + ci * 16384 + (size_t)(64 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 64; ++i) pre[i] = Bg[(size_t)i * 128];
            }
            float x[64];
            if (s == 0) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    x[i] = init ? init[((size_t)bh * 128 + 64 * hh + i) * 128 + dv] : 0.f;
            } else {
                ok = warp_ok(wyc_wait(&bars[CB_XDONE], (s - 1) & 1, 4u, tmo));
                if (!ok) break;
                tc_fence_after_sync();
                uint32_t r[4][16];
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld16(tmem + lb + TM_X + 64 * hh + 16 * j, r[j]);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[16 * j + i] = __uint_as_float(r[j][i]);
            }
            {  // the snapshot, and X^T as its hi | lo operand (key block hh)
                float *sn = snap + ci * 16384 + (size_t)(64 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 64; ++i) sn[(size_t)i * 128] = x[i];
                uint8_t *xo = sm + C_XOP + hh * 16384;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 hi, lo;
                    split8(x + 8 * c, hi, lo);
                    const uint32_t off = sw128_offset((uint32_t)dv, (uint32_t)(8 * c));
                    *reinterpret_cast<uint4 *>(xo + off) = hi;
                    *reinterpret_cast<uint4 *>(xo + 32768 + off) = lo;
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bars[CB_XREADY]);
            }
            // e^{gl} X^T (+ B^T) back into TMEM for the update (the Z product
            // reads only the operand tiles)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    r[i] = __float_as_uint(role == 0 ? el * x[16 * j + i] : el * x[16 * j + i] + pre[16 * j + i]);
                tmem_st16(tmem + lb + TM_X + 64 * hh + 16 * j, r);
            }
            ok = warp_ok(wyc_wait(&bars[CB_ZDONE], s & 1, 4u, tmo));
            if (!ok) break;
            tc_fence_after_sync();
            float z[32];
            {
                uint32_t r[2][16];
                tmem_ld16(tmem + lb + TM_Z + 32 * hh, r[0]);
                tmem_ld16(tmem + lb + TM_Z + 32 * hh + 16, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(r[i >> 4][i & 15]);
            }
            if (role == 0) {  // Vn = U - W S, kept
                float *Vg = p.Vnw + ci * (kRows * 128) + (size_t)(32 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    z[i] = pre[i] - z[i];
                    Vg[(size_t)i * 128] = z[i];
                }
            } else if (p.Yw) {
                // Y = Kd dS', kept for the gradient kernel over this chunk's B, which every
                // thread loaded before arriving on CB_XREADY (ordered before this write)
                float *Yg = p.Yw + ci * 16384 + (size_t)(32 * hh) * 128 + dv;
#pragma unroll
                for (int i = 0; i < 32; ++i) Yg[(size_t)i * 128] = z[i];
            }
            {  // Z'^T as its hi | lo operand (rows 32hh.. of the chunk)
                uint8_t *zo = sm + C_ZOP;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 hi, lo;
                    split8(z + 8 * c, hi, lo);
                    const uint32_t off = sw128_offset((uint32_t)dv, (uint32_t)(32 * hh + 8 * c));
                    *reinterpret_cast<uint4 *>(zo + off) = hi;
                    *reinterpret_cast<uint4 *>(zo + 16384 + off) = lo;
                }
            }
            tmem_wait_st();  // the decayed state is in place before the update reads it
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bars[CB_ZREADY]);
        }
        float *out = role == 0 ? p.sf : p.ds0;
        if (ok && NT > 0) {
            ok = warp_ok(wyc_wait(&bars[CB_XDONE], (NT - 1) & 1, 4u, tmo));
            if (ok && out) {
                tc_fence_after_sync();
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lb + TM_X + 64 * hh + 16 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        out[((size_t)bh * 128 + 64 * hh + 16 * j + i) * 128 + dv] = __uint_as_float(r[i]);
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int launch_wy_chain_tc(const WyChainTcArgs &a, cudaStream_t st) {
    if (a.BH <= 0 || a.NT <= 0 || a.roles < 1 || a.roles > 2) return GDN_ERR_INVALID_ARG;
    WyChainTcArgs p = a;
    p.timeout_ns = wait_limit_ns();
    if (cudaFuncSetAttribute(wy_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    wy_chain_tc_kernel<<<dim3((unsigned)a.BH, (unsigned)a.roles), kCThr, C_SMEM, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int wy_chain_tc_read_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_wyc_error, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_wyc_error, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
    return v ? GDN_ERR_TIMEOUT : GDN_OK;
}


// ======================= the state products of the gradient kernels (tcgen05)
// chunk_products_tc_kernel: per (head, chunk), after both chains, with S the
// state entering the chunk, dS' the gradient leaving it, Vn [64][128], the
// chunk's nq query rows of dO (bf16), P^ and T [64][64] from the WY kernel
// and Y = Kd dS' from the reverse chain, four batches of MMAs (M = 128):
//   1. Z^T = dS' Vn^T and t1^T = S dO^T, Yw^T = dO^T P^ and DOV = dO Vn^T;
//   2. dR^T = dVn^T T, with dVn^T = Y^T + Yw^T as a K-major operand;
//   3. dR Vn^T (dR^T's image read as an MN-major operand) and t2^T = S dR^T;
//   4. X1^T = Q^T P~ + Kr^T L, X2^T = Kw^T L^T and (P~ Kw)^T, with P~ formed
//      from DOV and L from dR Vn^T (both decay-masked, as the gradient kernels
//      define them) and the unit-normalised queries and keys.
// Each fp32 operand is split into bf16 hi | lo tiles (hi.hi + hi.lo + lo.hi,
// about 2^-16 relative; two terms where the other operand, dO, is exact).
// P~ and L serve as MN-major operands (rows K) and as K-major ones (rows N) in
// the same bytes.  The results go over slots that nothing reads afterwards
// (the layout is listed with ChunkProductsTcArgs).
namespace {

constexpr int kCpThr = 512;
constexpr int kCpCG = kCpThr / 128, kCpCW = 64 / kCpCG;  // epilogue column groups (warp / 4), columns of each
constexpr uint32_t CP_S = 0;          // S hi | lo: [2 value blocks][128 key rows][128 B], 32 KB each;
                                      //   batch 4: Kr hi | lo [2 key blocks][64 rows][128 B] (at 0), Kw (at 32768)
constexpr uint32_t CP_DS = 65536;     // dS' hi | lo, likewise; after batch 1 dVn^T hi | lo [128 value rows][128 B],
                                      //   after batch 2 Q hi | lo [2 key blocks][64 rows][128 B]
constexpr uint32_t CP_DR = 98304;     // dR^T hi | lo [128 value rows][128 B] (over dS' lo)
constexpr uint32_t CP_VN = 131072;    // Vn hi | lo: [2 value blocks][64 rows][128 B], 16 KB each
constexpr uint32_t CP_DO = 163840;    // dO: [2 value blocks][nq2 rows][128 B], 16 KB at most; then P~ hi | lo [64 rows][128 B]
constexpr uint32_t CP_P = 180224;     // P^ hi | lo as an MN-major operand: [64 query rows][128 B]; then L hi | lo
constexpr uint32_t CP_T = 196608;     // T hi | lo as an MN-major operand: [64 rows][128 B], 8 KB each
constexpr uint32_t CP_BAR = 212992;   // 4 mbarriers
constexpr uint32_t CP_VEC = CP_BAR + 32;   // gamma, beta (per sub-row), n (per sub-row), m (per query), mask
constexpr uint32_t CP_MISC = CP_VEC + 5 * 256;  // TMEM address, then the warps' sums
constexpr uint32_t CP_SMEM = CP_MISC + 16 + 4 * (kCpThr / 32) + 1024;
// The M = 128 products whose operand has fewer than 128 rows read past it for
// the rest (the next block or region, or stale staging); those rows of the
// product are not used.
static_assert(CP_DR + 32768 == CP_VN && CP_VN + 32768 == CP_DO && CP_T + 16384 <= CP_BAR, "products map");
constexpr uint32_t CT_Z = 0, CT_T1 = 64, CT_YW = 128, CT_DOV = 192, CT_DR = 256, CT_DA = 320, CT_T2 = 384;
constexpr uint32_t CT_X1 = 64, CT_X2 = 128, CT_DQ = 192;  // batch 4, over columns read in batch 1's epilogue

__device__ __forceinline__ float sum16p(float x) {  // over the 16 lanes that differ in bits 0..3
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void unpack8p(const uint4 &w, float *x) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 ldg16p(const unsigned short *p) { return *reinterpret_cast<const uint4 *>(p); }

template <bool MASKED>
__global__ void __launch_bounds__(kCpThr, 1) chunk_products_tc_kernel(ChunkProductsTcArgs p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + CP_BAR);
    float *gam = reinterpret_cast<float *>(sm + CP_VEC), *bet = gam + 64, *nk = bet + 64, *mq = nk + 64, *msk = mq + 64;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + CP_MISC);
    float *wsum = reinterpret_cast<float *>(sm + CP_MISC + 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q4 = warp & 3, cg = warp >> 2;
    const uint32_t lb = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
    const int c = blockIdx.x, bh = blockIdx.y, r = p.r;
    const size_t ci = (size_t)bh * p.NT + c;
    const int nq2 = p.nq2;  // query rows of the dO products (a multiple of 16; rows past the chunk are zero)
    const int t0 = c * p.Ct, ntok = min(p.Ct, p.T - t0), nrows = ntok * r;
    const size_t htok = (size_t)bh * p.T + t0, hrow = htok * r;
    float *Sg = p.Sw + ci * 16384, *dSg = p.dSw + ci * 16384, *Vg = p.Vnw + ci * 8192, *Bg = p.Bw + ci * 16384;
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1u);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid < 64) {
        gam[tid] = p.Gw[ci * 64 + tid];
        bet[tid] = tid < nrows ? __uint_as_float((uint32_t)p.beta[MASKED ? htok + tid / r : hrow + tid] << 16) : 0.f;
        if (MASKED && tid < r * r) msk[tid] = p.mask[tid];
    }
    // S and dS' split (row m, columns 8 g ..: hi at +0, lo at +32 KB), with <dS', S>;
    // every pass issues a batch of loads before its shared stores
    float dot = 0.f;
#pragma unroll 1
    for (int e0 = tid; e0 < 128 * 16; e0 += 4 * kCpThr) {
        float4 v[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + kCpThr * u, m2 = e >> 4, k0 = 8 * (e & 15);
            v[u][0] = *reinterpret_cast<const float4 *>(dSg + m2 * 128 + k0);
            v[u][1] = *reinterpret_cast<const float4 *>(dSg + m2 * 128 + k0 + 4);
            v[u][2] = *reinterpret_cast<const float4 *>(Sg + m2 * 128 + k0);
            v[u][3] = *reinterpret_cast<const float4 *>(Sg + m2 * 128 + k0 + 4);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + kCpThr * u, m2 = e >> 4, k0 = 8 * (e & 15);
            const float x[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
            const float y[8] = {v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w, v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w};
#pragma unroll
            for (int i = 0; i < 8; ++i) dot += x[i] * y[i];
            const uint32_t off = (uint32_t)(k0 >> 6) * 16384u + sw128_offset((uint32_t)m2, (uint32_t)(k0 & 63));
            uint4 hi, lo;
            split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(sm + CP_DS + off) = hi;
            *reinterpret_cast<uint4 *>(sm + CP_DS + 32768 + off) = lo;
            split8(y, hi, lo);
            *reinterpret_cast<uint4 *>(sm + CP_S + off) = hi;
            *reinterpret_cast<uint4 *>(sm + CP_S + 32768 + off) = lo;
        }
    }
    {  // Vn split (row b, columns 8 g ..), with Y_b . Vn_b (the 16 lanes of a row)
        constexpr int U = 1024 / kCpThr;
        float4 v[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + kCpThr * u, t = e >> 4, k0 = 8 * (e & 15);
            v[u][0] = *reinterpret_cast<const float4 *>(Vg + t * 128 + k0);
            v[u][1] = *reinterpret_cast<const float4 *>(Vg + t * 128 + k0 + 4);
            v[u][2] = *reinterpret_cast<const float4 *>(Bg + t * 128 + k0);
            v[u][3] = *reinterpret_cast<const float4 *>(Bg + t * 128 + k0 + 4);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + kCpThr * u, t = e >> 4, k0 = 8 * (e & 15);
            const float4 a0 = v[u][0], a1 = v[u][1], y0 = v[u][2], y1 = v[u][3];
            const float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float yv = y0.x * a0.x + y0.y * a0.y + y0.z * a0.z + y0.w * a0.w + y1.x * a1.x + y1.y * a1.y +
                       y1.z * a1.z + y1.w * a1.w;
            yv = sum16p(yv);
            if ((e & 15) == 0) Bg[8256 + t] = yv;
            const uint32_t off = (uint32_t)(k0 >> 6) * 8192u + sw128_offset((uint32_t)t, (uint32_t)(k0 & 63));
            uint4 hi, lo;
            split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(sm + CP_VN + off) = hi;
            *reinterpret_cast<uint4 *>(sm + CP_VN + 16384 + off) = lo;
        }
    }
    const unsigned short *dO = p.dout + htok * 128;
    {  // dO: query row q < nq2, columns 8 g .. (exact in bf16)
        constexpr int U = 1024 / kCpThr;
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + kCpThr * u, q = e >> 4, k0 = 8 * (e & 15);
            w[u] = q < ntok ? *reinterpret_cast<const uint4 *>(dO + (size_t)q * 128 + k0) : z4;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + kCpThr * u, q = e >> 4, k0 = 8 * (e & 15);
            if (q < nq2)
                *reinterpret_cast<uint4 *>(sm + CP_DO + (uint32_t)(k0 >> 6) * (uint32_t)(nq2 * 128) +
                                           sw128_offset((uint32_t)q, (uint32_t)(k0 & 63))) = w[u];
        }
    }
    {  // T (row b) and P^ (query row t < nq2), columns 8 g .., split as MN-major operands
        const float *Tg = p.Tw + ci * 4096, *Pg = p.Pw + ci * 4096;
        constexpr int U = 512 / kCpThr;
        float4 v[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + kCpThr * u, rr = e >> 3, k0 = 8 * (e & 7);
            v[u][0] = *reinterpret_cast<const float4 *>(Tg + rr * 64 + k0);
            v[u][1] = *reinterpret_cast<const float4 *>(Tg + rr * 64 + k0 + 4);
            v[u][2] = *reinterpret_cast<const float4 *>(Pg + rr * 64 + k0);
            v[u][3] = *reinterpret_cast<const float4 *>(Pg + rr * 64 + k0 + 4);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + kCpThr * u, rr = e >> 3, k0 = 8 * (e & 7);
            const uint32_t off = sw128_offset((uint32_t)rr, (uint32_t)k0);
            const float x[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
            uint4 hi, lo;
            split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(sm + CP_T + off) = hi;
            *reinterpret_cast<uint4 *>(sm + CP_T + 8192 + off) = lo;
            if (rr < nq2) {
                const float y[8] = {v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w, v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w};
                split8(y, hi, lo);
                *reinterpret_cast<uint4 *>(sm + CP_P + off) = hi;
                *reinterpret_cast<uint4 *>(sm + CP_P + 8192 + off) = lo;
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) wsum[warp] = dot;
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    if (tid == 0) {
        float d = 0.f;
        for (int w = 0; w < kCpThr / 32; ++w) d += wsum[w];
        Bg[8192] = d;
        // Z^T = dS' Vn^T, t1^T = S dO^T
        const uint32_t idZ = idesc_bf16(128, 64, false, false), idT = idesc_bf16(128, nq2, false, false);
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t a = sb + CP_DS + (pr == 2 ? 32768u : 0u), b = sb + CP_VN + (pr == 1 ? 16384u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(tmem + CT_Z, smem_desc(a + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                            smem_desc(b + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), idZ, (pr | ks) != 0);
        }
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            const uint32_t a = sb + CP_S + (pr == 1 ? 32768u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(tmem + CT_T1, smem_desc(a + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                            smem_desc(sb + CP_DO + (ks >> 2) * (nq2 * 128) + (ks & 3) * 32, 16, 1024), idT,
                            (pr | ks) != 0);
        }
        // Yw^T = dO^T P^ (dO as an MN-major operand: K = query rows, M = value columns)
        const uint32_t idY = idesc_bf16(128, 64, true, true);
        for (int pr = 0; pr < 2; ++pr)
            for (int ks = 0; ks < nq2 / 16; ++ks)
                mma_bf16_ss(tmem + CT_YW, smem_desc(sb + CP_DO + ks * 2048, nq2 * 128, 1024),
                            smem_desc(sb + CP_P + 8192u * pr + ks * 2048, 8192, 1024), idY, (pr | ks) != 0);
        // DOV = dO Vn^T (rows: the query rows of dO)
        const uint32_t idV = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            const uint32_t b = sb + CP_VN + 16384u * pr;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(tmem + CT_DOV, smem_desc(sb + CP_DO + (ks >> 2) * (nq2 * 128) + (ks & 3) * 32, 16, 1024),
                            smem_desc(b + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), idV, (pr | ks) != 0);
        }
        mma_commit(&bar[0]);
    }
    bool ok = warp_ok(wyc_wait(&bar[0], 0, 8u, p.timeout_ns));
    const int m = 32 * q4 + lane;  // TMEM lane
    if (ok) {
        tc_fence_after_sync();
        for (int j = cg; j < nq2 / 16; j += kCpCG) {  // t1 rows q = 16 j ..
            uint32_t rg[16];
            tmem_ld16(tmem + lb + CT_T1 + 16 * j, rg);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) dSg[8192 + (size_t)(16 * j + i) * 128 + m] = __uint_as_float(rg[i]);
        }
        {  // dVn^T row dv = m, columns b = CW cg ..: Y^T + Yw^T as a K-major operand (over dS' hi)
            uint32_t rg[kCpCW];
#pragma unroll
            for (int h = 0; h < kCpCW / 16; ++h)
                tmem_ld16(tmem + lb + CT_YW + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(rg + 16 * h));
            tmem_wait_ld();
            float x[kCpCW];
#pragma unroll
            for (int i = 0; i < kCpCW; ++i) x[i] = Bg[(size_t)(kCpCW * cg + i) * 128 + m] + __uint_as_float(rg[i]);
#pragma unroll
            for (int h = 0; h < kCpCW / 8; ++h) {
                uint4 hi, lo;
                split8(x + 8 * h, hi, lo);
                const uint32_t off = sw128_offset((uint32_t)m, (uint32_t)(kCpCW * cg + 8 * h));
                *reinterpret_cast<uint4 *>(sm + CP_DS + off) = hi;
                *reinterpret_cast<uint4 *>(sm + CP_DS + 16384 + off) = lo;
            }
        }
        if (q4 < 2) {  // DOV row i = m, columns b = CW cg ..: to the Vn slot (float 4096 on), and P~ (over dO)
            uint32_t rg[kCpCW];
#pragma unroll
            for (int h = 0; h < kCpCW / 16; ++h)
                tmem_ld16(tmem + lb + CT_DOV + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(rg + 16 * h));
            tmem_wait_ld();
            const int i = m;
            const bool live = i < ntok;
            const float gi = live ? gam[i * r] : 0.f;
            float x[kCpCW];
#pragma unroll
            for (int j = 0; j < kCpCW; ++j) {
                const int b = kCpCW * cg + j;
                const float dv = __uint_as_float(rg[j]);
                if (i < nq2) Vg[4096 + (size_t)i * 64 + b] = dv;
                x[j] = (live && b / r <= i) ? p.scale * expf(gi - gam[b]) * dv : 0.f;
            }
#pragma unroll
            for (int h = 0; h < kCpCW / 8; ++h) {
                uint4 hi, lo;
                split8(x + 8 * h, hi, lo);
                const uint32_t off = sw128_offset((uint32_t)i, (uint32_t)(kCpCW * cg + 8 * h));
                *reinterpret_cast<uint4 *>(sm + CP_DO + off) = hi;
                *reinterpret_cast<uint4 *>(sm + CP_DO + 8192 + off) = lo;
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (tid == 0) {  // dR^T = dVn^T T
        const uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t a = sb + CP_DS + (pr == 2 ? 16384u : 0u), b = sb + CP_T + (pr == 1 ? 8192u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tmem + CT_DR, smem_desc(a + ks * 32, 16, 1024), smem_desc(b + ks * 2048, 8192, 1024), id,
                            (pr | ks) != 0);
        }
        mma_commit(&bar[1]);
    }
    // the keys and queries of batch 4 (element e: row e / 16, 8-column group e % 16), loaded while dR forms
    constexpr int UK = 1024 / kCpThr;
    uint4 kg[UK], qg4[UK];
#pragma unroll
    for (int u = 0; u < UK; ++u) {
        const int e = tid + kCpThr * u, row = e >> 4, g = e & 15;
        const size_t ks = MASKED ? htok + row / r : hrow + row;
        kg[u] = row < nrows ? ldg16p(p.k + ks * 128 + 8 * g) : z4;
        qg4[u] = row < ntok ? ldg16p(p.q + (htok + row) * 128 + 8 * g) : z4;
    }
#pragma unroll
    for (int u = 0; u < UK; ++u) {  // norms (the 16 lanes of a row)
        const int e = tid + kCpThr * u, row = e >> 4, g = e & 15;
        float x[8];
        unpack8p(kg[u], x);
        float sk = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) sk += x[i] * x[i];
        unpack8p(qg4[u], x);
        float sq = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) sq += x[i] * x[i];
        sk = sum16p(sk);
        sq = sum16p(sq);
        if (g == 0) {
            nk[row] = p.l2 ? 1.f / fmaxf(sqrtf(sk), 1e-12f) : 1.f;
            mq[row] = p.l2 ? 1.f / fmaxf(sqrtf(sq), 1e-12f) : 1.f;
        }
    }
    ok = warp_ok(wyc_wait(&bar[1], 0, 8u, p.timeout_ns));
    if (ok) {  // dR^T row dv = m, columns a = CW cg ..: dR[a][dv] over S's slot, and dR^T's image
        tc_fence_after_sync();
        uint32_t rg[kCpCW];
#pragma unroll
        for (int h = 0; h < kCpCW / 16; ++h)
            tmem_ld16(tmem + lb + CT_DR + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(rg + 16 * h));
        tmem_wait_ld();
        float x[kCpCW];
#pragma unroll
        for (int i = 0; i < kCpCW; ++i) {
            x[i] = __uint_as_float(rg[i]);
            Sg[(size_t)(kCpCW * cg + i) * 128 + m] = x[i];
        }
#pragma unroll
        for (int h = 0; h < kCpCW / 8; ++h) {
            uint4 hi, lo;
            split8(x + 8 * h, hi, lo);
            const uint32_t off = sw128_offset((uint32_t)m, (uint32_t)(kCpCW * cg + 8 * h));
            *reinterpret_cast<uint4 *>(sm + CP_DR + off) = hi;
            *reinterpret_cast<uint4 *>(sm + CP_DR + 16384 + off) = lo;
        }
    }
    __syncthreads();  // the norms; dVn^T's image has been read
#pragma unroll
    for (int u = 0; u < UK; ++u) {  // Q = diag(m) q (hi | lo) over dVn^T's image
        const int e = tid + kCpThr * u, row = e >> 4, g = e & 15;
        float x[8];
        unpack8p(qg4[u], x);
        const float f = mq[row];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= f;
        uint4 hi, lo;
        split8(x, hi, lo);
        const uint32_t off = (uint32_t)(g >> 3) * 8192u + sw128_offset((uint32_t)row, (uint32_t)((8 * g) & 63));
        *reinterpret_cast<uint4 *>(sm + CP_DS + off) = hi;
        *reinterpret_cast<uint4 *>(sm + CP_DS + 16384 + off) = lo;
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (tid == 0) {
        // dR Vn^T: dR^T's image as an MN-major operand (K = value rows, M = a; the second atom is not used)
        const uint32_t idA = idesc_bf16(128, 64, true, false), idT2 = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t a = sb + CP_DR + (pr == 2 ? 16384u : 0u), b = sb + CP_VN + (pr == 1 ? 16384u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(tmem + CT_DA, smem_desc(a + ks * 2048, 16384, 1024),
                            smem_desc(b + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), idA, (pr | ks) != 0);
        }
        // t2^T = S dR^T (dR^T's image as an MN-major operand: K = value rows, N = a)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t a = sb + CP_S + (pr == 2 ? 32768u : 0u), b = sb + CP_DR + (pr == 1 ? 16384u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(tmem + CT_T2, smem_desc(a + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                            smem_desc(b + ks * 2048, 8192, 1024), idT2, (pr | ks) != 0);
        }
        mma_commit(&bar[2]);
    }
    ok = warp_ok(wyc_wait(&bar[2], 0, 8u, p.timeout_ns));
    if (ok) {
        tc_fence_after_sync();
        uint32_t rg[kCpCW];
        if (q4 < 2) {  // row a = m of dR Vn^T, columns CW cg ..: to the Vn slot [a][c], and L (over P^)
#pragma unroll
            for (int h = 0; h < kCpCW / 16; ++h)
                tmem_ld16(tmem + lb + CT_DA + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(rg + 16 * h));
            tmem_wait_ld();
            const int a = m;
            const float fa = bet[a], ga = gam[a];
            float x[kCpCW];
#pragma unroll
            for (int j = 0; j < kCpCW; ++j) {
                const int cc = kCpCW * cg + j;
                const float da = __uint_as_float(rg[j]);
                Vg[(size_t)a * 64 + cc] = da;
                x[j] = (MASKED ? cc / r < a / r : cc < a) ? -da * fa * expf(ga - gam[cc]) : 0.f;
            }
#pragma unroll
            for (int h = 0; h < kCpCW / 8; ++h) {
                uint4 hi, lo;
                split8(x + 8 * h, hi, lo);
                const uint32_t off = sw128_offset((uint32_t)a, (uint32_t)(kCpCW * cg + 8 * h));
                *reinterpret_cast<uint4 *>(sm + CP_P + off) = hi;
                *reinterpret_cast<uint4 *>(sm + CP_P + 8192 + off) = lo;
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();  // S's image has been read
    // Kr and Kw (hi | lo) of the rows (sub-rows), unit-normalised when asked, over S's image
#pragma unroll
    for (int u = 0; u < UK; ++u) {
        const int e = tid + kCpThr * u, row = e >> 4, g = e & 15;
        float x[8], y[8];
        unpack8p(kg[u], x);
        const float f = nk[row];
        float fr = f, fw = f;
        if (MASKED) {
            const int ib = row % r, j = (g * r) >> 4;
            fr = f * msk[ib * r + j];
            fw = j == ib ? f : 0.f;
        }
        const uint32_t off = (uint32_t)(g >> 3) * 8192u + sw128_offset((uint32_t)row, (uint32_t)((8 * g) & 63));
        uint4 hi, lo;
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = x[i] * fr;
        split8(y, hi, lo);
        *reinterpret_cast<uint4 *>(sm + CP_S + off) = hi;
        *reinterpret_cast<uint4 *>(sm + CP_S + 16384 + off) = lo;
        if (MASKED) {
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = x[i] * fw;
            split8(y, hi, lo);
            *reinterpret_cast<uint4 *>(sm + CP_S + 32768 + off) = hi;
            *reinterpret_cast<uint4 *>(sm + CP_S + 49152 + off) = lo;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (tid == 0) {  // X1^T = Q^T P~ + Kr^T L, X2^T = Kw^T L^T, (P~ Kw)^T
        const uint32_t kr = sb + CP_S, kw = sb + CP_S + (MASKED ? 32768u : 0u);
        const uint32_t idMM = idesc_bf16(128, 64, true, true), idMK = idesc_bf16(128, 64, true, false);
        const uint32_t idQ = idesc_bf16(128, nq2, true, false);
        int n = 0;
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t pa = pr == 2 ? 16384u : 0u, pb = pr == 1 ? 8192u : 0u;
            for (int ks = 0; ks < nq2 / 16; ++ks)  // Q^T P~ (K = query rows)
                mma_bf16_ss(tmem + CT_X1, smem_desc(sb + CP_DS + pa + ks * 2048, 8192, 1024),
                            smem_desc(sb + CP_DO + pb + ks * 2048, 8192, 1024), idMM, (n++) > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // Kr^T L (K = rows)
                mma_bf16_ss(tmem + CT_X1, smem_desc(kr + pa + ks * 2048, 8192, 1024),
                            smem_desc(sb + CP_P + pb + ks * 2048, 8192, 1024), idMM, 1u);
        }
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t pa = pr == 2 ? 16384u : 0u, pb = pr == 1 ? 8192u : 0u;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {  // Kw^T L^T and Kw^T P~^T (L and P~ as K-major operands)
                mma_bf16_ss(tmem + CT_X2, smem_desc(kw + pa + ks * 2048, 8192, 1024),
                            smem_desc(sb + CP_P + pb + ks * 32, 16, 1024), idMK, (pr | ks) != 0);
                mma_bf16_ss(tmem + CT_DQ, smem_desc(kw + pa + ks * 2048, 8192, 1024),
                            smem_desc(sb + CP_DO + pb + ks * 32, 16, 1024), idQ, (pr | ks) != 0);
            }
        }
        mma_commit(&bar[3]);
    }
    ok = warp_ok(wyc_wait(&bar[3], 0, 8u, p.timeout_ns));
    float *red = reinterpret_cast<float *>(sm + CP_T);  // [4 lane quarters][64 rows] (T's image is dead)
    if (ok) {  // row dk = m, columns a = CW cg ..: dk's share and the rows' kr . t2; (P~ Kw)[i][dk] (W slot)
        tc_fence_after_sync();
        float *DQg = p.Ww + ci * 8192;
        uint32_t z[kCpCW], x1[kCpCW], x2[kCpCW], t2[kCpCW];
#pragma unroll
        for (int h = 0; h < kCpCW / 16; ++h) {
            tmem_ld16(tmem + lb + CT_Z + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(z + 16 * h));
            tmem_ld16(tmem + lb + CT_X1 + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(x1 + 16 * h));
            tmem_ld16(tmem + lb + CT_X2 + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(x2 + 16 * h));
            tmem_ld16(tmem + lb + CT_T2 + kCpCW * cg + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(t2 + 16 * h));
        }
        tmem_wait_ld();
        // dk[a][m] = ww (e^{gl - gamma_a} Z + X1) + wr (X2 - beta_a e^{gamma_a} t2), with the
        // block-masked variant's weights ww (m in slice a % r) and wr = mask[a % r][slice of m]
        const float gl = gam[63];
        const int jm = MASKED ? m / (128 / r) : 0;
        const uint32_t kro = (uint32_t)(m >> 6) * 8192u;
#pragma unroll
        for (int i = 0; i < kCpCW; ++i) {
            const int a = kCpCW * cg + i;
            float ww = 1.f, wr = 1.f;
            if (MASKED) {
                ww = jm == a % r ? 1.f : 0.f;
                wr = msk[(a % r) * r + jm];
            }
            const float t2v = __uint_as_float(t2[i]);
            Bg[(size_t)a * 128 + m] =
                ww * (expf(gl - gam[a]) * __uint_as_float(z[i]) + __uint_as_float(x1[i])) +
                wr * (__uint_as_float(x2[i]) - bet[a] * expf(gam[a]) * t2v);
            // kr[a][m] from its split image (hi + lo), times t2, summed over the warp's 32 key columns
            const uint32_t off = kro + sw128_offset((uint32_t)a, (uint32_t)(m & 63));
            const float kr = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(sm + CP_S + off)) << 16) +
                             __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(sm + CP_S + 16384 + off)) << 16);
            float v = kr * t2v;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[q4 * 64 + a] = v;
        }
        for (int j = cg; j < nq2 / 16; j += kCpCG) {
            uint32_t r16[16];
            tmem_ld16(tmem + lb + CT_DQ + 16 * j, r16);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) DQg[(size_t)(16 * j + i) * 128 + m] = __uint_as_float(r16[i]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 64) Bg[8320 + tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];  // kr_a . t2_a
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

int launch_chunk_products_tc(const ChunkProductsTcArgs &a, cudaStream_t st) {
    if (a.BH <= 0 || a.NT <= 0 || a.Ct <= 0 || a.Ct > 64 || a.r < 1 || a.Ct * a.r > 64) return GDN_ERR_INVALID_ARG;
    if (a.masked && (a.r > 8 || 64 % a.r != 0)) return GDN_ERR_INVALID_ARG;
    ChunkProductsTcArgs p = a;
    p.nq2 = (a.Ct + 15) / 16 * 16;
    p.timeout_ns = wait_limit_ns();
    void (*kern)(ChunkProductsTcArgs) = a.masked ? chunk_products_tc_kernel<true> : chunk_products_tc_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CP_SMEM) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<dim3((unsigned)a.NT, (unsigned)a.BH), kCpThr, CP_SMEM, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// The chunk-local WY factors on tcgen05 for bf16 at Dk = Dv = 128, for the
// block-masked DeltaProduct forward and for the backward passes of the chunk
// GDN / DeltaProduct and of the block-masked variant (gated_deltaproduct
// test.py: `gated_chunk_scaled_dot_kkt_fwd_kernel` with its mask_ij coupling,
// the triangular solve, `gated_fwd_recompute_w_u_kernel`,
// `gated_bwd_prepare_wy_repr_kernel` and the chunk output of
// `gated_chunk_fwd_o_fn`).  Sub-row b of a 64-row chunk of Ct = 64 / r tokens
// belongs to token t_b = b / r.  GDN / DeltaProduct: sub-row b has its own key
// (read and write key alike), value and beta.  Block-masked: kw_b is slice
// i_b = b % r of k_{t_b} (zero elsewhere) and kr_b is k_{t_b} with slice j
// scaled by mask[i_b][j].  With the unit-norm flag n_b = 1/||key of b|| and
// m_t = 1/||q_t|| (else 1) stay scalar factors, so the raw bf16 keys and
// queries enter the products exactly.
//
// wy_tc_kernel, one CTA per chunk:
//   1. [K; Q] Kw^T as one exact product (M = 128: the sub-rows' raw read keys
//      in rows 0..63, the queries in rows 64..127; N = 64 sub-rows), since
//      kr_a . kw_b is mask[i_a][i_b] times the dot product of k_{t_a} and kw_b;
//   2. A[a][b] = beta_a e^{gamma_a - gamma_b} kr_a . kw_b below the diagonal
//      (earlier tokens for the block-masked variant), the output factors
//      P[t][b] = scale e^{gamma_{t r} - gamma_b} m_t q_t . kw_b for t_b <= t,
//      and for the backward kr_a . kw_b itself;
//   3. T = (I + A)^-1 on the CUDA cores (tri_inverse.cuh);
//   4. W = T diag(beta e^gamma) Kr as three split products (both operands
//      rounded) and U = T diag(beta) V as two (v is exact), M = 128 with rows
//      0..63 used, N = 128;
//   5. W and Kd = diag(e^{gl - gamma}) Kw as the chain's operand images, U, P,
//      gamma in fp32; the backward also T, kr . kw and the chunk's term of the
//      state gradient B = Q^T diag(scale e^{gamma_{t r}} m) dO - W^T P^T dO, as
//      B^T = dO^T Q' (two split products: dO is exact) - Y^T W (three), with
//      Y^T = dO^T P formed while T is inverted.
// masked_out_tc_kernel, one CTA of 256 threads per chunk (three per SM), with
// S the state entering it:  o_t = scale e^{gamma_{t r}} m_t q_t S + (P Vn)_t,
// as o^T = S^T Q^T + Vn^T P^T with bf16 operands (S, Vn and P rounded once, as
// in the fused forward; q exact), M = 128 value rows, N = the chunk's query
// rows rounded up to 16.
namespace {

// Shared memory of wy_tc_kernel, reused by the phases (byte offsets):
//   loads, [K; Q] Kw^T:  X = [sub-row read keys, rows 0..63 | queries q_t, rows 64..127] K-major,
//                        2 key blocks of 16 KB, at 0; Kw [2 key blocks][64 sub-rows][128 B] (exact)
//                        at 32768; Kd's image (hi | lo), staged for one bulk copy, at 49152
//   A, the inverse:      A, T fp32 [64][68] at 0 and 17408, scratch (1024 floats) at 34816;
//                        P's rows (68-float stride), staged for bulk copies, at 81920
//   W and U:             Tw hi | Tw lo | Tu hi | Tu lo [64 rows][128 B] K-major (8 KB each) at 0,
//                        Kr hi | lo [2 key blocks][64 sub-rows][128 B] at 32768,
//                        the sub-rows' values [2 value blocks][64 sub-rows][128 B] (exact) at 65536
//   the results:         W's image at 0, U's rows (132-float stride) at 32768, both for bulk copies
// and for the backward, from 99328 on: K K^T's rows (68-float stride, staged),
// P as an MN-major operand (rows t, hi | lo), dO (rows t, 2 value blocks,
// exact), Q' = diag(scale e^gamma m) Q (rows t, 2 key blocks, hi | lo), and Y^T
// = (P^T dO)^T as a K-major operand (rows dv, hi | lo) over the staging of P
// and K K^T once those have left.  The padded row strides keep the
// row-per-lane stores of the staging free of bank conflicts.
constexpr uint32_t MW_X = 0, MW_KW = 32768, MW_KD = 49152;
constexpr int kMwLA = 68;  // fp32 row stride of A and T (16-byte aligned rows)
constexpr uint32_t MW_AF = 0, MW_TF = 64 * kMwLA * 4, MW_X4 = 2 * 64 * kMwLA * 4, MW_PS = 81920;
constexpr uint32_t MW_TW = 0, MW_KR = 32768, MW_VS = 65536;
constexpr uint32_t MW_WS = 0, MW_US = 32768;
constexpr int kMwLP = 68, kMwLU = 132;  // staging row strides (floats)
constexpr uint32_t MW_KKS = 99328, MW_PI = 116736, MW_DOI = 133120, MW_QP = 149504, MW_YI = 81920;
__host__ __device__ constexpr uint32_t mw_vec(bool bwd) { return bwd ? 182272u : 99328u; }  // gamma, beta, n, m, mask: 64 floats each
__host__ __device__ constexpr uint32_t mw_bar(bool bwd) { return mw_vec(bwd) + 5 * 256; }     // 4 mbarriers, then the TMEM address
__host__ __device__ constexpr uint32_t mw_smem(bool bwd) { return mw_bar(bwd) + 48 + 1024; }
// The M = 128 products read A rows 64..127 from the 8 KB after the start of
// their 64-row operand: W's rows past Tw are Tw lo and Tu hi, and U's
// operand starts 8 KB before Tu hi (lo), so that Tu sits in rows 64..127 and
// U lands in TMEM lanes 64..127; every row read is finite and the rows not
// wanted are not used.
static_assert(MW_X4 + 4096 <= MW_PS && MW_KD + 32768 <= MW_PS && MW_PS + 64 * kMwLP * 4 <= MW_KKS &&
                  MW_VS + 16384 <= MW_PS && MW_US + 64 * kMwLU * 4 <= MW_PS && MW_KKS + 64 * kMwLP * 4 <= MW_PI &&
                  MW_PI + 16384 <= MW_DOI && MW_DOI + 16384 <= MW_QP && MW_QP + 32768 <= mw_vec(true) &&
                  MW_YI + 32768 <= MW_PI && mw_vec(false) >= MW_PS + 64 * kMwLP * 4,
              "WY map");
static_assert(2 * (mw_smem(false) + 1024) <= 233472 && mw_smem(true) <= 232448, "WY kernels fit shared memory");

__device__ __forceinline__ void unpack8(const uint4 &w, float *x) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ float sum16(float x) {  // over the 16 lanes that differ in bits 0..3
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ uint4 ldg16(const unsigned short *p) { return *reinterpret_cast<const uint4 *>(p); }

// wy_tc_kernel<R, MASKED, BWD>: one CTA per chunk; 256 threads and two CTAs
// per SM for the forward, 512 threads and one CTA per SM for the backward.
// MASKED: the sub-rows' keys are the token keys' slices (read keys scaled by
// the mask); otherwise each sub-row has its own key, value and beta.
template <int R, bool MASKED, bool BWD>
__global__ void __launch_bounds__(BWD ? 512 : 256, BWD ? 1 : 2) wy_tc_kernel(WyTcArgs p) {
    constexpr int NT = BWD ? 512 : 256, CG = NT / 128, Ct = 64 / R, NQ2 = (Ct + 15) / 16 * 16;
    constexpr uint32_t VEC = mw_vec(BWD), BAR = mw_bar(BWD), TCOLS = BWD ? 512u : 256u;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *Af = reinterpret_cast<float *>(sm + MW_AF), *Tf = reinterpret_cast<float *>(sm + MW_TF);
    float *X4 = reinterpret_cast<float *>(sm + MW_X4), *Ps = reinterpret_cast<float *>(sm + MW_PS);
    float *Us = reinterpret_cast<float *>(sm + MW_US), *KKs = reinterpret_cast<float *>(sm + MW_KKS);
    float *gam = reinterpret_cast<float *>(sm + VEC), *bet = gam + 64, *nk = bet + 64, *mq = nk + 64, *msk = mq + 64;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + BAR);  // [K; Q] Kw^T | W, U (and Y) | B
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + BAR + 32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q4 = warp & 3;
    const uint32_t lb = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
    const int c = blockIdx.x, bh = blockIdx.y;
    const int t0 = c * Ct, ntok = min(Ct, p.T - t0), nrows = ntok * R;
    const size_t htok = (size_t)bh * p.T + t0, hrow = htok * R, ci = (size_t)bh * p.NT + c;
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1u);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, TCOLS);
        tmem_relinquish();
    }
    if (tid < 64) {
        bet[tid] = tid < nrows ? __uint_as_float((uint32_t)p.beta[MASKED ? htok + tid / R : hrow + tid] << 16) : 0.f;
        if (MASKED && tid < R * R) msk[tid] = p.mask[tid];
    }
    if (warp == 1) {  // gamma: inclusive cumulative sum over the sub-rows; g_t enters on (t, 0)
        const int a0 = lane, a1 = lane + 32;
        float x0 = (a0 < nrows && a0 % R == 0) ? p.g[htok + a0 / R] : 0.f;
        float x1 = (a1 < nrows && a1 % R == 0) ? p.g[htok + a1 / R] : 0.f;
        for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) {
                x0 += y0;
                x1 += y1;
            }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        gam[a0] = x0;
        gam[a1] = x1;
    }
    // X: sub-row a's read key in row a, query t in row 64 + t (zero past the
    // sequence), and the norms; element e: matrix e / 1024, row (e / 16) % 64,
    // 8-column group e % 16
    {
        constexpr int U = 2048 / NT;
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + NT * u, mat = e >> 10, row = (e >> 4) & 63, g = e & 15;
            const size_t src = mat ? htok + row : (MASKED ? htok + row / R : hrow + row);
            w[u] = (mat ? row : row / R) < ntok ? ldg16((mat ? p.q : p.k) + src * 128 + 8 * g) : z4;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + NT * u, mat = e >> 10, row = (e >> 4) & 63, g = e & 15;
            float x[8];
            unpack8(w[u], x);
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
            ss = sum16(ss);
            if (g == 0) (mat ? mq : nk)[row] = p.l2 ? 1.f / fmaxf(sqrtf(ss), 1e-12f) : 1.f;
            *reinterpret_cast<uint4 *>(sm + MW_X + (uint32_t)(g >> 3) * 16384u +
                                       sw128_offset((uint32_t)(row + 64 * mat), (uint32_t)((8 * g) & 63))) = w[u];
        }
    }
    if constexpr (BWD) {  // dO rows t (exact) as an MN-major operand: [2 value blocks][64 rows][128 B]
        constexpr int U = 1024 / NT;
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + NT * u, t = e >> 4, g = e & 15;
            w[u] = t < ntok ? ldg16(p.dout + (htok + t) * 128 + 8 * g) : z4;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + NT * u, t = e >> 4, g = e & 15;
            *reinterpret_cast<uint4 *>(sm + MW_DOI + (uint32_t)(g >> 3) * 8192u +
                                       sw128_offset((uint32_t)t, (uint32_t)((8 * g) & 63))) = w[u];
        }
    }
    __syncthreads();
    // Kw (exact) and Kd = diag(e^{gl - gamma} n) Kw's image (hi | lo), staged;
    // element e: sub-row e / 16, 8-column group e % 16 (in slice g R / 16).  The
    // backward also forms Q' = diag(scale e^{gamma_{t r}} m) Q (hi | lo).
    {
        const float gl = gam[63];
        constexpr int U = 1024 / NT;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = tid + NT * u, b = e >> 4, g = e & 15;
            const bool own = !MASKED || ((g * R) >> 4) == b % R;
            const uint32_t off = (uint32_t)(g >> 3) * 8192u + sw128_offset((uint32_t)b, (uint32_t)((8 * g) & 63));
            const uint4 kx = *reinterpret_cast<const uint4 *>(sm + MW_X + (uint32_t)(g >> 3) * 16384u +
                                                              sw128_offset((uint32_t)b, (uint32_t)((8 * g) & 63)));
            *reinterpret_cast<uint4 *>(sm + MW_KW + off) = own ? kx : z4;
            float x[8];
            unpack8(kx, x);
            const float fd = own ? expf(gl - gam[b]) * nk[b] : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] *= fd;
            uint4 hi, lo;
            split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(sm + MW_KD + off) = hi;
            *reinterpret_cast<uint4 *>(sm + MW_KD + 16384 + off) = lo;
            if constexpr (BWD) {  // query row t = b
                const int t = b;
                const uint4 qx = *reinterpret_cast<const uint4 *>(
                    sm + MW_X + (uint32_t)(g >> 3) * 16384u + sw128_offset((uint32_t)(64 + t), (uint32_t)((8 * g) & 63)));
                unpack8(qx, x);
                const float fq = t < ntok ? p.scale * expf(gam[t * R]) * mq[t] : 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] *= fq;
                split8(x, hi, lo);
                *reinterpret_cast<uint4 *>(sm + MW_QP + off) = hi;
                *reinterpret_cast<uint4 *>(sm + MW_QP + 16384 + off) = lo;
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    if (tid == 0) {  // Kd's image out; [K; Q] Kw^T into columns 0..63
        bulk_store_global(p.Kdw + ci * 8192, sm + MW_KD, 32768u);
        tma_store_commit();
        const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(tmem, smem_desc(sb + MW_X + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                        smem_desc(sb + MW_KW + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), id, ks > 0);
        mma_commit(&bar[0]);
    }
    bool ok = warp_ok(wyc_wait(&bar[0], 0, 16u, p.timeout_ns));
    if (ok) {  // warp: TMEM lanes 32 (warp % 4) .., columns CW (warp / 4) ..  (A is written over X)
        constexpr int CW = 64 / CG;
        tc_fence_after_sync();
        const int c0 = CW * (warp >> 2);
        uint32_t x[CW];
#pragma unroll
        for (int h = 0; h < CW / 16; ++h)
            tmem_ld16(tmem + lb + c0 + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(x + 16 * h));
        tmem_wait_ld();
        if (q4 < 2) {  // row a of A (and of the read keys against the write keys)
            const int a = 32 * q4 + lane, ta = a / R, ia = a % R;
            const float fa = bet[a], na = nk[a], ga = gam[a];
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
                const int b = c0 + jj;
                const float kk = (MASKED ? msk[ia * R + b % R] : 1.f) * na * nk[b] * __uint_as_float(x[jj]);
                Af[a * kMwLA + b] = (MASKED ? b / R < ta : b < a) ? fa * expf(ga - gam[b]) * kk : 0.f;
                if constexpr (BWD) KKs[a * kMwLP + b] = kk;
            }
        } else {  // token t's query: row t of P, staged (and, for the backward, as an operand)
            const int t = 32 * (q4 - 2) + lane;
            const bool live = t < ntok;
            const float ga = live ? gam[t * R] : 0.f, fq = p.scale * mq[t];
            float pv[CW];
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
                const int b = c0 + jj;
                pv[jj] = (live && b / R <= t) ? fq * nk[b] * expf(ga - gam[b]) * __uint_as_float(x[jj]) : 0.f;
            }
            float4 *Pr = reinterpret_cast<float4 *>(Ps + t * kMwLP + c0);
#pragma unroll
            for (int h = 0; h < CW / 4; ++h) Pr[h] = make_float4(pv[4 * h], pv[4 * h + 1], pv[4 * h + 2], pv[4 * h + 3]);
            if constexpr (BWD) {
#pragma unroll
                for (int h = 0; h < CW / 8; ++h) {
                    uint4 hi, lo;
                    split8(pv + 8 * h, hi, lo);
                    const uint32_t off = sw128_offset((uint32_t)t, (uint32_t)(c0 + 8 * h));
                    *reinterpret_cast<uint4 *>(sm + MW_PI + off) = hi;
                    *reinterpret_cast<uint4 *>(sm + MW_PI + 8192 + off) = lo;
                }
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {  // P's rows (and K K^T's) out (lane: rows lane, lane + 32)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = lane + 32 * h;
            bulk_store_global(p.Pw + ci * 4096 + (size_t)t * 64, Ps + t * kMwLP, 256u);
            if constexpr (BWD) bulk_store_global(p.KKw + ci * 4096 + (size_t)t * 64, KKs + t * kMwLP, 256u);
        }
        tma_store_commit();
    }
    unit_lower_inverse64_v4<NT>(Af, Tf, X4, kMwLA);
    if constexpr (BWD) {  // T's rows out
        fence_proxy_async_smem();
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = lane + 32 * h;
                bulk_store_global(p.Tw + ci * 4096 + (size_t)t * 64, Tf + t * kMwLA, 256u);
            }
            tma_store_commit();
        }
    }
    // Tw = T diag(beta e^gamma) and Tu = T diag(beta) (rows a, columns 8 g ..,
    // item e: a = e / 8, g = e % 8) and the global loads of the sub-rows'
    // keys and values, all held in registers until T has been read
    constexpr int UT = 512 / NT, UK = 1024 / NT;
    uint4 th[UT][4];
    uint4 kg[UK], vg[UK];
#pragma unroll
    for (int u = 0; u < UK; ++u) {
        const int e = tid + NT * u, b = e >> 4, g = e & 15;
        const size_t src = MASKED ? htok + b / R : hrow + b;
        kg[u] = b < nrows ? ldg16(p.k + src * 128 + 8 * g) : z4;
        vg[u] = b < nrows ? ldg16(p.v + src * 128 + 8 * g) : z4;
    }
#pragma unroll
    for (int u = 0; u < UT; ++u) {
        const int e = tid + NT * u, a = e >> 3, g = e & 7;
        float w8[8], u8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b = 8 * g + i;
            const float t = b <= a ? Tf[a * kMwLA + b] : 0.f;
            u8[i] = t * bet[b];
            w8[i] = u8[i] * expf(gam[b]);
        }
        split8(w8, th[u][0], th[u][1]);
        split8(u8, th[u][2], th[u][3]);
    }
    if (warp == 0) tma_store_wait_read<0>();  // the staged Kd, P (K K^T, T) are overwritten below
    __syncthreads();
#pragma unroll
    for (int u = 0; u < UT; ++u) {
        const int e = tid + NT * u, a = e >> 3, g = e & 7;
        const uint32_t off = sw128_offset((uint32_t)a, (uint32_t)(8 * g));
#pragma unroll
        for (int h = 0; h < 4; ++h) *reinterpret_cast<uint4 *>(sm + MW_TW + 8192u * h + off) = th[u][h];
    }
    // Kr (hi | lo) and the sub-rows' values
#pragma unroll
    for (int u = 0; u < UK; ++u) {
        const int e = tid + NT * u, b = e >> 4, g = e & 15;
        const uint32_t off = (uint32_t)(g >> 3) * 8192u + sw128_offset((uint32_t)b, (uint32_t)((8 * g) & 63));
        *reinterpret_cast<uint4 *>(sm + MW_VS + off) = vg[u];
        float x[8];
        unpack8(kg[u], x);
        const float fr = nk[b] * (MASKED ? msk[(b % R) * R + ((g * R) >> 4)] : 1.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= fr;
        uint4 hi, lo;
        split8(x, hi, lo);
        *reinterpret_cast<uint4 *>(sm + MW_KR + off) = hi;
        *reinterpret_cast<uint4 *>(sm + MW_KR + 16384 + off) = lo;
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (tid == 0) {  // W = Tw Kr into columns 0..127 (lanes 0..63), U = Tu V into 128..255 (lanes 64..127)
        const uint32_t id = idesc_bf16(128, 128, false, true);
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t a = sb + MW_TW + (pr == 2 ? 8192u : 0u), b = sb + MW_KR + (pr == 1 ? 16384u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tmem, smem_desc(a + ks * 32, 16, 1024), smem_desc(b + ks * 2048, 8192, 1024), id,
                            (pr | ks) != 0);
        }
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            const uint32_t a = sb + MW_TW + 8192u + 8192u * pr;  // rows 64..127: Tu hi, then Tu lo
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tmem + 128, smem_desc(a + ks * 32, 16, 1024), smem_desc(sb + MW_VS + ks * 2048, 8192, 1024),
                            id, (pr | ks) != 0);
        }
        if constexpr (BWD) {  // Y^T = dO^T P (P^ hi | lo) into columns 256..319
            const uint32_t idy = idesc_bf16(128, 64, true, true);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr)
#pragma unroll
                for (int ks = 0; ks < NQ2 / 16; ++ks)
                    mma_bf16_ss(tmem + 256, smem_desc(sb + MW_DOI + ks * 2048, 8192, 1024),
                                smem_desc(sb + MW_PI + 8192u * pr + ks * 2048, 8192, 1024), idy, (pr | ks) != 0);
        }
        mma_commit(&bar[1]);
    }
    ok = warp_ok(wyc_wait(&bar[1], 0, 16u, p.timeout_ns));
    if (ok) {  // warp: lanes 32 (warp % 4) .. (W rows for quarters 0, 1; U rows for 2, 3), columns CW (warp / 4) ..
        constexpr int CW = 128 / CG;
        tc_fence_after_sync();
        const int c0 = CW * (warp >> 2), a = 32 * (q4 & 1) + lane;
        uint32_t x[CW];
#pragma unroll
        for (int h = 0; h < CW / 16; ++h)
            tmem_ld16(tmem + lb + (q4 < 2 ? 0u : 128u) + c0 + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(x + 16 * h));
        tmem_wait_ld();
        if (q4 < 2) {  // W's image, staged
#pragma unroll
            for (int h = 0; h < CW / 8; ++h) {
                float y[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = __uint_as_float(x[8 * h + i]);
                uint4 hi, lo;
                split8(y, hi, lo);
                const int c8 = c0 + 8 * h;
                const uint32_t off = (uint32_t)(c8 >> 6) * 8192u + sw128_offset((uint32_t)a, (uint32_t)(c8 & 63));
                *reinterpret_cast<uint4 *>(sm + MW_WS + off) = hi;
                *reinterpret_cast<uint4 *>(sm + MW_WS + 16384 + off) = lo;
            }
        } else {  // U's row a, staged
            float4 *Ur = reinterpret_cast<float4 *>(Us + a * kMwLU + c0);
#pragma unroll
            for (int h = 0; h < CW / 4; ++h)
                Ur[h] = make_float4(__uint_as_float(x[4 * h]), __uint_as_float(x[4 * h + 1]),
                                    __uint_as_float(x[4 * h + 2]), __uint_as_float(x[4 * h + 3]));
        }
        if constexpr (BWD) {  // Y^T row dv = lane of this quarter, columns 16 (warp / 4) ..: K-major operand
            uint32_t y[16];
            const int dv = 32 * q4 + lane, cy = 16 * (warp >> 2);
            tmem_ld16(tmem + lb + 256 + cy, y);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(y[8 * h + i]);
                uint4 hi, lo;
                split8(f, hi, lo);
                const uint32_t off = sw128_offset((uint32_t)dv, (uint32_t)(cy + 8 * h));
                *reinterpret_cast<uint4 *>(sm + MW_YI + off) = hi;
                *reinterpret_cast<uint4 *>(sm + MW_YI + 16384 + off) = lo;
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {  // W's image and U's rows out (lane: rows lane, lane + 32)
        if (lane == 0) bulk_store_global(p.Ww + ci * 8192, sm + MW_WS, 32768u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = lane + 32 * h;
            bulk_store_global(p.Uw + ci * 8192 + (size_t)r * 128, Us + r * kMwLU, 512u);
        }
        tma_store_commit();
    }
    if constexpr (BWD) {
        tc_fence_after_sync();
        if (tid == 0) {  // B^T = dO^T Q' - Y^T W into columns 384..511
            const uint32_t id1 = idesc_bf16(128, 128, true, true), id2 = idesc_bf16(128, 128, false, true, true);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr)
#pragma unroll
                for (int ks = 0; ks < NQ2 / 16; ++ks)
                    mma_bf16_ss(tmem + 384, smem_desc(sb + MW_DOI + ks * 2048, 8192, 1024),
                                smem_desc(sb + MW_QP + 16384u * pr + ks * 2048, 8192, 1024), id1, (pr | ks) != 0);
#pragma unroll
            for (int pr = 0; pr < 3; ++pr) {
                const uint32_t a = sb + MW_YI + (pr == 2 ? 16384u : 0u), b = sb + MW_WS + (pr == 1 ? 16384u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ss(tmem + 384, smem_desc(a + ks * 32, 16, 1024), smem_desc(b + ks * 2048, 8192, 1024),
                                id2, 1u);
            }
            mma_commit(&bar[2]);
        }
        ok = warp_ok(wyc_wait(&bar[2], 0, 16u, p.timeout_ns));
        if (ok) {  // B^T row dv = lane of this quarter, key columns 32 (warp / 4) ..: B[dk][dv]
            tc_fence_after_sync();
            const int dv = 32 * q4 + lane, k0 = 32 * (warp >> 2);
            float *Bg = p.Bw + ci * 16384 + dv;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t y[16];
                tmem_ld16(tmem + lb + 384 + k0 + 16 * h, y);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) Bg[(size_t)(k0 + 16 * h + i) * 128] = __uint_as_float(y[i]);
            }
        }
    }
    if (tid < 64) p.Gw[ci * 64 + tid] = gam[tid];
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tma_store_wait_all<0>();
        tc_fence_after_sync();
        tmem_dealloc(tmem, TCOLS);
    }
}

constexpr int kMoThr = 256;  // three CTAs per SM
constexpr uint32_t MO_S = 0;         // S: [2 value blocks][128 key rows][128 B] (bf16), 32 KB
constexpr uint32_t MO_VN = 32768;    // Vn: [2 value blocks][64 sub-rows][128 B] (bf16), 16 KB
constexpr uint32_t MO_Q = 49152;     // Q: [2 key blocks][nq2 query rows][128 B] (exact), 16 KB at most
constexpr uint32_t MO_P = 65536;     // P: [nq2 query rows][128 B] (bf16), 8 KB at most
constexpr uint32_t MO_VEC = 73728;   // gamma (64), query norms, then output row scales (64)
constexpr uint32_t MO_BAR = MO_VEC + 512;
constexpr uint32_t MO_SMEM = MO_BAR + 16 + 1024;
static_assert(3 * (MO_SMEM + 1024) <= 233472, "three output CTAs fit the shared memory of one SM");

__device__ __forceinline__ uint4 pack8(const float *x) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

// The output products take their operands in bf16 as the fused forward does
// (S, Vn and P rounded once; q exact), with fp32 accumulation.
__global__ void __launch_bounds__(kMoThr, 3) masked_out_tc_kernel(WyTcArgs p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *gam = reinterpret_cast<float *>(sm + MO_VEC), *sc = gam + 64;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + MO_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + MO_BAR + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, bh = blockIdx.y, r = p.r, Ct = p.Ct, nq2 = (Ct + 15) / 16 * 16;
    const int t0 = c * Ct, ntok = min(Ct, p.T - t0);
    const size_t htok = (size_t)bh * p.T + t0, ci = (size_t)bh * p.NT + c;

    if (tid == 0) {
        mbar_init(bar, 1u);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    if (tid < 64) gam[tid] = p.Gw[ci * 64 + tid];
    {  // S: key row m, value columns 8 g .. (element e: m = e / 16, g = e % 16), two batches of loads
        const float *Sg = p.Sw + ci * 16384;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = tid + kMoThr * (4 * half + u), m = e >> 4, k0 = 8 * (e & 15);
                v[2 * u] = *reinterpret_cast<const float4 *>(Sg + m * 128 + k0);
                v[2 * u + 1] = *reinterpret_cast<const float4 *>(Sg + m * 128 + k0 + 4);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = tid + kMoThr * (4 * half + u), m = e >> 4, k0 = 8 * (e & 15);
                const float x[8] = {v[2 * u].x,     v[2 * u].y,     v[2 * u].z,     v[2 * u].w,
                                    v[2 * u + 1].x, v[2 * u + 1].y, v[2 * u + 1].z, v[2 * u + 1].w};
                *reinterpret_cast<uint4 *>(sm + MO_S + (uint32_t)(k0 >> 6) * 16384u +
                                           sw128_offset((uint32_t)m, (uint32_t)(k0 & 63))) = pack8(x);
            }
        }
    }
    {  // Vn (sub-row b, value columns 8 g ..), P (query row t < nq2, columns 8 g ..) and Q
        const float *Vg = p.Vnw + ci * 8192, *Pg = p.Pw + ci * 4096;
        float4 v[8], pv[4];
        uint4 qw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = tid + kMoThr * u, b = e >> 4, k0 = 8 * (e & 15);
            v[2 * u] = *reinterpret_cast<const float4 *>(Vg + b * 128 + k0);
            v[2 * u + 1] = *reinterpret_cast<const float4 *>(Vg + b * 128 + k0 + 4);
            const int q = e >> 4;  // query row of Q (16 groups of 8 per row)
            qw[u] = q < ntok ? ldg16(p.q + (htok + q) * 128 + k0) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = tid + kMoThr * u, t = e >> 3, k0 = 8 * (e & 7);
            const bool in = t < nq2;
            pv[2 * u] = in ? *reinterpret_cast<const float4 *>(Pg + t * 64 + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
            pv[2 * u + 1] = in ? *reinterpret_cast<const float4 *>(Pg + t * 64 + k0 + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = tid + kMoThr * u, b = e >> 4, k0 = 8 * (e & 15);
            const float x[8] = {v[2 * u].x,     v[2 * u].y,     v[2 * u].z,     v[2 * u].w,
                                v[2 * u + 1].x, v[2 * u + 1].y, v[2 * u + 1].z, v[2 * u + 1].w};
            *reinterpret_cast<uint4 *>(sm + MO_VN + (uint32_t)(k0 >> 6) * 8192u +
                                       sw128_offset((uint32_t)b, (uint32_t)(k0 & 63))) = pack8(x);
            // Q row q = b and the query's norm
            const int q = b;
            float y[8];
            unpack8(qw[u], y);
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss += y[i] * y[i];
            ss = sum16(ss);
            if ((e & 15) == 0) sc[q] = p.l2 ? 1.f / fmaxf(sqrtf(ss), 1e-12f) : 1.f;  // m_q; the scale follows
            if (q < nq2)
                *reinterpret_cast<uint4 *>(sm + MO_Q + (uint32_t)(k0 >> 6) * (uint32_t)(nq2 * 128) +
                                           sw128_offset((uint32_t)q, (uint32_t)(k0 & 63))) = qw[u];
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = tid + kMoThr * u, t = e >> 3, k0 = 8 * (e & 7);
            if (t < nq2) {
                const float x[8] = {pv[2 * u].x,     pv[2 * u].y,     pv[2 * u].z,     pv[2 * u].w,
                                    pv[2 * u + 1].x, pv[2 * u + 1].y, pv[2 * u + 1].z, pv[2 * u + 1].w};
                *reinterpret_cast<uint4 *>(sm + MO_P + sw128_offset((uint32_t)t, (uint32_t)k0)) = pack8(x);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    if (tid == 0) {  // S^T Q^T into columns 0.., Vn^T P^T into 64..
        const uint32_t id = idesc_bf16(128, nq2, true, false);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(tmem, smem_desc(sb + MO_S + ks * 2048, 16384, 1024),
                        smem_desc(sb + MO_Q + (ks >> 2) * (nq2 * 128) + (ks & 3) * 32, 16, 1024), id, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem + 64, smem_desc(sb + MO_VN + ks * 2048, 8192, 1024),
                        smem_desc(sb + MO_P + ks * 32, 16, 1024), id, ks > 0);
        mma_commit(bar);
    }
    if (tid < 64) sc[tid] = tid < ntok ? p.scale * expf(gam[tid * r]) * sc[tid] : 0.f;  // row scales
    __syncthreads();
    const bool ok = warp_ok(wyc_wait(bar, 0, 16u, p.timeout_ns));
    if (ok) {  // value row dv = TMEM lane; query columns 16 j .. for j = warp / 4, + 2, ..
        tc_fence_after_sync();
        const int q4 = warp & 3, dv = 32 * q4 + lane;
        const uint32_t lb = (uint32_t)(32 * q4) << 16;
        unsigned short *op = p.o + htok * 128 + dv;
        for (int j = warp >> 2; j < nq2 / 16; j += 2) {
            uint32_t x1[16], x2[16];
            tmem_ld16(tmem + lb + 16 * j, x1);
            tmem_ld16(tmem + lb + 64 + 16 * j, x2);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = 16 * j + i;
                if (t < ntok)
                    op[(size_t)t * 128] = __bfloat16_as_ushort(
                        __float2bfloat16_rn(sc[t] * __uint_as_float(x1[i]) + __uint_as_float(x2[i])));
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 128);
    }
}

bool wy_tc_args_ok(const WyTcArgs &a) {
    return a.BH > 0 && a.NT > 0 && a.r >= 1 && a.r <= 8 && 64 % a.r == 0 && a.Ct == 64 / a.r;
}

template <bool MASKED, bool BWD>
void (*wy_tc_pick(int r))(WyTcArgs) {
    return r == 1 ? wy_tc_kernel<1, MASKED, BWD>
           : r == 2 ? wy_tc_kernel<2, MASKED, BWD>
           : r == 4 ? wy_tc_kernel<4, MASKED, BWD>
                    : wy_tc_kernel<8, MASKED, BWD>;
}

}  // namespace

int launch_wy_tc(const WyTcArgs &a, cudaStream_t st) {
    if (!wy_tc_args_ok(a)) return GDN_ERR_INVALID_ARG;
    if (!a.masked && !a.bwd) return GDN_ERR_UNSUPPORTED;  // the GDN / DeltaProduct forward is fused (scan_tc.cu)
    WyTcArgs p = a;
    p.timeout_ns = wait_limit_ns();
    void (*kern)(WyTcArgs) = a.bwd ? (a.masked ? wy_tc_pick<true, true>(a.r) : wy_tc_pick<false, true>(a.r))
                                   : wy_tc_pick<true, false>(a.r);
    const uint32_t smem = mw_smem(a.bwd != 0);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<dim3((unsigned)a.NT, (unsigned)a.BH), a.bwd ? 512 : 256, smem, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int launch_masked_out_tc(const WyTcArgs &a, cudaStream_t st) {
    if (!wy_tc_args_ok(a)) return GDN_ERR_INVALID_ARG;
    WyTcArgs p = a;
    p.timeout_ns = wait_limit_ns();
    if (cudaFuncSetAttribute(masked_out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MO_SMEM) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    masked_out_tc_kernel<<<dim3((unsigned)a.NT, (unsigned)a.BH), kMoThr, MO_SMEM, st>>>(p);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
