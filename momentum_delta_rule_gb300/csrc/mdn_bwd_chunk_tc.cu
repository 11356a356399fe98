// MDN gradient pass — the per-chunk products on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA-staged operands), bf16 inputs, head
// size 64 or 128.  One CTA per (chunk, head), after the reverse chain has
// left dR (= dV) and the state adjoints dS, dM at every chunk's end.
//
// The vector-Jacobian product of the chunk equations ("MDN: Parallelizing
// Stepwise Momentum for Delta Linear Attention" slides, frames "Solve the
// unknown residuals with a lower triangular system", Eqs. (15)-(18), and
// "Chunk outputs combine incoming states and local writes", Appendix C
// Eqs. (40)-(42)), with P = Diag(alpha) K, Kh = Diag(eta) K and the chunk's
// entry states S0, M0 (saved by the forward in bf16, copied straight into
// their operand tiles), as seven products over operands in their stored
// layouts (the [K; Q] and [dO; dR] tiles in the tc_row order):
//
//   MMA1  [K; Q] S0, [K; Q] M0   R  = V - Diag(abar_m) P S0 + Diag(b_m) P M0
//   MMA3  [dO; dR] S0^T, M0^T    dQs = Diag(abar) dO S0^T - Diag(b) dO M0^T
//                                dPs = -Diag(abar_m) dR S0^T + Diag(b_m) dR M0^T
//   MMA2  T R                    Vres
//   MMA4  Vres dS^T, Vres dM^T   dKc = Diag(gS) Vres dS^T - Diag(mu_tail) Vres dM^T
//   MMA5  [dO; dR] Vres^T        dA = dO Vres^T, dL = -dR Vres^T
//                                dY = dA . Gamma, dX = dL . Gamma_m
//   MMA6  [dQ; dP] += [dY Diag(eta); dX Diag(eta)] K
//   MMA7  dKh = dKc + dY^T Q + (Diag(alpha) dX)^T K   (over the 128 staged rows)
//         dK = Diag(alpha) dP + Diag(eta) dKh
//
// and the row sums the gates' gradients need (the adjoints of abar, b, their
// shifted copies, gS and mu_tail, d alpha|_P = rowsum(dP . K), d eta =
// rowsum(dKh . K)), the inner products <S0, dS>, <M0, dS>, <M0, dM>, and the
// products dA . Y and dL . X, written over matrices of the gradient block
// that are dead by then (see bwd_gates_kernel for the layout).
//
// Warp roles: warp 0 issues the TMA copies, warp 1 owns TMEM and issues the
// MMAs, warps 2-9 run the epilogues (two warps per 32-lane TMEM quadrant,
// each on half the columns).  Every wait is bounded.
#include <cudaTypedefs.h>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

using namespace sm100;
using BL = BwdLayout;
constexpr int C = kChunk;
constexpr uint32_t kHalf = 16384;      // 128 staged rows x 64 bf16 columns
constexpr uint32_t kTokHalf = 8192;    // 64 token rows x 64 bf16 columns

// Row sums, in the order of the gradient block's A slot.
enum { sAbar = 0, sB, sAbarM, sBM, sGLast, sMuTail, sDa, sDe, kSums = 8 };

template <int D>
struct GradCfg {
    static_assert(D == 64 || D == 128, "head size");
    static constexpr int kHalves = D / 64;
    static constexpr uint32_t kStage = kHalves * kHalf;     // [K; Q] or [dO; dR]
    static constexpr uint32_t kStateHalf = D * 128;         // D rows x 64 columns
    static constexpr uint32_t kState = kHalves * kStateHalf;
    static constexpr uint32_t kTok = kHalves * kTokHalf;    // 64 rows x D
    static constexpr uint32_t kOffKQ = 0;
    static constexpr uint32_t kOffOR = kOffKQ + kStage;
    static constexpr uint32_t kOffS0 = kOffOR + kStage;
    static constexpr uint32_t kOffM0 = kOffS0 + kState;
    static constexpr uint32_t kOffDS = kOffM0 + kState;
    static constexpr uint32_t kOffDM = kOffDS + kState;
    static constexpr uint32_t kOffV = kOffDM + kState;     // V, then R in place
    // Once MMA1 and MMA3 are done: the forward prep's [T; A_O T] tile and
    // Vres over S0, the key tile of the Gram product over M0 (then the
    // operands of MMA6 and MMA7 over M0 once the Gram product is done),
    // where the head size leaves those regions the room; else beside.
    static constexpr bool kOverlay = kState >= 2 * kHalf;
    static constexpr uint32_t kOffTile = kOverlay ? kOffS0 : kOffV + kTok;
    static constexpr uint32_t kOffVres = kOverlay ? kOffS0 + kHalf : kOffS0;
    static constexpr uint32_t kOffKt = kOffM0;
    static constexpr uint32_t kOffA6 = kOverlay ? kOffM0 : kOffTile + kHalf;
    static constexpr uint32_t kOffA7 = kOffA6 + kHalf;
    // Gamma (fp32 64 x 64) over V once MMA2 is done, where V has the room
    static constexpr uint32_t kOffGam = kOverlay ? kOffV : kOffA7 + kHalf;
    // dA . Y and dL . X (fp32, 64 x 64 each, in two 32-column boxes) staged
    // for their TMA stores over dS, dM once MMA4 is done, where those have
    // the room; dQ and dK (bf16) over [dO; dR] once MMA5 is done
    static constexpr uint32_t kOffWst = kOverlay ? kOffDS : kOffGam + 16384;
    static constexpr uint32_t kOffQKst = kOffOR;
    static constexpr uint32_t kOffCoef = kOverlay ? kOffV + kTok : kOffWst + 2 * kHalf;
    // coefficients (vector rows, alpha, eta), the two column halves' row sums,
    // per-warp inner products
    static constexpr int kCoefFloats = BL::kRows * C + 2 * C + 2 * kSums * C + 8 * 4;
    static constexpr uint32_t kOffBar = kOffCoef + ((kCoefFloats * 4 + 127) / 128) * 128;
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
    static_assert(kOffVres + kTok <= kOffM0 && kTok <= kState, "overlays");
    static_assert(!kOverlay || (kOffA7 + kHalf <= kOffDS && kTok >= 16384 && 2 * kState >= 2 * kHalf),
                  "overlays");
    static_assert(kStage == 2 * kTok, "dQ, dK staging");
    static constexpr uint32_t kColS1 = 0, kColM1 = D, kColS3 = 2 * D, kColM3 = 3 * D;
    static constexpr uint32_t kColG = 3 * D + 64 > 4 * D - 64 ? 4 * D : 3 * D + 64;  // Gram, 64 columns
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kThreads = 320;
    // copies: [K; Q] and the entry-state tiles (MMA1); [dO; dR] and V (MMA3,
    // the first epilogue); the adjoint tiles (MMA4)
    static constexpr uint32_t kTxFull = kStage + 2 * kState;
    static constexpr uint32_t kTxO = kStage + kTok;
    static constexpr uint32_t kTxAdj = 2 * kState;
    static constexpr uint32_t kTx2Bytes = kHalf + kTok;
    static_assert(kColG + 64 <= kTmemCols, "TMEM columns");
    static constexpr uint32_t kIdescKS = idesc_bf16(128, D, false, true);   // MMA1, MMA6
    static constexpr uint32_t kIdescKK = idesc_bf16(128, D, false, false);  // MMA3
    static constexpr uint32_t kIdescT = idesc_bf16(128, D, false, true);    // MMA2
    static constexpr uint32_t kIdescG = idesc_bf16(128, 64, false, false);  // Gram
    static constexpr uint32_t kIdescV = idesc_bf16(64, D, false, false);    // MMA4
    static constexpr uint32_t kIdescA = idesc_bf16(128, 64, false, false);  // MMA5
    static constexpr uint32_t kIdesc7 = idesc_bf16(64, D, true, true);      // MMA7
};

struct GradBars {
    uint64_t full, fullo, fulla, full2, full3, rd, d13, r, d2, v, d45, y, d67, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(GradBars) <= 256, "barrier block");

__device__ __forceinline__ uint32_t pk2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 16 bf16 values of row `row`, 16-byte chunks c0 and c0 + 1, of a
// 128-byte-swizzled tile, as fp32.
__device__ __forceinline__ void get16(const unsigned char *tile, int row, uint32_t c0, float *f) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(tile + sw128_offset((uint32_t)row, c0 + u));
        const __nv_bfloat162 *hv = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __bfloat1622float2(hv[i]);
            f[8 * u + 2 * i] = t.x;
            f[8 * u + 2 * i + 1] = t.y;
        }
    }
}

__device__ __forceinline__ void get8(const unsigned char *tile, int row, uint32_t chunk, float *f) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(tile + sw128_offset((uint32_t)row, chunk));
    const __nv_bfloat162 *hv = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(hv[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void put8(unsigned char *tile, int row, uint32_t chunk, const float *x) {
    *reinterpret_cast<uint4 *>(tile + sw128_offset((uint32_t)row, chunk)) =
        make_uint4(pk2(x[0], x[1]), pk2(x[2], x[3]), pk2(x[4], x[5]), pk2(x[6], x[7]));
}

__device__ __forceinline__ void put16(unsigned char *tile, int row, uint32_t c0, const float *x) {
    put8(tile, row, c0, x);
    put8(tile, row, c0 + 1, x + 8);
}

// 16 fp32 values of row t, columns 16 cc .. 16 cc + 15 of a 32-column box
// (64 rows x 128 bytes, 128-byte swizzled) staged for a TMA store.
__device__ __forceinline__ void stage_w(unsigned char *box, int t, int cc, const float *w) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(box + sw128_offset((uint32_t)t, (uint32_t)(4 * cc + i))) =
            make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// The same 16 values read back.
__device__ __forceinline__ void get_w(const unsigned char *box, int t, int cc, float *w) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 v =
            *reinterpret_cast<const float4 *>(box + sw128_offset((uint32_t)t, (uint32_t)(4 * cc + i)));
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
}

__device__ __forceinline__ void store16_bf16(void *g, const float *x) {
    uint4 *d = reinterpret_cast<uint4 *>(g);
    d[0] = make_uint4(pk2(x[0], x[1]), pk2(x[2], x[3]), pk2(x[4], x[5]), pk2(x[6], x[7]));
    d[1] = make_uint4(pk2(x[8], x[9]), pk2(x[10], x[11]), pk2(x[12], x[13]), pk2(x[14], x[15]));
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Named barrier of the eight epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(GradCfg<D>::kThreads, 1)
bwd_chunk_tc_kernel(const BwdProblem p, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_o,
                    const __grid_constant__ CUtensorMap map_r,
                    const __grid_constant__ CUtensorMap map_v,
                    const __grid_constant__ CUtensorMap map_kt,
                    const __grid_constant__ CUtensorMap map_dq,
                    const __grid_constant__ CUtensorMap map_dk,
                    const __grid_constant__ CUtensorMap map_wy,
                    const __grid_constant__ CUtensorMap map_wx,
                    const __grid_constant__ CUtensorMap map_gam,
                    const __grid_constant__ CUtensorMap map_s0,
                    const __grid_constant__ CUtensorMap map_m0) {
    using G = GradCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem_1024(smem_raw);
    GradBars *bars = reinterpret_cast<GradBars *>(smem + G::kOffBar);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int gc, h;
    chunk_head_of_block(p.loc.H, gc, h);
    const int H = p.loc.H;
    ChunkLoc loc;
    if (!locate_chunk_cta(p.loc, gc, loc)) return;      // the whole CTA, before any barrier
    const int n = loc.n, t0 = loc.t0;
    float *blk = reinterpret_cast<float *>(p.prep + ((size_t)gc * H + h) * BL::kBytes);

    if (threadIdx.x == 0) {
        mbar_init(&bars->full, 1);
        mbar_init(&bars->fullo, 1);
        mbar_init(&bars->fulla, 1);
        mbar_init(&bars->rd, 8);
        mbar_init(&bars->full2, 1);
        mbar_init(&bars->full3, 1);
        mbar_init(&bars->d13, 1);
        mbar_init(&bars->r, 8);
        mbar_init(&bars->d2, 1);
        mbar_init(&bars->v, 8);
        mbar_init(&bars->d45, 1);
        mbar_init(&bars->y, 8);
        mbar_init(&bars->d67, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_o);
        prefetch_tensormap(&map_r);
        prefetch_tensormap(&map_v);
        prefetch_tensormap(&map_kt);
        prefetch_tensormap(&map_gam);
        prefetch_tensormap(&map_s0);
        prefetch_tensormap(&map_m0);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, G::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars->full, G::kTxFull);
            unsigned char *kq = smem + G::kOffKQ, *orr = smem + G::kOffOR;
            const int bi = gc * H + h;
            // [K; Q] and the chunk's entry states (bf16 [dk, dv] rows; the
            // copy lays them out as the swizzled MN-major operand tiles)
#pragma unroll
            for (int hh = 0; hh < G::kHalves; ++hh) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint32_t off = hh * kHalf + g * 4096;
                    tma_load_3d(kq + off, &map_k, &bars->full, 64 * hh, h, t0 + 16 * g);
                    tma_load_3d(kq + off + 2048, &map_q, &bars->full, 64 * hh, h, t0 + 16 * g);
                }
                tma_load_3d(smem + G::kOffS0 + hh * G::kStateHalf, &map_s0, &bars->full, 64 * hh, 0, bi);
                tma_load_3d(smem + G::kOffM0 + hh * G::kStateHalf, &map_m0, &bars->full, 64 * hh, 0, bi);
            }
            // [dO; dR] and V
            mbar_arrive_expect_tx(&bars->fullo, G::kTxO);
#pragma unroll
            for (int hh = 0; hh < G::kHalves; ++hh) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint32_t off = hh * kHalf + g * 4096;
                    tma_load_3d(orr + off, &map_o, &bars->fullo, 64 * hh, h, t0 + 16 * g);
                    tma_load_3d(orr + off + 2048, &map_r, &bars->fullo, 64 * hh, h, t0 + 16 * g);
                }
                tma_load_3d(smem + G::kOffV + hh * kTokHalf, &map_v, &bars->fullo, 64 * hh, h, t0);
            }
            // the adjoints at the chunk's end as the reverse chain left them
            // (bf16 operand tiles dS, dM)
            mbar_arrive_expect_tx(&bars->fulla, G::kTxAdj);
            const unsigned char *adj = reinterpret_cast<const unsigned char *>(p.adj) +
                                       ((size_t)gc * H + h) * 2 * G::kState;
            bulk_load(smem + G::kOffDS, adj, G::kState, &bars->fulla);
            bulk_load(smem + G::kOffDM, adj + G::kState, G::kState, &bars->fulla);
            // once MMA1, MMA3 and the epilogue have read the states: the
            // operand tile of the forward prep and the 64 key rows of the
            // Gram product, over them
            bool go = mbar_wait(&bars->d13, 0, abort) && mbar_wait(&bars->rd, 0, abort);
            if (go) {
                mbar_arrive_expect_tx(&bars->full2, G::kTx2Bytes);
                const unsigned char *tile =
                    p.fwd_tile ? p.fwd_tile + ((size_t)gc * H + h) * p.fwd_tile_stride
                               : p.tcblk + ((size_t)gc * H + h) * BwdChainLayout::kBytes;
                bulk_load(smem + G::kOffTile, tile + BwdChainLayout::kOffTile, kHalf, &bars->full2);
#pragma unroll
                for (int hh = 0; hh < G::kHalves; ++hh)
                    tma_load_3d(smem + G::kOffKt + hh * kTokHalf, &map_kt, &bars->full2, 64 * hh, h, t0);
            }
            // once MMA2 has read R: Gamma over V
            bool go3 = go && mbar_wait(&bars->d2, 0, abort);
            if (go3) {
                // Gamma as two 32-column boxes, 128-byte swizzled (a row per
                // lane reads without bank conflicts)
                mbar_arrive_expect_tx(&bars->full3, 16384);
                tma_load_3d(smem + G::kOffGam, &map_gam, &bars->full3, 0, 0, gc * H + h);
                tma_load_3d(smem + G::kOffGam + 8192, &map_gam, &bars->full3, 32, 0, gc * H + h);
            }
            int dummy = 0;
            mbar_wait(&bars->full, 0, &dummy);     // no copy in flight at exit
            mbar_wait(&bars->fullo, 0, &dummy);
            mbar_wait(&bars->fulla, 0, &dummy);
            if (go) mbar_wait(&bars->full2, 0, &dummy);
            if (go3) mbar_wait(&bars->full3, 0, &dummy);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        const bool l0 = lane == 0;
        const uint32_t kq = smem_u32(smem + G::kOffKQ), orr = smem_u32(smem + G::kOffOR);
        const uint32_t s0 = smem_u32(smem + G::kOffS0), m0 = smem_u32(smem + G::kOffM0);
        const uint32_t ds = smem_u32(smem + G::kOffDS), dm = smem_u32(smem + G::kOffDM);
        const uint32_t vt = smem_u32(smem + G::kOffV), tt = smem_u32(smem + G::kOffTile);
        const uint32_t kt = smem_u32(smem + G::kOffKt);
        const uint32_t vr = smem_u32(smem + G::kOffVres);
        const uint32_t a6 = smem_u32(smem + G::kOffA6), a7 = smem_u32(smem + G::kOffA7);
        constexpr uint32_t kLboS = G::kHalves > 1 ? G::kStateHalf : 8192;
        constexpr int kSteps = D / 16;
        bool ok = warp_wait(&bars->full, 0, abort);
        if (ok) {
            tc_fence_after();
            if (l0) {
                // MMA1: [K; Q] S0 and [K; Q] M0 (B: the state tiles, rows k)
#pragma unroll
                for (int s = 0; s < kSteps; ++s) {
                    const uint64_t a = sdesc_sw128(kq + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024);
                    mma_bf16(tmem + G::kColS1, a, sdesc_sw128(s0 + s * 2048, kLboS, 1024), G::kIdescKS, s != 0);
                    mma_bf16(tmem + G::kColM1, a, sdesc_sw128(m0 + s * 2048, kLboS, 1024), G::kIdescKS, s != 0);
                }
            }
            __syncwarp();
            ok = warp_wait(&bars->fullo, 0, abort);
        }
        if (ok) {
            tc_fence_after();
            if (l0) {
                // MMA3: [dO; dR] S0^T and [dO; dR] M0^T (B: the same tiles, K-major)
#pragma unroll
                for (int s = 0; s < kSteps; ++s) {
                    const uint32_t kofs = (s >> 2) * G::kStateHalf + (s & 3) * 32;
                    const uint64_t a = sdesc_sw128(orr + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024);
                    mma_bf16(tmem + G::kColS3, a, sdesc_sw128(s0 + kofs, 16, 1024), G::kIdescKK, s != 0);
                    mma_bf16(tmem + G::kColM3, a, sdesc_sw128(m0 + kofs, 16, 1024), G::kIdescKK, s != 0);
                }
                mma_commit(&bars->d13);
            }
            __syncwarp();
            ok = warp_wait(&bars->r, 0, abort) && warp_wait(&bars->full2, 0, abort);
        }
        if (ok) {
            tc_fence_after();
            if (l0) {
                // MMA2: [T; A_O T] R (the T rows give Vres); the Gram
                // product [K; Q] K^T (B: the key tile, K-major)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + G::kColS1, sdesc_sw128(tt + s * 32, 16, 1024),
                             sdesc_sw128(vt + s * 2048, kTokHalf, 1024), G::kIdescT, s != 0);
#pragma unroll
                for (int s = 0; s < kSteps; ++s)
                    mma_bf16(tmem + G::kColG, sdesc_sw128(kq + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024),
                             sdesc_sw128(kt + (s >> 2) * kTokHalf + (s & 3) * 32, 16, 1024), G::kIdescG,
                             s != 0);
                mma_commit(&bars->d2);
            }
            __syncwarp();
            ok = warp_wait(&bars->v, 0, abort) && warp_wait(&bars->fulla, 0, abort);
        }
        if (ok) {
            tc_fence_after();
            if (l0) {
                // MMA4: Vres dS^T, Vres dM^T; MMA5: [dO; dR] Vres^T
#pragma unroll
                for (int s = 0; s < kSteps; ++s) {
                    const uint32_t kofs = (s >> 2) * G::kStateHalf + (s & 3) * 32;
                    const uint64_t a = sdesc_sw128(vr + (s >> 2) * kTokHalf + (s & 3) * 32, 16, 1024);
                    mma_bf16(tmem + G::kColS1, a, sdesc_sw128(ds + kofs, 16, 1024), G::kIdescV, s != 0);
                    mma_bf16(tmem + G::kColM1, a, sdesc_sw128(dm + kofs, 16, 1024), G::kIdescV, s != 0);
                }
#pragma unroll
                for (int s = 0; s < kSteps; ++s)
                    mma_bf16(tmem + G::kColM3, sdesc_sw128(orr + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024),
                             sdesc_sw128(vr + (s >> 2) * kTokHalf + (s & 3) * 32, 16, 1024), G::kIdescA,
                             s != 0);
                mma_commit(&bars->d45);
            }
            __syncwarp();
            ok = warp_wait(&bars->y, 0, abort);
        }
        if (ok) {
            tc_fence_after();
            if (l0) {
                // MMA6: [dQ; dP] += [dY eta; dX eta] K (B: the key rows of the
                // [K; Q] tile, 16 tokens per step)
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    mma_bf16(tmem + G::kColS3, sdesc_sw128(a6 + g * 32, 16, 1024),
                             sdesc_sw128(kq + g * 4096, kHalf, 1024), G::kIdescKS, 1);
                // MMA7: dKh += [alpha dX | dY]^T [K; Q] over the 128 staged rows
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16(tmem + G::kColS1, sdesc_sw128(a7 + s * 2048, kHalf, 1024),
                             sdesc_sw128(kq + s * 2048, kHalf, 1024), G::kIdesc7, 1);
                mma_commit(&bars->d67);
                // dA . Y and dL . X, staged by every epilogue warp before it
                // arrived: into the gradient block
                const int bi = gc * H + h;
                const unsigned char *wst = smem + G::kOffWst;
                tma_store_3d(&map_wy, wst, 0, 0, bi);
                tma_store_3d(&map_wy, wst + 8192, 32, 0, bi);
                tma_store_3d(&map_wx, wst + kHalf, 0, 0, bi);
                tma_store_3d(&map_wx, wst + kHalf + 8192, 32, 0, bi);
                bulk_commit_group();
            }
            __syncwarp();
        }
        if (l0) {
            mma_commit(&bars->drain);
            int dummy = 0;
            mbar_wait(&bars->drain, 0, &dummy);
            bulk_wait_group_read0();     // the staged W tiles stay until read
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps
        const int e = threadIdx.x - 64;
        const int q = warp & 3, ch = (warp - 2) >> 2;
        const bool first = lane < 16;            // K / dO row (else Q / dR row) of token t
        const int t = 16 * q + (lane & 15);
        const bool in = t < n;
        const int rowK = tc_row(t), rowQ = tc_row(C + t);
        const uint32_t lb = tmem + ((uint32_t)(32 * q) << 16);
        float *vec = reinterpret_cast<float *>(smem + G::kOffCoef);
        float *ga = vec + BL::kRows * C, *ge = ga + C;
        float *rowpart = ge + C, *red = rowpart + 2 * kSums * C;
        const unsigned char *kq = smem + G::kOffKQ, *orr = smem + G::kOffOR;
        float sc[3] = {0.f, 0.f, 0.f};

        // ---- the entry-state tiles (bf16), the inner products with the
        //      adjoint tiles, the coefficients
        {
            // the coefficients first (their latency overlaps the states')
            float vpre[BL::kRows * C / 256];
#pragma unroll
            for (int u = 0; u < BL::kRows * C / 256; ++u) vpre[u] = blk[BL::kMats * BL::kMat + e + 256 * u];
            float g_a = 0.f, g_e = 0.f;
            if (e < n) {
                const size_t gi = (size_t)(t0 + e) * H + h;
                g_a = p.alpha[gi];
                g_e = p.eta[gi];
            }
            const unsigned char *s0t = smem + G::kOffS0, *m0t = smem + G::kOffM0;
            const unsigned char *dst = smem + G::kOffDS, *dmt = smem + G::kOffDM;
            constexpr int kCh = D / 8;
            constexpr int kIter = D * kCh / 256;         // 16-byte chunks of a tile per thread
            float s[kIter][8], m[kIter][8];
            bool have = warp_wait(&bars->full, 0, abort);
            if (have) {
#pragma unroll
                for (int u = 0; u < kIter; ++u) {
                    const int idx = e + 256 * u;
                    const int k = idx / kCh, c8 = idx % kCh;
                    const uint32_t off = (c8 >> 3) * G::kStateHalf;
                    get8(s0t + off, k, c8 & 7, s[u]);
                    get8(m0t + off, k, c8 & 7, m[u]);
                }
            }
            // the state tiles are read: later copies may land over them
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->rd);
            // <S0, dS>, <M0, dS>, <M0, dM> while MMA1 and MMA3 run
            if (have && mbar_wait(&bars->fulla, 0, abort)) {
#pragma unroll
                for (int u = 0; u < kIter; ++u) {
                    const int idx = e + 256 * u;
                    const int k = idx / kCh, c8 = idx % kCh;
                    const uint32_t off = (c8 >> 3) * G::kStateHalf;
                    float a[8], b[8];
                    get8(dst + off, k, c8 & 7, a);
                    get8(dmt + off, k, c8 & 7, b);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        sc[0] = fmaf(s[u][v], a[v], sc[0]);
                        sc[1] = fmaf(m[u][v], a[v], sc[1]);
                        sc[2] = fmaf(m[u][v], b[v], sc[2]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < BL::kRows * C / 256; ++u) vec[e + 256 * u] = vpre[u];
            if (e < C) {
                ga[e] = g_a;
                ge[e] = g_e;
            }
        }
        epi_sync();                          // the coefficients are in shared memory
        const float a_t = ga[t], e_t = ge[t];
        const float abar = vec[BL::vAbar * C + t], bb = vec[BL::vB * C + t];
        const float abm = vec[BL::vAbarM * C + t], bm = vec[BL::vBM * C + t];
        const float gs = vec[BL::vGS * C + t], mt = vec[BL::vMuTail * C + t];
        float acc0 = 0.f, acc1 = 0.f;        // first: d abar_m, d b_m; else d abar, d b
        float rg = 0.f, rm = 0.f;            // first: gS and mu_tail sums (before eta)
        float dsum = 0.f;                    // first: d eta; else d alpha|_P
        constexpr int kCC = D / 32;          // 16-column chunks of this thread's half
        const int j0 = ch * (D / 2);

        // ---- R and the state terms of dQ, dP
        bool ok = warp_wait(&bars->fullo, 0, abort) && warp_wait(&bars->d13, 0, abort);
        if (ok) {
            tc_fence_after();
            unsigned char *vt = smem + G::kOffV;
#pragma unroll 1
            for (int cc = 0; cc < kCC; ++cc) {
                const int j = j0 + 16 * cc;
                const int hh = j >> 6;
                const uint32_t c0 = (uint32_t)((j & 63) >> 3);
                float xs[16], xm[16], ys[16], ym[16];
                __syncwarp();
                tmem_ld16(lb + G::kColS1 + j, xs);
                tmem_ld16(lb + G::kColM1 + j, xm);
                tmem_ld16(lb + G::kColS3 + j, ys);
                tmem_ld16(lb + G::kColM3 + j, ym);
                tmem_ld_wait();
                if (first) {
                    float v[16], r[16];
                    get16(vt + hh * kTokHalf, t, c0, v);
                    get16(orr + hh * kHalf, rowQ, c0, r);          // dR row t
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float ps = a_t * xs[u], pm = a_t * xm[u];
                        v[u] = in ? v[u] - abm * ps + bm * pm : 0.f;
                        if (in) {
                            acc0 = fmaf(-r[u], ps, acc0);
                            acc1 = fmaf(r[u], pm, acc1);
                        }
                    }
                    put16(vt + hh * kTokHalf, t, c0, v);
                } else if (in) {
                    float o[16];
                    get16(orr + hh * kHalf, rowK, c0, o);          // dO row t
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        acc0 = fmaf(xs[u], o[u], acc0);
                        acc1 = fmaf(-xm[u], o[u], acc1);
                    }
                }
                const float cS = first ? abar : -abm, cM = first ? -bb : bm;
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 16; ++u) ys[u] = in ? cS * ys[u] + cM * ym[u] : 0.f;
                tmem_st16(lb + G::kColS3 + j, ys);
            }
            tmem_st_wait();
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->r);
        }

        // ---- Vres (bf16, rows past n zero)
        if (ok) ok = warp_wait(&bars->d2, 0, abort);
        if (ok) {
            tc_fence_after();
            unsigned char *vr = smem + G::kOffVres;
#pragma unroll 1
            for (int cc = 0; cc < kCC; ++cc) {
                const int j = j0 + 16 * cc;
                float x[16];
                __syncwarp();
                tmem_ld16(lb + G::kColS1 + j, x);
                tmem_ld_wait();
                if (first) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) x[u] = in ? x[u] : 0.f;
                    put16(vr + (j >> 6) * kTokHalf, t, (uint32_t)((j & 63) >> 3), x);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->v);
        }

        // ---- dKc, the carry sums, dY and dX
        if (ok) ok = warp_wait(&bars->d45, 0, abort);
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < kCC; ++cc) {
                const int j = j0 + 16 * cc;
                float u1[16], u2[16];
                __syncwarp();
                tmem_ld16(lb + G::kColS1 + j, u1);
                tmem_ld16(lb + G::kColM1 + j, u2);
                tmem_ld_wait();
                if (first && in) {
                    float kk[16];
                    get16(kq + (j >> 6) * kHalf, rowK, (uint32_t)((j & 63) >> 3), kk);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        rg = fmaf(kk[u], u1[u], rg);
                        rm = fmaf(-kk[u], u2[u], rm);
                        u1[u] = gs * u1[u] - mt * u2[u];
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) u1[u] = 0.f;
                }
                __syncwarp();
                tmem_st16(lb + G::kColS1 + j, u1);
            }
            tmem_st_wait();
            ok = warp_wait(&bars->full3, 0, abort);         // Gamma in shared memory
        }
        if (ok) {
            // W1 = dA . Y, Y = (Q K^T) Diag(eta), and W2 = dL . X, X = Diag(alpha)
            // (K K^T) Diag(eta), for the gates (the Gram rows of the other
            // half-warp: each token's key and query rows share a warp)
            const unsigned char *Gm = smem + G::kOffGam;
            // this thread's W rows: dA . Y in the first 16 KB, dL . X in the
            // second, column box ch
            unsigned char *wst = smem + G::kOffWst + (first ? 0u : (uint32_t)kHalf) + ch * 8192;
            unsigned char *a6 = smem + G::kOffA6, *a7 = smem + G::kOffA7;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int m0 = 32 * ch + 16 * cc;
                const uint32_t c0 = (uint32_t)(m0 >> 3);
                float x[16], g[16], w[16], y[16], ys[16];
                __syncwarp();
                tmem_ld16(lb + G::kColM3 + m0, x);
                tmem_ld16(lb + G::kColG + m0, w);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) w[u] = __shfl_xor_sync(0xffffffffu, w[u], 16);
                if (first) {
                    // dA row t: dY = dA . Gamma, and dA . Y for the gates
                    get_w(Gm + ch * 8192, t, cc, g);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int m = m0 + u;
                        const bool on = in && m <= t;
                        y[u] = on ? x[u] * g[u] : 0.f;
                        w[u] = on ? x[u] * w[u] * ge[m] : 0.f;
                        ys[u] = y[u] * ge[m];
                    }
                    stage_w(wst, t, cc, w);
                    put16(a6, rowK, c0, ys);
                    put16(a7, rowQ, c0, y);
                } else {
                    // dL row t (= -(dR Vres^T)): dX = dL . Gamma_m, and dL . X
                    get_w(Gm + ch * 8192, t > 0 ? t - 1 : 0, cc, g);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int m = m0 + u;
                        const bool on = in && m < t;
                        y[u] = on ? -x[u] * g[u] : 0.f;
                        w[u] = on ? -x[u] * w[u] * a_t * ge[m] : 0.f;
                        ys[u] = y[u] * ge[m];
                        g[u] = a_t * y[u];
                    }
                    stage_w(wst, t, cc, w);
                    put16(a6, rowQ, c0, ys);
                    put16(a7, rowK, c0, g);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->y);
        }

        // ---- dQ, dK and their row sums
        if (ok) ok = warp_wait(&bars->d67, 0, abort);
        if (ok) {
            tc_fence_after();
            const size_t row = ((size_t)(t0 + t) * H + h) * D;
            __nv_bfloat16 *dqg = static_cast<__nv_bfloat16 *>(p.dq) + row;
            __nv_bfloat16 *dkg = static_cast<__nv_bfloat16 *>(p.dk) + row;
            // rows of a 16-row group that the chunk end cuts are stored here;
            // the full groups go out as TMA boxes from the staging tiles
            const bool ragged = 16 * (t >> 4) + 16 > n;
            unsigned char *qkst = smem + G::kOffQKst;
#pragma unroll 1
            for (int cc = 0; cc < kCC; ++cc) {
                const int j = j0 + 16 * cc;
                float x[16], kh[16], pv[16], kk[16];
                __syncwarp();
                tmem_ld16(lb + G::kColS3 + j, x);
                tmem_ld16(lb + G::kColS1 + j, kh);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) pv[u] = __shfl_down_sync(0xffffffffu, x[u], 16);
                get16(kq + (j >> 6) * kHalf, rowK, (uint32_t)((j & 63) >> 3), kk);
                if (first) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        dsum = fmaf(kh[u], kk[u], dsum);
                        pv[u] = a_t * pv[u] + e_t * kh[u];
                    }
                    const uint32_t hq = (uint32_t)(j >> 6) * kTokHalf, c0 = (uint32_t)((j & 63) >> 3);
                    put16(qkst + hq, t, c0, x);
                    put16(qkst + G::kTok + hq, t, c0, pv);
                    if (in && ragged) {
                        store16_bf16(dqg + j, x);
                        store16_bf16(dkg + j, pv);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) dsum = fmaf(x[u], kk[u], dsum);
                }
            }
        }

        fence_proxy_async();                 // the staged tiles, for the TMA stores
        // ---- the row sums of both column halves and the inner products to
        //      the gradient block's A slot
        {
            float *rp = rowpart + ch * kSums * C;
            if (first) {
                rp[sAbarM * C + t] = acc0;
                rp[sBM * C + t] = acc1;
                rp[sGLast * C + t] = rg;
                rp[sMuTail * C + t] = rm;
                rp[sDe * C + t] = dsum;
            } else {
                rp[sAbar * C + t] = acc0;
                rp[sB * C + t] = acc1;
                rp[sDa * C + t] = dsum;
            }
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                float x = sc[a];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                sc[a] = x;
            }
            if (lane == 0)
#pragma unroll
                for (int a = 0; a < 3; ++a) red[(warp - 2) * 4 + a] = sc[a];
        }
        epi_sync();
        if (!*abort) {
            if (e == 0) {
                // dQ and dK rows of the full 16-row groups
                const unsigned char *qkst = smem + G::kOffQKst;
                for (int g = 0; g < 4 && 16 * g + 16 <= n; ++g)
#pragma unroll
                    for (int hh = 0; hh < G::kHalves; ++hh) {
                        tma_store_3d(&map_dq, qkst + hh * kTokHalf + g * 2048, 64 * hh, h, t0 + 16 * g);
                        tma_store_3d(&map_dk, qkst + G::kTok + hh * kTokHalf + g * 2048, 64 * hh, h,
                                     t0 + 16 * g);
                    }
                bulk_commit_group();
            }
            float *ra = blk + BL::kA * BL::kMat;
            for (int idx = e; idx < kSums * C; idx += 256) {
                const int k = idx / C, tt = idx - k * C;
                float v = rowpart[idx] + rowpart[kSums * C + idx];
                if (k == sGLast || k == sMuTail) v *= ge[tt];
                ra[idx] = tt < n ? v : 0.f;
            }
            if (e < 3) {
                float s = 0.f;
                for (int w = 0; w < 8; ++w) s += red[w * 4 + e];
                ra[kSums * C + e] = s;
            }
            if (e == 0) bulk_wait_group_read0();   // the staging tiles stay until read
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, G::kTmemCols);
    if (threadIdx.x == 0 && *abort && p.loc.status)
        atomicExch(p.loc.status, (int)MDN_ERR_DEVICE_TIMEOUT);
}

template <int D>
cudaError_t launch_chunk_tc_d(const BwdProblem &p, cudaStream_t st, const CUtensorMap *maps) {
    using G = GradCfg<D>;
    auto kern = bwd_chunk_tc_kernel<D>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)G::kSmemBytes);
    if (err != cudaSuccess) return err;
    dim3 grid;
    if (!chunk_head_grid(p.loc.max_chunks, p.loc.H, grid)) return cudaErrorInvalidConfiguration;
    kern<<<grid, G::kThreads, G::kSmemBytes, st>>>(
        p, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9],
        maps[10], maps[11], maps[12]);
    return cudaGetLastError();
}

}  // namespace

// bf16 inputs: the chunk products of the gradient on the tensor cores, after
// the gradient prep and the reverse chain.
cudaError_t launch_bwd_chunk_tc(const BwdProblem &p, cudaStream_t st) {
    if ((p.D != 64 && p.D != 128) || p.dtype != MDN_BF16 || !p.prep || !p.adj || !p.tcblk)
        return cudaErrorInvalidValue;
    if (p.loc.max_chunks <= 0 || p.loc.T_total <= 0) return cudaSuccess;
    CUtensorMap maps[13];
    const void *src[8] = {p.k, p.q, p.dout, p.dv, p.v, p.k, p.dq, p.dk};
    const int box[8] = {16, 16, 16, 16, 64, 64, 16, 16};
    for (int i = 0; i < 8; ++i)
        if (!make_token_map_bf16(&maps[i], src[i], p.loc.T_total, p.loc.H, p.D, box[i]))
            return cudaErrorInvalidValue;
    // the gradient blocks' Y and X slots as [block][64 rows][64 columns] fp32
    const uint64_t blocks = (uint64_t)p.loc.max_chunks * p.loc.H;
    const uint64_t dims[3] = {64, 64, blocks};
    const uint64_t strides[2] = {64 * sizeof(float), BL::kBytes};
    const uint32_t wbox[3] = {32, 64, 1};
    if (!make_map_3d(&maps[8], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.prep + BL::kY * BL::kMat * sizeof(float),
                     dims, strides, wbox) ||
        !make_map_3d(&maps[9], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.prep + BL::kX * BL::kMat * sizeof(float),
                     dims, strides, wbox) ||
        !make_map_3d(&maps[10], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.prep + BL::kG * BL::kMat * sizeof(float),
                     dims, strides, wbox))
        return cudaErrorInvalidValue;
    // the chunk entry states, bf16 [block][dk rows][dv columns], as 64-column
    // boxes of all dk rows
    const uint64_t sdims[3] = {(uint64_t)p.D, (uint64_t)p.D, blocks};
    const uint64_t sstrides[2] = {(uint64_t)p.D * 2, (uint64_t)p.D * p.D * 2};
    const uint32_t sbox[3] = {64, (uint32_t)p.D, 1};
    if (!make_map_3d(&maps[11], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.S_chunks, sdims, sstrides, sbox) ||
        !make_map_3d(&maps[12], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.M_chunks, sdims, sstrides, sbox))
        return cudaErrorInvalidValue;
    return p.D == 128 ? launch_chunk_tc_d<128>(p, st, maps) : launch_chunk_tc_d<64>(p, st, maps);
}

}  // namespace mdn
