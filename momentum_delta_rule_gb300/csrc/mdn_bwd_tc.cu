// MDN gradient pass — the reverse chain over chunks on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA-staged operands), bf16
// inputs, head size 64 or 128.
//
// Per chunk of n tokens, walking the chunks from the last, with the state
// adjoints dS, dM at the chunk's end in TMEM (fp32) and the chunk's
// operand block (the forward prep's [T; A_O T] tile, read transposed as an
// MN-major operand, and the per-token coefficients):
//
//   MMA-U  D2  = (A T)^T dO                            (state-independent)
//   MMA1   D1  = [K; Q] [dS | dM]                      (K rows used)
//          R'' = Diag(gS eta) K dS - Diag(mu_tail eta) K dM
//   MMA2   D2 += T^T R''     ->  dR = T^T (A^T dO + WS dS - WM dM)  (= dV)
//   MMA3   [dS | dM] += [K; Q]^T [ -Diag(abar_m alpha) dR | Diag(b_m alpha) dR ;
//                                   Diag(abar) dO          | -Diag(b) dO      ]
//          after the in-place rescale dS <- abar_n dS, dM <- mubar_n dM - b_n dS
//
// which is the vector-Jacobian product of the chunk equations ("MDN:
// Parallelizing Stepwise Momentum for Delta Linear Attention" slides,
// frames "Solve the unknown residuals with a lower triangular system",
// Eqs. (15)-(18), and "Chunk outputs combine incoming states and local
// writes", Appendix C Eqs. (40)-(42)): the forward's state pass run
// backwards, with the adjoint of each product its transpose.  The structure
// follows the forward state pass (one CTA per (sequence, head, NS-column
// slice) - the adjoint states are column-independent like the states -,
// warp roles, TMEM layout, tc_row interleaving, bounded waits); MMA3 here
// runs over all 128 staged rows, the K rows against dR and the Q rows
// against dO.  Writes dV (= dR) in the input dtype, and the adjoints at
// every chunk's end as bf16 operand tiles for the chunk kernel.
#include <cudaTypedefs.h>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn_b() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// A [T_total, H, D] bf16 token tensor as a 3-D TMA map (D innermost, then
// the head, then the token), boxes of 64 columns x 1 head x box_t tokens,
// 128-byte swizzle.
bool make_token_map_bf16(CUtensorMap *map, const void *base, int T_total, int H, int D,
                         int box_t) {
    auto fn = encode_fn_b();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_t};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap *map, CUtensorMapDataType type, const void *base,
                 const uint64_t dims[3], const uint64_t strides[2], const uint32_t box[3]) {
    auto fn = encode_fn_b();
    if (!fn) return false;
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t st[2] = {strides[0], strides[1]};
    cuuint32_t b[3] = {box[0], box[1], box[2]};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, type, 3, const_cast<void *>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

using namespace sm100;

constexpr int kEpiCols = 16;
constexpr uint32_t kKQHalf = 16384;
constexpr uint32_t kOBytes = 8192;       // dO tile, 64 tokens x 64 columns, swizzled
using CL = BwdChainLayout;

template <int D, int NS>
struct ChainCfg {
    static_assert(NS == 16 || NS == 32 || NS == 64, "slice width");
    static_assert(D == 64 || D == 128, "head size");
    static constexpr int kHalves = D / 64;
    static constexpr int kStages = 2;
    static constexpr int kSlices = D / NS;
    static constexpr int kEpiWarps = 4 * NS / kEpiCols;
    static constexpr int kThreads = 32 * (2 + kEpiWarps);
    static constexpr uint32_t kKQBytes = kHalves * kKQHalf;
    static constexpr uint32_t kOffO = kKQBytes;
    static constexpr uint32_t kOffBlk = kOffO + kOBytes;
    static constexpr uint32_t kBlkBytes = (uint32_t)CL::kBytes;
    static constexpr uint32_t kStageBytes = kOffBlk + kBlkBytes;
    static_assert(kStageBytes % 1024 == 0, "stage alignment");
    static constexpr uint32_t kOffB1 = kStages * kStageBytes;   // [dS | dM] bf16, dk rows x 2NS
    static constexpr uint32_t kB1Bytes = (NS == 64 ? 2 : 1) * D * 128;
    static constexpr uint32_t kB1M = NS == 64 ? D * 128 : 0;
    static constexpr uint32_t kOffR = kOffB1 + kB1Bytes;       // R'' bf16, 64 token rows x NS
    static constexpr uint32_t kRBytes = 8192;
    static constexpr uint32_t kOffB3 = kOffR + kRBytes;        // 128 rows x 2NS (tc_row order)
    static constexpr uint32_t kB3Bytes = (NS == 64 ? 2 : 1) * 128 * 128;
    static constexpr uint32_t kB3M = NS == 64 ? 128 * 128 : 0;
    static constexpr uint32_t kChM = NS == 64 ? 0 : NS / 8;
    static constexpr uint32_t kOffBar = kOffB3 + kB3Bytes;
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
    static constexpr uint32_t kColD1 = 0;
    static constexpr uint32_t kColD2 = 2 * NS;
    static constexpr uint32_t kColSt = 4 * NS;
    static constexpr uint32_t kTmemCols = 8 * NS;
    static constexpr uint32_t kIdesc1 = idesc_bf16(128, 2 * NS, false, true);
    static constexpr uint32_t kIdesc2 = idesc_bf16(64, NS, true, true);
    static constexpr uint32_t kIdesc3 = idesc_bf16(D, 2 * NS, true, true);
};

struct ChainBars {
    uint64_t full[2], empty[2];
    uint64_t d1, r, d2, v, d3, state, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(ChainBars) <= 256, "barrier block");

__device__ __forceinline__ uint32_t pk2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void unpack8(const uint4 &raw, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void put8s(unsigned char *tile, uint32_t row, uint32_t chunk,
                                      const float *x, float s) {
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, chunk)) =
        make_uint4(pk2(s * x[0], s * x[1]), pk2(s * x[2], s * x[3]), pk2(s * x[4], s * x[5]),
                   pk2(s * x[6], s * x[7]));
}

__device__ __forceinline__ void store_row16(unsigned char *tile, uint32_t row, uint32_t chunk0,
                                            const float *x) {
    put8s(tile, row, chunk0, x, 1.f);
    put8s(tile, row, chunk0 + 1, x + 8, 1.f);
}

// dS <- abar_n dS, dM <- mubar_n dM - b_n dS (both from the old values): the
// adjoint of the forward's carry rescale.
__device__ __forceinline__ void rescale_adjoint(uint32_t st_s, uint32_t st_m, const float *cv) {
    const float ab_n = cv[CL::vScal * kChunk + 0];
    const float b_n = cv[CL::vScal * kChunk + 1];
    const float mb_n = cv[CL::vScal * kChunk + 2];
    float S[kEpiCols], M[kEpiCols];
    tmem_ld16(st_s, S);
    tmem_ld16(st_m, M);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < kEpiCols; ++j) {
        const float s_old = S[j];
        S[j] = ab_n * s_old;
        M[j] = mb_n * M[j] - b_n * s_old;
    }
    tmem_st16(st_s, S);
    tmem_st16(st_m, M);
    tmem_st_wait();
}

__device__ __forceinline__ bool warp_wait_c(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// One thread's 16 columns (from column j) of row d of the adjoints at the
// end of chunk slot `slot`, as the chunk kernel's bf16 operand tiles: per
// (slot, head) dS then dM, each D rows x D columns in 64-column halves of
// D rows x 128 bytes, 128-byte swizzled.
template <int D>
__device__ __forceinline__ void store_adjoint(const BwdProblem &p, int slot, int h, int d, int j,
                                              const float *S, const float *M) {
    unsigned char *base = reinterpret_cast<unsigned char *>(p.adj) +
                          ((size_t)slot * p.loc.H + h) * 2 * D * D * sizeof(__nv_bfloat16);
    const uint32_t off = (uint32_t)(j >> 6) * (D * 128);
    const uint32_t c0 = (uint32_t)((j & 63) >> 3);
    store_row16(base + off, d, c0, S);
    store_row16(base + (size_t)D * D * sizeof(__nv_bfloat16) + off, d, c0, M);
}

template <int D, int NS>
__global__ void __launch_bounds__(ChainCfg<D, NS>::kThreads, 1)
bwd_chain_tc_kernel(const BwdProblem p, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_o) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem_1024(smem_raw);
    using C = ChainCfg<D, NS>;
    ChainBars *bars = reinterpret_cast<ChainBars *>(smem + C::kOffBar);
    volatile int *abort = &bars->abort;
    constexpr int kEpiWarps = C::kEpiWarps;
    const ChunkProblem &L = p.loc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x % C::kSlices;
    const int kh = blockIdx.x / C::kSlices;
    const int s = ordered_sequence(L, kh / L.H), h = kh % L.H;
    const int sh = s * L.H + h;
    const int col0 = slice * NS;
    int start, len, slot0;
    sequence_range(L, s, start, len, slot0);
    const int nch = (len + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 1 + kEpiWarps);
        }
        mbar_init(&bars->d1, 1);
        mbar_init(&bars->r, kEpiWarps);
        mbar_init(&bars->d2, 1);
        mbar_init(&bars->v, kEpiWarps);
        mbar_init(&bars->d3, 1);
        mbar_init(&bars->state, kEpiWarps);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_o);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer, chunks in reverse
        if (lane == 0) {
            int last_use[2] = {-1, -1};
            for (int i = 0; i < nch; ++i) {
                const int c = nch - 1 - i;
                const int st = i & 1, use = i >> 1;
                if (!mbar_wait(&bars->empty[st], (use & 1) ^ 1, abort)) break;
                unsigned char *stage = smem + st * C::kStageBytes;
                const int t0 = start + c * kChunk;
                const unsigned char *blk = p.tcblk + ((size_t)(slot0 + c) * L.H + h) * CL::kBytes;
                mbar_arrive_expect_tx(&bars->full[st], C::kStageBytes);
#pragma unroll
                for (int hh = 0; hh < C::kHalves; ++hh)
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        unsigned char *dst = stage + hh * kKQHalf + g * 4096;
                        tma_load_3d(dst, &map_k, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                        tma_load_3d(dst + 2048, &map_q, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                    }
                tma_load_3d(stage + C::kOffO, &map_o, &bars->full[st], col0, h, t0);
                if (p.fwd_tile) {
                    // the tile from the forward's prepared block, the
                    // coefficient rows from the operand block
                    const unsigned char *ft = p.fwd_tile + ((size_t)(slot0 + c) * L.H + h) * p.fwd_tile_stride;
                    bulk_load(stage + C::kOffBlk, ft + CL::kOffTile, (uint32_t)CL::kOffVec, &bars->full[st]);
                    bulk_load(stage + C::kOffBlk + CL::kOffVec, blk + CL::kOffVec,
                              C::kBlkBytes - (uint32_t)CL::kOffVec, &bars->full[st]);
                } else {
                    bulk_load(stage + C::kOffBlk, blk, C::kBlkBytes, &bars->full[st]);
                }
                last_use[st] = use;
            }
            for (int st = 0; st < C::kStages; ++st) {
                if (last_use[st] < 0) continue;
                int dummy = 0;
                mbar_wait(&bars->full[st], last_use[st] & 1, &dummy);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        const bool l0 = lane == 0;
        const uint32_t b1 = smem_u32(smem + C::kOffB1);
        const uint32_t rr = smem_u32(smem + C::kOffR);
        const uint32_t b3 = smem_u32(smem + C::kOffB3);
        constexpr uint32_t kLbo1 = C::kB1M ? C::kB1M : 16384;
        constexpr uint32_t kLbo3 = C::kB3M ? C::kB3M : 16384;
        for (int i = 0; i < nch; ++i) {
            const int st = i & 1, use = i >> 1;
            const uint32_t kq = smem_u32(smem + st * C::kStageBytes);
            const uint32_t ob = kq + C::kOffO;
            const uint32_t blk = kq + C::kOffBlk;
            if (!warp_wait_c(&bars->full[st], use & 1, abort)) break;
            if (!warp_wait_c(&bars->state, i & 1, abort)) break;
            tc_fence_after();
            if (l0) {
                // MMA-U: D2 = (A T)^T dO (A: the A_O T rows of the tile, read
                // MN-major, 16 rows i per step), then MMA1: D1 = [K; Q] [dS | dM]
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sdesc_sw128(blk + CL::kOffTile + kk * 4096 + 2048, kKQHalf, 1024);
                    const uint64_t b = sdesc_sw128(ob + kk * 2048, 8192, 1024);
                    mma_bf16(tmem + C::kColD2, a, b, C::kIdesc2, kk != 0);
                }
#pragma unroll
                for (int kb = 0; kb < C::kHalves; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(kq + kb * kKQHalf + kk * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(b1 + (kb * 4 + kk) * 2048, kLbo1, 1024);
                        mma_bf16(tmem + C::kColD1, a, b, C::kIdesc1, (kb | kk) != 0);
                    }
                mma_commit(&bars->d1);
                if constexpr (NS == 64) {
                    // the adjoints at this chunk's end leave as they sit in
                    // B1: one 64-column half of the chunk kernel's dS and dM
                    // operand tiles each
                    const int c = nch - 1 - i;
                    unsigned char *dst = reinterpret_cast<unsigned char *>(p.adj) +
                                         ((size_t)(slot0 + c) * L.H + h) * 2 * D * D * 2 +
                                         (size_t)slice * D * 128;
                    bulk_store(dst, smem + C::kOffB1, D * 128);
                    bulk_store(dst + (size_t)D * D * 2, smem + C::kOffB1 + C::kB1M, D * 128);
                    bulk_commit_group();
                }
            }
            __syncwarp();
            if (!warp_wait_c(&bars->r, i & 1, abort)) break;
            tc_fence_after();
            if (l0) {
                // MMA2: D2 += T^T R'' (A: the T rows of the tile, MN-major)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sdesc_sw128(blk + CL::kOffTile + kk * 4096, kKQHalf, 1024);
                    const uint64_t b = sdesc_sw128(rr + kk * 2048, 8192, 1024);
                    mma_bf16(tmem + C::kColD2, a, b, C::kIdesc2, 1);
                }
                mma_commit(&bars->d2);
            }
            __syncwarp();
            if (!warp_wait_c(&bars->v, i & 1, abort)) break;
            tc_fence_after();
            if (l0) {
                // MMA3: [dS | dM] += [K; Q]^T B3 over all 128 staged rows
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t a = sdesc_sw128(kq + kk * 2048, kKQHalf, 1024);
                    const uint64_t b = sdesc_sw128(b3 + kk * 2048, kLbo3, 1024);
                    mma_bf16(tmem + C::kColSt, a, b, C::kIdesc3, 1);
                }
                // B1 is rewritten once MMA3 is done: its copy-out has read it
                if constexpr (NS == 64) bulk_wait_group_read0();
                mma_commit(&bars->d3);
                mma_commit(&bars->empty[st]);
            }
            __syncwarp();
        }
        if (l0) {
            mma_commit(&bars->drain);
            int dummy = 0;
            mbar_wait(&bars->drain, 0, &dummy);
            if constexpr (NS == 64) bulk_wait_group0();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;
        const int qc = (warp - 2) >> 2;
        const int c0 = qc * kEpiCols;
        const uint32_t ch0 = qc * 2;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const bool row_ok = D == 128 || lane < 16;
        const int d = D == 128 ? 32 * q + lane : 16 * q + (lane & 15);
        const uint32_t st_s = lane_base + C::kColSt + c0;
        const uint32_t st_m = lane_base + C::kColSt + NS + c0;
        const size_t st_row = (size_t)d * D + col0 + c0;        // within one [dk, dv] state
        const size_t st_off = (size_t)sh * D * D + st_row;
        unsigned char *b1 = smem + C::kOffB1;
        unsigned char *rt = smem + C::kOffR;
        unsigned char *b3 = smem + C::kOffB3;
        {
            float S[kEpiCols], M[kEpiCols];
#pragma unroll
            for (int j = 0; j < kEpiCols; j += 4) {
                float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), mv = sv;
                if (p.dS_T && row_ok) sv = *reinterpret_cast<const float4 *>(p.dS_T + st_off + j);
                if (p.dM_T && row_ok) mv = *reinterpret_cast<const float4 *>(p.dM_T + st_off + j);
                S[j] = sv.x; S[j + 1] = sv.y; S[j + 2] = sv.z; S[j + 3] = sv.w;
                M[j] = mv.x; M[j + 1] = mv.y; M[j + 2] = mv.z; M[j + 3] = mv.w;
            }
            tmem_st16(st_s, S);
            tmem_st16(st_m, M);
            tmem_st_wait();
            if (nch > 0) {
                if (row_ok) {
                    store_row16(b1, d, ch0, S);
                    store_row16(b1 + C::kB1M, d, ch0 + C::kChM, M);
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->state);
                if (NS != 64 && row_ok) store_adjoint<D>(p, slot0 + nch - 1, h, d, col0 + c0, S, M);
            }
        }
        const int tok = 16 * q + (lane & 15);
        const int cg = c0 + 8 * (lane >> 4);
        const uint32_t chk = (uint32_t)(cg >> 3);
        const uint32_t lk = tmem + ((uint32_t)(32 * q) << 16);
        const size_t rs = (size_t)L.H * D;
        const int rk = tc_row(tok), rq = tc_row(kChunk + tok);     // B3 rows of this token
        __nv_bfloat16 *dvg = static_cast<__nv_bfloat16 *>(p.dv) + (size_t)h * D + col0 + cg;
        for (int i = 0; i < nch; ++i) {
            const int c = nch - 1 - i;
            const int st = i & 1, use = i >> 1;
            unsigned char *stage = smem + st * C::kStageBytes;
            const float *cv = reinterpret_cast<const float *>(stage + C::kOffBlk + CL::kOffVec);
            const int n = min(kChunk, len - c * kChunk);
            const int t0 = start + c * kChunk;
            if (!warp_wait_c(&bars->full[st], use & 1, abort)) break;
            const bool in_chunk = tok < n;
            const float cs = cv[CL::vCS * kChunk + tok], cm = cv[CL::vCM * kChunk + tok];
            const float bs = cv[CL::vBS * kChunk + tok], bm = cv[CL::vBM * kChunk + tok];
            const float qs = cv[CL::vQS * kChunk + tok], qm = cv[CL::vQM * kChunk + tok];
            float dov[8];
            {
                uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                if (in_chunk) raw = *reinterpret_cast<const uint4 *>(stage + C::kOffO + sw128_offset(tok, chk));
                unpack8(raw, dov);
            }
            // ---- R'' = cS K dS + cM K dM: the critical step; beside it the
            //      query rows of MMA3's B operand, [abar dO | -b dO]
            if (!warp_wait_c(&bars->d1, i & 1, abort)) break;
            tc_fence_after();
            {
                float xs[8], xm[8], r[8];
                tmem_ld_16x2x8(lk + C::kColD1 + c0, xs);
                tmem_ld_16x2x8(lk + C::kColD1 + NS + c0, xm);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = in_chunk ? cs * xs[e] + cm * xm[e] : 0.f;
                put8s(rt, tok, chk, r, 1.f);
                put8s(b3, rq, chk, dov, qs);
                put8s(b3 + C::kB3M, rq, chk + C::kChM, dov, qm);
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->r);
            }
            rescale_adjoint(st_s, st_m, cv);
            // ---- dR = T^T (A^T dO + R''): the key rows of MMA3's B operand,
            //      [-abar_m alpha dR | b_m alpha dR], and dV
            if (!warp_wait_c(&bars->d2, i & 1, abort)) break;
            tc_fence_after();
            {
                float x[8];
                tmem_ld_16x2x8(lk + C::kColD2 + c0, x);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = in_chunk ? x[e] : 0.f;
                put8s(b3, rk, chk, x, bs);
                put8s(b3 + C::kB3M, rk, chk + C::kChM, x, bm);
                fence_proxy_async();
                if (in_chunk)
                    *reinterpret_cast<uint4 *>(dvg + (size_t)(t0 + tok) * rs) =
                        make_uint4(pk2(x[0], x[1]), pk2(x[2], x[3]), pk2(x[4], x[5]), pk2(x[6], x[7]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->v);
            }
            // ---- the adjoints at this chunk's start: bf16 copy for the next
            //      (earlier) chunk's MMA1, and to the workspace as the
            //      previous chunk's end adjoints (bf16 operand tiles)
            if (!warp_wait_c(&bars->d3, i & 1, abort)) break;
            tc_fence_after();
            {
                const bool more = c > 0;
                float S[kEpiCols], M[kEpiCols];
                if (more) {
                    tmem_ld16(st_s, S);
                    tmem_ld16(st_m, M);
                    tmem_ld_wait();
                    if (row_ok) {
                        store_row16(b1, d, ch0, S);
                        store_row16(b1 + C::kB1M, d, ch0 + C::kChM, M);
                    }
                    fence_proxy_async();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (more) mbar_arrive(&bars->state);
                    mbar_arrive(&bars->empty[st]);
                }
                if (NS != 64 && more && row_ok) store_adjoint<D>(p, slot0 + c - 1, h, d, col0 + c0, S, M);
            }
        }
        if (!*abort) {
            float S[kEpiCols], M[kEpiCols];
            tmem_ld16(st_s, S);
            tmem_ld16(st_m, M);
            tmem_ld_wait();
            if (row_ok) {
#pragma unroll
                for (int j = 0; j < kEpiCols; j += 4) {
                    if (p.dS0)
                        *reinterpret_cast<float4 *>(p.dS0 + st_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                    if (p.dM0)
                        *reinterpret_cast<float4 *>(p.dM0 + st_off + j) = make_float4(M[j], M[j + 1], M[j + 2], M[j + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    if (threadIdx.x == 0 && *abort && L.status) atomicExch(L.status, (int)MDN_ERR_DEVICE_TIMEOUT);
}

template <int D, int NS>
cudaError_t launch_chain_tc_t(const BwdProblem &p, cudaStream_t st, const CUtensorMap &mk,
                              const CUtensorMap &mq, const CUtensorMap &mo) {
    using C = ChainCfg<D, NS>;
    auto kern = bwd_chain_tc_kernel<D, NS>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)C::kSmemBytes);
    if (err != cudaSuccess) return err;
    const long blocks = (long)p.loc.n_seq * p.loc.H * C::kSlices;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)blocks, C::kThreads, C::kSmemBytes, st>>>(p, mk, mq, mo);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_chain_tc_d(const BwdProblem &p, cudaStream_t st, const CUtensorMap &mk,
                              const CUtensorMap &mq, const CUtensorMap &mo) {
    const long chains = (long)p.loc.n_seq * p.loc.H;
    const int sms = device_sm_count();
    const int ns = (sms > 0 && chains * (D / 16) <= sms) ? 16
                 : (sms > 0 && chains * (D / 32) <= sms) ? 32 : 64;
    if (ns == 16) return launch_chain_tc_t<D, 16>(p, st, mk, mq, mo);
    if (ns == 32) return launch_chain_tc_t<D, 32>(p, st, mk, mq, mo);
    return launch_chain_tc_t<D, 64>(p, st, mk, mq, mo);
}

}  // namespace

// bf16 inputs: the reverse chain on the tensor cores (after the gradient
// prep has written the chain's operand blocks).
cudaError_t launch_bwd_chain_tc(const BwdProblem &p, cudaStream_t st) {
    if ((p.D != 64 && p.D != 128) || p.dtype != MDN_BF16 || !p.tcblk) return cudaErrorInvalidValue;
    const int Tt = p.loc.T_total > 0 ? p.loc.T_total : 1;
    CUtensorMap mk, mq, mo;
    if (!make_token_map_bf16(&mk, p.k, Tt, p.loc.H, p.D, 16) ||
        !make_token_map_bf16(&mq, p.q, Tt, p.loc.H, p.D, 16) ||
        !make_token_map_bf16(&mo, p.dout, Tt, p.loc.H, p.D, 64))
        return cudaErrorInvalidValue;
    return p.D == 128 ? launch_chain_tc_d<128>(p, st, mk, mq, mo)
                      : launch_chain_tc_d<64>(p, st, mk, mq, mo);
}

}  // namespace mdn
