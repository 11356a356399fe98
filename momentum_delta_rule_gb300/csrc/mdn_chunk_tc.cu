// MDN chunkwise forward — sequential state pass on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA-staged operands), bf16 inputs, head
// size 128.
//
// Chunk equations ("MDN: Parallelizing Stepwise Momentum for Delta Linear
// Attention" slides, frames "Solve the unknown residuals with a lower
// triangular system", Eqs. (15)-(18), and "Chunk outputs combine incoming
// states and local writes", Appendix C Eqs. (40)-(42); reading notes 2.4-2.5),
// with the chunk-local matrices T and A_O T and the coefficient vectors taken
// from the prepared block of the prep kernel:
//
//   MMA1  D1 = [K; Q] [S_0 | M_0]          (M=128 rows, N=2 NS, K=dk)
//         R  = V - Diag(abar) K S_0 + Diag(b_{i-1} alpha_i) K M_0
//         O_inter = Diag(abar) Q S_0 - Diag(b) Q M_0
//   MMA2  D2 = [T; A_O T] R                 (M=128, N=NS, K=64 tokens)
//         Vres = the T rows,  O = O_inter + the A_O T rows
//   MMA3  [S | M] += K^T [Diag(gS) Vres | -Diag(gM) Vres]  (M=dk, N=2 NS, K=64)
//
// with gS_i = gamma_{n,i} eta_i and gM_i = prod_{u>i} mu_u eta_i.  The fp32
// state [S | M] of the slice lives in TMEM as MMA3's accumulator; before MMA3
// the epilogue rescales it in place to [abar_n S - b_n M | mubar_n M] (both
// carries use the old S_0, M_0), off the critical path while MMA2 runs.  Only
// a bf16 copy of the state goes to shared memory, as MMA1's B operand.
//
// One CTA owns one (sequence, head, NS-column slice), NS = 64, 32 or 16 (the
// launcher takes the narrowest whose grid still fits one CTA per SM, else
// 64): columns of S and M evolve independently (column j of Vres depends
// only on column j of S_0 and M_0), so the slices of a head never
// communicate.  A second instantiation also stores every chunk's entry state
// (S, M) for a gradient pass; the plain forward's kernel carries none of it.
//
// Warp roles (2 + NS / 4 warps, 18 for NS = 64): 0 TMA producer, 1 MMA
// issuer + TMEM owner (all lanes wait, lane 0 issues), the rest epilogue
// (TMEM lane quadrant = warp % 4, 16-column group of the slice =
// (warp-2)/4).  A warp reaches only the TMEM lanes of
// its quadrant, and the warps of a quadrant share one scheduler; [K; Q] and
// [T; A_O T] rows are therefore interleaved in blocks of 16 (tc_row), so that
// every quadrant holds 16 token rows and 16 query rows and the token-row
// steps (R, Vres) use all four schedulers (16x32bx2 TMEM loads: lanes t and
// t + 16 take 8 columns each).
// Every wait is bounded (1 s); on expiry the CTA records
// MDN_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

using namespace sm100;

constexpr int kD = 128;                  // head size (dk = dv)
constexpr int kStages = 2;
constexpr int kEpiCols = 16;             // state columns per epilogue thread

// shared memory of one pipeline stage (byte offsets from the stage base)
constexpr uint32_t kKQBytes = 32768;     // per 64-wide dk half: K rows, then Q rows
constexpr uint32_t kVBytes = 8192;       // V tile, 64 tokens x 64 columns, swizzled
constexpr uint32_t kPrepBytes = (uint32_t)PrepLayoutTC::kBytes;   // 18432
constexpr uint32_t kOffV = kKQBytes;
constexpr uint32_t kOffPrep = kKQBytes + kVBytes;
constexpr uint32_t kStageBytes = kKQBytes + kVBytes + kPrepBytes;  // 59392

// Everything that depends on the slice width NS (state columns per CTA).
// In the N dimension of [S | M]-shaped operands, S takes columns [0, NS) and
// M [NS, 2NS); operands are MN-major in blocks of 64 columns, so for NS = 64
// the M half is a second block and for NS = 32 or 16 it shares the block.
template <int NS>
struct Cfg {
    static_assert(NS == 16 || NS == 32 || NS == 64, "slice width");
    static constexpr int kSlices = kD / NS;
    static constexpr int kEpiWarps = 4 * NS / kEpiCols;      // 4 lane quadrants
    static constexpr int kThreads = 32 * (2 + kEpiWarps);
    static constexpr uint32_t kOffB1 = kStages * kStageBytes;  // [S | M] bf16, dk rows x 2NS
    static constexpr uint32_t kB1Bytes = NS == 64 ? 32768 : 16384;
    static constexpr uint32_t kB1M = NS == 64 ? 16384 : 0;    // byte offset of the M half
    static constexpr uint32_t kOffR = kOffB1 + kB1Bytes;      // R bf16, 64 token rows x NS
    static constexpr uint32_t kRBytes = 8192;
    static constexpr uint32_t kOffB3 = kOffR + kRBytes;       // [gS Vres | -gM Vres]
    static constexpr uint32_t kB3Bytes = NS == 64 ? 16384 : 8192;
    static constexpr uint32_t kB3M = NS == 64 ? 8192 : 0;
    static constexpr uint32_t kChM = NS == 64 ? 0 : NS / 8;   // chunk offset of the M half
    static constexpr uint32_t kOffBar = kOffB3 + kB3Bytes;
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
    // tensor memory columns
    static constexpr uint32_t kColD1 = 0;                     // 2NS columns
    static constexpr uint32_t kColD2 = 2 * NS;                // NS columns
    static constexpr uint32_t kColSt = 4 * NS;                // fp32 state [S | M], 2NS columns
    static constexpr uint32_t kTmemCols = 8 * NS;
    static constexpr uint32_t kIdesc1 = idesc_bf16(128, 2 * NS, false, true);
    static constexpr uint32_t kIdesc2 = idesc_bf16(128, NS, false, true);
    static constexpr uint32_t kIdesc3 = idesc_bf16(128, 2 * NS, true, true);
};

struct Bars {
    uint64_t full[kStages];    // TMA bytes of a stage landed
    uint64_t empty[kStages];   // stage free again (MMA commit + every epilogue warp)
    uint64_t d1, r, d2, v, d3, state, drain;   // d3: the state accumulation finished
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");


__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &raw, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// Write 16 fp32 values as bf16 into row `row`, 16-byte chunks [chunk0,
// chunk0+2) of a 128-byte-swizzled tile.
__device__ __forceinline__ void store_row16(unsigned char *tile, uint32_t row, uint32_t chunk0,
                                            const float *x, float scale) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        uint4 w;
        w.x = pack_bf16x2(scale * x[8 * cc + 0], scale * x[8 * cc + 1]);
        w.y = pack_bf16x2(scale * x[8 * cc + 2], scale * x[8 * cc + 3]);
        w.z = pack_bf16x2(scale * x[8 * cc + 4], scale * x[8 * cc + 5]);
        w.w = pack_bf16x2(scale * x[8 * cc + 6], scale * x[8 * cc + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, chunk0 + cc)) = w;
    }
}

// In-place rescale of this thread's 16 columns of the TMEM state for the
// carry of the current chunk: S <- abar_n S - b_n M, M <- mubar_n M.
__device__ __forceinline__ void rescale_state(uint32_t st_s, uint32_t st_m, const float *vec) {
    const float ab_n = vec[kVecScal * kChunk + 0];
    const float b_n = vec[kVecScal * kChunk + 1];
    const float mb_n = vec[kVecScal * kChunk + 2];
    float S[kEpiCols], M[kEpiCols];
    tmem_ld16(st_s, S);
    tmem_ld16(st_m, M);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < kEpiCols; ++j) {
        const float s_old = S[j];
        S[j] = ab_n * s_old - b_n * M[j];
        M[j] = mb_n * M[j];
    }
    tmem_st16(st_s, S);
    tmem_st16(st_m, M);
    tmem_st_wait();
}

// One thread's 16 columns of row d of the entry state of chunk slot `slot`
// (layout [slot, H, dk, dv]); `off` = d * dk + first column.
__device__ __forceinline__ void store_chunk_state(const ChunkProblem &p, int slot, int h, size_t off,
                                                  const float *S, const float *M) {
    const size_t base = ((size_t)slot * p.H + h) * kD * kD + off;
#pragma unroll
    for (int j = 0; j < kEpiCols; j += 4) {
        *reinterpret_cast<float4 *>(p.S_chunks + base + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        *reinterpret_cast<float4 *>(p.M_chunks + base + j) = make_float4(M[j], M[j + 1], M[j + 2], M[j + 3]);
    }
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// kChunkStates: also write the entry state of every chunk (a separate
// instantiation, so the plain forward carries none of its registers).
template <int NS, bool kChunkStates>
__global__ void __launch_bounds__(Cfg<NS>::kThreads, 1)
chunk_state_tc_kernel(const ChunkProblem p, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_v) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Bars *bars = reinterpret_cast<Bars *>(smem + Cfg<NS>::kOffBar);
    volatile int *abort = &bars->abort;

    using C = Cfg<NS>;
    constexpr int kEpiWarps = C::kEpiWarps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x % C::kSlices;
    const int kh = blockIdx.x / C::kSlices;
    // This grid may start while the prep kernel finishes (programmatic
    // dependent launch).  Packed sequences read the chunk offsets first: wait
    // for the preceding grids right away.  Fixed-length batches run their
    // setup and initial-state loads first; the producer waits before its
    // first prepared-block copy.
    if (p.cu_seqlens != nullptr) grid_dependency_wait();
    const int s = ordered_sequence(p, kh / p.H), h = kh % p.H;
    const int sh = s * p.H + h;                 // (sequence, head) of the states
    const int col0 = slice * NS;
    int start, len, slot0;
    sequence_range(p, s, start, len, slot0);
    const int nchunks = (len + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
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
        prefetch_tensormap(&map_v);
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
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_use[kStages] = {-1, -1};
            for (int c = 0; c < nchunks; ++c) {
                const int st = c & 1, use = c >> 1;
                if (c == 0) grid_dependency_wait();   // the prepared blocks are complete
                if (!mbar_wait(&bars->empty[st], (use & 1) ^ 1, abort)) break;
                unsigned char *stage = smem + st * kStageBytes;
                const int t0 = start + c * kChunk;
                const unsigned char *blk =
                    p.prep + ((size_t)(slot0 + c) * p.H + h) * p.prep_stride;
                mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
                // [K; Q] rows interleaved by 16 (tc_row): 16-token boxes
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        unsigned char *dst = stage + hh * 16384 + g * 4096;
                        tma_load_3d(dst, &map_k, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                        tma_load_3d(dst + 2048, &map_q, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                    }
                tma_load_3d(stage + kOffV, &map_v, &bars->full[st], col0, h, t0);
                bulk_load(stage + kOffPrep, blk, kPrepBytes, &bars->full[st]);
                last_use[st] = use;
            }
            // drain: every issued copy must land before the CTA may exit
            for (int st = 0; st < kStages; ++st) {
                if (last_use[st] < 0) continue;
                int dummy = 0;
                mbar_wait(&bars->full[st], last_use[st] & 1, &dummy);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (the
        // whole warp waits, lane 0 issues and commits)
        {
            const bool l0 = lane == 0;
            const uint32_t b1 = smem_u32(smem + C::kOffB1);
            const uint32_t rr = smem_u32(smem + C::kOffR);
            const uint32_t b3 = smem_u32(smem + C::kOffB3);
            for (int c = 0; c < nchunks; ++c) {
                const int st = c & 1, use = c >> 1;
                const uint32_t kq = smem_u32(smem + st * kStageBytes);
                const uint32_t prep = kq + kOffPrep;
                if (!warp_wait(&bars->full[st], use & 1, abort)) break;
                if (!warp_wait(&bars->state, c & 1, abort)) break;
                tc_fence_after();
                if (l0) {
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = sdesc_sw128(kq + kb * 16384 + kk * 32, 16, 1024);
                            const uint64_t b = sdesc_sw128(b1 + (kb * 4 + kk) * 2048, 16384, 1024);
                            mma_bf16(tmem + C::kColD1, a, b, C::kIdesc1, (kb | kk) != 0);
                        }
                    mma_commit(&bars->d1);
                }
                __syncwarp();
                if (!warp_wait(&bars->r, c & 1, abort)) break;
                tc_fence_after();
                if (l0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(prep + kk * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(rr + kk * 2048, 8192, 1024);
                        mma_bf16(tmem + C::kColD2, a, b, C::kIdesc2, kk != 0);
                    }
                    mma_commit(&bars->d2);
                }
                __syncwarp();
                if (!warp_wait(&bars->v, c & 1, abort)) break;
                tc_fence_after();
                if (l0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(kq + kk * 4096, 16384, 1024);
                        const uint64_t b = sdesc_sw128(b3 + kk * 2048, 8192, 1024);
                        mma_bf16(tmem + C::kColSt, a, b, C::kIdesc3, 1);
                    }
                    mma_commit(&bars->d3);
                    mma_commit(&bars->empty[st]);
                }
                __syncwarp();
            }
            // drain: all issued MMAs complete before TMEM is freed
            if (l0) {
                mma_commit(&bars->drain);
                int dummy = 0;
                mbar_wait(&bars->drain, 0, &dummy);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quadrant
        const int qc = (warp - 2) >> 2;         // 16-column quarter of the slice
        const int c0 = qc * kEpiCols;           // first column (within the slice)
        const uint32_t ch0 = qc * 2;            // first 16-byte chunk of those columns
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const int row = 32 * q + lane;          // TMEM lane = D row
        const int d = row;                      // state row (dk index)
        const uint32_t st_s = lane_base + C::kColSt + c0;       // S columns of this thread
        const uint32_t st_m = lane_base + C::kColSt + NS + c0;  // M columns
        const size_t st_off = (size_t)sh * kD * kD + (size_t)d * kD + col0 + c0;
        unsigned char *b1 = smem + C::kOffB1;
        unsigned char *rt = smem + C::kOffR;
        unsigned char *b3 = smem + C::kOffB3;
        {
            float S[kEpiCols], M[kEpiCols];
#pragma unroll
            for (int j = 0; j < kEpiCols; j += 4) {
                float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), mv = sv;
                if (p.S0) sv = *reinterpret_cast<const float4 *>(p.S0 + st_off + j);
                if (p.M0) mv = *reinterpret_cast<const float4 *>(p.M0 + st_off + j);
                S[j] = sv.x; S[j + 1] = sv.y; S[j + 2] = sv.z; S[j + 3] = sv.w;
                M[j] = mv.x; M[j + 1] = mv.y; M[j + 2] = mv.z; M[j + 3] = mv.w;
            }
            tmem_st16(st_s, S);
            tmem_st16(st_m, M);
            tmem_st_wait();
            if (nchunks > 0) {
                store_row16(b1, d, ch0, S, 1.f);
                store_row16(b1 + C::kB1M, d, ch0 + C::kChM, M, 1.f);
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->state);
                if (kChunkStates) store_chunk_state(p, slot0, h, st_off - (size_t)sh * kD * kD, S, M);
            }
        }
        // Token rows: the lower 16 lanes of this warp's quadrant hold the K
        // rows of tokens tok = 16 q + lane % 16, the upper 16 the Q rows of
        // the same tokens (tc_row order); lanes t and t + 16 split the
        // warp's 16 columns into two halves of 8 (16x32bx2 TMEM loads).
        const int tok = 16 * q + (lane & 15);
        const int cg = c0 + 8 * (lane >> 4);          // first of this thread's 8 columns
        const uint32_t chk = (uint32_t)(cg >> 3);     // their 16-byte chunk
        const uint32_t lk = tmem + ((uint32_t)(32 * q) << 16);        // K / T rows
        const uint32_t lq = tmem + ((uint32_t)(32 * q + 16) << 16);   // Q / A_O T rows
        const size_t rs = (size_t)p.H * kD;
        __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.o) + (size_t)h * kD + col0 + cg;
        __nv_bfloat16 *vg = p.vres ? static_cast<__nv_bfloat16 *>(p.vres) + (size_t)h * kD + col0 + cg
                                   : nullptr;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c & 1, use = c >> 1;
            unsigned char *stage = smem + st * kStageBytes;
            const float *vec = reinterpret_cast<const float *>(stage + kOffPrep + PrepLayoutTC::kOffVec);
            const int n = min(kChunk, len - c * kChunk);
            const int t0 = start + c * kChunk;
            if (!warp_wait(&bars->full[st], use & 1, abort)) break;
            // Everything that depends only on the staged inputs is read before
            // waiting on the MMAs, so the critical path sees no shared loads.
            // Past the chunk end the coefficients and V are zero, so R is too.
            const bool in_chunk = tok < n;
            const float ab = vec[kVecAbar * kChunk + tok];
            const float cbk = in_chunk ? vec[kVecBmA * kChunk + tok] : 0.f;
            const float abk = in_chunk ? ab : 0.f;
            const float cbq = vec[kVecB * kChunk + tok];
            const float gs = vec[kVecGS * kChunk + tok];
            const float gm = vec[kVecGM * kChunk + tok];
            uint4 vraw = make_uint4(0u, 0u, 0u, 0u);
            if (in_chunk) vraw = *reinterpret_cast<const uint4 *>(stage + kOffV + sw128_offset(tok, chk));

            // ---- R = V - abar K S_0 + b_{i-1} alpha_i K M_0: the critical step
            if (!warp_wait(&bars->d1, c & 1, abort)) break;
            tc_fence_after();
            {
                float xs[8], xm[8], vv[8], r[8];
                tmem_ld_16x2x8(lk + C::kColD1 + c0, xs);
                tmem_ld_16x2x8(lk + C::kColD1 + NS + c0, xm);
                tmem_ld_wait();
                unpack_bf16x8(vraw, vv);
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = vv[e] - abk * xs[e] + cbk * xm[e];
                uint4 w;
                w.x = pack_bf16x2(r[0], r[1]);
                w.y = pack_bf16x2(r[2], r[3]);
                w.z = pack_bf16x2(r[4], r[5]);
                w.w = pack_bf16x2(r[6], r[7]);
                *reinterpret_cast<uint4 *>(rt + sw128_offset(tok, chk)) = w;
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->r);
            }
            // ---- O_inter = abar Q S_0 - b Q M_0, then the state rescale (both
            //      overlap MMA2)
            float oint[8];
            {
                float xs[8], xm[8];
                tmem_ld_16x2x8(lq + C::kColD1 + c0, xs);
                tmem_ld_16x2x8(lq + C::kColD1 + NS + c0, xm);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) oint[e] = ab * xs[e] - cbq * xm[e];
            }
            rescale_state(st_s, st_m, vec);
            // ---- Vres rows scaled by gS and -gM: MMA3's B operand; O_intra
            if (!warp_wait(&bars->d2, c & 1, abort)) break;
            tc_fence_after();
            {
                float x[8];
                tmem_ld_16x2x8(lk + C::kColD2 + c0, x);
                tmem_ld_wait();
                uint4 w;
                w.x = pack_bf16x2(gs * x[0], gs * x[1]);
                w.y = pack_bf16x2(gs * x[2], gs * x[3]);
                w.z = pack_bf16x2(gs * x[4], gs * x[5]);
                w.w = pack_bf16x2(gs * x[6], gs * x[7]);
                *reinterpret_cast<uint4 *>(b3 + sw128_offset(tok, chk)) = w;
                w.x = pack_bf16x2(-gm * x[0], -gm * x[1]);
                w.y = pack_bf16x2(-gm * x[2], -gm * x[3]);
                w.z = pack_bf16x2(-gm * x[4], -gm * x[5]);
                w.w = pack_bf16x2(-gm * x[6], -gm * x[7]);
                *reinterpret_cast<uint4 *>(b3 + C::kB3M + sw128_offset(tok, chk + C::kChM)) = w;
                fence_proxy_async();
                if (vg && in_chunk) {
                    // the residuals themselves, for a gradient pass
                    w.x = pack_bf16x2(x[0], x[1]);
                    w.y = pack_bf16x2(x[2], x[3]);
                    w.z = pack_bf16x2(x[4], x[5]);
                    w.w = pack_bf16x2(x[6], x[7]);
                    *reinterpret_cast<uint4 *>(vg + (size_t)(t0 + tok) * rs) = w;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->v);
            }
            {
                float x[8];
                tmem_ld_16x2x8(lq + C::kColD2 + c0, x);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) oint[e] += x[e];     // O = O_inter + O_intra
            }

            // ---- new state: bf16 copy for the next chunk's MMA1
            if (!warp_wait(&bars->d3, c & 1, abort)) break;
            tc_fence_after();
            {
                const bool more = c + 1 < nchunks;
                float S[kEpiCols], M[kEpiCols];
                if (more) {
                    tmem_ld16(st_s, S);
                    tmem_ld16(st_m, M);
                    tmem_ld_wait();
                    store_row16(b1, d, ch0, S, 1.f);
                    store_row16(b1 + C::kB1M, d, ch0 + C::kChM, M, 1.f);
                    fence_proxy_async();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (more) mbar_arrive(&bars->state);
                    mbar_arrive(&bars->empty[st]);
                }
                // the next chunk's entry state, after the chain has moved on
                if (kChunkStates && more)
                    store_chunk_state(p, slot0 + c + 1, h, st_off - (size_t)sh * kD * kD, S, M);
            }
            // ---- outputs of this chunk (off the critical path)
            if (in_chunk) {
                uint4 w;
                w.x = pack_bf16x2(oint[0], oint[1]);
                w.y = pack_bf16x2(oint[2], oint[3]);
                w.z = pack_bf16x2(oint[4], oint[5]);
                w.w = pack_bf16x2(oint[6], oint[7]);
                *reinterpret_cast<uint4 *>(og + (size_t)(t0 + tok) * rs) = w;
            }
        }
        if (!*abort) {
            float S[kEpiCols], M[kEpiCols];
            tmem_ld16(st_s, S);
            tmem_ld16(st_m, M);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < kEpiCols; j += 4) {
                if (p.S_T)
                    *reinterpret_cast<float4 *>(p.S_T + st_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                if (p.M_T)
                    *reinterpret_cast<float4 *>(p.M_T + st_off + j) = make_float4(M[j], M[j + 1], M[j + 2], M[j + 3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    if (threadIdx.x == 0 && *abort && p.status) atomicExch(p.status, (int)MDN_ERR_DEVICE_TIMEOUT);
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [T_total, H, 128] bf16 viewed as a 3-D tensor (d, h, t); box 64 x 1 x box_t.
bool make_map(CUtensorMap *map, const void *base, int T_total, int H, bool swizzle,
              int box_t = 64) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_t};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int NS, bool kChunkStates>
cudaError_t launch_state_tc_t(const ChunkProblem &p, cudaStream_t st, const CUtensorMap &mk,
                              const CUtensorMap &mq, const CUtensorMap &mv) {
    using C = Cfg<NS>;
    auto kern = chunk_state_tc_kernel<NS, kChunkStates>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)C::kSmemBytes);
    if (err != cudaSuccess) return err;
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.maxThreadsPerBlock < C::kThreads) return cudaErrorLaunchOutOfResources;
    const long blocks = (long)p.n_seq * p.H * C::kSlices;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    // programmatic dependent launch: may start while the prep kernel drains
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, mk, mq, mv);
}

}  // namespace

// The slice width trades per-chunk latency (narrow slices: smaller MMAs and
// epilogues) against CTA count: the narrowest slices (16, 32 or 64 columns)
// whose CTAs still fit on the GPU in one wave.
cudaError_t launch_chunk_state_tc(const ChunkProblem &p, cudaStream_t st) {
    if (p.D != kD || p.dtype != MDN_BF16) return cudaErrorInvalidValue;
    if (p.prep_stride % 16 != 0) return cudaErrorInvalidValue;
    CUtensorMap mk, mq, mv;
    const int Tt = p.T_total > 0 ? p.T_total : 1;
    if (!make_map(&mk, p.k, Tt, p.H, true, 16) || !make_map(&mq, p.q, Tt, p.H, true, 16) ||
        !make_map(&mv, p.v, Tt, p.H, true))
        return cudaErrorInvalidValue;
    const long chains = (long)p.n_seq * p.H;
    const int sms = device_sm_count();
    const int ns = (sms > 0 && chains * Cfg<16>::kSlices <= sms) ? 16
                 : (sms > 0 && chains * Cfg<32>::kSlices <= sms) ? 32 : 64;
    if (p.S_chunks) {
        if (ns == 16) return launch_state_tc_t<16, true>(p, st, mk, mq, mv);
        if (ns == 32) return launch_state_tc_t<32, true>(p, st, mk, mq, mv);
        return launch_state_tc_t<64, true>(p, st, mk, mq, mv);
    }
    if (ns == 16) return launch_state_tc_t<16, false>(p, st, mk, mq, mv);
    if (ns == 32) return launch_state_tc_t<32, false>(p, st, mk, mq, mv);
    return launch_state_tc_t<64, false>(p, st, mk, mq, mv);
}

}  // namespace mdn
