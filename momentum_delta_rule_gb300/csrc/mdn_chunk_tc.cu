// MDN chunkwise forward — sequential state pass on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA-staged operands), head size 64 or
// 128, bf16 inputs, or fp32 inputs through split bf16 operands.
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
// fp32 inputs (kSplit): every operand X is held as two bf16 parts, X_hi =
// bf16(X) and X_lo = bf16(X - X_hi), which carry about 16 significant bits,
// and each product is taken as A_hi B_hi + A_hi B_lo + A_lo B_hi (three MMA
// groups into the same fp32 accumulator); the dropped A_lo B_lo and the
// parts' own rounding leave relative errors near 1e-5.  The q, k, v parts
// come from a conversion kernel, T and A_O T's parts from the fp32 prep.  The
// stage is single-buffered there (the split operands double its size).
//
// One CTA owns one (sequence, head, NS-column slice): columns of S and M
// evolve independently (column j of Vres depends only on column j of S_0 and
// M_0), so the slices of a head never communicate.  A second instantiation
// also stores every chunk's entry state (S, M) for a gradient pass.
//
// Warp roles (2 + NS / 4 warps, 18 for NS = 64): 0 TMA producer, 1 MMA
// issuer + TMEM owner (all lanes wait, lane 0 issues), the rest epilogue
// (TMEM lane quadrant = warp % 4, 16-column group of the slice =
// (warp-2)/4).  A warp reaches only the TMEM lanes of its quadrant, and the
// warps of a quadrant share one scheduler; [K; Q] and [T; A_O T] rows are
// therefore interleaved in blocks of 16 (tc_row), so that every quadrant
// holds 16 token rows and 16 query rows and the token-row steps (R, Vres)
// use all four schedulers (16x32bx2 TMEM loads: lanes t and t + 16 take 8
// columns each).  With head size 64, MMA3 is an M = 64 product, whose row r
// sits in TMEM lane 32 (r / 16) + r % 16: lanes 0..15 of each quadrant hold
// the state rows.
// Every wait is bounded (1 s); on expiry the CTA records
// MDN_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <type_traits>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

using namespace sm100;

constexpr int kEpiCols = 16;             // state columns per epilogue thread
constexpr uint32_t kKQHalf = 16384;      // one 64-wide dk half: 64 K rows + 64 Q rows, swizzled
constexpr uint32_t kVBytes = 8192;       // V tile, 64 tokens x 64 columns, swizzled

// Everything that depends on the head size D, the slice width NS (state
// columns per CTA) and the operand form (kSplit: hi and lo bf16 parts).
// In the N dimension of [S | M]-shaped operands, S takes columns [0, NS) and
// M [NS, 2NS); operands are MN-major in blocks of 64 columns, so for NS = 64
// the M half is a second block and for NS = 32 or 16 it shares the block.
template <int D, int NS, bool kSplit>
struct Cfg {
    static_assert(NS == 16 || NS == 32 || NS == 64, "slice width");
    static_assert(D == 64 || D == 128, "head size");
    static constexpr int kHalves = D / 64;
    static constexpr int kStages = kSplit ? 1 : 2;
    static constexpr int kParts = kSplit ? 2 : 1;
    static constexpr int kSlices = D / NS;
    static constexpr int kEpiWarps = 4 * NS / kEpiCols;      // 4 lane quadrants
    static constexpr int kThreads = 32 * (2 + kEpiWarps);
    // one pipeline stage: [K; Q] parts, V parts, the prepared block
    static constexpr uint32_t kKQPart = kHalves * kKQHalf;
    static constexpr uint32_t kOffV = kParts * kKQPart;
    static constexpr uint32_t kOffPrep = kOffV + kParts * kVBytes;
    static constexpr uint32_t kPrepBytes =
        kSplit ? (uint32_t)PrepLayoutTC::kSplitBytes : (uint32_t)PrepLayoutTC::kBytes;
    static constexpr uint32_t kPrepLo = (uint32_t)PrepLayoutTC::kSplitLo;   // lo part (split)
    static constexpr uint32_t kPrepVec =
        kSplit ? (uint32_t)PrepLayoutTC::kSplitVec : (uint32_t)PrepLayoutTC::kOffVec;
    static constexpr uint32_t kStageBytes = kOffPrep + kPrepBytes;
    static_assert(kStageBytes % 1024 == 0, "stage alignment");
    // operands written by the epilogue
    static constexpr uint32_t kOffB1 = kStages * kStageBytes;  // [S | M] bf16, dk rows x 2NS
    static constexpr uint32_t kB1Part = (NS == 64 ? 2 : 1) * D * 128;
    static constexpr uint32_t kB1M = NS == 64 ? D * 128 : 0;    // byte offset of the M half
    static constexpr uint32_t kOffR = kOffB1 + kParts * kB1Part; // R bf16, 64 token rows x NS
    static constexpr uint32_t kRPart = 8192;
    static constexpr uint32_t kOffB3 = kOffR + kParts * kRPart;  // [gS Vres | -gM Vres]
    static constexpr uint32_t kB3Part = NS == 64 ? 16384 : 8192;
    static constexpr uint32_t kB3M = NS == 64 ? 8192 : 0;
    static constexpr uint32_t kChM = NS == 64 ? 0 : NS / 8;   // chunk offset of the M half
    static constexpr uint32_t kOffBar = kOffB3 + kParts * kB3Part;
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
    // tensor memory columns
    static constexpr uint32_t kColD1 = 0;                     // 2NS columns
    static constexpr uint32_t kColD2 = 2 * NS;                // NS columns
    static constexpr uint32_t kColSt = 4 * NS;                // fp32 state [S | M], 2NS columns
    static constexpr uint32_t kTmemCols = 8 * NS;
    static constexpr uint32_t kIdesc1 = idesc_bf16(128, 2 * NS, false, true);
    static constexpr uint32_t kIdesc2 = idesc_bf16(128, NS, false, true);
    static constexpr uint32_t kIdesc3 = idesc_bf16(D, 2 * NS, true, true);
};

struct Bars {
    uint64_t full[2];          // TMA bytes of a stage landed
    uint64_t empty[2];         // stage free again (MMA commit + every epilogue warp)
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

// Eight fp32 values (times `scale`) as one 16-byte chunk of bf16, and, for a
// split operand, the chunk of what the first rounding left over.
__device__ __forceinline__ void pack8(const float *x, float scale, uint4 &hi, uint4 &lo) {
    float y[8], r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        y[e] = scale * x[e];
        r[e] = y[e] - __bfloat162float(__float2bfloat16_rn(y[e]));
    }
    hi = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
    lo = make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                    pack_bf16x2(r[6], r[7]));
}

// Write 8 values into 16-byte chunk `chunk` of row `row` of a 128-byte-swizzled
// operand tile, and the lo part `part_bytes` further on (split operands).
template <bool kSplit>
__device__ __forceinline__ void put8(unsigned char *tile, uint32_t part_bytes, uint32_t row,
                                     uint32_t chunk, const float *x, float scale) {
    uint4 hi, lo;
    pack8(x, scale, hi, lo);
    const uint32_t off = sw128_offset(row, chunk);
    *reinterpret_cast<uint4 *>(tile + off) = hi;
    if (kSplit) *reinterpret_cast<uint4 *>(tile + part_bytes + off) = lo;
}

// Write 16 fp32 values into row `row`, 16-byte chunks [chunk0, chunk0+2).
template <bool kSplit>
__device__ __forceinline__ void store_row16(unsigned char *tile, uint32_t part_bytes, uint32_t row,
                                            uint32_t chunk0, const float *x) {
    put8<kSplit>(tile, part_bytes, row, chunk0, x, 1.f);
    put8<kSplit>(tile, part_bytes, row, chunk0 + 1, x + 8, 1.f);
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

// The same rescale eight columns at a time: half the registers at its peak
// (the dual-slice pass runs it while one slice's O_inter is still held).
__device__ __forceinline__ void rescale_state_halves(uint32_t st_s, uint32_t st_m, const float *vec) {
    const float ab_n = vec[kVecScal * kChunk + 0];
    const float b_n = vec[kVecScal * kChunk + 1];
    const float mb_n = vec[kVecScal * kChunk + 2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float S[8], M[8];
        tmem_ld8(st_s + 8 * hf, S);
        tmem_ld8(st_m + 8 * hf, M);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float s_old = S[j];
            S[j] = ab_n * s_old - b_n * M[j];
            M[j] = mb_n * M[j];
        }
        tmem_st8(st_s + 8 * hf, S);
        tmem_st8(st_m + 8 * hf, M);
    }
    tmem_st_wait();
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Eight consecutive outputs (o or the residuals) of one token row.
__device__ __forceinline__ void store_out8(__nv_bfloat16 *dst, const float *x) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                                 pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
}
__device__ __forceinline__ void store_out8(float *dst, const float *x) {
    *reinterpret_cast<float4 *>(dst) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
}

// One thread's 16 columns of row d of the entry state of chunk slot `slot`
// (layout [slot, H, dk, dv], element type Ts: bf16 for bf16 inputs, fp32
// for fp32 inputs); `off` = d * dk + first column.
template <int D, typename Ts>
__device__ __forceinline__ void store_chunk_state(const ChunkProblem &p, int slot, int h, size_t off,
                                                  const float *S, const float *M) {
    const size_t base = ((size_t)slot * p.H + h) * D * D + off;
    Ts *sd = static_cast<Ts *>(p.S_chunks) + base, *md = static_cast<Ts *>(p.M_chunks) + base;
#pragma unroll
    for (int j = 0; j < kEpiCols; j += 8) {
        store_out8(sd + j, S + j);
        store_out8(md + j, M + j);
    }
}

// The tensor maps of one launch: K, Q, V, for split operands their lo
// parts, and for the saved chunk states of bf16 inputs the bf16 [block, dk,
// dv] arrays as boxes of 64 columns by all dk rows (the layout of a 64-column
// state operand tile).
struct Maps {
    CUtensorMap k, q, v, k_lo, q_lo, v_lo, sc, mc;
};

// kChunkStates: also write the entry state of every chunk (a separate
// instantiation, so the plain forward carries none of its registers).
template <int D, int NS, bool kChunkStates, bool kSplit, bool kSeg>
__global__ void __launch_bounds__(Cfg<D, NS, kSplit>::kThreads, 1)
chunk_state_tc_kernel(const ChunkProblem p, const __grid_constant__ Maps maps) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem_1024(smem_raw);
    using C = Cfg<D, NS, kSplit>;
    using Tio = typename std::conditional<kSplit, float, __nv_bfloat16>::type;
    constexpr int kStages = C::kStages;
    // bf16 entry states of 64-column slices leave as tensor stores of the
    // operand tile; narrower slices (S and M share a tile row) and fp32
    // store from the epilogue's registers
    constexpr bool kTmaStates = kChunkStates && !kSplit && NS == 64;
    Bars *bars = reinterpret_cast<Bars *>(smem + C::kOffBar);
    volatile int *abort = &bars->abort;

    constexpr int kEpiWarps = C::kEpiWarps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x % C::kSlices;
    const int kh = blockIdx.x / C::kSlices;
    // This grid may start while the prep kernel finishes (programmatic
    // dependent launch).  Packed sequences read the chunk offsets first: wait
    // for the preceding grids right away.  Fixed-length batches run their
    // setup and initial-state loads first; the producer waits before its
    // first prepared-block copy.  A later time segment reads the states the
    // previous one left, so it waits first too; a segment with a successor
    // lets that successor's prep start as soon as all its CTAs run.
    if constexpr (kSeg) {
        if (p.seg_mode & kSegStateTrigger) grid_launch_dependents();
        if (p.seg_mode & kSegStateWaitFirst) grid_dependency_wait();
    }
    if (p.cu_seqlens != nullptr) grid_dependency_wait();
    const int s = ordered_sequence(p, kh / p.H), h = kh % p.H;
    const int sh = s * p.H + h;                 // (sequence, head) of the states
    const int col0 = slice * NS;
    int start, len, slot0;
    sequence_range(p, s, start, len, slot0);
    if constexpr (kSeg) {
        // a time segment: chunks [seg_c0, seg_c1) of the sequence, whole
        // chunks but for the sequence's last
        const int all = (len + kChunk - 1) / kChunk;
        const int c0 = min(p.seg_c0, all), c1 = min(p.seg_c1, all);
        start += c0 * kChunk;
        slot0 += c0;
        len = min(len - c0 * kChunk, (c1 - c0) * kChunk);
    }
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
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.v);
        if (kSplit) {
            prefetch_tensormap(&maps.k_lo);
            prefetch_tensormap(&maps.q_lo);
            prefetch_tensormap(&maps.v_lo);
        }
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
            int last_use[2] = {-1, -1};
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kStages, use = c / kStages;
                if (c == 0) grid_dependency_wait();   // the prepared blocks are complete
                if (!mbar_wait(&bars->empty[st], (use & 1) ^ 1, abort)) break;
                unsigned char *stage = smem + st * C::kStageBytes;
                const int t0 = start + c * kChunk;
                const unsigned char *blk =
                    p.prep + ((size_t)(slot0 + c) * p.H + h) * p.prep_stride;
                mbar_arrive_expect_tx(&bars->full[st], C::kStageBytes);
                // [K; Q] rows interleaved by 16 (tc_row): 16-token boxes
#pragma unroll
                for (int part = 0; part < C::kParts; ++part) {
                    const CUtensorMap *mk = part ? &maps.k_lo : &maps.k;
                    const CUtensorMap *mq = part ? &maps.q_lo : &maps.q;
#pragma unroll
                    for (int hh = 0; hh < C::kHalves; ++hh)
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            unsigned char *dst = stage + part * C::kKQPart + hh * kKQHalf + g * 4096;
                            tma_load_3d(dst, mk, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                            tma_load_3d(dst + 2048, mq, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                        }
                    tma_load_3d(stage + C::kOffV + part * kVBytes, part ? &maps.v_lo : &maps.v,
                                &bars->full[st], col0, h, t0);
                }
                bulk_load(stage + C::kOffPrep, blk, C::kPrepBytes, &bars->full[st]);
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
        // whole warp waits, lane 0 issues and commits).  Split operands take
        // three passes per product: (hi, hi), (hi, lo), (lo, hi).
        {
            const bool l0 = lane == 0;
            const uint32_t b1 = smem_u32(smem + C::kOffB1);
            const uint32_t rr = smem_u32(smem + C::kOffR);
            const uint32_t b3 = smem_u32(smem + C::kOffB3);
            constexpr uint32_t kLbo1 = C::kB1M ? C::kB1M : 16384;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kStages, use = c / kStages;
                const uint32_t kq = smem_u32(smem + st * C::kStageBytes);
                const uint32_t prep = kq + C::kOffPrep;
                if (!warp_wait(&bars->full[st], use & 1, abort)) break;
                if (!warp_wait(&bars->state, c & 1, abort)) break;
                tc_fence_after();
                if (l0) {
#pragma unroll
                    for (int pass = 0; pass < (kSplit ? 3 : 1); ++pass) {
                        const uint32_t a0 = kq + (pass == 2 ? C::kKQPart : 0u);
                        const uint32_t bb = b1 + (pass == 1 ? C::kB1Part : 0u);
#pragma unroll
                        for (int kb = 0; kb < C::kHalves; ++kb)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t a = sdesc_sw128(a0 + kb * kKQHalf + kk * 32, 16, 1024);
                                const uint64_t b = sdesc_sw128(bb + (kb * 4 + kk) * 2048, kLbo1, 1024);
                                mma_bf16(tmem + C::kColD1, a, b, C::kIdesc1, (pass | kb | kk) != 0);
                            }
                    }
                    mma_commit(&bars->d1);
                    if constexpr (kTmaStates) {
                        // the chunk's entry state, already the bf16 operand
                        // tile: out to its slot by tensor stores
                        const int z = (slot0 + c) * p.H + h;
                        tma_store_3d(&maps.sc, smem + C::kOffB1, col0, 0, z);
                        tma_store_3d(&maps.mc, smem + C::kOffB1 + C::kB1M, col0, 0, z);
                        bulk_commit_group();
                    }
                }
                __syncwarp();
                if (!warp_wait(&bars->r, c & 1, abort)) break;
                tc_fence_after();
                if (l0) {
#pragma unroll
                    for (int pass = 0; pass < (kSplit ? 3 : 1); ++pass) {
                        const uint32_t a0 = prep + (pass == 2 ? C::kPrepLo : 0u);
                        const uint32_t bb = rr + (pass == 1 ? C::kRPart : 0u);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = sdesc_sw128(a0 + kk * 32, 16, 1024);
                            const uint64_t b = sdesc_sw128(bb + kk * 2048, 8192, 1024);
                            mma_bf16(tmem + C::kColD2, a, b, C::kIdesc2, (pass | kk) != 0);
                        }
                    }
                    mma_commit(&bars->d2);
                }
                __syncwarp();
                if (!warp_wait(&bars->v, c & 1, abort)) break;
                tc_fence_after();
                if (l0) {
#pragma unroll
                    for (int pass = 0; pass < (kSplit ? 3 : 1); ++pass) {
                        const uint32_t a0 = kq + (pass == 2 ? C::kKQPart : 0u);
                        const uint32_t bb = b3 + (pass == 1 ? C::kB3Part : 0u);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = sdesc_sw128(a0 + kk * 4096, kKQHalf, 1024);
                            const uint64_t b = sdesc_sw128(bb + kk * 2048, 8192, 1024);
                            mma_bf16(tmem + C::kColSt, a, b, C::kIdesc3, 1);
                        }
                    }
                    // the epilogue rewrites the state tile after d3
                    if constexpr (kTmaStates) bulk_wait_group_read0();
                    mma_commit(&bars->d3);
                    mma_commit(&bars->empty[st]);
                }
                __syncwarp();
            }
            // drain: all issued MMAs complete before TMEM is freed, the
            // state stores before the CTA exits
            if (l0) {
                mma_commit(&bars->drain);
                int dummy = 0;
                mbar_wait(&bars->drain, 0, &dummy);
                if constexpr (kTmaStates) bulk_wait_group0();
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
        // state row of this thread: lane = row for head size 128; lanes
        // 0..15 of each quadrant for 64 (the M = 64 product's rows)
        const bool row_ok = D == 128 || lane < 16;
        const int d = D == 128 ? 32 * q + lane : 16 * q + (lane & 15);
        const uint32_t st_s = lane_base + C::kColSt + c0;       // S columns of this thread
        const uint32_t st_m = lane_base + C::kColSt + NS + c0;  // M columns
        const size_t st_off = (size_t)sh * D * D + (size_t)d * D + col0 + c0;
        unsigned char *b1 = smem + C::kOffB1;
        unsigned char *rt = smem + C::kOffR;
        unsigned char *b3 = smem + C::kOffB3;
        {
            float S[kEpiCols], M[kEpiCols];
#pragma unroll
            for (int j = 0; j < kEpiCols; j += 4) {
                float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), mv = sv;
                if (p.S0 && row_ok) sv = *reinterpret_cast<const float4 *>(p.S0 + st_off + j);
                if (p.M0 && row_ok) mv = *reinterpret_cast<const float4 *>(p.M0 + st_off + j);
                S[j] = sv.x; S[j + 1] = sv.y; S[j + 2] = sv.z; S[j + 3] = sv.w;
                M[j] = mv.x; M[j + 1] = mv.y; M[j + 2] = mv.z; M[j + 3] = mv.w;
            }
            tmem_st16(st_s, S);
            tmem_st16(st_m, M);
            tmem_st_wait();
            if (nchunks > 0) {
                if (row_ok) {
                    store_row16<kSplit>(b1, C::kB1Part, d, ch0, S);
                    store_row16<kSplit>(b1 + C::kB1M, C::kB1Part, d, ch0 + C::kChM, M);
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->state);
                if (kChunkStates && !kTmaStates && row_ok)
                    store_chunk_state<D, Tio>(p, slot0, h, st_off - (size_t)sh * D * D, S, M);
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
        const size_t rs = (size_t)p.H * D;
        Tio *og = static_cast<Tio *>(p.o) + (size_t)h * D + col0 + cg;
        Tio *vg = p.vres ? static_cast<Tio *>(p.vres) + (size_t)h * D + col0 + cg : nullptr;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kStages, use = c / kStages;
            unsigned char *stage = smem + st * C::kStageBytes;
            const float *vec = reinterpret_cast<const float *>(stage + C::kOffPrep + C::kPrepVec);
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
            float vv[8];
            {
                uint4 vraw = make_uint4(0u, 0u, 0u, 0u), vlo = vraw;
                if (in_chunk) {
                    vraw = *reinterpret_cast<const uint4 *>(stage + C::kOffV + sw128_offset(tok, chk));
                    if (kSplit)
                        vlo = *reinterpret_cast<const uint4 *>(stage + C::kOffV + kVBytes +
                                                               sw128_offset(tok, chk));
                }
                unpack_bf16x8(vraw, vv);
                if (kSplit) {
                    float vl[8];
                    unpack_bf16x8(vlo, vl);
#pragma unroll
                    for (int e = 0; e < 8; ++e) vv[e] += vl[e];
                }
            }

            // ---- R = V - abar K S_0 + b_{i-1} alpha_i K M_0: the critical step
            if (!warp_wait(&bars->d1, c & 1, abort)) break;
            tc_fence_after();
            {
                float xs[8], xm[8], r[8];
                tmem_ld_16x2x8(lk + C::kColD1 + c0, xs);
                tmem_ld_16x2x8(lk + C::kColD1 + NS + c0, xm);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = vv[e] - abk * xs[e] + cbk * xm[e];
                put8<kSplit>(rt, C::kRPart, tok, chk, r, 1.f);
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
                put8<kSplit>(b3, C::kB3Part, tok, chk, x, gs);
                put8<kSplit>(b3 + C::kB3M, C::kB3Part, tok, chk + C::kChM, x, -gm);
                fence_proxy_async();
                // the residuals themselves, for a gradient pass
                if (vg && in_chunk) store_out8(vg + (size_t)(t0 + tok) * rs, x);
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
                    if (row_ok) {
                        store_row16<kSplit>(b1, C::kB1Part, d, ch0, S);
                        store_row16<kSplit>(b1 + C::kB1M, C::kB1Part, d, ch0 + C::kChM, M);
                    }
                    fence_proxy_async();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (more) mbar_arrive(&bars->state);
                    mbar_arrive(&bars->empty[st]);
                }
                // the next chunk's entry state, after the chain has moved on
                if (kChunkStates && !kTmaStates && more && row_ok)
                    store_chunk_state<D, Tio>(p, slot0 + c + 1, h, st_off - (size_t)sh * D * D, S, M);
            }
            // ---- outputs of this chunk (off the critical path)
            if (in_chunk) store_out8(og + (size_t)(t0 + tok) * rs, oint);
        }
        if (!*abort) {
            // every lane takes part in the warp's loads; lanes with a state
            // row store it
            float S[kEpiCols], M[kEpiCols];
            tmem_ld16(st_s, S);
            tmem_ld16(st_m, M);
            tmem_ld_wait();
            if (row_ok) {
#pragma unroll
                for (int j = 0; j < kEpiCols; j += 4) {
                    if (p.S_T)
                        *reinterpret_cast<float4 *>(p.S_T + st_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                    if (p.M_T)
                        *reinterpret_cast<float4 *>(p.M_T + st_off + j) = make_float4(M[j], M[j + 1], M[j + 2], M[j + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    if (threadIdx.x == 0 && *abort && p.status) atomicExch(p.status, (int)MDN_ERR_DEVICE_TIMEOUT);
}

// ------------------------------------------------------------------ dual

// Both 64-column slices of a head (d = 128, bf16 inputs) in one CTA, as two
// chains A (columns 0..63) and B (64..127) whose steps interleave: while the
// epilogue warps work on one slice's step, the tensor cores run the other
// slice's product.  Per chunk the MMA thread issues MMA1_A, MMA1_B, MMA2_A,
// MMA2_B, MMA3_A, MMA3_B and the epilogue runs R_A, R_B, Vres_A, Vres_B,
// state_A, state_B, each waiting only on its own slice's barrier.  TMEM:
// slice X owns columns [256 X, 256 X + 256): MMA1's [S | M] products at
// +0 (MMA2's product later over their S part, once the R step has read both
// the key and the query rows), the fp32 state [S | M] at +128.  Shared
// memory holds one V tile (both slices' columns) apart from the double-
// buffered [K; Q] stages: the next chunk's V is copied in once both R steps
// have read the current one; and each slice's R sits over the S half of its
// MMA3 operand, which is written only after MMA2 has read R and read by MMA3
// before the next R.
struct DualCfg {
    static constexpr int D = 128, NS = 64;
    static constexpr int kHalves = 2;
    static constexpr int kEpiWarps = 16;
    static constexpr int kThreads = 32 * (2 + kEpiWarps);
    static constexpr uint32_t kOffPrep = kHalves * kKQHalf;          // [K; Q], then the block
    static constexpr uint32_t kPrepBytes = (uint32_t)PrepLayoutTC::kBytes;
    static constexpr uint32_t kPrepVec = (uint32_t)PrepLayoutTC::kOffVec;
    static constexpr uint32_t kStageBytes = kOffPrep + kPrepBytes;
    static_assert(kStageBytes % 1024 == 0, "stage alignment");
    static constexpr uint32_t kOffB1 = 2 * kStageBytes;             // per slice [S | M] bf16
    static constexpr uint32_t kB1Bytes = 2 * D * 128;
    static constexpr uint32_t kB1M = D * 128;
    static constexpr uint32_t kOffB3 = kOffB1 + 2 * kB1Bytes;       // per slice [gS Vres | -gM Vres];
    static constexpr uint32_t kB3Bytes = 16384;                     // R over its S half
    static constexpr uint32_t kB3M = 8192;
    static constexpr uint32_t kOffV = kOffB3 + 2 * kB3Bytes;        // V, 64 tokens x 128 columns
    static constexpr uint32_t kVTile = 2 * kVBytes;
    static constexpr uint32_t kOffBar = kOffV + kVTile;
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kSliceCols = 256;                    // per slice
    static constexpr uint32_t kColSt = 128;                        // state, within a slice
    static constexpr uint32_t kIdesc1 = idesc_bf16(128, 2 * NS, false, true);
    static constexpr uint32_t kIdesc2 = idesc_bf16(128, NS, false, true);
    static constexpr uint32_t kIdesc3 = idesc_bf16(D, 2 * NS, true, true);
};

struct DualBars {
    uint64_t full[2], empty[2], vfull, vempty;
    uint64_t d1[2], r[2], d2[2], v[2], d3[2], state[2];   // per slice
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(DualBars) <= 256, "barrier block");

template <bool kChunkStates, bool kVres>
__global__ void __launch_bounds__(DualCfg::kThreads, 1)
chunk_state_dual_kernel(const ChunkProblem p, const __grid_constant__ Maps maps) {
    using C = DualCfg;
    constexpr int D = C::D;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem_1024(smem_raw);
    DualBars *bars = reinterpret_cast<DualBars *>(smem + C::kOffBar);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (p.cu_seqlens != nullptr) grid_dependency_wait();
    const int kh = blockIdx.x;
    const int s = ordered_sequence(p, kh / p.H), h = kh % p.H;
    const int sh = s * p.H + h;
    int start, len, slot0;
    sequence_range(p, s, start, len, slot0);
    const int nchunks = (len + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 1 + C::kEpiWarps);
            mbar_init(&bars->d1[i], 1);
            mbar_init(&bars->r[i], C::kEpiWarps);
            mbar_init(&bars->d2[i], 1);
            mbar_init(&bars->v[i], C::kEpiWarps);
            mbar_init(&bars->d3[i], 1);
            mbar_init(&bars->state[i], C::kEpiWarps);
        }
        mbar_init(&bars->vfull, 1);
        mbar_init(&bars->vempty, C::kEpiWarps);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.v);
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
            int last_use[2] = {-1, -1}, v_last = -1;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c & 1, use = c >> 1;
                if (c == 0) grid_dependency_wait();
                if (!mbar_wait(&bars->empty[st], (use & 1) ^ 1, abort)) break;
                unsigned char *stage = smem + st * C::kStageBytes;
                const int t0 = start + c * kChunk;
                const unsigned char *blk = p.prep + ((size_t)(slot0 + c) * p.H + h) * p.prep_stride;
                mbar_arrive_expect_tx(&bars->full[st], C::kStageBytes);
#pragma unroll
                for (int hh = 0; hh < C::kHalves; ++hh)
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        unsigned char *dst = stage + hh * kKQHalf + g * 4096;
                        tma_load_3d(dst, &maps.k, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                        tma_load_3d(dst + 2048, &maps.q, &bars->full[st], 64 * hh, h, t0 + 16 * g);
                    }
                bulk_load(stage + C::kOffPrep, blk, C::kPrepBytes, &bars->full[st]);
                last_use[st] = use;
                // V of this chunk, once both R steps of the previous one are done
                if (!mbar_wait(&bars->vempty, (c & 1) ^ 1, abort)) break;
                mbar_arrive_expect_tx(&bars->vfull, C::kVTile);
                tma_load_3d(smem + C::kOffV, &maps.v, &bars->vfull, 0, h, t0);
                tma_load_3d(smem + C::kOffV + kVBytes, &maps.v, &bars->vfull, 64, h, t0);
                v_last = c;
            }
            for (int st = 0; st < 2; ++st) {
                if (last_use[st] < 0) continue;
                int dummy = 0;
                mbar_wait(&bars->full[st], last_use[st] & 1, &dummy);
            }
            if (v_last >= 0) {
                int dummy = 0;
                mbar_wait(&bars->vfull, v_last & 1, &dummy);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        const bool l0 = lane == 0;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c & 1, use = c >> 1;
            const uint32_t kq = smem_u32(smem + st * C::kStageBytes);
            const uint32_t prep = kq + C::kOffPrep;
            bool ok = warp_wait(&bars->full[st], use & 1, abort);
            // MMA1 of both slices: D = [K; Q] [S | M]
            for (int x = 0; x < 2 && ok; ++x) {
                ok = warp_wait(&bars->state[x], c & 1, abort);
                if (!ok) break;
                tc_fence_after();
                if (l0) {
                    const uint32_t b1 = smem_u32(smem + C::kOffB1 + x * C::kB1Bytes);
#pragma unroll
                    for (int kb = 0; kb < C::kHalves; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = sdesc_sw128(kq + kb * kKQHalf + kk * 32, 16, 1024);
                            const uint64_t b = sdesc_sw128(b1 + (kb * 4 + kk) * 2048, C::kB1M, 1024);
                            mma_bf16(tmem + x * C::kSliceCols, a, b, C::kIdesc1, (kb | kk) != 0);
                        }
                    mma_commit(&bars->d1[x]);
                    if constexpr (kChunkStates) {
                        // the chunk's entry state of this slice, already the
                        // bf16 operand tile: out to its slot by tensor stores
                        const unsigned char *bx = smem + C::kOffB1 + x * C::kB1Bytes;
                        const int z = (slot0 + c) * p.H + h;
                        tma_store_3d(&maps.sc, bx, 64 * x, 0, z);
                        tma_store_3d(&maps.mc, bx + C::kB1M, 64 * x, 0, z);
                        bulk_commit_group();
                    }
                }
                __syncwarp();
            }
            // MMA2 of both slices: D = [T; A_O T] R, over MMA1's S columns
            for (int x = 0; x < 2 && ok; ++x) {
                ok = warp_wait(&bars->r[x], c & 1, abort);
                if (!ok) break;
                tc_fence_after();
                if (l0) {
                    const uint32_t rr = smem_u32(smem + C::kOffB3 + x * C::kB3Bytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(prep + kk * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(rr + kk * 2048, 8192, 1024);
                        mma_bf16(tmem + x * C::kSliceCols, a, b, C::kIdesc2, kk != 0);
                    }
                    mma_commit(&bars->d2[x]);
                }
                __syncwarp();
            }
            // MMA3 of both slices: [S | M] += K^T [gS Vres | -gM Vres]
            for (int x = 0; x < 2 && ok; ++x) {
                ok = warp_wait(&bars->v[x], c & 1, abort);
                if (!ok) break;
                tc_fence_after();
                if (l0) {
                    const uint32_t b3 = smem_u32(smem + C::kOffB3 + x * C::kB3Bytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(kq + kk * 4096, kKQHalf, 1024);
                        const uint64_t b = sdesc_sw128(b3 + kk * 2048, 8192, 1024);
                        mma_bf16(tmem + x * C::kSliceCols + C::kColSt, a, b, C::kIdesc3, 1);
                    }
                    // the epilogue rewrites the state tiles after d3
                    if (kChunkStates && x == 0) bulk_wait_group_read0();
                    mma_commit(&bars->d3[x]);
                    if (x == 1) mma_commit(&bars->empty[st]);
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (l0) {
            mma_commit(&bars->drain);
            int dummy = 0;
            mbar_wait(&bars->drain, 0, &dummy);
            if (kChunkStates) bulk_wait_group0();    // the state stores land before exit
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;
        const int qc = (warp - 2) >> 2;
        const int c0 = qc * kEpiCols;                    // first column within a slice
        const uint32_t ch0 = qc * 2;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const int d = 32 * q + lane;                     // state row
        const size_t st_row = (size_t)d * D + c0;        // + 64 x for slice x
        unsigned char *b1 = smem + C::kOffB1;
        unsigned char *b3 = smem + C::kOffB3;
        auto st_s = [&](int x) { return lane_base + x * C::kSliceCols + C::kColSt + c0; };
        auto st_m = [&](int x) { return lane_base + x * C::kSliceCols + C::kColSt + C::NS + c0; };
#pragma unroll 1
        for (int x = 0; x < 2; ++x) {
            float S[kEpiCols], M[kEpiCols];
            const size_t off = (size_t)sh * D * D + st_row + 64 * x;
#pragma unroll
            for (int j = 0; j < kEpiCols; j += 4) {
                float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), mv = sv;
                if (p.S0) sv = *reinterpret_cast<const float4 *>(p.S0 + off + j);
                if (p.M0) mv = *reinterpret_cast<const float4 *>(p.M0 + off + j);
                S[j] = sv.x; S[j + 1] = sv.y; S[j + 2] = sv.z; S[j + 3] = sv.w;
                M[j] = mv.x; M[j + 1] = mv.y; M[j + 2] = mv.z; M[j + 3] = mv.w;
            }
            tmem_st16(st_s(x), S);
            tmem_st16(st_m(x), M);
            tmem_st_wait();
            if (nchunks > 0) {
                unsigned char *bx = b1 + x * C::kB1Bytes;
                store_row16<false>(bx, 0, d, ch0, S);
                store_row16<false>(bx + C::kB1M, 0, d, ch0, M);
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->state[x]);
            }
        }
        const int tok = 16 * q + (lane & 15);
        const int cg = c0 + 8 * (lane >> 4);
        const uint32_t chk = (uint32_t)(cg >> 3);
        const uint32_t lk = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t lq = tmem + ((uint32_t)(32 * q + 16) << 16);
        const size_t rs = (size_t)p.H * D;
        __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.o) + (size_t)h * D + cg;
        // the residual output is a separate instantiation (its pointer and
        // stores would cost the plain pass registers)
        __nv_bfloat16 *vg = kVres ? static_cast<__nv_bfloat16 *>(p.vres) + (size_t)h * D + cg : nullptr;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c & 1, use = c >> 1;
            unsigned char *stage = smem + st * C::kStageBytes;
            const float *vec = reinterpret_cast<const float *>(stage + C::kOffPrep + C::kPrepVec);
            const int n = min(kChunk, len - c * kChunk);
            const int t0 = start + c * kChunk;
            const bool in_chunk = tok < n;
            ok = warp_wait(&bars->full[st], use & 1, abort) && warp_wait(&bars->vfull, c & 1, abort);
            if (!ok) break;
            // V of this thread's token row, both slices (zero past the chunk end)
            uint4 vraw[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if (in_chunk) {
                vraw[0] = *reinterpret_cast<const uint4 *>(smem + C::kOffV + sw128_offset(tok, chk));
                vraw[1] = *reinterpret_cast<const uint4 *>(smem + C::kOffV + kVBytes +
                                                           sw128_offset(tok, chk));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->vempty);   // V read: the next one may land
            const float ab = vec[kVecAbar * kChunk + tok];
            const float cbk = in_chunk ? vec[kVecBmA * kChunk + tok] : 0.f;
            const float abk = in_chunk ? ab : 0.f;
            const float cbq = vec[kVecB * kChunk + tok];
            const float gs = vec[kVecGS * kChunk + tok];
            const float gm = vec[kVecGM * kChunk + tok];
            float oint[2][8];
            // ---- R and O_inter of each slice (both row sets of MMA1 read
            //      before MMA2 may overwrite them), then the state rescale
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                ok = warp_wait(&bars->d1[x], c & 1, abort);
                if (!ok) break;
                tc_fence_after();
                float vv[8], xs[8], xm[8], ys[8], ym[8], r[8];
                unpack_bf16x8(vraw[x], vv);
                const uint32_t dx = x * C::kSliceCols;
                tmem_ld_16x2x8(lk + dx + c0, xs);
                tmem_ld_16x2x8(lk + dx + C::NS + c0, xm);
                tmem_ld_16x2x8(lq + dx + c0, ys);
                tmem_ld_16x2x8(lq + dx + C::NS + c0, ym);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    r[e] = vv[e] - abk * xs[e] + cbk * xm[e];
                    oint[x][e] = ab * ys[e] - cbq * ym[e];
                }
                put8<false>(b3 + x * C::kB3Bytes, 0, tok, chk, r, 1.f);
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->r[x]);
                rescale_state_halves(st_s(x), st_m(x), vec);
            }
            if (!ok) break;
            // ---- Vres of each slice: MMA3's B operand; O = O_inter + O_intra
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                ok = warp_wait(&bars->d2[x], c & 1, abort);
                if (!ok) break;
                tc_fence_after();
                float xv[8], xo[8];
                const uint32_t dx = x * C::kSliceCols;
                tmem_ld_16x2x8(lk + dx + c0, xv);
                tmem_ld_16x2x8(lq + dx + c0, xo);
                tmem_ld_wait();
                unsigned char *bx = b3 + x * C::kB3Bytes;
                put8<false>(bx, 0, tok, chk, xv, gs);
                put8<false>(bx + C::kB3M, 0, tok, chk, xv, -gm);
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->v[x]);
                if (in_chunk) {
                    if constexpr (kVres) store_out8(vg + (size_t)(t0 + tok) * rs + 64 * x, xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xo[e] += oint[x][e];
                    store_out8(og + (size_t)(t0 + tok) * rs + 64 * x, xo);
                }
            }
            if (!ok) break;
            // ---- new state of each slice: bf16 copy for the next MMA1
            const bool more = c + 1 < nchunks;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                ok = warp_wait(&bars->d3[x], c & 1, abort);
                if (!ok) break;
                tc_fence_after();
                float S[kEpiCols], M[kEpiCols];
                if (more) {
                    tmem_ld16(st_s(x), S);
                    tmem_ld16(st_m(x), M);
                    tmem_ld_wait();
                    unsigned char *bx = b1 + x * C::kB1Bytes;
                    store_row16<false>(bx, 0, d, ch0, S);
                    store_row16<false>(bx + C::kB1M, 0, d, ch0, M);
                    fence_proxy_async();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (more) mbar_arrive(&bars->state[x]);
                    if (x == 1) mbar_arrive(&bars->empty[st]);
                }
            }
        }
        if (!*abort) {
#pragma unroll 1
            for (int x = 0; x < 2; ++x) {
                float S[kEpiCols], M[kEpiCols];
                tmem_ld16(st_s(x), S);
                tmem_ld16(st_m(x), M);
                tmem_ld_wait();
                const size_t off = (size_t)sh * D * D + st_row + 64 * x;
#pragma unroll
                for (int j = 0; j < kEpiCols; j += 4) {
                    if (p.S_T)
                        *reinterpret_cast<float4 *>(p.S_T + off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                    if (p.M_T)
                        *reinterpret_cast<float4 *>(p.M_T + off + j) = make_float4(M[j], M[j + 1], M[j + 2], M[j + 3]);
                }
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

// [T_total, H, D] bf16 viewed as a 3-D tensor (d, h, t); box 64 x 1 x box_t.
bool make_map(CUtensorMap *map, const void *base, int T_total, int H, int D, int box_t) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_t};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int NS, bool kChunkStates, bool kSplit>
cudaError_t launch_state_tc_t(const ChunkProblem &p, cudaStream_t st, const Maps &maps) {
    using C = Cfg<D, NS, kSplit>;
    // time segments (narrow slices of the plain forward only) are a separate
    // instantiation
    constexpr bool kSegOk = NS != 64 && !kChunkStates;
    if (is_segment(p) && !kSegOk) return cudaErrorInvalidValue;
    auto kern = (kSegOk && is_segment(p)) ? chunk_state_tc_kernel<D, NS, kChunkStates, kSplit, kSegOk>
                                          : chunk_state_tc_kernel<D, NS, kChunkStates, kSplit, false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)C::kSmemBytes);
    if (err != cudaSuccess) return err;
    if (is_segment(p)) {
        // the largest shared-memory carveout: the next segment's prep CTAs
        // fit beside this pass's CTAs
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
    }
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
    return cudaLaunchKernelEx(&cfg, kern, p, maps);
}

// Split operands at head size 128 leave no room for 64-column slices (their
// single stage and doubled operands exceed a CTA's shared memory): 32.
template <int D, bool kSplit>
constexpr int kWidestSlice = (kSplit && D == 128) ? 32 : 64;

template <bool kChunkStates>
cudaError_t launch_state_dual(const ChunkProblem &p, cudaStream_t st, const Maps &maps) {
    using C = DualCfg;
    auto kern = p.vres ? chunk_state_dual_kernel<kChunkStates, true>
                       : chunk_state_dual_kernel<kChunkStates, false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)C::kSmemBytes);
    if (err != cudaSuccess) return err;
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.maxThreadsPerBlock < C::kThreads) return cudaErrorLaunchOutOfResources;
    const long blocks = (long)p.n_seq * p.H;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
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
    return cudaLaunchKernelEx(&cfg, kern, p, maps);
}

// Slice width for a problem: 0 for both 64-column slices of a head in one
// CTA (bf16 at head size 128 with more 64-column slices than SMs), else the
// narrowest slices (16, 32 or 64 columns) whose CTAs fit on the GPU in one
// wave.
template <int D, bool kSplit>
int slice_width_d(const ChunkProblem &p) {
    const long chains = (long)p.n_seq * p.H;
    const int sms = device_sm_count();
    if (D == 128 && !kSplit && sms > 0 && chains * 2 > sms) return 0;
    return (sms > 0 && chains * (D / 16) <= sms) ? 16
           : ((sms > 0 && chains * (D / 32) <= sms) || kWidestSlice<D, kSplit> == 32) ? 32
                                                                                     : 64;
}

template <int D, bool kSplit>
cudaError_t launch_state_tc_d(const ChunkProblem &p, cudaStream_t st, const Maps &maps) {
    const int ns = slice_width_d<D, kSplit>(p);
    // both slices of a head in one CTA, their steps interleaved
    if constexpr (D == 128 && !kSplit) {
        if (ns == 0) {
            if (is_segment(p)) return cudaErrorInvalidValue;    // whole sequences only
            return p.S_chunks ? launch_state_dual<true>(p, st, maps) : launch_state_dual<false>(p, st, maps);
        }
    }
    if (p.S_chunks) {
        if (ns == 16) return launch_state_tc_t<D, 16, true, kSplit>(p, st, maps);
        if (ns == 32) return launch_state_tc_t<D, 32, true, kSplit>(p, st, maps);
        if constexpr (kWidestSlice<D, kSplit> == 64)
            return launch_state_tc_t<D, 64, true, kSplit>(p, st, maps);
        return cudaErrorInvalidConfiguration;
    }
    if (ns == 16) return launch_state_tc_t<D, 16, false, kSplit>(p, st, maps);
    if (ns == 32) return launch_state_tc_t<D, 32, false, kSplit>(p, st, maps);
    if constexpr (kWidestSlice<D, kSplit> == 64)
        return launch_state_tc_t<D, 64, false, kSplit>(p, st, maps);
    return cudaErrorInvalidConfiguration;
}

}  // namespace

int chunk_state_slice_width(const ChunkProblem &p) {
    const bool split = p.dtype == MDN_F32;
    if (p.D == 128) return split ? slice_width_d<128, true>(p) : slice_width_d<128, false>(p);
    return split ? slice_width_d<64, true>(p) : slice_width_d<64, false>(p);
}

// The slice width trades per-chunk latency (narrow slices: smaller MMAs and
// epilogues) against CTA count: the narrowest slices (16, 32 or 64 columns)
// whose CTAs still fit on the GPU in one wave.  bf16 inputs read q, k, v
// directly; fp32 inputs read their hi / lo bf16 parts.
cudaError_t launch_chunk_state_tc(const ChunkProblem &p, cudaStream_t st) {
    if (p.D != 64 && p.D != 128) return cudaErrorInvalidValue;
    const bool split = p.dtype == MDN_F32;
    if (split && !p.k_hi) return cudaErrorInvalidValue;
    if (p.prep_stride % 16 != 0) return cudaErrorInvalidValue;
    Maps maps;
    const int Tt = p.T_total > 0 ? p.T_total : 1;
    const void *k = split ? p.k_hi : p.k, *q = split ? p.q_hi : p.q;
    const void *v = split ? p.v_hi : p.v;
    if (!make_map(&maps.k, k, Tt, p.H, p.D, 16) || !make_map(&maps.q, q, Tt, p.H, p.D, 16) ||
        !make_map(&maps.v, v, Tt, p.H, p.D, 64))
        return cudaErrorInvalidValue;
    maps.k_lo = maps.k;
    maps.q_lo = maps.q;
    maps.v_lo = maps.v;
    if (split && (!make_map(&maps.k_lo, p.k_lo, Tt, p.H, p.D, 16) ||
                  !make_map(&maps.q_lo, p.q_lo, Tt, p.H, p.D, 16) ||
                  !make_map(&maps.v_lo, p.v_lo, Tt, p.H, p.D, 64)))
        return cudaErrorInvalidValue;
    maps.sc = maps.k;
    maps.mc = maps.k;
    if (p.S_chunks && !split) {
        const uint64_t blocks = (uint64_t)(p.max_chunks > 0 ? p.max_chunks : 1) * p.H;
        const uint64_t sdims[3] = {(uint64_t)p.D, (uint64_t)p.D, blocks};
        const uint64_t sstrides[2] = {(uint64_t)p.D * 2, (uint64_t)p.D * p.D * 2};
        const uint32_t sbox[3] = {64, (uint32_t)p.D, 1};
        if (!make_map_3d(&maps.sc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.S_chunks, sdims, sstrides, sbox) ||
            !make_map_3d(&maps.mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.M_chunks, sdims, sstrides, sbox))
            return cudaErrorInvalidValue;
    }
    if (p.D == 128)
        return split ? launch_state_tc_d<128, true>(p, st, maps)
                     : launch_state_tc_d<128, false>(p, st, maps);
    return split ? launch_state_tc_d<64, true>(p, st, maps)
                 : launch_state_tc_d<64, false>(p, st, maps);
}

}  // namespace mdn
