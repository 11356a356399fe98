// MDN chunkwise forward, the kernels around the tensor-core state pass that
// run mostly on the CUDA cores:
//
//   offsets  the chunk offsets and longest-first order of packed sequences,
//            with the device-side check of cu_seqlens;
//   prep     for fp32 inputs (one CTA per chunk and head, all chunks in
//            parallel): log-space prefix scans of alpha and mu, the
//            coefficient matrix Gamma, the Gram matrices K K^T and Q K^T on
//            the tensor cores (split operands: hi hi + hi lo + lo hi of the
//            bf16 parts, one fp32 accumulator), the unit-lower-triangular
//            system matrix, its inverse T and the intra-chunk output
//            operator A_O T in fp32 (an fp32-level error bound needs the
//            fp32 inverse), written as the hi / lo bf16 parts of the state
//            pass's operand [T; A_O T];
//   split    fp32 q, k, v as hi / lo bf16 parts for the state pass;
//   states   calls without tokens: final states = initial states.
//
// Equations: "MDN: Parallelizing Stepwise Momentum for Delta Linear
// Attention" slides, frames "Reorder the triangular sum ..." (Eqs. (7)-(9)),
// "Solve the unknown residuals with a lower triangular system" (Eqs.
// (15)-(18)), "Chunk outputs combine incoming states and local writes"
// (Appendix C Eqs. (40)-(42)), backup frames on the one-row shift and on the
// log-domain coefficients (Algorithm 1); reading notes sections 2.3-2.6.
#include <type_traits>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

constexpr int kThreads = 256;     // prep

// ------------------------------------------------------------- offsets

// off[s] = sum_{s' < s} ceil(len_{s'} / 64), s = 0..n_seq (one CTA), and
// order[] = the sequences sorted by decreasing length (ties by index): the
// rank of s counts the sequences that come before it.  Quadratic in n_seq,
// so beyond kMaxOrdered sequences the order is the identity.
//
// The offsets are checked first: cu[0] == 0, cu[s] <= cu[s + 1] and
// cu[n_seq] == T_total.  An offset array that breaks any of these would put
// chunk slots past the workspace and token rows past the tensors, so it is
// rejected on the device: MDN_ERR_INVALID_ARG goes to the status word, every
// chunk offset is written as 0 (every later kernel then finds no chunk to
// work on, and each state pass clamps its sequence to no tokens) and the
// order is the identity.
constexpr int kMaxOrdered = 4096;

__global__ void __launch_bounds__(1024)
chunk_offsets_kernel(const int32_t *cu, int n_seq, int T_total, int32_t *off, int32_t *order,
                     int *status) {
    int bad = 0;
    for (int s = threadIdx.x; s < n_seq; s += blockDim.x)
        bad |= cu[s] > cu[s + 1];
    if (threadIdx.x == 0) bad |= (cu[0] != 0) || (cu[n_seq] != T_total);
    if (__syncthreads_or(bad)) {
        for (int s = threadIdx.x; s <= n_seq; s += blockDim.x) {
            off[s] = 0;
            if (order && s < n_seq) order[s] = s;
        }
        if (threadIdx.x == 0 && status) atomicExch(status, (int)MDN_ERR_INVALID_ARG);
        return;
    }
    if (order) {
        for (int s = threadIdx.x; s < n_seq; s += blockDim.x) {
            int rank = s;
            if (n_seq <= kMaxOrdered) {
                const int ls = cu[s + 1] - cu[s];
                rank = 0;
                for (int t = 0; t < n_seq; ++t) {
                    const int lt = cu[t + 1] - cu[t];
                    rank += (lt > ls) || (lt == ls && t < s);
                }
            }
            order[rank] = s;
        }
    }
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = 0; base < n_seq; base += 1024) {
        const int s = base + threadIdx.x;
        int32_t x = 0;
        if (s < n_seq) x = (cu[s + 1] - cu[s] + kChunk - 1) / kChunk;
        int32_t incl = x;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int32_t wbase = 0;
        for (int w = 0; w < warp; ++w) wbase += warp_tot[w];
        const int32_t c0 = carry;
        if (s < n_seq) off[s] = c0 + wbase + incl - x;
        __syncthreads();
        if (threadIdx.x == 1023) carry = c0 + wbase + incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) off[n_seq] = carry;
}

// ---------------------------------------------------------------- prep
//
// Tile copies are fully unrolled loops (constant trip counts), so that every
// thread issues all of its loads of a tile before the first shared-memory
// store instead of one load round trip per iteration.

template <int D>
struct PrepSmem {
    static constexpr int LM = kChunk + 1;     // padded row stride of 64x64
    static constexpr int kHalves = D / 64;
    // The hi and lo [K; Q] tiles (bf16, 128 rows - the keys, then the
    // queries - x 64 columns per 16 KiB half, 128-byte swizzled) are read
    // only by the Gram products; L, T and A_O (fp32) take their place
    // afterwards, so that two (d = 128) or three (d = 64) CTAs share an SM.
    static constexpr size_t kTiles = 2 * kHalves * 16384;
    static constexpr size_t kLTA = sizeof(float) * 3 * kChunk * LM;
    static constexpr size_t kShared = ((kTiles > kLTA ? kTiles : kLTA) + 1023) / 1024 * 1024;
    static constexpr int kFloats = kChunk * LM + 12 * kChunk + 64;   // Gamma, vectors, exchange
    static constexpr size_t kOffBar = kShared + sizeof(float) * kFloats;
    static constexpr size_t kBytes = kOffBar + 64 + 1024;            // + barriers, alignment
};

struct PrepBars {
    uint64_t tma, gram;
    uint32_t tmem_base;
    int abort, issued;
};

constexpr uint32_t kTmemColsPS = 64;
constexpr uint32_t kIdescGramS = sm100::idesc_bf16(128, 64, false, false);

// Inclusive sum over the 64 lanes of warps 0 and 1.  Every thread of the
// block must call it (it synchronises the block).
__device__ __forceinline__ float scan64(float x, float *xch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (warp == 0 && lane == 31) *xch = x;
    __syncthreads();
    if (warp == 1) x += *xch;
    __syncthreads();
    return x;
}

// Inclusive composition of the affine maps x -> a x + c over the 64 lanes of
// warps 0 and 1 (token order); returns the composed map's c, i.e. the value
// of the recurrence x_i = a_i x_{i-1} + c_i started from x = 0.  Every thread
// of the block must call it (it synchronises the block).
__device__ __forceinline__ float scan64_affine(float a, float c, float *xch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float pa = __shfl_up_sync(0xffffffffu, a, d);
        const float pc = __shfl_up_sync(0xffffffffu, c, d);
        if (lane >= d) {
            c = a * pc + c;
            a = a * pa;
        }
    }
    if (warp == 0 && lane == 31) *xch = c;
    __syncthreads();
    if (warp == 1) c = a * *xch + c;
    __syncthreads();
    return c;
}

template <int D>
__global__ void __launch_bounds__(kThreads)
chunk_prep_split_kernel(ChunkProblem p, const __grid_constant__ CUtensorMap map_khi,
                        const __grid_constant__ CUtensorMap map_qhi,
                        const __grid_constant__ CUtensorMap map_klo,
                        const __grid_constant__ CUtensorMap map_qlo) {
    using SM = PrepSmem<D>;
    using namespace sm100;
    constexpr int LM = SM::LM;
    int gc, h;
    chunk_head_of_block(p.H, gc, h);
    ChunkLoc loc;
    if (!locate_chunk_cta(p, gc, loc)) return;
    const int n = loc.n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = align_smem_1024(smem_raw);
    float *L = reinterpret_cast<float *>(base);      // system matrix (strict lower), after the Grams
    float *Tm = L + kChunk * LM;           // its inverse
    float *AO = Tm + kChunk * LM;          // output operator (lower)
    float *G = reinterpret_cast<float *>(base + SM::kShared);   // Gamma [64][LM]
    float *va = G + kChunk * LM;           // alpha
    float *vb = va + kChunk;               // beta
    float *ve = vb + kChunk;               // eta
    float *vA = ve + kChunk;               // A_i = sum log alpha
    float *vU = vA + kChunk;               // U'_i = sum of finite log mu
    float *vZ = vU + kChunk;               // number of zero mu so far
    float *vbb = vZ + kChunk;              // b_i
    float *vm = vbb + kChunk;              // mu
    float *vgs = vm + kChunk;              // gamma_{n,j} (Gamma's last row, kept for the carry)
    float *xch = vgs + kChunk;             // scan exchange
    PrepBars *bars = reinterpret_cast<PrepBars *>(base + SM::kOffBar);
    volatile int *abort = &bars->abort;

    if (tid == 0) {
        mbar_init(&bars->tma, 1);
        mbar_init(&bars->gram, 1);
        bars->abort = 0;
        bars->issued = 0;
        fence_mbar_init();
        // the hi and lo parts of the chunk's keys (rows 0..63) and queries
        // (rows 64..127); their latency hides behind the scans and Gamma
        mbar_arrive_expect_tx(&bars->tma, (uint32_t)SM::kTiles);
#pragma unroll
        for (int hh = 0; hh < SM::kHalves; ++hh) {
            unsigned char *hi = base + hh * 16384, *lo = base + (SM::kHalves + hh) * 16384;
            tma_load_3d(hi, &map_khi, &bars->tma, 64 * hh, h, loc.t0);
            tma_load_3d(hi + 8192, &map_qhi, &bars->tma, 64 * hh, h, loc.t0);
            tma_load_3d(lo, &map_klo, &bars->tma, 64 * hh, h, loc.t0);
            tma_load_3d(lo + 8192, &map_qlo, &bars->tma, 64 * hh, h, loc.t0);
        }
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemColsPS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // ---- gates and log-space prefix scans (lanes 0..63 = tokens)
    float a = 1.f, mu = 0.f, be = 0.f, et = 0.f;
    if (tid < kChunk && tid < n) {
        const size_t gi = (size_t)(loc.t0 + tid) * p.H + h;
        a = p.alpha[gi];
        mu = p.mu[gi];
        et = p.eta[gi];
        be = p.beta ? p.beta[gi] : 1.f;
    }
    const bool zero_mu = (mu == 0.f);
    const float A = scan64(tid < kChunk ? logf(a) : 0.f, xch);
    const float U = scan64(tid < kChunk && !zero_mu ? logf(mu) : 0.f, xch);
    const float Z = scan64(tid < kChunk && zero_mu ? 1.f : 0.f, xch);
    // b_i = alpha_i b_{i-1} + beta_i mubar_i  (mubar_i = exp(U_i) without a zero mu)
    const float bsum = scan64_affine(tid < kChunk ? a : 1.f,
                                     (tid < kChunk && Z == 0.f) ? be * expf(U) : 0.f, xch);
    if (tid < kChunk) {
        va[tid] = a;
        vb[tid] = be;
        ve[tid] = et;
        vA[tid] = A;
        vU[tid] = U;
        vZ[tid] = Z;
        vbb[tid] = bsum;
        vm[tid] = mu;
    }
    __syncthreads();

    // ---- Gamma, column j per lane: gamma_{j,j} = beta_j and
    //      gamma_{i,j} = alpha_i gamma_{i-1,j} + beta_i m_{i,j} with the mu
    //      product m_{i,j} = prod_{u=j+1}^{i} mu_u carried as m <- mu_i m
    //      (exact for mu = 0, no exponential per entry)
    if (tid < kChunk) {
        const int j = tid;
        float g = vb[j], m = 1.f;
        for (int i = 0; i < j; ++i) G[i * LM + j] = 0.f;
        G[j * LM + j] = g;
        for (int i = j + 1; i < kChunk; ++i) {
            m *= vm[i];
            g = va[i] * g + vb[i] * m;
            G[i * LM + j] = g;
        }
        vgs[j] = (j < n) ? G[(n - 1) * LM + j] : 0.f;
    }
    __syncthreads();

    // ---- the Gram products [K; Q] K^T on the tensor cores, split operands:
    //      hi hi^T + hi lo^T + lo hi^T into one fp32 accumulator (M = 128: the
    //      key rows, then the query rows; N = 64: the tile's first 64 rows)
    if (tid == 32) {
        if (mbar_wait(&bars->tma, 0, abort)) {
            tc_fence_after();
            const uint32_t hi = smem_u32(base), lo = hi + SM::kHalves * 16384;
            const uint32_t as[3] = {hi, hi, lo}, bs[3] = {hi, lo, hi};
#pragma unroll
            for (int pr = 0; pr < 3; ++pr)
#pragma unroll
                for (int kb = 0; kb < SM::kHalves; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t off = kb * 16384 + kk * 32;
                        mma_bf16(tmem, sdesc_sw128(as[pr] + off, 16, 1024),
                                 sdesc_sw128(bs[pr] + off, 16, 1024), kIdescGramS,
                                 (pr | kb | kk) != 0);
                    }
            mma_commit(&bars->gram);
            bars->issued = 1;
        } else {
            int dummy = 0;               // the copy must land before the CTA exits
            mbar_wait(&bars->tma, 0, &dummy);
        }
    }
    {
        // the Gram rows -> L = (P Khat^T) . Gamma_shifted (key rows) and
        // A_O = (Q Khat^T) . Gamma (query rows), masked past the chunk end;
        // they overwrite the tiles, which the finished MMAs no longer read
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->gram, 0, abort));
        const int q = warp & 3, half = warp >> 2, row = 32 * q + lane;
        if (ok) {
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + half * 32, x);
            tmem_ld_wait();
            if (row < kChunk) {
                const int i = row;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    // alpha_i (k_i.k_j) eta_j gamma_{i-1,j}, j < i
                    L[i * LM + j] = (j < i && i < n) ? va[i] * x[jj] * ve[j] * G[(i - 1) * LM + j] : 0.f;
                }
            } else {
                const int i = row - kChunk;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    // (q_i.k_j) eta_j gamma_{i,j}, j <= i
                    AO[i * LM + j] = (j <= i && i < n) ? x[jj] * ve[j] * G[i * LM + j] : 0.f;
                }
            }
        }
        for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
            const int i = idx >> 6, j = idx & 63;
            Tm[i * LM + j] = (i == j) ? 1.f : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && bars->issued) {
            int dummy = 0;               // no MMA in flight when TMEM is freed
            mbar_wait(&bars->gram, 0, &dummy);
        }
        __syncwarp();
        tmem_dealloc(tmem, kTmemColsPS);
    }

    // ---- T = (I + L)^{-1}, blocked: diagonal 16x16 blocks by forward
    //      substitution in registers (one lane per column), then
    //      [[A, 0], [C, B]]^{-1} = [[A^-1, 0], [-B^-1 C A^-1, B^-1]] for the
    //      16-blocks inside each 32-block and for the two 32-blocks.  T holds
    //      the identity from the step above, so everything above the
    //      diagonal blocks stays zero.
    {
        const int warp = tid >> 5, lane = tid & 31;
        float *X = G;                      // scratch: Gamma is consumed
        constexpr int LX = 33;
        if (warp < 2) {
            const int blk = warp * 2 + (lane >> 4);
            const int c = lane & 15;
            const int base = blk * 16;
            float t[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < r; ++k) acc += L[(base + r) * LM + base + k] * t[k];
                t[r] = (r < c) ? 0.f : ((r == c) ? 1.f : -acc);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tm[(base + r) * LM + base + c] = t[r];
        }
        __syncthreads();
        // 16-blocks below the diagonal inside each 32-block (two of them);
        // each thread computes two adjacent outputs of one row
        {
            const int pb = tid >> 7, i = (tid >> 3) & 15, j = (tid & 7) * 2;
            const int r0 = 32 * pb + 16, c0 = 32 * pb;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float l = L[(r0 + i) * LM + c0 + k];
                const float *t = Tm + (c0 + k) * LM + c0 + j;
                a0 += l * t[0];
                a1 += l * t[1];
            }
            X[(pb * 16 + i) * LX + j] = a0;
            X[(pb * 16 + i) * LX + j + 1] = a1;
        }
        __syncthreads();
        {
            const int pb = tid >> 7, i = (tid >> 3) & 15, j = (tid & 7) * 2;
            const int r0 = 32 * pb + 16, c0 = 32 * pb;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float t = Tm[(r0 + i) * LM + r0 + k];
                a0 += t * X[(pb * 16 + k) * LX + j];
                a1 += t * X[(pb * 16 + k) * LX + j + 1];
            }
            Tm[(r0 + i) * LM + c0 + j] = -a0;
            Tm[(r0 + i) * LM + c0 + j + 1] = -a1;
        }
        __syncthreads();
        // the 32-block below the diagonal: -T_B (L_C T_A).  X = L_C T_A: warp
        // w owns columns [4w, 4w+4) of all 32 rows; k runs over T_A's nonzero
        // rows k >= 4w only
        {
            const int i = lane, j0 = warp * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = j0; k < 32; ++k) {
                const float l = L[(32 + i) * LM + k];
                const float *t = Tm + k * LM + j0;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] += l * t[e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) X[i * LX + j0 + e] = acc[e];
        }
        __syncthreads();
        // T_C = -T_B X: warp w owns rows [4w, 4w+4), lane = column; k runs
        // over T_B's nonzero columns k <= 4w+3 only
        {
            const int i0 = warp * 4, j = lane;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < i0 + 4; ++k) {
                const float x = X[k * LX + j];
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] += Tm[(32 + i0 + e) * LM + 32 + k] * x;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) Tm[(32 + i0 + e) * LM + j] = -acc[e];
        }
        __syncthreads();
    }

    // ---- write the prepared block: row-major fp32 T and A_O T, or, when the
    //      tensor-core state pass takes fp32 inputs (split operands), the
    //      operand [T; A_O T] of its second product as hi / lo bf16 parts in
    //      the 128-byte-swizzled layout, rows interleaved by tc_row
    unsigned char *blk = p.prep + ((size_t)gc * p.H + h) * p.prep_stride;
    float *vec = reinterpret_cast<float *>(blk + PrepLayoutTC::kSplitVec);
    auto put4 = [&](int op_row, int col4, const float *x) {
        // four consecutive columns col4..col4+3 = half of a 16-byte chunk
        float r[4];
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = x[e] - __bfloat162float(__float2bfloat16_rn(x[e]));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            __nv_bfloat162 a = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
            __nv_bfloat162 b = __floats2bfloat162_rn(r[2 * e], r[2 * e + 1]);
            hi[e] = *reinterpret_cast<uint32_t *>(&a);
            lo[e] = *reinterpret_cast<uint32_t *>(&b);
        }
        const uint32_t off = sm100::sw128_offset((uint32_t)op_row, (uint32_t)(col4 >> 3)) +
                             (uint32_t)(col4 & 4) * 2;
        *reinterpret_cast<uint2 *>(blk + off) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2 *>(blk + PrepLayoutTC::kSplitLo + off) = make_uint2(lo[0], lo[1]);
    };
    {
        const int ti = tid >> 4, tj = tid & 15;
        float acc[4][4] = {};
        for (int k = 0; k < kChunk; ++k) {
            float ar[4], tc[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                ar[r] = AO[(4 * ti + r) * LM + k];
                tc[r] = Tm[k * LM + 4 * tj + r];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] += ar[r] * tc[c];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * ti + r;
            const float t4[4] = {Tm[i * LM + 4 * tj], Tm[i * LM + 4 * tj + 1],
                                 Tm[i * LM + 4 * tj + 2], Tm[i * LM + 4 * tj + 3]};
            put4(tc_row(i), 4 * tj, t4);
            put4(tc_row(kChunk + i), 4 * tj, acc[r]);
        }
    }
    if (tid < kChunk) {
        const int i = tid;
        const bool valid = i < n;
        const int last = n - 1;
        const float abar = expf(vA[i]);
        vec[kVecAbar * kChunk + i] = valid ? abar : 0.f;
        vec[kVecBmA * kChunk + i] = (valid && i > 0) ? vbb[i - 1] * va[i] : 0.f;
        vec[kVecB * kChunk + i] = valid ? vbb[i] : 0.f;
        vec[kVecGS * kChunk + i] = valid ? vgs[i] * ve[i] : 0.f;
        const float mtail = (vZ[last] == vZ[i]) ? expf(vU[last] - vU[i]) : 0.f;
        vec[kVecGM * kChunk + i] = valid ? mtail * ve[i] : 0.f;
        float sc = 0.f;
        if (i == 0) sc = expf(vA[last]);
        if (i == 1) sc = vbb[last];
        if (i == 2) sc = (vZ[last] == 0.f) ? expf(vU[last]) : 0.f;
        if (i == 3) sc = (float)n;
        vec[kVecScal * kChunk + i] = sc;
    }
    if (tid == 0 && *abort && p.status) atomicExch(p.status, (int)MDN_ERR_DEVICE_TIMEOUT);
}

// ----------------------------------------------------- no-token calls

// With no tokens every sequence is empty: its final states are its initial
// states (zero when absent).  One thread per state element.
__global__ void __launch_bounds__(256)
states_passthrough_kernel(const float *S0, const float *M0, float *S_T, float *M_T, long n) {
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += stride) {
        if (S_T) S_T[i] = S0 ? S0[i] : 0.f;
        if (M_T) M_T[i] = M0 ? M0[i] : 0.f;
    }
}

template <int D>
cudaError_t launch_prep_t(const ChunkProblem &p, cudaStream_t st) {
    if (p.max_chunks == 0) return cudaSuccess;
    CUtensorMap mkh, mqh, mkl, mql;
    if (!make_token_map_bf16(&mkh, p.k_hi, p.T_total, p.H, D, 64) ||
        !make_token_map_bf16(&mqh, p.q_hi, p.T_total, p.H, D, 64) ||
        !make_token_map_bf16(&mkl, p.k_lo, p.T_total, p.H, D, 64) ||
        !make_token_map_bf16(&mql, p.q_lo, p.T_total, p.H, D, 64))
        return cudaErrorInvalidValue;
    auto kp = chunk_prep_split_kernel<D>;
    cudaError_t err = cudaFuncSetAttribute(
        kp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PrepSmem<D>::kBytes);
    if (err != cudaSuccess) return err;
    dim3 grid;
    if (!chunk_head_grid(p.max_chunks, p.H, grid)) return cudaErrorInvalidConfiguration;
    kp<<<grid, kThreads, PrepSmem<D>::kBytes, st>>>(p, mkh, mqh, mkl, mql);
    return cudaGetLastError();
}

// fp32 q, k, v -> their hi / lo bf16 parts (hi = bf16(x), lo = bf16(x - hi)),
// four elements per thread and tensor.
__global__ void __launch_bounds__(256)
split_inputs_kernel(const float4 *q, const float4 *k, const float4 *v, long n4, uint2 *q_hi,
                    uint2 *q_lo, uint2 *k_hi, uint2 *k_lo, uint2 *v_hi, uint2 *v_lo) {
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 *src[3] = {q, k, v};
        uint2 *hi[3] = {q_hi, k_hi, v_hi}, *lo[3] = {q_lo, k_lo, v_lo};
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const float4 x = src[t][i];
            const __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x, x.y);
            const __nv_bfloat162 h1 = __floats2bfloat162_rn(x.z, x.w);
            const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
            const __nv_bfloat162 l0 = __floats2bfloat162_rn(x.x - f0.x, x.y - f0.y);
            const __nv_bfloat162 l1 = __floats2bfloat162_rn(x.z - f1.x, x.w - f1.y);
            hi[t][i] = make_uint2(*reinterpret_cast<const uint32_t *>(&h0),
                                  *reinterpret_cast<const uint32_t *>(&h1));
            lo[t][i] = make_uint2(*reinterpret_cast<const uint32_t *>(&l0),
                                  *reinterpret_cast<const uint32_t *>(&l1));
        }
    }
}

}  // namespace

cudaError_t launch_split_inputs(const ChunkProblem &p, cudaStream_t st) {
    const long n4 = (long)p.T_total * p.H * p.D / 4;
    if (n4 == 0) return cudaSuccess;
    const int blocks = (int)((n4 + 255) / 256 < 152L * 8 ? (n4 + 255) / 256 : 152L * 8);
    split_inputs_kernel<<<blocks, 256, 0, st>>>(
        static_cast<const float4 *>(p.q), static_cast<const float4 *>(p.k),
        static_cast<const float4 *>(p.v), n4, static_cast<uint2 *>(p.q_hi),
        static_cast<uint2 *>(p.q_lo), static_cast<uint2 *>(p.k_hi), static_cast<uint2 *>(p.k_lo),
        static_cast<uint2 *>(p.v_hi), static_cast<uint2 *>(p.v_lo));
    return cudaGetLastError();
}

cudaError_t launch_chunk_offsets(const ChunkProblem &p, cudaStream_t st) {
    chunk_offsets_kernel<<<1, 1024, 0, st>>>(p.cu_seqlens, p.n_seq, p.T_total,
                                              p.chunk_offsets, p.seq_order, p.status);
    return cudaGetLastError();
}

// fp32 inputs, after their hi / lo parts are written (launch_split_inputs).
cudaError_t launch_chunk_prep_simt(const ChunkProblem &p, cudaStream_t st) {
    if (p.dtype != MDN_F32 || (p.D != 64 && p.D != 128)) return cudaErrorInvalidValue;
    if (p.max_chunks == 0) return cudaSuccess;
    if (!p.k_hi || !p.q_hi || !p.k_lo || !p.q_lo) return cudaErrorInvalidValue;
    return p.D == 128 ? launch_prep_t<128>(p, st) : launch_prep_t<64>(p, st);
}

cudaError_t launch_states_passthrough(const ChunkProblem &p, cudaStream_t st) {
    const long n = (long)p.n_seq * p.H * p.D * p.D;
    if (n == 0 || (!p.S_T && !p.M_T)) return cudaSuccess;
    const int blocks = (int)((n + 255) / 256 < 152L * 8 ? (n + 255) / 256 : 152L * 8);
    states_passthrough_kernel<<<blocks, 256, 0, st>>>(p.S0, p.M0, p.S_T, p.M_T, n);
    return cudaGetLastError();
}

}  // namespace mdn
