// MDN chunkwise forward — chunk-local preparation on the tensor cores
// (bf16 inputs, head size 64 or 128).  One CTA per (chunk, head); all chunks
// of all sequences in parallel.  The gradient pass runs it too, for the same
// T and A_O T.
//
// Per chunk of n <= 64 tokens ("MDN: Parallelizing Stepwise Momentum for
// Delta Linear Attention" slides, frames "Reorder the triangular sum ..."
// (Eqs. (7)-(9)), "Solve the unknown residuals with a lower triangular
// system" (Eqs. (15)-(18)), "Chunk outputs combine incoming states and local
// writes", backup frames on the row shift and the log-domain coefficients;
// reading notes 2.3-2.6):
//
//   A_i = sum_{r<=i} log alpha_r, U_i = sum_{r<=i, mu_r>0} log mu_r,
//   Z_i = #{r <= i : mu_r = 0}                       (warp-shuffle prefix scans)
//   Gt = Gamma Diag(eta): on the four diagonal 16-blocks by the column
//   recurrence
//       m_{j,j} = eta_j,           m_{i,j} = mu_i m_{i-1,j}  (= eta_j prod_{u=j+1}^{i} mu_u)
//       Gt_{j,j} = beta_j eta_j,   Gt_{i,j} = alpha_i Gt_{i-1,j} + beta_i m_{i,j},
//   left of them (rows of segment s starting at r0, columns j < r0) by the
//   exact split of that sum at r0
//       Gt_{r,j} = F_s(r) Gt_{r0-1,j} + c_j^(s) lambda_s(r),
//       F_s(r) = prod_{u=r0}^{r} alpha_u,  c_j^(s) = eta_j prod_{u=j+1}^{r0-1} mu_u,
//       lambda_s(r) = alpha_r lambda_s(r-1) + beta_r prod_{u=r0}^{r} mu_u;
//   no exponential per entry, no difference of prefix sums, so mu = 0 is
//   exact and nothing cancels
//   b_i = alpha_i b_{i-1} + beta_i mubar_i, F_s and lambda_s: one segmented
//     prefix scan (one token per lane) of the maps (b, mubar) -> (alpha b +
//     beta mu mubar, mu mubar), beside the log-space scans
//   MMA   G = [K; Q] K^T                                 (M=128, N=64, K=128)
//   L_{i,j}   = alpha_i G_K[i,j] Gt_{i-1,j}     (j < i: the row-shifted Gamma)
//   A_O[i,j]  = G_Q[i,j] Gt_{i,j}               (j <= i)
//   T = (I + L)^{-1} = D - N D + N^2 D - N^3 D with D the inverses of L's
//   diagonal 16-blocks (forward substitution, fp32) and N = D L_o (L_o: L
//   off those blocks, so N^4 = 0): three MMAs (M=64)
//   MMA   A_O T                                          (M=128, N=64, K=64)
//
// and writes the prepared block: T and A_O T in bf16 in the 128-byte-swizzled
// K-major operand layout of the state pass (rows interleaved by tc_row), then
// the fp32 carry vectors.  Rows and columns past the chunk end are masked (T
// is the identity there and every vector entry is zero).
#include <cudaTypedefs.h>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

using namespace sm100;

constexpr int kThreadsP = 256;
constexpr int LM = kChunk + 1;                 // padded fp32 row stride

// shared memory (bytes from the 1024-aligned base), under 56 KiB so that four
// CTAs share an SM.  Regions are reused once their last reader is done:
//   [0, 32768)       K/Q tiles (TMA), read by the Gram MMA only; then
//   [0, 8192)        L_o bf16 (off-diagonal 16-blocks of L, row-major); after
//                    the first hop of the inverse, bf16 T (row-major)
//   [8192, 16384)    Y bf16 (I - N, then the Horner iterates)
//   [16384, 20736)   diagonal 16-blocks of L fp32 [4][16][17], then D in place
//   [24576, 32768)   A_O bf16, K-major A operand (rows 0..63; the MMA's rows
//                    64..127 read the next region and are never used)
//   [32768, 49408)   Gt fp32 [64][65], computed while the copy and the Gram
//                    MMA are in flight; after L is built, D bf16 [32768,
//                    40960) and N bf16 [40960, 49152)
//   [49408, 50432)   (alpha, beta, mu, eta) per token
//   [50432, 53504)   per-token vectors (12 rows of 64 fp32)
constexpr int LB = 17;                         // padded row stride of a 16 x 16 block
constexpr uint32_t kOffKQ = 0;
constexpr uint32_t kOffLo = 0;
constexpr uint32_t kOffB2 = 0;
constexpr uint32_t kOffY = 8192;
constexpr uint32_t kOffLd = 16384;
constexpr uint32_t kOffAO = 24576;
constexpr uint32_t kOffG = 32768;
constexpr uint32_t kOffDbf = 32768;
constexpr uint32_t kOffN = 40960;
constexpr uint32_t kOffGate = 49408;
constexpr uint32_t kOffVec = 50432;
constexpr uint32_t kOffBarP = 53504;
constexpr uint32_t kSmemP = kOffBarP + 128 + 1024;
static_assert(kOffLd + 4 * 64 * LB <= kOffAO && kOffAO + 8192 <= kOffG, "prep layout");
static_assert(kOffG + 4 * 64 * LM <= kOffGate && kOffN + 8192 <= kOffGate, "prep layout");
static_assert(kOffGate + 16 * 64 <= kOffVec && kOffVec + 12 * 4 * 64 <= kOffBarP, "prep layout");
static_assert(kSmemP <= 57344, "four CTAs per SM");

constexpr uint32_t kTmemColsP = 128;
constexpr uint32_t kColG = 0;                  // Gram accumulator, 64 columns
constexpr uint32_t kColD2 = 64;                // A_O T accumulator, 64 columns

constexpr uint32_t kIdescGram = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescOut = idesc_bf16(128, 64, false, true);
constexpr uint32_t kIdescHop = idesc_bf16(64, 64, false, true);    // the inverse's products
constexpr uint32_t kIdescHop2 = idesc_bf16(64, 128, false, true);  // ... with two B blocks

struct BarsP {
    uint64_t tma, gram, hop, out, drain;
    uint32_t tmem_base;
    int abort;
};

// rows of the per-token vector block: prefix sums of log alpha / log mu,
// zero-mu counts, alpha products from each 16-row segment start, b, the
// scans' exchange slot, the segments' lambda, and the three segments' column
// factors
enum { vA = 0, vU, vZ, vF, vB, vScan, vLam, vC };   // vC .. vC + 2: one row per segment

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// One token per lane over lanes 0..63 (warps 0 and 1, named barrier 1):
// inclusive prefix sums of log alpha, log mu and the zero-mu count, and the
// prefix products of the per-token maps (b, mubar) -> (alpha b + beta mu
// mubar, mu mubar), i.e. upper-triangular 2 x 2 matrices [[a, c], [0, e]] =
// [[alpha, beta mu], [0, mu]] composed later-times-earlier.  The matrix
// products are taken within each segment of 16 tokens first (returned in
// (fa, fc): for a token r of segment s they are F_s(r) = prod_{u=r0}^{r}
// alpha_u and lambda_s(r)), then across segments; from the start (b_0 = 0,
// mubar_0 = 1) the chunk-wide product's c entry is b_r.
__device__ __forceinline__ void scan64_gates(float &A, float &U, float &Z, float &ta, float &tc,
                                             float &te, float &fa, float &fc, float *xch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 16; d <<= 1) {
        const float pA = __shfl_up_sync(0xffffffffu, A, d);
        const float pU = __shfl_up_sync(0xffffffffu, U, d);
        const float pZ = __shfl_up_sync(0xffffffffu, Z, d);
        const float pa = __shfl_up_sync(0xffffffffu, ta, d);
        const float pc = __shfl_up_sync(0xffffffffu, tc, d);
        const float pe = __shfl_up_sync(0xffffffffu, te, d);
        if ((lane & 15) >= d) {
            A += pA;
            U += pU;
            Z += pZ;
            tc = fmaf(ta, pc, tc * pe);
            ta *= pa;
            te *= pe;
        }
    }
    fa = ta;
    fc = tc;
    // the second segment of each warp joins the first
    {
        const float qA = __shfl_sync(0xffffffffu, A, 15);
        const float qU = __shfl_sync(0xffffffffu, U, 15);
        const float qZ = __shfl_sync(0xffffffffu, Z, 15);
        const float qa = __shfl_sync(0xffffffffu, ta, 15);
        const float qc = __shfl_sync(0xffffffffu, tc, 15);
        const float qe = __shfl_sync(0xffffffffu, te, 15);
        if (lane >= 16) {
            A += qA;
            U += qU;
            Z += qZ;
            tc = fmaf(ta, qc, tc * qe);
            ta *= qa;
            te *= qe;
        }
    }
    // warp 1 joins warp 0's total
    if (warp == 0 && lane == 31) {
        xch[0] = A; xch[1] = U; xch[2] = Z;
        xch[3] = ta; xch[4] = tc; xch[5] = te;
    }
    asm volatile("bar.sync 1, 64;" ::: "memory");
    if (warp == 1) {
        A += xch[0];
        U += xch[1];
        Z += xch[2];
        tc = fmaf(ta, xch[4], tc * xch[5]);
        ta *= xch[3];
        te *= xch[5];
    }
}

template <int D, bool kSeg>
__global__ void __launch_bounds__(kThreadsP, 4)
chunk_prep_tc_kernel(const ChunkProblem p, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_q) {
    constexpr int kHalves = D / 64;           // 64-wide d_k halves of the K and Q tiles
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem_1024(smem_raw);
    BarsP *bars = reinterpret_cast<BarsP *>(smem + kOffBarP);
    volatile int *abort = &bars->abort;
    float4 *gate = reinterpret_cast<float4 *>(smem + kOffGate);   // (alpha, beta, mu, eta)
    float *vec = reinterpret_cast<float *>(smem + kOffVec);
    float *Gt = reinterpret_cast<float *>(smem + kOffG);
    float *Ldg = reinterpret_cast<float *>(smem + kOffLd);     // [4][16][LB]
    unsigned char *Lo = smem + kOffLo;
    unsigned char *Ybf = smem + kOffY;
    unsigned char *Dbf = smem + kOffDbf;
    unsigned char *Nbf = smem + kOffN;
    unsigned char *AO = smem + kOffAO;
    unsigned char *B2 = smem + kOffB2;

    // The state pass may be scheduled as soon as every CTA of this grid has
    // started; it waits for this grid's completion before it reads a
    // prepared block.  The prep of a later time segment, which runs beside
    // the previous segment's state pass, lets no dependent start early, and
    // its last CTA outlives that state pass (SegMode).
    const bool follower = kSeg && (p.seg_mode & kSegPrepFollower) != 0;
    const bool last_cta = blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1;
    if (!follower) grid_launch_dependents();
    int gc = blockIdx.x;
    if constexpr (kSeg) {
        // the segment's chunks of every sequence (equal lengths), sequence-major
        const int len = p.seg_c1 - p.seg_c0, cps = (p.T + kChunk - 1) / kChunk;
        const int s = blockIdx.x / len;
        gc = s * cps + p.seg_c0 + (blockIdx.x - s * len);
    }
    const int h = blockIdx.y;
    ChunkLoc loc;
    if (!locate_chunk_cta(p, gc, loc)) {
        if constexpr (kSeg)
            if (follower && last_cta && threadIdx.x == 0) grid_dependency_wait();
        return;
    }
    const int n = loc.n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char *pblk = p.prep + ((size_t)gc * p.H + h) * p.prep_stride;
    float *gv = reinterpret_cast<float *>(pblk + PrepLayoutTC::kOffVec);
    // gates first: their latency overlaps the setup below (past the chunk
    // end alpha = 1 and beta = mu = eta = 0)
    float g_a = 1.f, g_mu = 0.f, g_be = 0.f, g_et = 0.f;
    if (tid < n) {
        const size_t gi = (size_t)(loc.t0 + tid) * p.H + h;
        g_a = p.alpha[gi];
        g_mu = p.mu[gi];
        g_et = p.eta[gi];
        g_be = p.beta ? p.beta[gi] : 1.f;
    }

    if (tid == 0) {
        mbar_init(&bars->tma, 1);
        mbar_init(&bars->gram, 1);
        mbar_init(&bars->hop, 1);
        mbar_init(&bars->out, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        // K and Q tiles: their latency gates only the Gram MMA
        mbar_arrive_expect_tx(&bars->tma, 16384 * kHalves);
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
            tma_load_3d(smem + kOffKQ + hh * 16384, &map_k, &bars->tma, 64 * hh, h, loc.t0);
            tma_load_3d(smem + kOffKQ + hh * 16384 + 8192, &map_q, &bars->tma, 64 * hh, h, loc.t0);
        }
    }
    if (warp == 2) {
        tmem_alloc(&bars->tmem_base, kTmemColsP);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // ---- gates, their log-space prefix scans, b and the segments' F and
    //      lambda (warps 0, 1)
    if (warp < 2) {
        const int i = tid;
        const bool zmu = (g_mu == 0.f);
        float A = logf(g_a), U = zmu ? 0.f : logf(g_mu), Z = zmu ? 1.f : 0.f;
        float ta = g_a, tc = g_be * g_mu, te = g_mu, fa, fc;
        scan64_gates(A, U, Z, ta, tc, te, fa, fc, vec + vScan * kChunk);
        gate[i] = make_float4(g_a, g_be, g_mu, g_et);
        vec[vA * kChunk + i] = A;
        vec[vU * kChunk + i] = U;
        vec[vZ * kChunk + i] = Z;
        vec[vB * kChunk + i] = tc;
        vec[vF * kChunk + i] = fa;
        vec[vLam * kChunk + i] = fc;
    }
    __syncthreads();

    if (warp == 1) {
        // ---- the Gram MMA: this warp waits for the K/Q tiles alone and joins
        //      the other warps again at the block barrier before L is built,
        //      so the copy's latency hides behind everything up to there
        __syncwarp();
        if (lane == 0) {
            const uint32_t kq = smem_u32(smem + kOffKQ);
            if (mbar_wait(&bars->tma, 0, abort)) {
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < kHalves; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(kq + kb * 16384 + kk * 32, 16, 1024);
                        mma_bf16(tmem + kColG, a, a, kIdescGram, (kb | kk) != 0);
                    }
                mma_commit(&bars->gram);
            } else {
                int dummy = 0;           // the copy must land before the CTA exits
                mbar_wait(&bars->tma, 0, &dummy);
            }
        }
        __syncwarp();
    } else {
        // every warp but warp 1 (224 threads, named barrier 2) from here to L
        const int t7 = warp == 0 ? lane : tid - 32;
        if (warp == 0) {
            // ---- the carry vectors that do not need Gamma (tokens 2l, 2l+1
            //      per lane), to the prepared block
            const int i0 = 2 * lane, i1 = i0 + 1;
            const float4 g0 = gate[i0], g1 = gate[i1];
            const float A0 = vec[vA * kChunk + i0], A1 = vec[vA * kChunk + i1];
            const float U0 = vec[vU * kChunk + i0], U1 = vec[vU * kChunk + i1];
            const float Z0 = vec[vZ * kChunk + i0], Z1 = vec[vZ * kChunk + i1];
            const float b0 = vec[vB * kChunk + i0], b1 = vec[vB * kChunk + i1];
            const float bprev = lane == 0 ? 0.f : vec[vB * kChunk + i0 - 1];   // b_0 = 0
            const int last = n - 1;
            const float Al = vec[vA * kChunk + last], Ul = vec[vU * kChunk + last];
            const float Zl = vec[vZ * kChunk + last], bl = vec[vB * kChunk + last];
            const bool v0 = i0 < n, v1 = i1 < n;
            auto put2 = [&](int row, float x0, float x1) {
                *reinterpret_cast<float2 *>(gv + row * kChunk + i0) =
                    make_float2(v0 ? x0 : 0.f, v1 ? x1 : 0.f);
            };
            put2(kVecAbar, __expf(A0), __expf(A1));
            put2(kVecBmA, bprev * g0.x, b0 * g1.x);
            put2(kVecB, b0, b1);
            put2(kVecGM, (Zl == Z0) ? __expf(Ul - U0) * g0.w : 0.f,
                 (Zl == Z1) ? __expf(Ul - U1) * g1.w : 0.f);
            {
                // [abar_n, b_n, mubar_n, n, 0, ...]
                const float s0 = lane == 0 ? __expf(Al) : (lane == 1 ? ((Zl == 0.f) ? __expf(Ul) : 0.f) : 0.f);
                const float s1 = lane == 0 ? bl : (lane == 1 ? (float)n : 0.f);
                *reinterpret_cast<float2 *>(gv + kVecScal * kChunk + 2 * lane) = make_float2(s0, s1);
            }
        } else if (warp == 2 || warp == 3) {
            // ---- Gt = Gamma Diag(eta) on the four diagonal 16-blocks: thread
            //      = (block b, column j = 16 b + jj), the column recurrence
            //      from its diagonal entry down to the block's last row
            //      (the column is kept in registers and stored after the
            //      loop, so no gate load waits behind a store)
            const int t = tid - 64, blk = t >> 4, j = 16 * blk + (t & 15);
            const float et = gate[j].w;
            float m = 0.f, g = 0.f, col[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = 16 * blk + rr;
                const float4 gr = gate[r];
                const bool diag = (r == j);
                m = diag ? et : gr.z * m;
                g = (diag ? 0.f : gr.x * g) + gr.y * m;
                col[rr] = g;
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (16 * blk + rr >= j) Gt[(16 * blk + rr) * LM + j] = col[rr];
        } else {
            // ---- column factors c_j^(s) = eta_j prod_{u=j+1}^{r0-1} mu_u for
            //      the columns j < r0 = 16 s left of segment s, from the
            //      prefix sums (0 across a zero mu)
            const int t = tid - 128;
            if (t < 96) {
                const int sg = t < 16 ? 1 : (t < 48 ? 2 : 3);
                const int j = t - (sg == 1 ? 0 : (sg == 2 ? 16 : 48));
                const int rp = 16 * sg - 1;
                const float c = (vec[vZ * kChunk + rp] == vec[vZ * kChunk + j])
                                    ? gate[j].w * __expf(vec[vU * kChunk + rp] - vec[vU * kChunk + j])
                                    : 0.f;
                vec[(vC + sg - 1) * kChunk + j] = c;
            }
        }
        asm volatile("bar.sync 2, 224;" ::: "memory");
        // Left of the diagonal blocks the recurrence is affine in a segment's
        // start row:  Gt_{r,j} = F_s(r) Gt_{r0-1,j} + c_j^(s) lambda_s(r)
        // (j < r0, every term non-negative).  Row r0 - 1 is itself in the
        // diagonal block of column j or follows from an earlier segment the
        // same way, so each entry is reached from the last row of its
        // column's diagonal block through whole segments (factors F and
        // lambda at the segment's last row) and then its own segment: one
        // thread per (row, 8 columns), segment 1 rows 16..31 x 2 groups,
        // segment 2 rows 32..47 x 4, segment 3 rows 48..63 x 6
        if (t7 < 32 + 64 + 96) {
            int sg, r, jg;
            if (t7 < 32) {
                sg = 1; r = 16 + (t7 >> 1); jg = t7 & 1;
            } else if (t7 < 96) {
                const int k = t7 - 32;
                sg = 2; r = 32 + (k >> 2); jg = k & 3;
            } else {
                const int k = t7 - 96;
                sg = 3; r = 48 + k / 6; jg = k - (k / 6) * 6;
            }
            const int j0 = 8 * jg, tb = j0 >> 4;
            const float *src = Gt + (16 * tb + 15) * LM + j0;
            float e[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) e[k] = src[k];
            for (int u = tb + 1; u < sg; ++u) {
                const float Fu = vec[vF * kChunk + 16 * u + 15], Lu = vec[vLam * kChunk + 16 * u + 15];
                const float4 c0 = *reinterpret_cast<const float4 *>(vec + (vC + u - 1) * kChunk + j0);
                const float4 c1 = *reinterpret_cast<const float4 *>(vec + (vC + u - 1) * kChunk + j0 + 4);
                const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) e[k] = Fu * e[k] + c[k] * Lu;
            }
            const float F = vec[vF * kChunk + r], lam = vec[vLam * kChunk + r];
            const float4 c0 = *reinterpret_cast<const float4 *>(vec + (vC + sg - 1) * kChunk + j0);
            const float4 c1 = *reinterpret_cast<const float4 *>(vec + (vC + sg - 1) * kChunk + j0 + 4);
            const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            float *dst = Gt + r * LM + j0;
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[k] = F * e[k] + c[k] * lam;
        }
    }
    __syncthreads();   // Gt complete

    // ---- Gram results -> L and A_O.  L is split: its off-diagonal 16-blocks
    //      L_o in bf16 (row-major, the B operand of N = D L_o), its diagonal
    //      16-blocks in fp32 for the forward substitution.  A_O in bf16
    //      (K-major A operand).
    {
        if (warp < 2) {
            const int i = tid;   // carry weight of S: gamma_{n,i} eta_i
            gv[kVecGS * kChunk + i] = i < n ? Gt[(n - 1) * LM + i] : 0.f;
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->gram, 0, abort));
        const int q = warp & 3, half = warp >> 2;
        const int row = 32 * q + lane;
        if (ok) {
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + kColG + half * 32, x);
            tmem_ld_wait();
            if (row < 64) {
                const int i = row, bi = i >> 4;
                const float ai = i < n ? gate[i].x : 0.f;      // rows past the chunk end: 0
                const float *gp = Gt + max(i - 1, 0) * LM + half * 32;
                float y[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    y[jj] = (j < i) ? ai * x[jj] * gp[jj] : 0.f;
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (half * 4 + cc < 2 * bi) {                  // left of the diagonal block
                        w.x = pack2(y[cc * 8 + 0], y[cc * 8 + 1]);
                        w.y = pack2(y[cc * 8 + 2], y[cc * 8 + 3]);
                        w.z = pack2(y[cc * 8 + 4], y[cc * 8 + 5]);
                        w.w = pack2(y[cc * 8 + 6], y[cc * 8 + 7]);
                    }
                    *reinterpret_cast<uint4 *>(Lo + sw128_offset(i, half * 4 + cc)) = w;
                }
                if ((bi >> 1) == half) {                           // the diagonal block
                    float *ld = Ldg + (bi * 16 + (i & 15)) * LB;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) ld[jj] = (bi & 1) ? y[16 + jj] : y[jj];
                }
            } else {
                const int i = row - 64;
                const float *gp = Gt + i * LM + half * 32;
                const bool vi = i < n;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = half * 32 + cc * 8 + e;
                        y[e] = (j <= i && vi) ? x[cc * 8 + e] * gp[cc * 8 + e] : 0.f;
                    }
                    uint4 w;
                    w.x = pack2(y[0], y[1]);
                    w.y = pack2(y[2], y[3]);
                    w.z = pack2(y[4], y[5]);
                    w.w = pack2(y[6], y[7]);
                    *reinterpret_cast<uint4 *>(AO + sw128_offset(i, half * 4 + cc)) = w;
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();   // L_o, the diagonal blocks and A_O ready; Gt no longer needed

    // ---- T = (I + L)^{-1}.  With D = (I + L_d)^{-1} (the inverses of the
    //      diagonal 16-blocks) and N = D L_o (strictly block-lower, so
    //      N^4 = 0):  I + L = (I + L_d)(I + N)  and
    //      T = (I + N)^{-1} D = D - N D + N^2 D - N^3 D.
    //      D by forward substitution in registers (one lane per column of a
    //      block), written in fp32 over L_d and in bf16 (row-major) as an MMA
    //      operand while the other warps zero that operand outside the
    //      diagonal blocks; then three MMAs, each epilogue writing the next
    //      bf16 operands.
    if (warp < 2) {
        const int blk = warp * 2 + (lane >> 4);
        const int c = lane & 15;
        const float *lb = Ldg + blk * 16 * LB;
        // column c of (I + L_d)^{-1}: right-looking forward substitution,
        // every row's update at step k independent of the others
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) t[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < 15; ++k)
#pragma unroll
            for (int r = k + 1; r < 16; ++r) t[r] = fmaf(-lb[r * LB + k], t[k], t[r]);
        asm volatile("bar.sync 1, 64;" ::: "memory");    // every lane has read its block of L
        float *db = Ldg + blk * 16 * LB;                  // D replaces L_d in place
        const int col = 16 * blk + c;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            db[r * LB + c] = t[r];
            *reinterpret_cast<__nv_bfloat16 *>(Dbf + sw128_offset(16 * blk + r, (uint32_t)(col >> 3)) +
                                               2 * (col & 7)) = __float2bfloat16_rn(t[r]);
        }
    } else {
        // the 16-byte pieces of D off its diagonal blocks: rows r, pieces
        // cc with cc / 2 != r / 16 (six per row)
        for (int idx = tid - 64; idx < kChunk * 6; idx += kThreadsP - 64) {
            const int r = idx / 6, k = idx - (idx / 6) * 6;
            const int cc = k + (k >= 2 * (r >> 4) ? 2 : 0);
            *reinterpret_cast<uint4 *>(Dbf + sw128_offset(r, cc)) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Three hops, T = D - N D + N^2 D - N^3 D: N = D L_o; [N D | N^2] =
    // N [D | N]; [N^2 D | N^3 D] = N^2 [D | N D].  Each an M = 64 MMA (the 64
    // result rows sit in lanes 16 q .. 16 q + 15 of quadrant q) whose B
    // operand is two 64-column blocks 8 KiB apart (D, then N or N D), read by
    // all eight warps: quadrant warp % 4, column half warp / 4.
    uint32_t hop_parity = 0;
    const int hq = warp & 3, hhalf = warp >> 2;
    const int hr = 16 * hq + (lane & 15);                      // result row of this thread
    const int hc1 = hhalf * 32 + 8 * (lane >> 4);              // first column of its two groups of 8
    const uint32_t hta = tmem + ((uint32_t)(32 * hq) << 16) + hhalf * 32;
#pragma unroll 1
    for (int hop = 0; hop < 3; ++hop) {
        if (warp == 2 && lane == 0 && !*abort) {
            const uint32_t aop = hop == 0 ? smem_u32(Dbf) : (hop == 1 ? smem_u32(Nbf) : smem_u32(Ybf));
            const uint32_t bop = hop == 0 ? smem_u32(Lo) : smem_u32(Dbf);
            const uint32_t idesc = hop == 0 ? kIdescHop : kIdescHop2;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = sdesc_sw128(aop + kk * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(bop + kk * 2048, 8192, 1024);
                mma_bf16(tmem + kColG, a, b, idesc, kk != 0);
            }
            mma_commit(&bars->hop);
        }
        __syncwarp();
        {
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->hop, hop_parity, abort));
            hop_parity ^= 1;
            if (ok) {
                tc_fence_after();
                float v[16], w2[16];
                tmem_ld_16x2x8(hta, v);                        // first 64 columns
                tmem_ld_16x2x8(hta + 16, v + 8);
                if (hop > 0) {
                    tmem_ld_16x2x8(hta + 64, w2);              // second 64 columns
                    tmem_ld_16x2x8(hta + 64 + 16, w2 + 8);
                }
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const int cb = hc1 + 16 * g;
                    const uint32_t off = sw128_offset(hr, (uint32_t)(cb >> 3));
                    const float *x = v + 8 * g, *y = w2 + 8 * g;
                    uint4 o;
                    if (hop == 0) {
                        // N
                        o.x = pack2(x[0], x[1]); o.y = pack2(x[2], x[3]);
                        o.z = pack2(x[4], x[5]); o.w = pack2(x[6], x[7]);
                        *reinterpret_cast<uint4 *>(Nbf + off) = o;
                    } else if (hop == 1) {
                        // N D replaces N (its MMA is complete); N^2
                        o.x = pack2(x[0], x[1]); o.y = pack2(x[2], x[3]);
                        o.z = pack2(x[4], x[5]); o.w = pack2(x[6], x[7]);
                        *reinterpret_cast<uint4 *>(Nbf + off) = o;
                        o.x = pack2(y[0], y[1]); o.y = pack2(y[2], y[3]);
                        o.z = pack2(y[4], y[5]); o.w = pack2(y[6], y[7]);
                        *reinterpret_cast<uint4 *>(Ybf + off) = o;
                    } else {
                        // T = D - N D + N^2 D - N^3 D (D exact in fp32, block diagonal)
                        const uint4 ndr = *reinterpret_cast<const uint4 *>(Nbf + off);
                        const __nv_bfloat162 *nd2 = reinterpret_cast<const __nv_bfloat162 *>(&ndr);
                        const bool in_blk = (cb >> 4) == (hr >> 4);
                        const float *drow = Ldg + ((hr >> 4) * 16 + (hr & 15)) * LB + (cb & 15);
                        float t[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 nd = __bfloat1622float2(nd2[e]);
                            t[2 * e] = (in_blk ? drow[2 * e] : 0.f) - nd.x + x[2 * e] - y[2 * e];
                            t[2 * e + 1] = (in_blk ? drow[2 * e + 1] : 0.f) - nd.y + x[2 * e + 1] - y[2 * e + 1];
                        }
                        o.x = pack2(t[0], t[1]); o.y = pack2(t[2], t[3]);
                        o.z = pack2(t[4], t[5]); o.w = pack2(t[6], t[7]);
                        *reinterpret_cast<uint4 *>(B2 + off) = o;
                    }
                }
                fence_proxy_async();
            }
            tc_fence_before();
        }
        __syncthreads();
        tc_fence_after();
    }

    // ---- MMA A_O T (rows 0..63 of an M = 128 product: the A rows past A_O
    //      read the next region and are never used); the T rows of the
    //      prepared block leave in bulk: each group of 16 rows of the
    //      row-major T is one 2 KiB piece there (prepared rows 32 g .. 32 g +
    //      15, same row mod 8, so the same swizzle)
    if (warp == 2 && lane == 0 && !*abort) {
        const uint32_t a2 = smem_u32(AO), b2 = smem_u32(B2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = sdesc_sw128(a2 + kk * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(b2 + kk * 2048, 8192, 1024);
            mma_bf16(tmem + kColD2, a, b, kIdescOut, kk != 0);
        }
        mma_commit(&bars->out);
#pragma unroll
        for (int g = 0; g < 4; ++g)
            bulk_store(pblk + PrepLayoutTC::kOffT + g * 4096, B2 + g * 2048, 2048);
        bulk_commit_group();
    }
    __syncwarp();

    // ---- A_O T (accumulator rows 0..63: lane quadrants 0, 1) -> bf16 rows
    //      staged in the A_O buffer (the MMA that read it is complete), then
    //      copied out in bulk: rows 16 g .. 16 g + 15 to prepared rows
    //      32 g + 16 .. 32 g + 31
    if ((warp & 3) < 2) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->out, 0, abort));
        const int q = warp & 3, half = warp >> 2;
        const int i = 32 * q + lane;
        if (ok) {
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + kColD2 + half * 32, x);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint4 w;
                w.x = pack2(x[cc * 8 + 0], x[cc * 8 + 1]);
                w.y = pack2(x[cc * 8 + 2], x[cc * 8 + 3]);
                w.z = pack2(x[cc * 8 + 4], x[cc * 8 + 5]);
                w.w = pack2(x[cc * 8 + 6], x[cc * 8 + 7]);
                *reinterpret_cast<uint4 *>(AO + sw128_offset(i, half * 4 + cc)) = w;
            }
            fence_proxy_async();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        if (lane == 0) {
            if (!*abort) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    bulk_store(pblk + PrepLayoutTC::kOffT + g * 4096 + 2048, AO + g * 2048, 2048);
                bulk_commit_group();
            }
            bulk_wait_group0();          // shared memory stays valid until the copies are done
            // every MMA issued by this CTA completes before TMEM is freed
            mma_commit(&bars->drain);
            int dummy = 0;
            mbar_wait(&bars->drain, 0, &dummy);
        }
        __syncwarp();
        tmem_dealloc(tmem, kTmemColsP);
    }
    if (tid == 0 && *abort && p.status) atomicExch(p.status, (int)MDN_ERR_DEVICE_TIMEOUT);
    if constexpr (kSeg)
        if (follower && last_cta && tid == 0) grid_dependency_wait();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_p() {
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

bool make_map_p(CUtensorMap *map, const void *base, int T_total, int H, int D) {
    auto fn = encode_fn_p();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_prep_tc_t(const ChunkProblem &p, cudaStream_t st) {
    CUtensorMap mk, mq;
    if (!make_map_p(&mk, p.k, p.T_total, p.H, D) || !make_map_p(&mq, p.q, p.T_total, p.H, D))
        return cudaErrorInvalidValue;
    // time segments are a separate instantiation
    auto kern = is_segment(p) ? chunk_prep_tc_kernel<D, true> : chunk_prep_tc_kernel<D, false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemP);
    if (err != cudaSuccess) return err;
    if (is_segment(p)) {
        // the largest shared-memory carveout, so that a CTA fits beside a
        // state-pass CTA (which needs most of it)
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
    }
    dim3 grid(p.max_chunks, p.H);
    if (is_segment(p)) grid.x = (unsigned)(p.n_seq * (p.seg_c1 - p.seg_c0));
    if (!(p.seg_mode & kSegPrepFollower)) {
        kern<<<grid, kThreadsP, kSmemP, st>>>(p, mk, mq);
        return cudaGetLastError();
    }
    // a later segment's prep: a programmatic dependent of the previous
    // segment's state pass, so it starts once that pass's CTAs all run
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = kSmemP;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, mk, mq);
}

}  // namespace

// bf16 inputs, head size 64 or 128.
cudaError_t launch_chunk_prep_tc(const ChunkProblem &p, cudaStream_t st) {
    if ((p.D != 64 && p.D != 128) || p.dtype != MDN_BF16) return cudaErrorInvalidValue;
    if (p.max_chunks == 0) return cudaSuccess;
    return p.D == 128 ? launch_prep_tc_t<128>(p, st) : launch_prep_tc_t<64>(p, st);
}

}  // namespace mdn
