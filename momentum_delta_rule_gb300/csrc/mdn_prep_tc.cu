// MDN chunkwise forward — chunk-local preparation on the tensor cores
// (bf16 inputs, head size 128).  One CTA per (chunk, head); all chunks of all
// sequences in parallel.
//
// Per chunk of n <= 64 tokens ("MDN: Parallelizing Stepwise Momentum for
// Delta Linear Attention" slides, frames "Reorder the triangular sum ..."
// (Eqs. (7)-(9)), "Solve the unknown residuals with a lower triangular
// system" (Eqs. (15)-(18)), "Chunk outputs combine incoming states and local
// writes", backup frames on the row shift and the log-domain coefficients;
// reading notes 2.3-2.6):
//
//   A_i = sum_{r<=i} log alpha_r, U_i = sum_{r<=i, mu_r>0} log mu_r,
//   Z_i = #{r <= i : mu_r = 0}            (warp-shuffle prefix scans)
//   gamma_{j,j} = beta_j,  gamma_{i,j} = alpha_i gamma_{i-1,j}
//                 + beta_i [Z_i = Z_j] exp(U_i - U_j)       (column recurrence)
//   b_i = sum_{r<=i} beta_r [Z_r = 0] exp(A_i - A_r + U_r)
//   MMA   G = [K; Q] K^T                                   (M=128, N=64, K=128)
//   L_{i,j}   = alpha_i G_K[i,j] eta_j gamma_{i-1,j}   (j < i, the shifted Gamma)
//   A_O[i,j]  = G_Q[i,j] eta_j gamma_{i,j}             (j <= i)
//   T = (I + L)^{-1}                     (forward substitution, fp32)
//   MMA   [T; A_O T] = [I; A_O] T                          (M=128, N=64, K=64)
//
// and writes the prepared block: [T; A_O T] in bf16 in the 128-byte-swizzled
// K-major operand layout of the state pass (rows interleaved by tc_row), then
// the fp32 carry vectors.
// Rows and columns past the chunk end are masked (T is the identity there and
// every vector entry is zero).
#include <cudaTypedefs.h>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kThreadsP = 256;
constexpr int LM = kChunk + 1;                 // padded fp32 row stride

// shared memory (bytes from the 1024-aligned base), 55 KiB so that four CTAs
// share an SM.  Regions are reused once their last reader is done:
//   [0, 32768)       K/Q tiles (TMA), read by the Gram MMA only; then
//   [0, 16640)       Gamma fp32 [64][65], later T fp32 [64][65]
//   [17408, 34048)   L fp32 [64][65]; after the inverse, bf16(T) (8 KiB)
//   [34048, 38272)   the per-token vectors (2 KiB); after L is built, the
//                    inverse's 32 x 33 fp32 scratch
//   [38912, 55296)   [I; A_O] bf16, K-major A operand
constexpr uint32_t kOffKQ = 0;
constexpr uint32_t kOffG = 0;
constexpr uint32_t kOffL = 17408;
constexpr uint32_t kOffB2 = 17408;
constexpr uint32_t kOffVec = 34048;
constexpr uint32_t kOffXs = 34048;
constexpr uint32_t kOffA2 = 38912;
constexpr uint32_t kOffBarP = kOffA2 + 16384;
constexpr uint32_t kSmemP = kOffBarP + 128 + 1024;
static_assert(kOffL + 4 * 64 * 65 <= kOffVec + 0 && kOffXs + 4 * 32 * 33 <= kOffA2, "prep layout");
static_assert(kSmemP <= 57344, "four CTAs per SM");

constexpr uint32_t kTmemColsP = 128;
constexpr uint32_t kColG = 0;                  // Gram accumulator, 64 columns
constexpr uint32_t kColD2 = 64;                // [T; A_O T] accumulator, 64 columns

constexpr uint32_t kIdescGram = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescOut = idesc_bf16(128, 64, false, true);

struct BarsP {
    uint64_t tma, gram, out, drain;
    uint32_t tmem_base;
    int abort;
};

enum { vAlpha = 0, vBeta, vEta, vA, vU, vZ, vB, vScan };

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Inclusive prefix sum over lanes 0..63 (warps 0 and 1).  Called by those two
// warps only; they synchronise on named barrier 1.
__device__ __forceinline__ float scan64(float x, float *xch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (warp == 0 && lane == 31) *xch = x;
    asm volatile("bar.sync 1, 64;" ::: "memory");
    if (warp == 1) x += *xch;
    asm volatile("bar.sync 1, 64;" ::: "memory");
    return x;
}

__global__ void __launch_bounds__(kThreadsP, 4)
chunk_prep_tc_kernel(const ChunkProblem p, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_q) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    BarsP *bars = reinterpret_cast<BarsP *>(smem + kOffBarP);
    volatile int *abort = &bars->abort;
    float *vec = reinterpret_cast<float *>(smem + kOffVec);    // [8][64]
    float *G = reinterpret_cast<float *>(smem + kOffG);        // Gamma, then T
    float *L = reinterpret_cast<float *>(smem + kOffL);
    unsigned char *A2 = smem + kOffA2;
    unsigned char *B2 = smem + kOffB2;

    // The state pass may be scheduled as soon as every CTA of this grid has
    // started; it waits for this grid's completion before it reads a
    // prepared block.
    grid_launch_dependents();
    const int gc = blockIdx.x, h = blockIdx.y;
    ChunkLoc loc;
    if (!locate_chunk(p, gc, loc)) return;
    const int n = loc.n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // gates first: their latency overlaps the setup below
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
        mbar_init(&bars->out, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        // K and Q tiles: issued before the block-wide setup, their latency
        // gates the Gram MMA and with it Gamma
        mbar_arrive_expect_tx(&bars->tma, 32768);
        tma_load_3d(smem + kOffKQ + 0, &map_k, &bars->tma, 0, h, loc.t0);
        tma_load_3d(smem + kOffKQ + 8192, &map_q, &bars->tma, 0, h, loc.t0);
        tma_load_3d(smem + kOffKQ + 16384, &map_k, &bars->tma, 64, h, loc.t0);
        tma_load_3d(smem + kOffKQ + 24576, &map_q, &bars->tma, 64, h, loc.t0);
    }
    if (warp == 2) {
        tmem_alloc(&bars->tmem_base, kTmemColsP);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 2) {
        // ---- the Gram MMA once the K/Q tiles land
        if (lane == 0) {
            // Gram MMA G = [K; Q] K^T as soon as the tiles land: Gamma reuses
            // their space
            const uint32_t kq = smem_u32(smem + kOffKQ);
            if (mbar_wait(&bars->tma, 0, abort)) {
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
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
    } else if (warp < 2) {
        // ---- gates, log-space prefix scans, Gamma, b, carry vectors
        const int i = tid;                 // token 0..63
        const float a = g_a, mu = g_mu, be = g_be, et = g_et;
        const bool zmu = (mu == 0.f);
        float *xch = vec + vScan * kChunk;
        const float A = scan64(logf(a), xch);
        const float U = scan64(zmu ? 0.f : logf(mu), xch);
        const float Z = scan64(zmu ? 1.f : 0.f, xch);
        vec[vAlpha * kChunk + i] = a;
        vec[vBeta * kChunk + i] = be;
        vec[vEta * kChunk + i] = et;
        vec[vA * kChunk + i] = A;
        vec[vU * kChunk + i] = U;
        vec[vZ * kChunk + i] = Z;
        asm volatile("bar.sync 1, 64;" ::: "memory");
    } else {
        // ---- identity rows of [I; A_O] while the others work (warps 3..7)
        for (int idx = tid - 96; idx < 64 * 8; idx += kThreadsP - 96) {
            const int r = idx >> 3, c = idx & 7;
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if ((r >> 3) == c) {
                const int e = r & 7;                       // 1.0 at column r
                const uint32_t one = 0x3F80u;              // bf16 1.0
                uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
                wp[e >> 1] = (e & 1) ? (one << 16) : one;
            }
            *reinterpret_cast<uint4 *>(A2 + sw128_offset(r, c)) = w;
        }
    }
    __syncthreads();   // gates and prefix scans are in shared memory

    // ---- Gamma: gamma_{j,j} = beta_j, gamma_{r,j} = alpha_r gamma_{r-1,j} +
    //      beta_r m_{r,j} with m_{r,j} = [Z_r = Z_j] exp(U_r - U_j), in four
    //      row segments of 16 run side by side (thread = segment x column).
    //      Each segment starts from zero; as the recurrence is affine,
    //      gamma_{r,j} = local_{r,j} + (prod_{u=r0..r} alpha_u) gamma_{r0-1,j}
    //      restores the exact values (segment ends first, in order).  Only
    //      the lower triangle is ever read.
    float *F = vec + vB * kChunk;      // prod of alpha from the segment start (b comes later)
    // Gamma overwrites the K/Q tiles: the Gram MMA must have read them
    const bool gram_ok = __all_sync(0xffffffffu, mbar_wait(&bars->gram, 0, abort));
    if (gram_ok) {
        tc_fence_after();
    }
    {
        const int j = tid & 63, r0 = 16 * (tid >> 6);
        const float Uj = vec[vU * kChunk + j], Zj = vec[vZ * kChunk + j];
        float gl = 0.f, pa = 1.f;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const int r = r0 + rr;
            const float ar = vec[vAlpha * kChunk + r], br = vec[vBeta * kChunk + r];
            const float ur = vec[vU * kChunk + r], zr = vec[vZ * kChunk + r];
            pa *= ar;
            const float m = (zr == Zj) ? __expf(ur - Uj) : 0.f;
            const float gn = (r == j) ? br : ar * gl + br * m;
            if (r >= j) {
                gl = gn;
                G[r * LM + j] = gl;
            }
            if (j == 0) F[r] = pa;
        }
    }
    __syncthreads();
    if (tid < 64) {
        // exact values at rows 31 and 47 (row 15 is exact already)
        const int j = tid;
        float e = G[15 * LM + j];
#pragma unroll
        for (int g = 1; g < 4; ++g) {
            const int rend = 16 * g + 15;
            if (j < 16 * g) {
                e = G[rend * LM + j] + F[rend] * e;
                G[rend * LM + j] = e;
            } else if (j <= rend) {
                e = G[rend * LM + j];
            }
        }
    }
    __syncthreads();
    {
        const int j = tid & 63, r0 = 16 * (tid >> 6);
        if (j < r0) {
            const float e = G[(r0 - 1) * LM + j];
#pragma unroll
            for (int rr = 0; rr < 15; ++rr) {
                const int r = r0 + rr;
                G[r * LM + j] += F[r] * e;
            }
        }
    }
    __syncthreads();   // Gamma complete
    if (warp < 2) {
        const int i = tid;
        const float a = vec[vAlpha * kChunk + i], be = vec[vBeta * kChunk + i];
        const float et = vec[vEta * kChunk + i];
        const float A = vec[vA * kChunk + i], U = vec[vU * kChunk + i], Z = vec[vZ * kChunk + i];
        // b_i = alpha_i b_{i-1} + beta_i mubar_i as an affine prefix scan:
        // each lane holds the map x -> ca x + cb of its token; maps compose.
        float ca = a;
        float cb = (Z == 0.f) ? be * __expf(U) : 0.f;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float pa = __shfl_up_sync(0xffffffffu, ca, d);
            const float pb = __shfl_up_sync(0xffffffffu, cb, d);
            if ((i & 31) >= d) {
                cb = ca * pb + cb;
                ca = ca * pa;
            }
        }
        if (warp == 0 && lane == 31) vec[vScan * kChunk] = cb;
        asm volatile("bar.sync 1, 64;" ::: "memory");
        const float bsum = (warp == 1) ? ca * vec[vScan * kChunk] + cb : cb;
        vec[vB * kChunk + i] = bsum;
        asm volatile("bar.sync 1, 64;" ::: "memory");
        // carry vectors of the prepared block
        const int last = n - 1;
        const bool valid = i < n;
        float *gv = reinterpret_cast<float *>(
            p.prep + ((size_t)gc * p.H + h) * p.prep_stride + PrepLayoutTC::kOffVec);
        gv[kVecAbar * kChunk + i] = valid ? expf(A) : 0.f;
        gv[kVecBmA * kChunk + i] = (valid && i > 0) ? vec[vB * kChunk + i - 1] * a : 0.f;
        gv[kVecB * kChunk + i] = valid ? bsum : 0.f;
        gv[kVecGS * kChunk + i] = valid ? G[last * LM + i] * et : 0.f;
        const float mtail =
            (vec[vZ * kChunk + last] == Z) ? expf(vec[vU * kChunk + last] - U) : 0.f;
        gv[kVecGM * kChunk + i] = valid ? mtail * et : 0.f;
        float sc = 0.f;
        if (i == 0) sc = expf(vec[vA * kChunk + last]);
        if (i == 1) sc = vec[vB * kChunk + last];
        if (i == 2) sc = (vec[vZ * kChunk + last] == 0.f) ? expf(vec[vU * kChunk + last]) : 0.f;
        if (i == 3) sc = (float)n;
        gv[kVecScal * kChunk + i] = sc;
    }
    __syncthreads();   // vectors ready

    // ---- Gram results -> L (fp32) and A_O (bf16 rows 64..127 of A2)
    {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->gram, 0, abort));
        const int q = warp & 3, half = warp >> 2;
        const int row = 32 * q + lane;
        if (ok) {
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + kColG + half * 32, x);
            tmem_ld_wait();
            const float *va = vec + vAlpha * kChunk;
            const float *ve = vec + vEta * kChunk;
            if (row < 64) {
                const int i = row;
                const float ai = va[i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    float v = 0.f;
                    if (j < i && i < n) v = ai * x[jj] * ve[j] * G[(i - 1) * LM + j];
                    L[i * LM + j] = v;       // padded stride: lanes hit distinct banks
                }
            } else {
                const int i = row - 64;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = half * 32 + cc * 8 + e;
                        y[e] = (j <= i && i < n) ? x[cc * 8 + e] * ve[j] * G[i * LM + j] : 0.f;
                    }
                    uint4 w;
                    w.x = pack2(y[0], y[1]);
                    w.y = pack2(y[2], y[3]);
                    w.z = pack2(y[4], y[5]);
                    w.w = pack2(y[6], y[7]);
                    *reinterpret_cast<uint4 *>(A2 + sw128_offset(row, half * 4 + cc)) = w;
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();   // L ready; Gamma no longer needed

    // ---- T = (I + L)^{-1}, blocked:
    //   diagonal 16x16 blocks by forward substitution in registers (one lane
    //   per column), then [[A,0],[C,B]]^{-1} = [[A^-1,0],[-B^-1 C A^-1, B^-1]]
    //   for the 16-blocks inside each 32-block and for the two 32-blocks.
    //   The blocks above the diagonal 16-blocks are never read; bf16(T)
    //   writes zeros there.
    float *Tm = G;
    float *X = reinterpret_cast<float *>(smem + kOffXs);    // scratch (the vectors are consumed)
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
    // 16-blocks below the diagonal inside each 32-block (two of them); each
    // thread computes two adjacent outputs of one row
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
    // the 32-block below the diagonal: -T_B (L_C T_A).  X = L_C T_A: warp w
    // owns columns [4w, 4w+4) of all 32 rows, so k runs over T_A's nonzero
    // rows k >= 4w only (warp-uniform trip count).
    {
        const int i = lane, j0 = warp * 4;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = j0; k < 32; ++k) {
            const float l = L[(32 + i) * LM + k];
            const float *t = Tm + k * LM + j0;
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] += l * t[e];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) X[i * LX + j0 + e] = a[e];
    }
    __syncthreads();
    // T_C = -T_B X: warp w owns rows [4w, 4w+4), lane = column; k runs over
    // T_B's nonzero columns k <= 4w+3 only.
    {
        const int i0 = warp * 4, j = lane;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < i0 + 4; ++k) {
            const float x = X[k * LX + j];
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] += Tm[(32 + i0 + e) * LM + 32 + k] * x;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) Tm[(32 + i0 + e) * LM + j] = -a[e];
    }
    __syncthreads();

    // ---- bf16(T) as the MN-major B operand (rows k, columns j)
    for (int idx = tid; idx < kChunk * 8; idx += kThreadsP) {
        const int r = idx >> 3, c = idx & 7;
        const float *src = Tm + r * LM + c * 8;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if ((c >> 1) <= (r >> 4)) {              // above the diagonal blocks T is zero
            w.x = pack2(src[0], src[1]);
            w.y = pack2(src[2], src[3]);
            w.z = pack2(src[4], src[5]);
            w.w = pack2(src[6], src[7]);
        }
        *reinterpret_cast<uint4 *>(B2 + sw128_offset(r, c)) = w;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2 && lane == 0 && !*abort) {
        const uint32_t a2 = smem_u32(A2), b2 = smem_u32(B2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = sdesc_sw128(a2 + kk * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(b2 + kk * 2048, 8192, 1024);
            mma_bf16(tmem + kColD2, a, b, kIdescOut, kk != 0);
        }
        mma_commit(&bars->out);
    }
    __syncwarp();

    // ---- [T; A_O T] -> bf16 swizzled rows of the prepared block
    {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->out, 0, abort));
        const int q = warp & 3, half = warp >> 2;
        const int row = 32 * q + lane;
        if (ok) {
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + kColD2 + half * 32, x);
            tmem_ld_wait();
            // staged in shared memory (the MMA that read [I; A_O] is done),
            // then one bulk copy writes whole lines of the prepared block
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint4 w;
                w.x = pack2(x[cc * 8 + 0], x[cc * 8 + 1]);
                w.y = pack2(x[cc * 8 + 2], x[cc * 8 + 3]);
                w.z = pack2(x[cc * 8 + 4], x[cc * 8 + 5]);
                w.w = pack2(x[cc * 8 + 6], x[cc * 8 + 7]);
                *reinterpret_cast<uint4 *>(A2 + sw128_offset(tc_row(row), half * 4 + cc)) = w;
            }
            fence_proxy_async();
        }
        tc_fence_before();
    }
    __syncthreads();
    if (tid == 0 && !*abort) {
        bulk_store(p.prep + ((size_t)gc * p.H + h) * p.prep_stride + PrepLayoutTC::kOffT, A2, 16384);
        bulk_commit_group();
        bulk_wait_group0();
    }
    if (warp == 2) {
        // every MMA issued by this CTA completes before TMEM is freed
        if (lane == 0) {
            mma_commit(&bars->drain);
            int dummy = 0;
            mbar_wait(&bars->drain, 0, &dummy);
        }
        __syncwarp();
        tmem_dealloc(tmem, kTmemColsP);
    }
    if (tid == 0 && *abort && p.status) atomicExch(p.status, (int)MDN_ERR_DEVICE_TIMEOUT);
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

bool make_map_p(CUtensorMap *map, const void *base, int T_total, int H) {
    auto fn = encode_fn_p();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_prep_tc(const ChunkProblem &p, cudaStream_t st) {
    if (p.D != kD || p.dtype != MDN_BF16) return cudaErrorInvalidValue;
    if (p.max_chunks == 0) return cudaSuccess;
    CUtensorMap mk, mq;
    if (!make_map_p(&mk, p.k, p.T_total, p.H) || !make_map_p(&mq, p.q, p.T_total, p.H))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(chunk_prep_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemP);
    if (err != cudaSuccess) return err;
    dim3 grid(p.max_chunks, p.H);
    chunk_prep_tc_kernel<<<grid, kThreadsP, kSmemP, st>>>(p, mk, mq);
    return cudaGetLastError();
}

}  // namespace mdn
