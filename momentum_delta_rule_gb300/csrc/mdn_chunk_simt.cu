// MDN chunkwise forward, CUDA-core (FFMA) path.
//
// Serves fp32 inputs (where one bf16/tf32 tensor-core pass would not hold an
// fp32-level error) and head size 64.  It follows the same two-stage plan as
// the tensor-core path:
//
//   prep  (one CTA per chunk and head, all chunks in parallel)
//         log-space prefix scans of alpha and mu, the coefficient matrix
//         Gamma, the Gram matrices K K^T and Q K^T, the unit-lower-triangular
//         system matrix, its inverse T and the intra-chunk output operator
//         A_O T, written to a prepared block in the workspace;
//   state (one CTA per sequence, head and 32-column slice, chunks in order)
//         the state-dependent part of each chunk: residual right-hand side,
//         residuals, outputs and the carry of S and M.
//
// Equations: "MDN: Parallelizing Stepwise Momentum for Delta Linear
// Attention" slides, frames "Reorder the triangular sum ..." (Eqs. (7)-(9)),
// "Solve the unknown residuals with a lower triangular system" (Eqs.
// (15)-(18)), "Chunk outputs combine incoming states and local writes"
// (Appendix C Eqs. (40)-(42)), backup frames on the one-row shift and on the
// log-domain coefficients (Algorithm 1); reading notes sections 2.3-2.6.
//
// With p_i = alpha_i k_i the residual right-hand side simplifies:
// Diag(abar_shifted) P = Diag(abar) K and Diag(b_shifted) P = Diag(b_{i-1}
// alpha_i) K, so the state pass needs only K S_0 and K M_0.  Writing
// R = V - Diag(abar) K S_0 + Diag(b_{i-1} alpha_i) K M_0, the residuals are
// Vres = T R and the in-chunk output term is (A_O T) R.
#include <type_traits>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

constexpr int kThreads = 256;     // prep
// state pass: 16 row groups of 4 token rows and D/16 state rows, x 32 or 64 columns

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
    static constexpr int LD = D + 1;          // padded row stride of K, Q
    static constexpr int LM = kChunk + 1;     // padded row stride of 64x64
    // K and Q are read only by the Gram products; L, T and A_O take their
    // place afterwards, so that two (d = 128) or three (d = 64) CTAs share an SM
    static constexpr int kKQ = 2 * kChunk * LD, kLTA = 3 * kChunk * LM;
    static constexpr int kShared = kKQ > kLTA ? kKQ : kLTA;
    static constexpr int kFloats = kShared + kChunk * LM + 12 * kChunk + 64;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

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

template <int D, typename Tin>
__global__ void __launch_bounds__(kThreads)
chunk_prep_simt_kernel(ChunkProblem p) {
    using SM = PrepSmem<D>;
    constexpr int LD = SM::LD, LM = SM::LM;
    const int gc = blockIdx.x, h = blockIdx.y;
    ChunkLoc loc;
    if (!locate_chunk(p, gc, loc)) return;
    const int n = loc.n;
    const int tid = threadIdx.x;

    extern __shared__ float smem[];
    float *Ks = smem;                      // [64][LD], until the Gram products
    float *Qs = Ks + kChunk * LD;          // [64][LD], until the Gram products
    float *L = smem;                       // system matrix (strict lower), after them
    float *Tm = L + kChunk * LM;           // its inverse
    float *AO = Tm + kChunk * LM;          // output operator (lower)
    float *G = smem + SM::kShared;         // Gamma [64][LM]
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

    const size_t rs = (size_t)p.H * D;     // token row stride
    const Tin *kg = static_cast<const Tin *>(p.k) + (size_t)loc.t0 * rs + (size_t)h * D;
    const Tin *qg = static_cast<const Tin *>(p.q) + (size_t)loc.t0 * rs + (size_t)h * D;
#pragma unroll
    for (int idx = tid; idx < kChunk * D; idx += kThreads) {
        const int i = idx / D, d = idx - i * D;
        float kv = 0.f, qv = 0.f;
        if (i < n) {
            kv = to_f32(kg[(size_t)i * rs + d]);
            qv = to_f32(qg[(size_t)i * rs + d]);
        }
        Ks[i * LD + d] = kv;
        Qs[i * LD + d] = qv;
    }

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

    // ---- Gram tiles: thread owns a 4 x 4 block of both 64 x 64 products
    {
        const int ti = tid >> 4, tj = tid & 15;
        float gk[4][4] = {}, gq[4][4] = {};
        for (int d = 0; d < D; ++d) {
            float kr[4], qr[4], kc[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                kr[r] = Ks[(4 * ti + r) * LD + d];
                qr[r] = Qs[(4 * ti + r) * LD + d];
                kc[r] = Ks[(4 * tj + r) * LD + d];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    gk[r][c] += kr[r] * kc[c];
                    gq[r][c] += qr[r] * kc[c];
                }
        }
        __syncthreads();   // every thread is done with K and Q: L, T, A_O replace them
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = 4 * ti + r, j = 4 * tj + c;
                // (P Khat^T) . Gamma_shifted: alpha_i (k_i.k_j) eta_j gamma_{i-1,j}, j < i
                L[i * LM + j] = (j < i) ? va[i] * gk[r][c] * ve[j] * G[(i - 1) * LM + j] : 0.f;
                // (Q Khat^T) . Gamma: (q_i.k_j) eta_j gamma_{i,j}, j <= i
                AO[i * LM + j] = (j <= i) ? gq[r][c] * ve[j] * G[i * LM + j] : 0.f;
                Tm[i * LM + j] = (i == j) ? 1.f : 0.f;
            }
    }
    __syncthreads();

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
    float *Tg = reinterpret_cast<float *>(blk + PrepLayout<float>::kOffT);
    float *AOTg = reinterpret_cast<float *>(blk + PrepLayout<float>::kOffAOT);
    float *vec = reinterpret_cast<float *>(blk + PrepLayout<float>::kOffVec);
    static_assert(PrepLayout<float>::kOffVec == PrepLayoutTC::kSplitVec, "vector rows");
    const bool split_tc = p.k_hi != nullptr;
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
        if (split_tc) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * ti + r;
                const float t4[4] = {Tm[i * LM + 4 * tj], Tm[i * LM + 4 * tj + 1],
                                     Tm[i * LM + 4 * tj + 2], Tm[i * LM + 4 * tj + 3]};
                put4(tc_row(i), 4 * tj, t4);
                put4(tc_row(kChunk + i), 4 * tj, acc[r]);
            }
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int i = 4 * ti + r, j = 4 * tj + c;
                    AOTg[i * kChunk + j] = acc[r][c];
                    Tg[i * kChunk + j] = Tm[i * LM + j];
                }
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
}

// --------------------------------------------------------------- state

// The state pass runs 16 row groups x NSC state columns per CTA (NSC = 32:
// 512 threads; NSC = 64: 1024 threads, so that fp32 prefills with many
// (sequence, head) chains at d = 128 fit the GPU in one wave).  With
// NSC = 32 the next chunk's K and vectors are double-buffered.
template <int D, int NSC>
struct StateSmem {
    static constexpr bool kPrefetchK = NSC == 32;
    static constexpr int kFloats = 2 * kChunk * D        // K, Q
                                 + kChunk * NSC          // V slice
                                 + 2 * kChunk * kChunk   // T, AOT
                                 + kVecRows * kChunk     // vectors
                                 + 2 * D * NSC           // S, M slices
                                 + 2 * kChunk * NSC      // R, scaled residuals
                                 + (kPrefetchK ? kChunk * D + kVecRows * kChunk : 0);
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

// 16-byte asynchronous copy global -> shared; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int D, typename Tin, int NSC>
__global__ void __launch_bounds__(16 * NSC)
chunk_state_simt_kernel(ChunkProblem p) {
    constexpr int kNS = NSC;                            // state columns of this CTA
    constexpr int kThreadsS = 16 * NSC;                 // 16 row groups x kNS columns
    constexpr int kSlices = D / kNS;
    constexpr int kRowsA = kChunk / 16;                 // token rows per row group
    constexpr int kRowsC = D / 16;                      // state rows per row group
    const int slice = blockIdx.x % kSlices;
    const int kh = blockIdx.x / kSlices;
    const int s = ordered_sequence(p, kh / p.H), h = kh % p.H;
    const int sh = s * p.H + h;
    // thread = (row group wg, column cc); a warp is 32 adjacent columns of one
    // row group, so the row group's K, Q and T rows are warp-wide broadcasts
    const int tid = threadIdx.x;
    const int cc = ((tid >> 5) % (kNS / 32)) * 32 + (tid & 31), wg = (tid >> 5) / (kNS / 32);
    const int col0 = slice * kNS;

    extern __shared__ float smem[];
    float *Ks = smem;
    float *Qs = Ks + kChunk * D;
    float *Vs = Qs + kChunk * D;
    float *Ts = Vs + kChunk * kNS;
    float *AOTs = Ts + kChunk * kChunk;
    float *vec = AOTs + kChunk * kChunk;
    float *Ss = vec + kVecRows * kChunk;
    float *Ms = Ss + D * kNS;
    float *Rs = Ms + D * kNS;
    float *Vr = Rs + kChunk * kNS;
    float *Kalt = Vr + kChunk * kNS;           // the next chunk's K ...
    float *vecalt = Kalt + kChunk * D;         // ... and vectors
    // fp32 inputs are copied as they are, so the next chunk's tiles stream in
    // with asynchronous copies while this chunk computes (K and the vectors
    // double-buffered, Q and V once the residuals are formed, T and A_O T once
    // the outputs are); bf16 inputs are converted by plain loads per chunk.
    constexpr bool kAsync = std::is_same<Tin, float>::value;
    constexpr bool kPrefK = kAsync && StateSmem<D, NSC>::kPrefetchK;

    int start, len, slot0;
    sequence_range(p, s, start, len, slot0);
    const int nchunks = (len + kChunk - 1) / kChunk;
    const size_t st_off = (size_t)sh * D * D;

#pragma unroll
    for (int idx = tid; idx < D * kNS; idx += kThreadsS) {
        const int d = idx / kNS, c = idx - d * kNS;
        const size_t g = st_off + (size_t)d * D + col0 + c;
        Ss[idx] = p.S0 ? p.S0[g] : 0.f;
        Ms[idx] = p.M0 ? p.M0[g] : 0.f;
    }

    const size_t rs = (size_t)p.H * D;
    const Tin *kg0 = static_cast<const Tin *>(p.k) + (size_t)h * D;
    const Tin *qg0 = static_cast<const Tin *>(p.q) + (size_t)h * D;
    const Tin *vg0 = static_cast<const Tin *>(p.v) + (size_t)h * D + col0;
    Tin *og0 = static_cast<Tin *>(p.o) + (size_t)h * D + col0;
    Tin *rg0 = p.vres ? static_cast<Tin *>(p.vres) + (size_t)h * D + col0 : nullptr;

    // asynchronous copies of chunk cn's tiles (fp32 inputs only); rows past
    // the chunk end are zero-filled
    auto rows_of = [&](int cn, int &t0n, int &nn) {
        t0n = start + cn * kChunk;
        nn = min(kChunk, len - cn * kChunk);
    };
    auto copy_kq = [&](int cn, float *dst, const Tin *src0) {
        int t0n, nn;
        rows_of(cn, t0n, nn);
        for (int idx = tid; idx < kChunk * D / 4; idx += kThreadsS) {
            const int i = idx / (D / 4), q4 = idx - i * (D / 4);
            const bool v = i < nn;
            const Tin *src = src0 + (size_t)(t0n + (v ? i : 0)) * rs + 4 * q4;
            cp_async16(dst + i * D + 4 * q4, src, v ? 16u : 0u);
        }
    };
    auto copy_v = [&](int cn) {
        int t0n, nn;
        rows_of(cn, t0n, nn);
        for (int idx = tid; idx < kChunk * kNS / 4; idx += kThreadsS) {
            const int i = idx / (kNS / 4), q4 = idx - i * (kNS / 4);
            const bool v = i < nn;
            const Tin *src = vg0 + (size_t)(t0n + (v ? i : 0)) * rs + 4 * q4;
            cp_async16(Vs + i * kNS + 4 * q4, src, v ? 16u : 0u);
        }
    };
    auto block_of = [&](int cn) {
        return p.prep + ((size_t)(slot0 + cn) * p.H + h) * p.prep_stride;
    };
    auto copy_floats = [&](float *dst, const unsigned char *src, int nfloats) {
        for (int idx = tid; idx < nfloats / 4; idx += kThreadsS)
            cp_async16(dst + 4 * idx, src + 16 * (size_t)idx, 16u);
    };
    if (kAsync && nchunks > 0) {
        const unsigned char *b0 = block_of(0);
        copy_kq(0, Ks, kg0);
        copy_kq(0, Qs, qg0);
        copy_v(0);
        copy_floats(Ts, b0 + PrepLayout<float>::kOffT, kChunk * kChunk);
        copy_floats(AOTs, b0 + PrepLayout<float>::kOffAOT, kChunk * kChunk);
        copy_floats(vec, b0 + PrepLayout<float>::kOffVec, kVecRows * kChunk);
        cp_async_commit();
    }

    for (int c = 0; c < nchunks; ++c) {
        const int t0 = start + c * kChunk;
        const int n = min(kChunk, len - c * kChunk);
        const unsigned char *blk = p.prep + ((size_t)(slot0 + c) * p.H + h) * p.prep_stride;
        const float *Tg = reinterpret_cast<const float *>(blk + PrepLayout<float>::kOffT);
        const float *AOTg = reinterpret_cast<const float *>(blk + PrepLayout<float>::kOffAOT);
        const float *vg = reinterpret_cast<const float *>(blk + PrepLayout<float>::kOffVec);

        if (kAsync) cp_async_wait_all();   // this chunk's tiles have landed
        __syncthreads();   // previous chunk finished with every buffer
        if (kAsync && !kPrefK && c > 0) {
            // K and the vectors have no second buffer at this width
            copy_kq(c, Ks, kg0);
            copy_floats(vec, block_of(c) + PrepLayout<float>::kOffVec, kVecRows * kChunk);
            cp_async_commit();
            cp_async_wait_all();
            __syncthreads();
        }
        if (p.S_chunks) {
            // the entry state of this chunk, at its chunk slot
            const size_t cs = ((size_t)(slot0 + c) * p.H + h) * D * D;
            for (int idx = tid; idx < D * kNS; idx += kThreadsS) {
                const int d = idx / kNS, cx = idx - d * kNS;
                const size_t g = cs + (size_t)d * D + col0 + cx;
                p.S_chunks[g] = Ss[idx];
                p.M_chunks[g] = Ms[idx];
            }
        }
        if (!kAsync) {
#pragma unroll
            for (int idx = tid; idx < kChunk * D; idx += kThreadsS) {
                const int i = idx / D, d = idx - i * D;
                float kv = 0.f, qv = 0.f;
                if (i < n) {
                    kv = to_f32(kg0[(size_t)(t0 + i) * rs + d]);
                    qv = to_f32(qg0[(size_t)(t0 + i) * rs + d]);
                }
                Ks[idx] = kv;
                Qs[idx] = qv;
            }
#pragma unroll
            for (int idx = tid; idx < kChunk * kNS; idx += kThreadsS) {
                const int i = idx / kNS, cx = idx - i * kNS;
                Vs[idx] = (i < n) ? to_f32(vg0[(size_t)(t0 + i) * rs + cx]) : 0.f;
            }
#pragma unroll
            for (int idx = tid; idx < kChunk * kChunk; idx += kThreadsS) {
                Ts[idx] = Tg[idx];
                AOTs[idx] = AOTg[idx];
            }
#pragma unroll
            for (int idx = tid; idx < kVecRows * kChunk; idx += kThreadsS) vec[idx] = vg[idx];
        }
        __syncthreads();

        // ---- K S_0, K M_0, Q S_0, Q M_0 for kRowsA token rows x 1 column;
        //      the K and Q rows (the same for the whole warp) four at a time
        float ks[kRowsA] = {}, km[kRowsA] = {}, qs[kRowsA] = {}, qm[kRowsA] = {};
        for (int d = 0; d < D; d += 4) {
            float sv[4], mv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                sv[u] = Ss[(d + u) * kNS + cc];
                mv[u] = Ms[(d + u) * kNS + cc];
            }
#pragma unroll
            for (int r = 0; r < kRowsA; ++r) {
                const int i = wg * kRowsA + r;
                const float4 kv = *reinterpret_cast<const float4 *>(Ks + i * D + d);
                const float4 qv = *reinterpret_cast<const float4 *>(Qs + i * D + d);
                ks[r] += kv.x * sv[0] + kv.y * sv[1] + kv.z * sv[2] + kv.w * sv[3];
                km[r] += kv.x * mv[0] + kv.y * mv[1] + kv.z * mv[2] + kv.w * mv[3];
                qs[r] += qv.x * sv[0] + qv.y * sv[1] + qv.z * sv[2] + qv.w * sv[3];
                qm[r] += qv.x * mv[0] + qv.y * mv[1] + qv.z * mv[2] + qv.w * mv[3];
            }
        }
        float oint[kRowsA];
#pragma unroll
        for (int r = 0; r < kRowsA; ++r) {
            const int i = wg * kRowsA + r;
            Rs[i * kNS + cc] = Vs[i * kNS + cc] - vec[kVecAbar * kChunk + i] * ks[r]
                               + vec[kVecBmA * kChunk + i] * km[r];
            oint[r] = vec[kVecAbar * kChunk + i] * qs[r] - vec[kVecB * kChunk + i] * qm[r];
        }
        __syncthreads();
        if (kAsync && c + 1 < nchunks) {
            // Q and V are free now; K and the vectors go to the other buffers
            copy_kq(c + 1, Qs, qg0);
            copy_v(c + 1);
            if (kPrefK) {
                copy_kq(c + 1, Kalt, kg0);
                copy_floats(vecalt, block_of(c + 1) + PrepLayout<float>::kOffVec, kVecRows * kChunk);
            }
        }

        // ---- residuals Vres = T R, outputs O = O_inter + (A_O T) R: the
        //      warp's rows i0 .. i0 + kRowsA - 1 share every R column j < i0
        //      (read once, four at a time with the rows of T and A_O T), then
        //      the triangle j = i0 .. i
        static_assert(kRowsA == 4, "four token rows per warp");
        const int i0 = wg * kRowsA;
        float vrr[kRowsA] = {}, oir[kRowsA] = {};
        for (int j = 0; j < i0; j += 4) {
            float rv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) rv[u] = Rs[(j + u) * kNS + cc];
#pragma unroll
            for (int r = 0; r < kRowsA; ++r) {
                const float4 tv = *reinterpret_cast<const float4 *>(Ts + (i0 + r) * kChunk + j);
                const float4 av = *reinterpret_cast<const float4 *>(AOTs + (i0 + r) * kChunk + j);
                vrr[r] += tv.x * rv[0] + tv.y * rv[1] + tv.z * rv[2] + tv.w * rv[3];
                oir[r] += av.x * rv[0] + av.y * rv[1] + av.z * rv[2] + av.w * rv[3];
            }
        }
#pragma unroll
        for (int u = 0; u < kRowsA; ++u) {
            const float rv = Rs[(i0 + u) * kNS + cc];
#pragma unroll
            for (int r = u; r < kRowsA; ++r) {
                vrr[r] += Ts[(i0 + r) * kChunk + i0 + u] * rv;
                oir[r] += AOTs[(i0 + r) * kChunk + i0 + u] * rv;
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsA; ++r) {
            const int i = i0 + r;
            const float vr = vrr[r], oi = oir[r];
            Vr[i * kNS + cc] = vr;
            if (i < n) og0[(size_t)(t0 + i) * rs + cc] = from_f32<Tin>(oint[r] + oi);
            if (rg0 && i < n) rg0[(size_t)(t0 + i) * rs + cc] = from_f32<Tin>(vr);
        }
        __syncthreads();
        if (kAsync && c + 1 < nchunks) {
            // T and A_O T are free now
            const unsigned char *bn = block_of(c + 1);
            copy_floats(Ts, bn + PrepLayout<float>::kOffT, kChunk * kChunk);
            copy_floats(AOTs, bn + PrepLayout<float>::kOffAOT, kChunk * kChunk);
            cp_async_commit();
        }

        // ---- carry, both from the old S_0, M_0:
        //      S <- abar_n S - b_n M + sum_i k_i gamma_{n,i} eta_i vres_i^T
        //      M <- mubar_n M - sum_i k_i (prod_{u>i} mu_u) eta_i vres_i^T
        const float abar_n = vec[kVecScal * kChunk + 0];
        const float b_n = vec[kVecScal * kChunk + 1];
        const float mubar_n = vec[kVecScal * kChunk + 2];
        // the warp's kRowsC state rows d0 .. d0 + kRowsC - 1 at once: per
        // token, its weighted residuals once and the K row four at a time
        static_assert(kRowsC % 4 == 0, "state rows per warp");
        const int d0 = wg * kRowsC;
        float as[kRowsC] = {}, am[kRowsC] = {};
        for (int i = 0; i < n; ++i) {
            const float vv = Vr[i * kNS + cc];
            const float gsv = vec[kVecGS * kChunk + i] * vv;
            const float gmv = vec[kVecGM * kChunk + i] * vv;
#pragma unroll
            for (int r = 0; r < kRowsC; r += 4) {
                const float4 kv = *reinterpret_cast<const float4 *>(Ks + i * D + d0 + r);
                as[r] += kv.x * gsv; as[r + 1] += kv.y * gsv; as[r + 2] += kv.z * gsv; as[r + 3] += kv.w * gsv;
                am[r] += kv.x * gmv; am[r + 1] += kv.y * gmv; am[r + 2] += kv.z * gmv; am[r + 3] += kv.w * gmv;
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsC; ++r) {
            const int d = d0 + r;
            const float so = Ss[d * kNS + cc], mo = Ms[d * kNS + cc];
            Ss[d * kNS + cc] = abar_n * so - b_n * mo + as[r];
            Ms[d * kNS + cc] = mubar_n * mo - am[r];
        }
        if (kPrefK) {               // the next chunk's K and vectors are in the other buffers
            float *t = Ks; Ks = Kalt; Kalt = t;
            t = vec; vec = vecalt; vecalt = t;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < D * kNS; idx += kThreadsS) {
        const int d = idx / kNS, cx = idx - d * kNS;
        const size_t g = st_off + (size_t)d * D + col0 + cx;
        if (p.S_T) p.S_T[g] = Ss[idx];
        if (p.M_T) p.M_T[g] = Ms[idx];
    }
}

template <int D, typename Tin>
cudaError_t launch_prep_t(const ChunkProblem &p, cudaStream_t st) {
    if (p.max_chunks == 0) return cudaSuccess;
    auto kp = chunk_prep_simt_kernel<D, Tin>;
    cudaError_t err = cudaFuncSetAttribute(
        kp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PrepSmem<D>::kBytes);
    if (err != cudaSuccess) return err;
    dim3 grid(p.max_chunks, p.H);
    kp<<<grid, kThreads, PrepSmem<D>::kBytes, st>>>(p);
    return cudaGetLastError();
}

template <int D, typename Tin, int NSC>
cudaError_t launch_state_t(const ChunkProblem &p, cudaStream_t st) {
    auto ks = chunk_state_simt_kernel<D, Tin, NSC>;
    cudaError_t err = cudaFuncSetAttribute(
        ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)StateSmem<D, NSC>::kBytes);
    if (err != cudaSuccess) return err;
    const long blocks = (long)p.n_seq * p.H * (D / NSC);
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    ks<<<(unsigned)blocks, 16 * NSC, StateSmem<D, NSC>::kBytes, st>>>(p);
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

cudaError_t launch_chunk_prep_simt(const ChunkProblem &p, cudaStream_t st) {
    if (p.D == 128) {
        return p.dtype == MDN_BF16 ? launch_prep_t<128, __nv_bfloat16>(p, st)
                                   : launch_prep_t<128, float>(p, st);
    }
    return p.dtype == MDN_BF16 ? launch_prep_t<64, __nv_bfloat16>(p, st)
                               : launch_prep_t<64, float>(p, st);
}

cudaError_t launch_chunk_state_simt(const ChunkProblem &p, cudaStream_t st) {
    if (p.D == 128) {
        if (p.dtype == MDN_BF16) return launch_state_t<128, __nv_bfloat16, 32>(p, st);
        // 64-column CTAs once 32-column ones would need more than one wave
        const long chains = (long)p.n_seq * p.H;
        const int sms = device_sm_count();
        if (sms > 0 && chains * (128 / 32) > sms) return launch_state_t<128, float, 64>(p, st);
        return launch_state_t<128, float, 32>(p, st);
    }
    return p.dtype == MDN_BF16 ? launch_state_t<64, __nv_bfloat16, 32>(p, st)
                               : launch_state_t<64, float, 32>(p, st);
}

}  // namespace mdn
