// MDN chunkwise gradient pass: the CUDA-core kernels (all of them for fp32
// inputs, in fp32; for bf16 inputs the coefficient and gate kernels around
// the tensor-core chain and chunk kernels).
//
// The pages give the storage policy of training, not the gradient formulas:
// the forward keeps what the backward needs so that the states need not be
// stored token by token ("MDN: Parallelizing Stepwise Momentum for Delta
// Linear Attention" slides, frame "The implementation trades saved residuals
// for throughput" and the "Backward computation" block; reading notes, end of
// section 2.6).  Here the forward's per-chunk entry states (mdn_chunk_fwd_states)
// are that saved data, and the gradient is the vector-Jacobian product of
// the chunk equations (frames "Solve the unknown residuals with a lower
// triangular system", Eqs. (15)-(18), and "Chunk outputs combine incoming
// states and local writes", Appendix C Eqs. (40)-(42)).  Per chunk of n
// tokens, with P = Diag(alpha) K, Kh = Diag(eta) K, X = P Kh^T, Y = Q Kh^T,
// T = (I + X . Gamma_m)^{-1}, A = Y . Gamma and the carry rows
// WS = Diag(Gamma_{n,:}) Kh, WM = Diag(mu_tail) Kh:
//
//   reverse chain over chunks (state adjoints dS, dM at the chunk's end):
//     dVres = WS dS - WM dM + A^T dO,   dR = T^T dVres   (= dV)
//     dS   <- abar_n dS + (Diag(abar) Q)^T dO - (Diag(abar_m) P)^T dR
//     dM   <- mubar_n dM - b_n dS + ... - (Diag(b) Q)^T dO + (Diag(b_m) P)^T dR
//   per chunk, from its entry states S0, M0 and end adjoints dS, dM:
//     Vres = T (V - Diag(abar_m) P S0 + Diag(b_m) P M0)
//     dQ   = Diag(abar) dO S0^T - Diag(b) dO M0^T + ((dO Vres^T) . Gamma) Kh
//     dP   = -Diag(abar_m) dR S0^T + Diag(b_m) dR M0^T + ((-dR Vres^T) . Gamma_m) Kh
//     dKh  = Diag(Gamma_{n,:}) Vres dS^T - Diag(mu_tail) Vres dM^T
//            + ((dO Vres^T) . Gamma)^T Q + ((-dR Vres^T) . Gamma_m)^T P
//     dK = Diag(alpha) dP + Diag(eta) dKh,  d alpha|_P = rowsum(dP . K),
//     d eta = rowsum(dKh . K)
//   and the gates' gradients through the chunk coefficients (Gamma, its row
//   shift, abar, b, their shifted copies, mu_tail and the chunk totals): each
//   coefficient is a sum of products in which a gate appears at most once,
//   and its partial with respect to a gate is the product of the factors on
//   either side of it.  The sums over Gamma's index triangle follow one-step
//   recurrences along each row (O(C^2) per chunk, no division by a gate, so
//   mu = 0 is exact).
//
// fp32 inputs, three kernels after the packed-offset kernel:
//   bwd_prep   (chunk, head)            coefficients, Grams, T, A -> workspace
//   bwd_chain  (sequence, head, 32 cols) the reverse chain; dV; every chunk's
//                                       end adjoints -> workspace
//   bwd_chunk  (chunk, head)            the state products in 32-column slabs,
//                                       then dQ, dK and the gate gradients
// bf16 inputs: the forward's tensor-core prep (T, A_O T), bwd_vec (Gamma and
// the vectors), the reverse chain and the chunk products on the tensor cores
// (mdn_bwd_tc.cu, mdn_bwd_chunk_tc.cu), then bwd_gates (the gate gradients
// through the coefficients, as at the end of bwd_chunk).
#include <type_traits>

#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

constexpr int C = kChunk;
constexpr int LP = C + 1;       // padded row stride of 64 x 64 fp32 tiles
constexpr int NSB = 32;         // state columns per chain CTA / per slab
constexpr int LS = NSB + 1;     // padded row stride of 32-column tiles
using BL = BwdLayout;

__device__ __forceinline__ float *bwd_block(const BwdProblem &p, int slot, int h) {
    return reinterpret_cast<float *>(p.prep + ((size_t)slot * p.loc.H + h) * BL::kBytes);
}

template <typename T>
__device__ __forceinline__ T cvt_out(float x) { return from_f32<T>(x); }

// ------------------------------------------------------------------ prep

template <int D>
struct PrepBwdSmem {
    static constexpr int LD = D + 1;
    static constexpr int kFloats = 2 * C * LD + 4 * C * LP + 4 * C + BL::kRows * C;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int D, typename Tin>
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const BwdProblem p) {
    constexpr int LD = D + 1;
    extern __shared__ float sm[];
    float *Kf = sm, *Qf = Kf + C * LD;
    float *G = Qf + C * LD, *X = G + C * LP, *Y = X + C * LP, *Tm = Y + C * LP;
    float *ga = Tm + C * LP, *gm = ga + C, *ge = gm + C, *gb = ge + C, *vec = gb + C;

    int gc, h;
    chunk_head_of_block(p.loc.H, gc, h);
    const int tid = threadIdx.x;
    ChunkLoc loc;
    if (!locate_chunk_cta(p.loc, gc, loc)) return;
    const int n = loc.n, H = p.loc.H;
    if (tid < C) {
        float a = 1.f, m = 0.f, e = 0.f, b = 0.f;
        if (tid < n) {
            const size_t gi = (size_t)(loc.t0 + tid) * H + h;
            a = p.alpha[gi];
            m = p.mu[gi];
            e = p.eta[gi];
            b = p.beta ? p.beta[gi] : 1.f;
        }
        ga[tid] = a; gm[tid] = m; ge[tid] = e; gb[tid] = b;
    }
    const Tin *kg = static_cast<const Tin *>(p.k), *qg = static_cast<const Tin *>(p.q);
    for (int idx = tid; idx < C * D; idx += blockDim.x) {
        const int i = idx / D, c = idx - i * D;
        float kv = 0.f, qv = 0.f;
        if (i < n) {
            const size_t g = ((size_t)(loc.t0 + i) * H + h) * D + c;
            kv = to_f32(kg[g]);
            qv = to_f32(qg[g]);
        }
        Kf[i * LD + c] = kv;
        Qf[i * LD + c] = qv;
    }
    __syncthreads();

    if (tid < C) {
        // column j of Gamma by its recurrence: Gamma_{j,j} = beta_j,
        // Gamma_{i,j} = alpha_i Gamma_{i-1,j} + beta_i prod_{u=j+1}^{i} mu_u
        const int j = tid;
        float g = 0.f, mm = 1.f;
        for (int i = 0; i < C; ++i) {
            float out = 0.f;
            if (i >= j && i < n) {
                mm = (i == j) ? 1.f : mm * gm[i];
                g = (i == j) ? gb[i] : ga[i] * g + gb[i] * mm;
                out = g;
            }
            G[i * LP + j] = out;
        }
        float mt = 1.f;                         // mu_tail_j = prod_{u=j+1}^{n-1} mu_u
        for (int u = j + 1; u < n; ++u) mt *= gm[u];
        vec[BL::vMuTail * C + j] = j < n ? mt : 0.f;
    } else if (tid == C) {
        // abar, b (the origin's column: b_i = alpha_i b_{i-1} + beta_i mubar_i),
        // their one-row shifts and the chunk totals
        float ab = 1.f, bb = 0.f, mub = 1.f;
        for (int i = 0; i < C; ++i) {
            const float abm = ab, bm = bb;
            if (i < n) {
                ab *= ga[i];
                mub *= gm[i];
                bb = ga[i] * bb + gb[i] * mub;
            }
            const bool in = i < n;
            vec[BL::vAbarM * C + i] = in ? abm : 0.f;
            vec[BL::vBM * C + i] = in ? bm : 0.f;
            vec[BL::vAbar * C + i] = in ? ab : 0.f;
            vec[BL::vB * C + i] = in ? bb : 0.f;
        }
        vec[BL::vScal * C + 0] = ab;
        vec[BL::vScal * C + 1] = bb;
        vec[BL::vScal * C + 2] = mub;
        vec[BL::vScal * C + 3] = (float)n;
        for (int i = 4; i < C; ++i) vec[BL::vScal * C + i] = 0.f;
    }
    // X = P Kh^T (X_ij = alpha_i eta_j (K K^T)_ij), Y = Q Kh^T
    {
        const int i = tid >> 2, jq = tid & 3;
        float xk[16], yq[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) xk[jj] = yq[jj] = 0.f;
        for (int c = 0; c < D; ++c) {
            const float ki = Kf[i * LD + c], qi = Qf[i * LD + c];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const float kj = Kf[(jq + 4 * jj) * LD + c];
                xk[jj] = fmaf(ki, kj, xk[jj]);
                yq[jj] = fmaf(qi, kj, yq[jj]);
            }
        }
        __syncthreads();      // the gates above are read below
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int j = jq + 4 * jj;
            X[i * LP + j] = ga[i] * ge[j] * xk[jj];
            Y[i * LP + j] = ge[j] * yq[jj];
        }
    }
    __syncthreads();
    if (tid < C) {
        const int j = tid;
        vec[BL::vGS * C + j] = j < n ? G[(n - 1) * LP + j] : 0.f;
        // column c = j of T = (I + L)^{-1}, L_{r,k} = X_{r,k} Gamma_{r-1,k} (k < r)
        const int c = j;
        for (int r = 0; r < C; ++r) {
            float t;
            if (r < c) {
                t = 0.f;
            } else if (r == c) {
                t = 1.f;
            } else {
                float s = 0.f;
                for (int k = c; k < r; ++k) s = fmaf(X[r * LP + k] * G[(r - 1) * LP + k], Tm[k * LP + c], s);
                t = -s;
            }
            Tm[r * LP + c] = t;
        }
    }
    __syncthreads();
    float *blk = bwd_block(p, gc, h);
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int i = idx >> 6, j = idx & 63;
        blk[BL::kT * BL::kMat + idx] = Tm[i * LP + j];
        blk[BL::kA * BL::kMat + idx] = Y[i * LP + j] * G[i * LP + j];
        blk[BL::kX * BL::kMat + idx] = X[i * LP + j];
        blk[BL::kY * BL::kMat + idx] = Y[i * LP + j];
        blk[BL::kG * BL::kMat + idx] = G[i * LP + j];
    }
    for (int idx = tid; idx < BL::kRows * C; idx += blockDim.x)
        blk[BL::kMats * BL::kMat + idx] = idx < 7 * C ? vec[idx] : 0.f;
}

// The coefficients of the tensor-core gradient (bf16 inputs), whose matrices
// T and A_O T come from the forward's tensor-core prep: Gamma and the vector
// rows into the gradient block, and the reverse chain's per-token
// coefficients into the operand block, over the forward's carry vectors.
__global__ void __launch_bounds__(128)
bwd_vec_kernel(const BwdProblem p) {
    using CL = BwdChainLayout;
    __shared__ float ga[C], gm[C], ge[C], gb[C], vec[BL::kRows * C];
    int gc, h;
    chunk_head_of_block(p.loc.H, gc, h);
    const int tid = threadIdx.x, H = p.loc.H;
    ChunkLoc loc;
    if (!locate_chunk_cta(p.loc, gc, loc)) return;
    const int n = loc.n;
    if (tid < C) {
        float a = 1.f, m = 0.f, e = 0.f, b = 0.f;
        if (tid < n) {
            const size_t gi = (size_t)(loc.t0 + tid) * H + h;
            a = p.alpha[gi];
            m = p.mu[gi];
            e = p.eta[gi];
            b = p.beta ? p.beta[gi] : 1.f;
        }
        ga[tid] = a; gm[tid] = m; ge[tid] = e; gb[tid] = b;
    }
    __syncthreads();
    float *blk = bwd_block(p, gc, h);
    if (tid < C) {
        // column j of Gamma by its recurrence (as in the prep above), its
        // last row gS and mu_tail_j
        const int j = tid;
        float *G = blk + BL::kG * BL::kMat;
        float g = 0.f, mm = 1.f, gl = 0.f;
        for (int i = 0; i < C; ++i) {
            float out = 0.f;
            if (i >= j && i < n) {
                mm = (i == j) ? 1.f : mm * gm[i];
                g = (i == j) ? gb[i] : ga[i] * g + gb[i] * mm;
                out = g;
                if (i == n - 1) gl = g;
            }
            G[i * C + j] = out;
        }
        float mt = 1.f;
        for (int u = j + 1; u < n; ++u) mt *= gm[u];
        vec[BL::vGS * C + j] = j < n ? gl : 0.f;
        vec[BL::vMuTail * C + j] = j < n ? mt : 0.f;
    } else if (tid == C) {
        float ab = 1.f, bb = 0.f, mub = 1.f;
        for (int i = 0; i < C; ++i) {
            const float abm = ab, bm = bb;
            if (i < n) {
                ab *= ga[i];
                mub *= gm[i];
                bb = ga[i] * bb + gb[i] * mub;
            }
            const bool in = i < n;
            vec[BL::vAbarM * C + i] = in ? abm : 0.f;
            vec[BL::vBM * C + i] = in ? bm : 0.f;
            vec[BL::vAbar * C + i] = in ? ab : 0.f;
            vec[BL::vB * C + i] = in ? bb : 0.f;
        }
        vec[BL::vScal * C + 0] = ab;
        vec[BL::vScal * C + 1] = bb;
        vec[BL::vScal * C + 2] = mub;
        vec[BL::vScal * C + 3] = (float)n;
        for (int i = 4; i < C; ++i) vec[BL::vScal * C + i] = 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < BL::kRows * C; idx += blockDim.x)
        blk[BL::kMats * BL::kMat + idx] = idx < 7 * C ? vec[idx] : 0.f;
    if (tid < C) {
        const int t = tid;
        const bool in = t < n;
        float *cv = reinterpret_cast<float *>(p.tcblk + ((size_t)gc * H + h) * CL::kBytes + CL::kOffVec);
        cv[CL::vCS * C + t] = in ? vec[BL::vGS * C + t] * ge[t] : 0.f;
        cv[CL::vCM * C + t] = in ? -vec[BL::vMuTail * C + t] * ge[t] : 0.f;
        cv[CL::vBS * C + t] = in ? -vec[BL::vAbarM * C + t] * ga[t] : 0.f;
        cv[CL::vBM * C + t] = in ? vec[BL::vBM * C + t] * ga[t] : 0.f;
        cv[CL::vQS * C + t] = in ? vec[BL::vAbar * C + t] : 0.f;
        cv[CL::vQM * C + t] = in ? -vec[BL::vB * C + t] : 0.f;
        cv[CL::vScal * C + t] = t < 4 ? vec[BL::vScal * C + t] : 0.f;
        cv[7 * C + t] = 0.f;
    }
}

// ------------------------------------------------------------------ chain

template <int D>
struct ChainSmem {
    static constexpr int LD = D + 1;
    static constexpr int kFloats = 2 * D * LS + 2 * C * LD + 2 * C * LP + 3 * C * LS +
                                   BL::kRows * C + 2 * C;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

// Loads the chunk's K and Q rows (zero past n) as fp32.
template <int D, typename Tin>
__device__ __forceinline__ void load_kq(const BwdProblem &p, int t0, int n, int h, float *Kf,
                                        float *Qf) {
    constexpr int LD = D + 1;
    const Tin *kg = static_cast<const Tin *>(p.k), *qg = static_cast<const Tin *>(p.q);
    for (int idx = threadIdx.x; idx < C * D; idx += blockDim.x) {
        const int i = idx / D, c = idx - i * D;
        float kv = 0.f, qv = 0.f;
        if (i < n) {
            const size_t g = ((size_t)(t0 + i) * p.loc.H + h) * D + c;
            kv = to_f32(kg[g]);
            qv = to_f32(qg[g]);
        }
        Kf[i * LD + c] = kv;
        Qf[i * LD + c] = qv;
    }
}

template <int D, typename Tin>
__global__ void __launch_bounds__(512, 1)
bwd_chain_kernel(const BwdProblem p) {
    constexpr int LD = D + 1, kSlices = D / NSB;
    constexpr int kJ = D * NSB / 512;           // state entries per thread in the update
    constexpr int kTpr = NSB / kJ;              // threads per state row
    extern __shared__ float sm[];
    float *dS = sm, *dM = dS + D * LS;
    float *Kf = dM + D * LS, *Qf = Kf + C * LD;
    float *Tm = Qf + C * LD, *Am = Tm + C * LP;
    float *dO = Am + C * LP, *dV = dO + C * LS, *dRs = dV + C * LS;
    float *vec = dRs + C * LS, *ga = vec + BL::kRows * C, *ge = ga + C;

    const int tid = threadIdx.x, H = p.loc.H;
    const int slice = blockIdx.x % kSlices, kh = blockIdx.x / kSlices;
    const int s = ordered_sequence(p.loc, kh / H), h = kh % H;
    const int col0 = slice * NSB;
    int start, len, slot0;
    sequence_range(p.loc, s, start, len, slot0);
    const int nch = (len + C - 1) / C;
    const size_t st_off = ((size_t)s * H + h) * D * D;
    for (int idx = tid; idx < D * NSB; idx += blockDim.x) {
        const int k = idx / NSB, j = idx - k * NSB;
        const size_t g = st_off + (size_t)k * D + col0 + j;
        dS[k * LS + j] = p.dS_T ? p.dS_T[g] : 0.f;
        dM[k * LS + j] = p.dM_T ? p.dM_T[g] : 0.f;
    }
    const Tin *dog = static_cast<const Tin *>(p.dout);
    Tin *dvg = static_cast<Tin *>(p.dv);
    for (int c = nch - 1; c >= 0; --c) {
        const int slot = slot0 + c, t0 = start + c * C, n = min(C, len - c * C);
        const float *blk = bwd_block(p, slot, h);
        __syncthreads();                    // the previous chunk is done with every tile
        load_kq<D, Tin>(p, t0, n, h, Kf, Qf);
        for (int idx = tid; idx < C * C; idx += blockDim.x) {
            const int i = idx >> 6, j = idx & 63;
            Tm[i * LP + j] = blk[BL::kT * BL::kMat + idx];
            Am[i * LP + j] = blk[BL::kA * BL::kMat + idx];
        }
        for (int idx = tid; idx < BL::kRows * C; idx += blockDim.x)
            vec[idx] = blk[BL::kMats * BL::kMat + idx];
        for (int idx = tid; idx < C * NSB; idx += blockDim.x) {
            const int i = idx / NSB, j = idx - i * NSB;
            dO[i * LS + j] = i < n ? to_f32(dog[((size_t)(t0 + i) * H + h) * D + col0 + j]) : 0.f;
        }
        if (tid < C) {
            const size_t gi = (size_t)(t0 + tid) * H + h;
            ga[tid] = tid < n ? p.alpha[gi] : 0.f;
            ge[tid] = tid < n ? p.eta[gi] : 0.f;
        }
        // the adjoints at this chunk's end, for the chunk kernel
        float *adj = p.adj + ((size_t)slot * H + h) * 2 * D * D;
        for (int idx = tid; idx < D * NSB; idx += blockDim.x) {
            const int k = idx / NSB, j = idx - k * NSB;
            adj[(size_t)k * D + col0 + j] = dS[k * LS + j];
            adj[(size_t)D * D + (size_t)k * D + col0 + j] = dM[k * LS + j];
        }
        __syncthreads();
        // dVres = WS dS - WM dM + A^T dO
        {
            const int t = tid >> 3, jq = tid & 7;
            float xs[4] = {0.f, 0.f, 0.f, 0.f}, xm[4] = {0.f, 0.f, 0.f, 0.f}, xa[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < D; ++k) {
                const float kt = Kf[t * LD + k];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    xs[jj] = fmaf(kt, dS[k * LS + jq + 8 * jj], xs[jj]);
                    xm[jj] = fmaf(kt, dM[k * LS + jq + 8 * jj], xm[jj]);
                }
            }
            for (int i = 0; i < C; ++i) {
                const float a_it = Am[i * LP + t];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) xa[jj] = fmaf(a_it, dO[i * LS + jq + 8 * jj], xa[jj]);
            }
            const float ws = vec[BL::vGS * C + t] * ge[t], wm = vec[BL::vMuTail * C + t] * ge[t];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                dV[t * LS + jq + 8 * jj] = t < n ? ws * xs[jj] - wm * xm[jj] + xa[jj] : 0.f;
        }
        __syncthreads();
        // dR = T^T dVres (= dV of the inputs)
        {
            const int t = tid >> 3, jq = tid & 7;
            float xr[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = 0; i < C; ++i) {
                const float tt = Tm[i * LP + t];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) xr[jj] = fmaf(tt, dV[i * LS + jq + 8 * jj], xr[jj]);
            }
            float *dRg = p.dR + ((size_t)slot * H + h) * C * D;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = jq + 8 * jj;
                const float r = t < n ? xr[jj] : 0.f;
                dRs[t * LS + j] = r;
                if (t < n) {
                    dRg[(size_t)t * D + col0 + j] = r;
                    dvg[((size_t)(t0 + t) * H + h) * D + col0 + j] = cvt_out<Tin>(r);
                }
            }
        }
        __syncthreads();
        // the adjoints at the chunk's start
        {
            const int k = tid / kTpr, jq = tid - k * kTpr;
            float cS[kJ], cM[kJ];
#pragma unroll
            for (int jj = 0; jj < kJ; ++jj) cS[jj] = cM[jj] = 0.f;
            for (int t = 0; t < C; ++t) {
                const float q = Qf[t * LD + k], kk = Kf[t * LD + k] * ga[t];
                const float qa = vec[BL::vAbar * C + t] * q, qb = vec[BL::vB * C + t] * q;
                const float pa = vec[BL::vAbarM * C + t] * kk, pb = vec[BL::vBM * C + t] * kk;
#pragma unroll
                for (int jj = 0; jj < kJ; ++jj) {
                    const int j = jq + kTpr * jj;
                    const float o = dO[t * LS + j], r = dRs[t * LS + j];
                    cS[jj] = fmaf(qa, o, fmaf(-pa, r, cS[jj]));
                    cM[jj] = fmaf(-qb, o, fmaf(pb, r, cM[jj]));
                }
            }
            const float abn = vec[BL::vScal * C + 0], bn = vec[BL::vScal * C + 1];
            const float mbn = vec[BL::vScal * C + 2];
#pragma unroll
            for (int jj = 0; jj < kJ; ++jj) {
                const int j = jq + kTpr * jj;
                const float so = dS[k * LS + j], mo = dM[k * LS + j];
                dS[k * LS + j] = abn * so + cS[jj];
                dM[k * LS + j] = mbn * mo - bn * so + cM[jj];
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < D * NSB; idx += blockDim.x) {
        const int k = idx / NSB, j = idx - k * NSB;
        const size_t g = st_off + (size_t)k * D + col0 + j;
        if (p.dS0) p.dS0[g] = dS[k * LS + j];
        if (p.dM0) p.dM0[g] = dM[k * LS + j];
    }
}

// ------------------------------------------------------------------ chunk

// Row sums the slab phase accumulates per token row i (indices into rowacc).
enum { rAbar = 0, rB, rAbarM, rBM, rGLast, rMuTail, kRowAcc = 8 };

// The gates' gradients through the chunk coefficients, from dG (the adjoint
// of Gamma with the row-shifted copy's folded in, rows < n, C x LP; F
// replaces it in place), the per-row sums `rowacc` (kRowAcc rows), the
// adjoints of the chunk totals dcs = (d abar_n, d b_n, d mubar_n) and the
// chunk's vectors abar_{i-1} and mu_tail_i.  The products A(r, i) =
// prod_{u=r+1}^{i} alpha_u are formed as running products along the loops.
// `scr` holds kGateScratch floats: I and G' (C rows of LP floats, so that a
// warp's threads walking rows or columns hit distinct banks) and two
// vectors.  Every thread of a CTA of at least 128 threads takes part;
// writes dalpha, dmu, deta and dbeta of the chunk's tokens.
constexpr int kGateScratch = 2 * C * LP + 2 * C;

__device__ void gate_gradients(const BwdProblem &p, int t0, int n, int h, float *dGF, float *scr,
                               const float *ga, const float *gm, const float *gb,
                               const float *rowacc, const float *dcs, const float *abar_m,
                               const float *mu_tail) {
    const int tid = threadIdx.x, H = p.loc.H;
    float *Im = scr, *Gg = Im + C * LP;
    float *dab = Gg + C * LP, *Tl = dab + C;
    if (tid < C) {
        const int r = tid;                       // row r of the triangle
        // the folded vector adjoints: d abar_r plus the shifted copy's (at
        // r + 1) and the chunk total's (at n - 1); d b_r likewise
        float va = 0.f, vb = 0.f;
        if (r < n) {
            va = rowacc[rAbar * C + r];
            vb = rowacc[rB * C + r];
            if (r + 1 < n) {
                va += rowacc[rAbarM * C + r + 1];
                vb += rowacc[rBM * C + r + 1];
            }
            if (r == n - 1) {
                va += dcs[0];
                vb += dcs[1];
            }
        }
        dab[r] = va;
        // F[r, m + 1] = mu_m F[r, m] + dG[r, m], F[r, 0] = db_r, over dG's row
        // (each dG entry is read before its slot is written)
        float *row = dGF + r * LP;
        float f = vb, nxt = row[0];
        row[0] = f;
        for (int m = 0; m < C; ++m) {
            const float cur = nxt;
            if (m + 1 < C) nxt = row[m + 1];
            f = (m <= r && r < n) ? gm[m] * f + cur : 0.f;
            row[m + 1] = f;
        }
    } else if (tid == C) {
        // Tl_u = sum_{j<u} dmu_tail_j Mu(j, u-1), started from d mubar_n
        float tl = dcs[2];
        for (int u = 0; u < C; ++u) {
            Tl[u] = tl;
            if (u < n) tl = gm[u] * tl + rowacc[rMuTail * C + u];
        }
    }
    __syncthreads();
    const float *Fm = dGF;
    if (tid < C) {
        // I[r, u] = sum_{v<u} beta_v A(v, u-1) F[r, v+1] (alpha's inner sum)
        const int r = tid;
        float inner = 0.f;
        for (int u = 0; u < C; ++u) {
            const bool in = u <= r && r < n;
            Im[r * LP + u] = in ? inner : 0.f;
            if (in) inner = ga[u] * inner + gb[u] * Fm[r * LP + u + 1];
        }
    } else if (tid < 2 * C) {
        // G'[r, u] = sum_{v=u}^{r} beta_v A(v, r) Mu(u, v) (mu's), u = r .. 0,
        // with the running product P = A(u - 1, r) = prod_{w=u}^{r} alpha_w
        const int r = tid - C;
        float g = r < n ? gb[r] : 0.f, P = 1.f;
        for (int u = C - 1; u >= 0; --u) {
            if (u <= r && r < n) {
                Gg[r * LP + u] = g;
                P *= ga[u];
                if (u > 0) g = gb[u - 1] * P + gm[u] * g;
            } else {
                Gg[r * LP + u] = 0.f;
            }
        }
    }
    __syncthreads();
    if (tid < n) {
        const int u = tid;
        float db = 0.f, dal = 0.f, dmu = 0.f, Aur = 1.f;    // A(u, r), r = u first
        const float a_prev = abar_m[u];                      // A(-1, u-1)
        for (int r = u; r < n; ++r) {
            if (r > u) Aur *= ga[r];
            db = fmaf(Aur, Fm[r * LP + u + 1], db);
            dal = fmaf(Aur, Im[r * LP + u] + dab[r] * a_prev, dal);
            dmu = fmaf(Fm[r * LP + u], Gg[r * LP + u], dmu);
        }
        dmu = fmaf(Tl[u], mu_tail[u], dmu);                  // Mu(u, n-1)
        const size_t gi = (size_t)(t0 + u) * H + h;
        p.dalpha[gi] = rowacc[6 * C + u] + dal;
        p.dmu[gi] = dmu;
        p.deta[gi] = rowacc[7 * C + u];
        if (p.dbeta) p.dbeta[gi] = db;
    }
}

template <int D>
struct ChunkSmem {
    static constexpr int LD = D + 1;
    static constexpr int kSlab = 4 * D * LS + 4 * C * LS;
    static constexpr int kPh4 = 5 * C * LP;
    static constexpr int kPh5 = C * LP + kGateScratch;
    static constexpr int kUnion = kSlab > kPh4 ? (kSlab > kPh5 ? kSlab : kPh5) : (kPh4 > kPh5 ? kPh4 : kPh5);
    static constexpr int kFloats = 2 * C * LD + C * LP + BL::kRows * C + 4 * C + kRowAcc * C +
                                   16 * 4 + kUnion;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int D, typename Tin>
__global__ void __launch_bounds__(512, 1)
bwd_chunk_kernel(const BwdProblem p) {
    constexpr int LD = D + 1;
    constexpr int kKK = D / 8;                  // state rows per thread (k = q8 + 8 kk)
    extern __shared__ float sm[];
    float *Kf = sm, *Qf = Kf + C * LD, *Tm = Qf + C * LD;
    float *vec = Tm + C * LP, *ga = vec + BL::kRows * C, *gm = ga + C, *ge = gm + C, *gb = ge + C;
    float *rowacc = gb + C, *red = rowacc + kRowAcc * C, *U = red + 16 * 4;
    // slab phase
    float *S0s = U, *M0s = S0s + D * LS, *dSs = M0s + D * LS, *dMs = dSs + D * LS;
    float *Vs = dMs + D * LS, *dOs = Vs + C * LS, *dRs = dOs + C * LS, *Rs = dRs + C * LS;

    int gc, h;
    chunk_head_of_block(p.loc.H, gc, h);
    const int tid = threadIdx.x, H = p.loc.H;
    ChunkLoc loc;
    if (!locate_chunk_cta(p.loc, gc, loc)) return;
    const int n = loc.n, t0 = loc.t0;
    const float *blk = bwd_block(p, gc, h);
    load_kq<D, Tin>(p, t0, n, h, Kf, Qf);
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int i = idx >> 6, j = idx & 63;
        Tm[i * LP + j] = blk[BL::kT * BL::kMat + idx];
    }
    for (int idx = tid; idx < BL::kRows * C; idx += blockDim.x) vec[idx] = blk[BL::kMats * BL::kMat + idx];
    if (tid < C) {
        float a = 0.f, m = 0.f, e = 0.f, b = 0.f;
        if (tid < n) {
            const size_t gi = (size_t)(t0 + tid) * H + h;
            a = p.alpha[gi];
            m = p.mu[gi];
            e = p.eta[gi];
            b = p.beta ? p.beta[gi] : 1.f;
        }
        ga[tid] = a; gm[tid] = m; ge[tid] = e; gb[tid] = b;
    }
    __syncthreads();

    const int i = tid >> 3, q8 = tid & 7;
    const float a_i = ga[i], e_i = ge[i];
    const float abar_i = vec[BL::vAbar * C + i], b_i = vec[BL::vB * C + i];
    const float abm_i = vec[BL::vAbarM * C + i], bm_i = vec[BL::vBM * C + i];
    const float gs_i = vec[BL::vGS * C + i], mt_i = vec[BL::vMuTail * C + i];
    float dQs[kKK], dPs[kKK], dKc[kKK], dA[8], dL[8];
#pragma unroll
    for (int kk = 0; kk < kKK; ++kk) dQs[kk] = dPs[kk] = dKc[kk] = 0.f;
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) dA[mm] = dL[mm] = 0.f;
    float racc[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float sc[3] = {0.f, 0.f, 0.f};      // <S0, dS>, <M0, dS>, <M0, dM>

    const size_t sbase = ((size_t)gc * H + h) * D * D;
    const float *adj = p.adj + ((size_t)gc * H + h) * 2 * D * D;
    const float *dRg = p.dR + ((size_t)gc * H + h) * C * D;
    const Tin *vg = static_cast<const Tin *>(p.v), *dog = static_cast<const Tin *>(p.dout);
    for (int c0 = 0; c0 < D; c0 += NSB) {
        __syncthreads();
        for (int idx = tid; idx < D * NSB; idx += blockDim.x) {
            const int k = idx / NSB, j = idx - k * NSB;
            const size_t g = (size_t)k * D + c0 + j;
            const float s0 = static_cast<const float *>(p.S_chunks)[sbase + g];
            const float m0 = static_cast<const float *>(p.M_chunks)[sbase + g];
            const float ds = adj[g], dm = adj[(size_t)D * D + g];
            S0s[k * LS + j] = s0;
            M0s[k * LS + j] = m0;
            dSs[k * LS + j] = ds;
            dMs[k * LS + j] = dm;
            sc[0] = fmaf(s0, ds, sc[0]);
            sc[1] = fmaf(m0, ds, sc[1]);
            sc[2] = fmaf(m0, dm, sc[2]);
        }
        for (int idx = tid; idx < C * NSB; idx += blockDim.x) {
            const int r = idx / NSB, j = idx - r * NSB;
            const bool in = r < n;
            const size_t g = ((size_t)(t0 + r) * H + h) * D + c0 + j;
            Vs[r * LS + j] = in ? to_f32(vg[g]) : 0.f;
            dOs[r * LS + j] = in ? to_f32(dog[g]) : 0.f;
            dRs[r * LS + j] = in ? dRg[(size_t)r * D + c0 + j] : 0.f;
        }
        __syncthreads();
        // P S0, P M0, Q S0, Q M0, Kh dS, Kh dM for (i, j = q8 + 8 jj); R
        float kds[4], kdm[4];
        {
            float ps[4], pm[4], qs[4], qm[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) ps[jj] = pm[jj] = qs[jj] = qm[jj] = kds[jj] = kdm[jj] = 0.f;
            for (int k = 0; k < D; ++k) {
                const float kv = Kf[i * LD + k], qv = Qf[i * LD + k];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = q8 + 8 * jj;
                    const float s0 = S0s[k * LS + j], m0 = M0s[k * LS + j];
                    const float ds = dSs[k * LS + j], dm = dMs[k * LS + j];
                    ps[jj] = fmaf(kv, s0, ps[jj]);
                    pm[jj] = fmaf(kv, m0, pm[jj]);
                    qs[jj] = fmaf(qv, s0, qs[jj]);
                    qm[jj] = fmaf(qv, m0, qm[jj]);
                    kds[jj] = fmaf(kv, ds, kds[jj]);
                    kdm[jj] = fmaf(kv, dm, kdm[jj]);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = q8 + 8 * jj;
                const float PS = a_i * ps[jj], PM = a_i * pm[jj];
                const float o = dOs[i * LS + j], r = dRs[i * LS + j];
                Rs[i * LS + j] = Vs[i * LS + j] - abm_i * PS + bm_i * PM;
                racc[rAbar] = fmaf(qs[jj], o, racc[rAbar]);
                racc[rB] = fmaf(-qm[jj], o, racc[rB]);
                racc[rAbarM] = fmaf(-r, PS, racc[rAbarM]);
                racc[rBM] = fmaf(r, PM, racc[rBM]);
                kds[jj] *= e_i;
                kdm[jj] *= e_i;
            }
        }
        __syncthreads();
        // Vres = T R (overwrites V)
        {
            float vr[4] = {0.f, 0.f, 0.f, 0.f};
            for (int m = 0; m < C; ++m) {
                const float tt = Tm[i * LP + m];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) vr[jj] = fmaf(tt, Rs[m * LS + q8 + 8 * jj], vr[jj]);
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                Vs[i * LS + q8 + 8 * jj] = vr[jj];
                racc[rGLast] = fmaf(vr[jj], kds[jj], racc[rGLast]);
                racc[rMuTail] = fmaf(-vr[jj], kdm[jj], racc[rMuTail]);
            }
        }
        __syncthreads();
        // the slab's share of the n x dk products and of dO Vres^T, -dR Vres^T
        for (int j = 0; j < NSB; ++j) {
            const float o = dOs[i * LS + j], r = dRs[i * LS + j], vr = Vs[i * LS + j];
            const float oa = o * abar_i, ob = o * b_i, ra = r * abm_i, rb = r * bm_i;
            const float vs = vr * gs_i, vm = vr * mt_i;
#pragma unroll
            for (int kk = 0; kk < kKK; ++kk) {
                const int k = q8 + 8 * kk;
                const float s0 = S0s[k * LS + j], m0 = M0s[k * LS + j];
                const float ds = dSs[k * LS + j], dm = dMs[k * LS + j];
                dQs[kk] = fmaf(oa, s0, fmaf(-ob, m0, dQs[kk]));
                dPs[kk] = fmaf(-ra, s0, fmaf(rb, m0, dPs[kk]));
                dKc[kk] = fmaf(vs, ds, fmaf(-vm, dm, dKc[kk]));
            }
#pragma unroll
            for (int mm = 0; mm < 8; ++mm) {
                const float v_m = Vs[(q8 + 8 * mm) * LS + j];
                dA[mm] = fmaf(o, v_m, dA[mm]);
                dL[mm] = fmaf(-r, v_m, dL[mm]);
            }
        }
    }
    // row sums over the eight threads of a row (consecutive lanes)
#pragma unroll
    for (int a = 0; a < 6; ++a) {
        float x = racc[a];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        racc[a] = x;
    }
    if (q8 == 0)
#pragma unroll
        for (int a = 0; a < 6; ++a) rowacc[a * C + i] = racc[a];
    // the three scalar sums: warp sums, then a fixed-order block sum
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        float x = sc[a];
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        sc[a] = x;
    }
    if ((tid & 31) == 0)
        for (int a = 0; a < 3; ++a) red[(tid >> 5) * 4 + a] = sc[a];
    __syncthreads();
    // ---- phase 4: dQ, dK and the coefficient adjoints
    float *G = U, *X = G + C * LP, *Y = X + C * LP, *dAm = Y + C * LP, *dLm = dAm + C * LP;
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int r = idx >> 6, j = idx & 63;
        G[r * LP + j] = blk[BL::kG * BL::kMat + idx];
        X[r * LP + j] = blk[BL::kX * BL::kMat + idx];
        Y[r * LP + j] = blk[BL::kY * BL::kMat + idx];
    }
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) {
        dAm[i * LP + q8 + 8 * mm] = dA[mm];
        dLm[i * LP + q8 + 8 * mm] = dL[mm];
    }
    __syncthreads();
    float dcs[3] = {0.f, 0.f, 0.f};       // d abar_n, d b_n, d mubar_n
    for (int w = 0; w < 16; ++w) {
        dcs[0] += red[w * 4 + 0];
        dcs[1] -= red[w * 4 + 1];
        dcs[2] += red[w * 4 + 2];
    }
    {
        // dY = dA . Gamma (row i), dX = dL . Gamma_m;  dQ = dQs + dY Kh,
        // dP = dPs + dX Kh, dKh = dKc + dY^T Q + dX^T P
        float dq[kKK], dp[kKK], dkh[kKK];
#pragma unroll
        for (int kk = 0; kk < kKK; ++kk) { dq[kk] = dQs[kk]; dp[kk] = dPs[kk]; dkh[kk] = dKc[kk]; }
        for (int m = 0; m < C; ++m) {
            const float dy_im = dAm[i * LP + m] * G[i * LP + m] * ge[m];
            const float dx_im = (m < i && i > 0) ? dLm[i * LP + m] * G[(i - 1) * LP + m] * ge[m] : 0.f;
            const float dy_mi = dAm[m * LP + i] * G[m * LP + i];
            const float dx_mi = (i < m) ? dLm[m * LP + i] * G[(m - 1) * LP + i] * ga[m] : 0.f;
#pragma unroll
            for (int kk = 0; kk < kKK; ++kk) {
                const int k = q8 + 8 * kk;
                const float km = Kf[m * LD + k], qm = Qf[m * LD + k];
                dq[kk] = fmaf(dy_im, km, dq[kk]);
                dp[kk] = fmaf(dx_im, km, dp[kk]);
                dkh[kk] = fmaf(dy_mi, qm, fmaf(dx_mi, km, dkh[kk]));
            }
        }
        float da = 0.f, de = 0.f;
        Tin *dqg = static_cast<Tin *>(p.dq), *dkg = static_cast<Tin *>(p.dk);
        const size_t row = ((size_t)(t0 + i) * H + h) * D;
#pragma unroll
        for (int kk = 0; kk < kKK; ++kk) {
            const int k = q8 + 8 * kk;
            const float kv = Kf[i * LD + k];
            da = fmaf(dp[kk], kv, da);
            de = fmaf(dkh[kk], kv, de);
            if (i < n) {
                dqg[row + k] = cvt_out<Tin>(dq[kk]);
                dkg[row + k] = cvt_out<Tin>(a_i * dp[kk] + e_i * dkh[kk]);
            }
        }
        da += __shfl_xor_sync(0xffffffffu, da, 1);
        da += __shfl_xor_sync(0xffffffffu, da, 2);
        da += __shfl_xor_sync(0xffffffffu, da, 4);
        de += __shfl_xor_sync(0xffffffffu, de, 1);
        de += __shfl_xor_sync(0xffffffffu, de, 2);
        de += __shfl_xor_sync(0xffffffffu, de, 4);
        if (q8 == 0) {
            rowacc[6 * C + i] = da;
            rowacc[7 * C + i] = de;
        }
    }
    // dG = dA . Y (+ the carry row), with the row-shifted copy's adjoint
    // dL . X folded one row up (dG_{r,m} += dL_{r+1,m} X_{r+1,m}); it
    // replaces G, which the loop above was the last to read
    {
        float vals[8];
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            const int m = q8 + 8 * mm;
            float v = 0.f;
            if (i < n && m <= i) {
                v = dAm[i * LP + m] * Y[i * LP + m];
                if (i == n - 1) v += rowacc[rGLast * C + m];
                if (i + 1 < n) v += dLm[(i + 1) * LP + m] * X[(i + 1) * LP + m];
            }
            vals[mm] = v;
        }
        __syncthreads();
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) G[i * LP + q8 + 8 * mm] = vals[mm];
    }
    __syncthreads();
    // ---- phase 5: the gates through the coefficients
    gate_gradients(p, t0, n, h, G, U + C * LP, ga, gm, gb, rowacc, dcs, vec + BL::vAbarM * C,
                   vec + BL::vMuTail * C);
}

// ------------------------------------------------------------------ gates

// The gate stage after the tensor-core chunk kernel (bf16 inputs), which
// leaves per (slot, head), over matrices of the gradient block it no longer
// needs: dA . Y in the Y slot, dL . X in the X slot (rows < n; the lower
// triangle), and in the A slot the kRowAcc row sums followed by the three
// state inner products <S0, dS>, <M0, dS>, <M0, dM>.  The two products and
// the row sums arrive by bulk copy (the products into the scratch area the
// gate recurrences use later): plain loads of them would be capped by the
// little L1 left beside four CTAs' shared memory.
constexpr size_t kGateSmem = sizeof(float) * (C * LP + kGateScratch + 5 * C + kRowAcc * C) + 16;
constexpr int kGateThreads = 128;

__global__ void __launch_bounds__(kGateThreads)
bwd_gates_kernel(const BwdProblem p) {
    using namespace sm100;
    extern __shared__ float sm[];
    float *dG = sm, *scr = dG + C * LP;
    float *ga = scr + kGateScratch, *gm = ga + C, *gb = gm + C, *abm = gb + C, *mtl = abm + C;
    float *rowacc = mtl + C;
    uint64_t *cbar = reinterpret_cast<uint64_t *>(rowacc + kRowAcc * C);
    volatile int *abort = reinterpret_cast<volatile int *>(cbar + 1);
    int gc, h;
    chunk_head_of_block(p.loc.H, gc, h);
    const int tid = threadIdx.x, H = p.loc.H;
    ChunkLoc loc;
    if (!locate_chunk_cta(p.loc, gc, loc)) return;
    const int n = loc.n, t0 = loc.t0;
    const float *blk = bwd_block(p, gc, h);
    const float *ra = blk + BL::kA * BL::kMat;
    const float *vec = blk + BL::kMats * BL::kMat;
    float *W1 = scr, *W2 = scr + C * C;      // dA . Y and dL . X as copied
    if (tid == 0) {
        mbar_init(cbar, 1);
        *abort = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(cbar, 2 * C * C * 4 + kRowAcc * C * 4);
        bulk_load(W1, blk + BL::kY * BL::kMat, C * C * 4, cbar);
        bulk_load(W2, blk + BL::kX * BL::kMat, C * C * 4, cbar);
        bulk_load(rowacc, ra, kRowAcc * C * 4, cbar);
    }
    if (tid < C) {
        float a = 0.f, m = 0.f, b = 0.f;
        if (tid < n) {
            const size_t gi = (size_t)(t0 + tid) * H + h;
            a = p.alpha[gi];
            m = p.mu[gi];
            b = p.beta ? p.beta[gi] : 1.f;
        }
        ga[tid] = a; gm[tid] = m; gb[tid] = b;
        abm[tid] = vec[BL::vAbarM * C + tid];
        mtl[tid] = vec[BL::vMuTail * C + tid];
    }
    const float dcs[3] = {ra[kRowAcc * C + 0], -ra[kRowAcc * C + 1], ra[kRowAcc * C + 2]};
    __syncthreads();                         // the barrier is initialised
    // dG = dA . Y, plus the carry row on the last row, plus dL . X one row up
    if (mbar_wait(cbar, 0, abort)) {
        for (int idx = tid; idx < C * C; idx += kGateThreads) {
            const int r = idx >> 6, m = idx & 63;
            float v = 0.f;
            if (r < n && m <= r) {
                v = W1[idx];
                if (r + 1 < n) v += W2[idx + C];
                if (r == n - 1) v += rowacc[rGLast * C + m];
            }
            dG[r * LP + m] = v;
        }
    }
    __syncthreads();
    if (*abort) {
        if (tid == 0) {
            int dummy = 0;                   // the copies land before the CTA exits
            mbar_wait(cbar, 0, &dummy);
            if (p.loc.status) atomicExch(p.loc.status, (int)MDN_ERR_DEVICE_TIMEOUT);
        }
        return;
    }
    gate_gradients(p, t0, n, h, dG, scr, ga, gm, gb, rowacc, dcs, abm, mtl);
}

template <int D, typename Tin>
cudaError_t launch_bwd_t(const BwdProblem &p, cudaStream_t st) {
    const int H = p.loc.H;
    if (p.tcblk) {
        // bf16 inputs: the forward's tensor-core prep writes T and A_O T into
        // the operand blocks, the coefficient kernel Gamma and the vectors;
        // the reverse chain and the chunk products run on the tensor cores,
        // the gates' partials on the CUDA cores
        ChunkProblem fp = p.loc;
        fp.q = p.q;
        fp.k = p.k;
        fp.alpha = p.alpha; fp.mu = p.mu; fp.eta = p.eta; fp.beta = p.beta;
        fp.prep = p.tcblk;
        fp.prep_stride = BwdChainLayout::kBytes;
        dim3 cg;
        if (!chunk_head_grid(p.loc.max_chunks, H, cg)) return cudaErrorInvalidConfiguration;
        // (the forward's own blocks, when the caller kept them, already hold
        // the same tiles)
        cudaError_t err = p.fwd_tile ? cudaSuccess : launch_chunk_prep_tc(fp, st);
        if (err != cudaSuccess) return err;
        bwd_vec_kernel<<<cg, 128, 0, st>>>(p);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        if ((err = launch_bwd_chain_tc(p, st)) != cudaSuccess) return err;
        if ((err = launch_bwd_chunk_tc(p, st)) != cudaSuccess) return err;
        auto kg = bwd_gates_kernel;
        if ((err = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kGateSmem)) != cudaSuccess)
            return err;
        kg<<<cg, kGateThreads, kGateSmem, st>>>(p);
        return cudaGetLastError();
    }
    // fp32 inputs (bf16 inputs reach here only without tokens: the chain
    // alone passes the final-state adjoints through)
    constexpr bool kF32 = std::is_same<Tin, float>::value;
    if constexpr (kF32) {
        if (p.loc.max_chunks > 0) {
            auto kp = bwd_prep_kernel<D, Tin>;
            cudaError_t err = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)PrepBwdSmem<D>::kBytes);
            if (err != cudaSuccess) return err;
            dim3 cg;
            if (!chunk_head_grid(p.loc.max_chunks, H, cg)) return cudaErrorInvalidConfiguration;
            kp<<<cg, 256, PrepBwdSmem<D>::kBytes, st>>>(p);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
    } else if (p.loc.max_chunks > 0) {
        return cudaErrorInvalidValue;
    }
    {
        auto kc = bwd_chain_kernel<D, Tin>;
        cudaError_t err = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)ChainSmem<D>::kBytes);
        if (err != cudaSuccess) return err;
        const long blocks = (long)p.loc.n_seq * H * (D / NSB);
        if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
        if (blocks > 0) kc<<<(unsigned)blocks, 512, ChainSmem<D>::kBytes, st>>>(p);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if constexpr (kF32) {
        if (p.loc.max_chunks > 0) {
            auto kk = bwd_chunk_kernel<D, Tin>;
            cudaError_t err = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)ChunkSmem<D>::kBytes);
            if (err != cudaSuccess) return err;
            dim3 cg;
            if (!chunk_head_grid(p.loc.max_chunks, H, cg)) return cudaErrorInvalidConfiguration;
            kk<<<cg, 512, ChunkSmem<D>::kBytes, st>>>(p);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_chunk_bwd(const BwdProblem &p, cudaStream_t st) {
    if (p.D == 128)
        return p.dtype == MDN_BF16 ? launch_bwd_t<128, __nv_bfloat16>(p, st)
                                   : launch_bwd_t<128, float>(p, st);
    return p.dtype == MDN_BF16 ? launch_bwd_t<64, __nv_bfloat16>(p, st)
                               : launch_bwd_t<64, float>(p, st);
}

}  // namespace mdn
