// MDN decode step: one token per sequence, both states updated in place.
//
// The token recurrence of "MDN: Parallelizing Stepwise Momentum for Delta
// Linear Attention" (slides, "MDN adds a momentum matrix to the delta update",
// Eqs. (3)-(5); reading notes section 2.2):
//   vres = v - alpha S^T k;  M' = mu M - eta k vres^T;  S' = alpha S - beta M';
//   o = S'^T q.
//
// Memory-bound: every (sequence, head) reads and writes two dk x dv fp32
// states once.  One CTA owns a 32-column slice of one (sequence, head):
// column slices evolve independently because column j of S' and M' depends
// only on column j of S and M (vres_j reads column j of S).  Each thread
// keeps its rows of both states in registers between the two reductions, so
// HBM sees exactly one read and one write of every state element.
#include "mdn_internal.cuh"

namespace mdn {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecCols = 32;          // columns per CTA
constexpr int kColGroups = kDecCols / 4;   // float4 groups: 8
constexpr int kRowGroups = kDecThreads / kColGroups;  // 32

template <int D, typename Tin>
__global__ void __launch_bounds__(kDecThreads)
decode_step_kernel(DecodeProblem p) {
    constexpr int kRowsPerThread = D / kRowGroups;   // 4 (D=128) or 2 (D=64)
    constexpr int kSlices = D / kDecCols;
    const int slice = blockIdx.x % kSlices;
    const int nh = blockIdx.x / kSlices;             // n * H + h
    const int tid = threadIdx.x;
    const int cg = tid % kColGroups;
    const int rg = tid / kColGroups;
    const int warp = tid >> 5;
    const int col = slice * kDecCols + cg * 4;

    const size_t st_base = (size_t)nh * D * D;
    const Tin *qp = static_cast<const Tin *>(p.q) + (size_t)nh * D;
    const Tin *kp = static_cast<const Tin *>(p.k) + (size_t)nh * D;
    const Tin *vp = static_cast<const Tin *>(p.v) + (size_t)nh * D;
    const float a = p.alpha[nh], m = p.mu[nh], e = p.eta[nh];
    const float b = p.beta ? p.beta[nh] : 1.0f;

    float4 S[kRowsPerThread], M[kRowsPerThread];
    float kr[kRowsPerThread], qr[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const int row = rg + r * kRowGroups;
        const size_t off = st_base + (size_t)row * D + col;
        S[r] = __ldcs(reinterpret_cast<const float4 *>(p.S + off));
        M[r] = __ldcs(reinterpret_cast<const float4 *>(p.M + off));
        kr[r] = to_f32(kp[row]);
        qr[r] = to_f32(qp[row]);
    }

    __shared__ float red[kDecThreads / 32][kDecCols];
    __shared__ float vres_s[kDecCols];

    // ---- vres = v - alpha S^T k  (column sums over all D rows)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        acc.x += S[r].x * kr[r];
        acc.y += S[r].y * kr[r];
        acc.z += S[r].z * kr[r];
        acc.w += S[r].w * kr[r];
    }
    // lanes with equal cg differ in bits 3 and 4 of the lane id
#pragma unroll
    for (int sh = 8; sh < 32; sh <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, sh);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, sh);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, sh);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, sh);
    }
    if ((tid & 31) < kColGroups) {
        red[warp][cg * 4 + 0] = acc.x;
        red[warp][cg * 4 + 1] = acc.y;
        red[warp][cg * 4 + 2] = acc.z;
        red[warp][cg * 4 + 3] = acc.w;
    }
    __syncthreads();
    if (tid < kDecCols) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) s += red[w][tid];
        vres_s[tid] = to_f32(vp[slice * kDecCols + tid]) - a * s;
    }
    __syncthreads();
    const float4 vr = make_float4(vres_s[cg * 4 + 0], vres_s[cg * 4 + 1],
                                  vres_s[cg * 4 + 2], vres_s[cg * 4 + 3]);

    // ---- M' = mu M - eta k vres^T ; S' = alpha S - beta M' ; o = S'^T q
    float4 oacc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const float ek = e * kr[r];
        float4 Mn, Sn;
        Mn.x = m * M[r].x - ek * vr.x;
        Mn.y = m * M[r].y - ek * vr.y;
        Mn.z = m * M[r].z - ek * vr.z;
        Mn.w = m * M[r].w - ek * vr.w;
        Sn.x = a * S[r].x - b * Mn.x;
        Sn.y = a * S[r].y - b * Mn.y;
        Sn.z = a * S[r].z - b * Mn.z;
        Sn.w = a * S[r].w - b * Mn.w;
        const int row = rg + r * kRowGroups;
        const size_t off = st_base + (size_t)row * D + col;
        __stcs(reinterpret_cast<float4 *>(p.M + off), Mn);
        __stcs(reinterpret_cast<float4 *>(p.S + off), Sn);
        oacc.x += Sn.x * qr[r];
        oacc.y += Sn.y * qr[r];
        oacc.z += Sn.z * qr[r];
        oacc.w += Sn.w * qr[r];
    }
#pragma unroll
    for (int sh = 8; sh < 32; sh <<= 1) {
        oacc.x += __shfl_xor_sync(0xffffffffu, oacc.x, sh);
        oacc.y += __shfl_xor_sync(0xffffffffu, oacc.y, sh);
        oacc.z += __shfl_xor_sync(0xffffffffu, oacc.z, sh);
        oacc.w += __shfl_xor_sync(0xffffffffu, oacc.w, sh);
    }
    __syncthreads();   // everyone is done reading red[] from the first pass
    if ((tid & 31) < kColGroups) {
        red[warp][cg * 4 + 0] = oacc.x;
        red[warp][cg * 4 + 1] = oacc.y;
        red[warp][cg * 4 + 2] = oacc.z;
        red[warp][cg * 4 + 3] = oacc.w;
    }
    __syncthreads();
    if (tid < kDecCols) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) s += red[w][tid];
        Tin *op = static_cast<Tin *>(p.o) + (size_t)nh * D + slice * kDecCols;
        op[tid] = from_f32<Tin>(s);
    }
}

template <int D, typename Tin>
cudaError_t launch_decode_t(const DecodeProblem &p, cudaStream_t st) {
    const long blocks = (long)p.N * p.H * (D / kDecCols);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    decode_step_kernel<D, Tin><<<(unsigned)blocks, kDecThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem &p, cudaStream_t st) {
    if (p.D == 128) {
        return p.dtype == MDN_BF16 ? launch_decode_t<128, __nv_bfloat16>(p, st)
                                   : launch_decode_t<128, float>(p, st);
    }
    return p.dtype == MDN_BF16 ? launch_decode_t<64, __nv_bfloat16>(p, st)
                               : launch_decode_t<64, float>(p, st);
}

}  // namespace mdn
