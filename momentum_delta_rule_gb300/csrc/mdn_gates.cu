// MDN layer inputs in one pass: the gates from their scalar projections and
// the query/key preparation (slides, frame "Coupled gates restrict the
// spectral region", Sec. 3.3; reading notes sections 2.8 and 2.9).
//
// Per (token, head) row:
//   eta   = 1 + tanh(z_eta / tau)
//   alpha = alpha_max exp(f(z_alpha)),  beta = sigmoid(z_beta) beta_max,
//   mu    = exp(max(f(z_mu), log_mu_min)),  f(z) = -a softplus(z + b),
// with alpha_max = cos^2(arctan(s eta)) = 1 / (1 + (s eta)^2) and
// beta_max = 1 - alpha_max = (s eta)^2 / (1 + (s eta)^2);
//   q_hat = (q - d k) / |q - d k|,  k_hat = k / |k|   (zero rows stay zero).
//
// One warp per row: 32 lanes hold the head's d elements, two shuffle
// reductions give the norms, lane 0 computes the four gates.  Memory bound:
// each row reads 2 d elements + 4 floats and writes as much.
#include <cuda_bf16.h>

#include "mdn_internal.cuh"

namespace mdn {
namespace {

constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ float softplus_f(float x) {
    // log(1 + e^x) = max(x, 0) + log(1 + e^{-|x|}): no overflow for large x
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

template <typename T, int E> struct Vec;
template <> struct Vec<float, 4> {
    static __device__ __forceinline__ void ld(const float *p, float *x) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    static __device__ __forceinline__ void st(float *p, const float *x) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <> struct Vec<float, 2> {
    static __device__ __forceinline__ void ld(const float *p, float *x) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        x[0] = v.x; x[1] = v.y;
    }
    static __device__ __forceinline__ void st(float *p, const float *x) {
        *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
    }
};
template <> struct Vec<__nv_bfloat16, 4> {
    static __device__ __forceinline__ void ld(const __nv_bfloat16 *p, float *x) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
        const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, const float *x) {
        uint2 v;
        __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        v.x = *reinterpret_cast<uint32_t *>(&a);
        v.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = v;
    }
};
template <> struct Vec<__nv_bfloat16, 2> {
    static __device__ __forceinline__ void ld(const __nv_bfloat16 *p, float *x) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
        x[0] = a.x; x[1] = a.y;
    }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, const float *x) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x[0], x[1]);
    }
};

template <int D, typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
prepare_inputs_kernel(InputsProblem p) {
    constexpr int E = D / 32;                   // elements per lane
    const long row = (long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.rows) return;
    const size_t off = (size_t)row * D + (size_t)lane * E;
    float q[E], k[E];
    Vec<T, E>::ld(static_cast<const T *>(p.q_in) + off, q);
    Vec<T, E>::ld(static_cast<const T *>(p.k_in) + off, k);
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        q[e] -= p.comba_d * k[e];
        sq += q[e] * q[e];
        sk += k[e] * k[e];
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
    }
    const float iq = sq > 0.f ? 1.f / sqrtf(sq) : 0.f;
    const float ik = sk > 0.f ? 1.f / sqrtf(sk) : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        q[e] *= iq;
        k[e] *= ik;
    }
    Vec<T, E>::st(static_cast<T *>(p.q_out) + off, q);
    Vec<T, E>::st(static_cast<T *>(p.k_out) + off, k);

    if (lane == 0) {
        const float eta = 1.f + tanhf(p.z_eta[row] / p.tau);
        const float x2 = (p.s * eta) * (p.s * eta);
        const float amax = 1.f / (1.f + x2);
        const float bmax = x2 / (1.f + x2);
        p.alpha[row] = amax * expf(-p.a * softplus_f(p.z_alpha[row] + p.b));
        p.beta[row] = bmax / (1.f + expf(-p.z_beta[row]));
        p.mu[row] = expf(fmaxf(-p.a * softplus_f(p.z_mu[row] + p.b), p.log_mu_min));
        p.eta[row] = eta;
    }
}

template <int D, typename T>
cudaError_t launch_t(const InputsProblem &p, cudaStream_t st) {
    const long blocks = (p.rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    prepare_inputs_kernel<D, T><<<(unsigned)blocks, 32 * kRowsPerBlock, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare_inputs(const InputsProblem &p, cudaStream_t st) {
    if (p.D == 128)
        return p.dtype == MDN_BF16 ? launch_t<128, __nv_bfloat16>(p, st) : launch_t<128, float>(p, st);
    return p.dtype == MDN_BF16 ? launch_t<64, __nv_bfloat16>(p, st) : launch_t<64, float>(p, st);
}

}  // namespace mdn
