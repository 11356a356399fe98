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
// Memory bound: each row reads 2 d elements + 4 floats and writes as much,
// in 16-byte packets with streaming cache hints.
#include <cuda_bf16.h>

#include "mdn_internal.cuh"

namespace mdn {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float softplus_f(float x) {
    // log(1 + e^x) = max(x, 0) + log(1 + e^{-|x|}): no overflow for large x
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

// 16-byte packets of 8 bf16 or 4 fp32 values
__device__ __forceinline__ void unpack16(const uint4 &u, float *x, const float *) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4 &u, float *x, const __nv_bfloat16 *) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        x[2 * i] = t.x;
        x[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 pack16(const float *x, const float *) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
}
__device__ __forceinline__ uint4 pack16(const float *x, const __nv_bfloat16 *) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&t);
    }
    return u;
}

// One warp covers kLoads x (32 / lanes-per-row) rows: every lane moves
// 16-byte packets (all loads issued before any arithmetic), a row's norm is a
// shuffle reduction over the lanes that hold it, and the first lanes of the
// warp turn the rows' projections into gates.
template <int D, typename T, int kLoads>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
prepare_inputs_kernel(InputsProblem p) {
    constexpr int EL = 16 / (int)sizeof(T);     // elements per packet
    constexpr int LR = D / EL;                  // lanes per row
    constexpr int RPI = 32 / LR;                // rows per load instruction
    constexpr int RW = RPI * kLoads;            // rows per warp
    const T *tag = nullptr;
    const int lane = threadIdx.x & 31;
    const long row0 = ((long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * RW;
    const int sub = lane / LR, li = lane % LR;
    uint4 qr[kLoads], kr[kLoads];
    float za = 0.f, zb = 0.f, zm = 0.f, ze = 0.f;
    const long grow = row0 + lane;
    if (lane < RW && grow < p.rows) {
        za = p.z_alpha[grow];
        zb = p.z_beta[grow];
        zm = p.z_mu[grow];
        ze = p.z_eta[grow];
    }
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
        const long row = row0 + i * RPI + sub;
        qr[i] = kr[i] = make_uint4(0u, 0u, 0u, 0u);
        if (row < p.rows) {
            const size_t off = (size_t)row * D + (size_t)li * EL;
            qr[i] = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const T *>(p.q_in) + off));
            kr[i] = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const T *>(p.k_in) + off));
        }
    }
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
        const long row = row0 + i * RPI + sub;
        float q[EL], k[EL];
        unpack16(qr[i], q, tag);
        unpack16(kr[i], k, tag);
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            q[e] -= p.comba_d * k[e];
            sq += q[e] * q[e];
            sk += k[e] * k[e];
        }
#pragma unroll
        for (int m = LR / 2; m > 0; m >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, m);
            sk += __shfl_xor_sync(0xffffffffu, sk, m);
        }
        const float iq = sq > 0.f ? 1.f / sqrtf(sq) : 0.f;
        const float ik = sk > 0.f ? 1.f / sqrtf(sk) : 0.f;
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            q[e] *= iq;
            k[e] *= ik;
        }
        if (row < p.rows) {
            const size_t off = (size_t)row * D + (size_t)li * EL;
            __stcs(reinterpret_cast<uint4 *>(static_cast<T *>(p.q_out) + off), pack16(q, tag));
            __stcs(reinterpret_cast<uint4 *>(static_cast<T *>(p.k_out) + off), pack16(k, tag));
        }
    }
    if (lane < RW && grow < p.rows) {
        const float eta = 1.f + tanhf(ze / p.tau);
        const float x2 = (p.s * eta) * (p.s * eta);
        const float amax = 1.f / (1.f + x2);
        const float bmax = x2 / (1.f + x2);
        p.alpha[grow] = amax * expf(-p.a * softplus_f(za + p.b));
        p.beta[grow] = bmax / (1.f + expf(-zb));
        p.mu[grow] = expf(fmaxf(-p.a * softplus_f(zm + p.b), p.log_mu_min));
        p.eta[grow] = eta;
    }
}

template <int D, typename T>
cudaError_t launch_t(const InputsProblem &p, cudaStream_t st) {
    constexpr int EL = 16 / (int)sizeof(T);
    constexpr int RPI = 32 / (D / EL);
    constexpr int kLoads = RPI >= 4 ? 1 : 4 / RPI;     // four rows per warp
    constexpr long kRowsPerBlock = (long)kWarpsPerBlock * RPI * kLoads;
    const long blocks = (p.rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    prepare_inputs_kernel<D, T, kLoads><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare_inputs(const InputsProblem &p, cudaStream_t st) {
    if (p.D == 128)
        return p.dtype == MDN_BF16 ? launch_t<128, __nv_bfloat16>(p, st) : launch_t<128, float>(p, st);
    return p.dtype == MDN_BF16 ? launch_t<64, __nv_bfloat16>(p, st) : launch_t<64, float>(p, st);
}

}  // namespace mdn
