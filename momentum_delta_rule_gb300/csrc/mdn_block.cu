// MDN token-mixer block around the memory core ("MDN: Parallelizing Stepwise
// Momentum for Delta Linear Attention" slides, frame "The memory sits inside
// a familiar language-model block" (Sec. 3.3, Fig. 3); reading notes 2.9):
//
//   P   = x W_in                      one projection GEMM: q, k, v, the
//                                     output-gate input g (H d columns each)
//                                     and the four gate projections (H each)
//   q, k, v = SiLU(ShortConv(.))      causal depthwise convolution along the
//                                     tokens (width 4, restarting at every
//                                     sequence start), then SiLU
//   q <- q - d k; q, k L2-normalised; the four gates    (mdn_prepare_inputs)
//   o   = MDN memory update                             (mdn_chunk_fwd)
//   u   = sigmoid(g) * RMSNorm(o)      per head over d_v, weight shared by
//                                     the heads
//   y   = u W_o                       the output projection GEMM
//
// The two projections are plain GEMMs and go to cuBLAS; the convolution and
// the norm-and-gate step are memory-bound kernels of this file; the rest
// reuses the library's own kernels.
#include <cublas_v2.h>

#include <algorithm>
#include <mutex>

#include "mdn_internal.cuh"

namespace mdn {
namespace {

constexpr int kConvWidth = 4;
constexpr size_t kCublasWorkspace = 4u << 20;

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

template <typename T> __device__ __forceinline__ void store4(T *dst, const float *v);
template <> __device__ __forceinline__ void store4<float>(float *dst, const float *v) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, const float *v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t *>(&a);
    w.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(dst) = w;
}

// First token of the sequence that token t belongs to.
__device__ __forceinline__ long seq_start(long t, const int32_t *cu, int n_seq, int T) {
    if (cu == nullptr) return T > 0 ? (t / T) * T : 0;
    int lo = 0, hi = n_seq;                 // largest s with cu[s] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return cu[lo];
}

// The short convolution and SiLU of the q, k, v channels (four channels per
// thread), and the gate projections copied out as [tokens, H] arrays.
template <typename Tout>
__global__ void __launch_bounds__(256)
block_conv_kernel(const float *proj, int ncol, const float *conv_w, int Hd, int H,
                  const int32_t *cu, int n_seq, int T, long T_total, Tout *qc, Tout *kc,
                  Tout *vc, float *za, float *zb, float *zm, float *ze) {
    const long groups = 3L * Hd / 4;
    const long total = T_total * groups;
    const long stride = (long)gridDim.x * blockDim.x;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const long t = idx / groups;
        const int c = (int)(idx - t * groups) * 4;
        const long start = max(seq_start(t, cu, n_seq, T), 0L);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kConvWidth; ++j) {
            const long src = t - (kConvWidth - 1) + j;   // tap j: (width - 1 - j) tokens back
            if (src < start) continue;
            const float4 pv = *reinterpret_cast<const float4 *>(proj + src * ncol + c);
            acc[0] = fmaf(conv_w[(c + 0) * kConvWidth + j], pv.x, acc[0]);
            acc[1] = fmaf(conv_w[(c + 1) * kConvWidth + j], pv.y, acc[1]);
            acc[2] = fmaf(conv_w[(c + 2) * kConvWidth + j], pv.z, acc[2]);
            acc[3] = fmaf(conv_w[(c + 3) * kConvWidth + j], pv.w, acc[3]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = silu(acc[e]);
        const int which = c / Hd, ch = c - which * Hd;
        Tout *dst = which == 0 ? qc : (which == 1 ? kc : vc);
        store4<Tout>(dst + t * Hd + ch, acc);
    }
    const long zt = T_total * H;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < zt; idx += stride) {
        const long t = idx / H;
        const int h = (int)(idx - t * H);
        const float *row = proj + t * ncol + 4L * Hd;
        za[idx] = row[h];
        zb[idx] = row[H + h];
        zm[idx] = row[2 * H + h];
        ze[idx] = row[3 * H + h];
    }
}

// u = sigmoid(g) * RMSNorm(o) per (token, head) row of d outputs, one warp
// per row.
template <typename T, int D>
__global__ void __launch_bounds__(256)
block_out_kernel(const T *o, const float *proj, int ncol, const float *rms_w, float eps, int Hd,
                 int H, long rows, T *u) {
    constexpr int E = D / 32;
    const long row = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const long t = row / H;
    const int h = (int)(row - t * H);
    float v[E];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        v[e] = to_f32(o[row * D + lane * E + e]);
        ss = fmaf(v[e], v[e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = rsqrtf(ss / (float)D + eps);
    const float *g = proj + t * ncol + 3L * Hd + (long)h * D;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int c = lane * E + e;
        const float gate = 1.f / (1.f + expf(-g[c]));
        u[row * D + c] = from_f32<T>(gate * v[e] * inv * rms_w[c]);
    }
}

// One cuBLAS handle per device, created on the device's first block call;
// calls on one device are serialised around the handle's stream and
// workspace settings.
struct CublasSlot {
    std::mutex mu;
    cublasHandle_t handle = nullptr;
};
CublasSlot g_cublas[64];

cudaError_t gemm_rowmajor(cublasHandle_t hnd, int M, int N, int K, const void *A, const void *B,
                          void *Cm, cudaDataType ab_type, cudaDataType c_type) {
    // row-major C[M, N] = A[M, K] B[K, N]: in cuBLAS's column-major terms
    // C^T (N x M) = B^T (N x K) A^T (K x M)
    const float one = 1.f, zero = 0.f;
    const cublasStatus_t st = cublasGemmEx(hnd, CUBLAS_OP_N, CUBLAS_OP_N, N, M, K, &one, B, ab_type, N,
                                           A, ab_type, K, &zero, Cm, c_type, N, CUBLAS_COMPUTE_32F,
                                           CUBLAS_GEMM_DEFAULT);
    return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

size_t round256b(size_t x) { return (x + 255) & ~(size_t)255; }

struct BlockWs {
    size_t proj, qc, kc, vc, z, gates, o, u, chunk, cublas, total;
};

BlockWs block_ws_layout(int n_seq, long T_total, int H, int d, mdn_dtype dtype) {
    const size_t el = dtype == MDN_BF16 ? 2 : 4;
    const size_t Hd = (size_t)H * d, ncol = 4 * Hd + 4 * (size_t)H;
    BlockWs w;
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t at = off; off += round256b(bytes); return at; };
    w.proj = take((size_t)T_total * ncol * 4);
    w.qc = take((size_t)T_total * Hd * el);
    w.kc = take((size_t)T_total * Hd * el);
    w.vc = take((size_t)T_total * Hd * el);
    w.z = take((size_t)T_total * H * 4 * 4);
    w.gates = take((size_t)T_total * H * 4 * 4);
    w.o = take((size_t)T_total * Hd * el);
    w.u = take((size_t)T_total * Hd * el);
    w.chunk = take(mdn_chunk_fwd_workspace_size(n_seq, (int)T_total, H, d, d, dtype));
    w.cublas = take(kCublasWorkspace);
    w.total = off;
    return w;
}

}  // namespace
}  // namespace mdn

extern "C" {

size_t mdn_block_fwd_workspace_size(int n_seq, int T_total, int H, int d, int d_model,
                                    mdn_dtype dtype) {
    if (n_seq < 0 || T_total < 0 || H <= 0 || d <= 0 || d_model <= 0) return 0;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return 0;
    return mdn::block_ws_layout(n_seq, T_total, H, d, dtype).total;
}

mdn_status mdn_block_fwd(const void *x, const void *W_in, const float *conv_w, const float *rms_w,
                         const void *W_o, float a, float b, float s, float tau, float log_mu_min,
                         float comba_d, float rms_eps, const float *S0, const float *M0, void *y,
                         float *S_T, float *M_T, const int32_t *cu_seqlens, int n_seq, int B,
                         int T, int H, int d, int d_model, mdn_dtype dtype, void *workspace,
                         size_t workspace_bytes, void *stream) {
    using namespace mdn;
    if (B < 0 || T < 0 || H <= 0 || n_seq < 0 || d_model <= 0) return MDN_ERR_INVALID_ARG;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return MDN_ERR_INVALID_ARG;
    if (cu_seqlens ? B != 1 : n_seq != B) return MDN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return MDN_ERR_UNSUPPORTED;
    if (d_model % 8 != 0) return MDN_ERR_UNSUPPORTED;
    if (!(rms_eps >= 0.f)) return MDN_ERR_INVALID_ARG;
    const long T_total = (long)B * T;
    if (T_total > 0x3fffffffL) return MDN_ERR_INVALID_ARG;
    if (T_total > 0) {
        const void *need[] = {x, W_in, conv_w, rms_w, W_o, y};
        for (const void *ptr : need)
            if (!ptr) return MDN_ERR_INVALID_ARG;
    }
    const void *al16[] = {x, W_in, W_o, y, S0, M0, S_T, M_T, conv_w, rms_w};
    for (const void *ptr : al16)
        if (ptr && ((uintptr_t)ptr & 15u)) return MDN_ERR_INVALID_ARG;
    if (cu_seqlens && ((uintptr_t)cu_seqlens & 3u)) return MDN_ERR_INVALID_ARG;
    const BlockWs L = block_ws_layout(n_seq, T_total, H, d, dtype);
    if (T_total > 0 && n_seq > 0 &&
        (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u)))
        return MDN_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) return MDN_ERR_UNSUPPORTED;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    const int Hd = H * d, ncol = 4 * Hd + 4 * H;
    const size_t el = dtype == MDN_BF16 ? 2 : 4;
    if (T_total == 0 || n_seq == 0) {
        // no tokens: the core only hands the initial states through
        return mdn_chunk_fwd(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, S0, M0,
                             nullptr, S_T, M_T, cu_seqlens, n_seq, B, T, H, d, d, dtype, 64,
                             nullptr, 0, stream);
    }
    float *proj = reinterpret_cast<float *>(ws + L.proj);
    void *qc = ws + L.qc, *kc = ws + L.kc, *vc = ws + L.vc, *o = ws + L.o, *u = ws + L.u;
    float *z = reinterpret_cast<float *>(ws + L.z);
    float *gt = reinterpret_cast<float *>(ws + L.gates);
    const size_t gn = (size_t)T_total * H;
    const cudaDataType ab = dtype == MDN_BF16 ? CUDA_R_16BF : CUDA_R_32F;

    CublasSlot &slot = g_cublas[dev];
    std::lock_guard<std::mutex> lock(slot.mu);
    if (!slot.handle && cublasCreate(&slot.handle) != CUBLAS_STATUS_SUCCESS) {
        slot.handle = nullptr;
        return MDN_ERR_CUDA;
    }
    if (cublasSetStream(slot.handle, cs) != CUBLAS_STATUS_SUCCESS ||
        cublasSetWorkspace(slot.handle, ws + L.cublas, kCublasWorkspace) != CUBLAS_STATUS_SUCCESS)
        return MDN_ERR_CUDA;
    // 1. P = x W_in (fp32 out)
    if (gemm_rowmajor(slot.handle, (int)T_total, ncol, d_model, x, W_in, proj, ab, CUDA_R_32F) !=
        cudaSuccess)
        return MDN_ERR_CUDA;
    // 2. short convolution + SiLU, gate projections
    {
        const long work = T_total * (3L * Hd / 4);
        const int blocks = (int)std::min<long>((work + 255) / 256, 152L * 16);
        if (dtype == MDN_BF16)
            block_conv_kernel<__nv_bfloat16><<<blocks, 256, 0, cs>>>(
                proj, ncol, conv_w, Hd, H, cu_seqlens, n_seq, T, T_total,
                static_cast<__nv_bfloat16 *>(qc), static_cast<__nv_bfloat16 *>(kc),
                static_cast<__nv_bfloat16 *>(vc), z, z + gn, z + 2 * gn, z + 3 * gn);
        else
            block_conv_kernel<float><<<blocks, 256, 0, cs>>>(
                proj, ncol, conv_w, Hd, H, cu_seqlens, n_seq, T, T_total, static_cast<float *>(qc),
                static_cast<float *>(kc), static_cast<float *>(vc), z, z + gn, z + 2 * gn, z + 3 * gn);
        if (cudaGetLastError() != cudaSuccess) return MDN_ERR_CUDA;
    }
    // 3. gates, Comba correction and L2 normalisation (in place on q, k)
    mdn_status st = mdn_prepare_inputs(qc, kc, z, z + gn, z + 2 * gn, z + 3 * gn, qc, kc, gt,
                                       gt + gn, gt + 2 * gn, gt + 3 * gn, (int)T_total, H, d, dtype,
                                       a, b, s, tau, log_mu_min, comba_d, stream);
    if (st != MDN_OK) return st;
    // 4. the memory update (gates: alpha, beta, mu, eta in that order)
    st = mdn_chunk_fwd(qc, kc, vc, gt, gt + 2 * gn, gt + 3 * gn, gt + gn, S0, M0, o, S_T, M_T,
                       cu_seqlens, n_seq, B, T, H, d, d, dtype, 64, ws + L.chunk,
                       mdn_chunk_fwd_workspace_size(n_seq, (int)T_total, H, d, d, dtype), stream);
    if (st != MDN_OK) return st;
    // 5. u = sigmoid(g) * RMSNorm(o)
    {
        const long rows = T_total * H;
        const long blocks = (rows * 32 + 255) / 256;
        if (dtype == MDN_BF16) {
            if (d == 128)
                block_out_kernel<__nv_bfloat16, 128><<<(unsigned)blocks, 256, 0, cs>>>(
                    static_cast<const __nv_bfloat16 *>(o), proj, ncol, rms_w, rms_eps, Hd, H, rows,
                    static_cast<__nv_bfloat16 *>(u));
            else
                block_out_kernel<__nv_bfloat16, 64><<<(unsigned)blocks, 256, 0, cs>>>(
                    static_cast<const __nv_bfloat16 *>(o), proj, ncol, rms_w, rms_eps, Hd, H, rows,
                    static_cast<__nv_bfloat16 *>(u));
        } else {
            if (d == 128)
                block_out_kernel<float, 128><<<(unsigned)blocks, 256, 0, cs>>>(
                    static_cast<const float *>(o), proj, ncol, rms_w, rms_eps, Hd, H, rows,
                    static_cast<float *>(u));
            else
                block_out_kernel<float, 64><<<(unsigned)blocks, 256, 0, cs>>>(
                    static_cast<const float *>(o), proj, ncol, rms_w, rms_eps, Hd, H, rows,
                    static_cast<float *>(u));
        }
        if (cudaGetLastError() != cudaSuccess) return MDN_ERR_CUDA;
    }
    // 6. y = u W_o
    if (gemm_rowmajor(slot.handle, (int)T_total, d_model, Hd, u, W_o, y, ab, ab) != cudaSuccess)
        return MDN_ERR_CUDA;
    (void)el;
    return MDN_OK;
}

}  // extern "C"
