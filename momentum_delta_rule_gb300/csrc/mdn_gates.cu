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
#include "mdn_sm100.cuh"

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

// ---------------------------------------------------------------- streaming

// Whole 16 KiB tiles of q and k stream through shared memory: a persistent
// grid of kStreamBlocksPerSM blocks per SM, each with two stages.  A producer
// warp moves tiles in and results out with bulk asynchronous copies (the
// bytes stay in flight without holding registers); eight compute warps
// normalise each tile in place.  Stage handshake: `full` (the tile landed,
// transaction bytes) and `done` (every compute warp has written its results
// back).  The producer stores a done stage, waits until that store has read
// shared memory, then loads the stage's next tile.
constexpr int kStreamComputeWarps = 8;
constexpr int kStreamThreads = 32 * (kStreamComputeWarps + 1);
constexpr int kStreamBlocksPerSM = 3;
constexpr uint32_t kTileBytes = 16384;              // of q, and of k
constexpr uint32_t kStreamSmem = 2 * 2 * kTileBytes + 64 + 1024;

struct StreamBars {
    uint64_t full[2], done[2];
    int abort;
};

template <int D, typename T>
__global__ void __launch_bounds__(kStreamThreads, kStreamBlocksPerSM)
prepare_inputs_stream_kernel(InputsProblem p, long ntiles) {
    constexpr int EL = 16 / (int)sizeof(T);           // elements per 16-byte packet
    constexpr int LR = D / EL;                        // lanes (packets) per row
    constexpr int RB = D * (int)sizeof(T);            // bytes per row
    constexpr int R = kTileBytes / RB;                // rows per tile
    constexpr int kPackets = kTileBytes / 16;         // packets per tile (of q, of k)
    constexpr int kPer = kPackets / (32 * kStreamComputeWarps);
    static_assert(kPackets % (32 * kStreamComputeWarps) == 0, "tile split");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = sm100::align_smem_1024(smem_raw);
    StreamBars *bars = reinterpret_cast<StreamBars *>(smem + 4 * kTileBytes);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T *tag = nullptr;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            sm100::mbar_init(&bars->full[i], 1);
            sm100::mbar_init(&bars->done[i], kStreamComputeWarps);
        }
        bars->abort = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    const long first = blockIdx.x;
    const long step = gridDim.x;
    const unsigned char *qin = static_cast<const unsigned char *>(p.q_in);
    const unsigned char *kin = static_cast<const unsigned char *>(p.k_in);
    unsigned char *qout = static_cast<unsigned char *>(p.q_out);
    unsigned char *kout = static_cast<unsigned char *>(p.k_out);

    if (warp == kStreamComputeWarps) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            int nload = 0;                 // loads issued; load j fills stage j % 2
            auto load = [&](long t, int st) {
                unsigned char *qs = smem + st * 2 * kTileBytes, *ks = qs + kTileBytes;
                sm100::mbar_arrive_expect_tx(&bars->full[st], 2 * kTileBytes);
                sm100::bulk_load(qs, qin + (size_t)t * kTileBytes, kTileBytes, &bars->full[st]);
                sm100::bulk_load(ks, kin + (size_t)t * kTileBytes, kTileBytes, &bars->full[st]);
                ++nload;
            };
            if (first < ntiles) load(first, 0);
            if (first + step < ntiles) load(first + step, 1);
            int i = 0;
            for (long t = first; t < ntiles; t += step, ++i) {
                const int st = i & 1;
                if (!sm100::mbar_wait(&bars->done[st], (i >> 1) & 1, abort)) break;
                unsigned char *qs = smem + st * 2 * kTileBytes, *ks = qs + kTileBytes;
                sm100::bulk_store(qout + (size_t)t * kTileBytes, qs, kTileBytes);
                sm100::bulk_store(kout + (size_t)t * kTileBytes, ks, kTileBytes);
                sm100::bulk_commit_group();
                const long tn = t + 2 * step;
                if (tn < ntiles) {
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    load(tn, st);
                }
            }
            sm100::bulk_wait_group0();     // every result is written before the block exits
            // after an expired wait the last two loads may be unconsumed: they
            // land before the block exits
            for (int j = nload - 2; j < nload; ++j) {
                if (j < 0) continue;
                int dummy = 0;
                sm100::mbar_wait(&bars->full[j & 1], (j >> 1) & 1, &dummy);
            }
        }
        return;
    }
    // ------------------------------------------------ compute
    const int ctid = threadIdx.x;                      // 0 .. 255
    int i = 0;
    for (long t = first; t < ntiles; t += step, ++i) {
        const int st = i & 1;
        unsigned char *qs = smem + st * 2 * kTileBytes, *ks = qs + kTileBytes;
        // gates of the tile's rows (plain loads, overlap the wait)
        const long grow = t * R + ctid;
        float za = 0.f, zb = 0.f, zm = 0.f, ze = 0.f;
        const bool gate_row = ctid < R;
        if (gate_row) {
            za = __ldcs(p.z_alpha + grow);
            zb = __ldcs(p.z_beta + grow);
            zm = __ldcs(p.z_mu + grow);
            ze = __ldcs(p.z_eta + grow);
        }
        if (!__all_sync(0xffffffffu, sm100::mbar_wait(&bars->full[st], (i >> 1) & 1, abort))) break;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            // packet index: consecutive lanes take consecutive packets of a row
            const int pk = (k * kStreamComputeWarps + warp) * 32 + lane;
            uint4 *qp = reinterpret_cast<uint4 *>(qs + pk * 16);
            uint4 *kp = reinterpret_cast<uint4 *>(ks + pk * 16);
            float qv[EL], kv[EL];
            unpack16(*qp, qv, tag);
            unpack16(*kp, kv, tag);
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < EL; ++e) {
                qv[e] -= p.comba_d * kv[e];
                sq += qv[e] * qv[e];
                sk += kv[e] * kv[e];
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
                qv[e] *= iq;
                kv[e] *= ik;
            }
            *qp = pack16(qv, tag);
            *kp = pack16(kv, tag);
        }
        sm100::fence_proxy_async();                    // results visible to the bulk store
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(&bars->done[st]);
        if (gate_row) {
            const float eta = 1.f + tanhf(ze / p.tau);
            const float x2 = (p.s * eta) * (p.s * eta);
            const float amax = 1.f / (1.f + x2);
            const float bmax = x2 / (1.f + x2);
            __stcs(p.alpha + grow, amax * expf(-p.a * softplus_f(za + p.b)));
            __stcs(p.beta + grow, bmax / (1.f + expf(-zb)));
            __stcs(p.mu + grow, expf(fmaxf(-p.a * softplus_f(zm + p.b), p.log_mu_min)));
            __stcs(p.eta + grow, eta);
        }
    }
}

template <int D, typename T>
cudaError_t launch_t(const InputsProblem &p, cudaStream_t st) {
    constexpr int EL = 16 / (int)sizeof(T);
    constexpr int RPI = 32 / (D / EL);
    constexpr int kLoads = RPI >= 4 ? 1 : 4 / RPI;     // four rows per warp
    constexpr long kRowsPerBlock = (long)kWarpsPerBlock * RPI * kLoads;
    constexpr long R = kTileBytes / (D * (long)sizeof(T));
    // whole tiles stream; the rows after the last whole tile take the
    // one-shot kernel
    const long ntiles = p.rows / R;
    if (ntiles > 0) {
        const int sms = device_sm_count();
        long blocks = (long)(sms > 0 ? sms : 1) * kStreamBlocksPerSM;
        if (blocks > ntiles) blocks = ntiles;
        auto k = prepare_inputs_stream_kernel<D, T>;
        cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kStreamSmem);
        if (err != cudaSuccess) return err;
        k<<<(unsigned)blocks, kStreamThreads, kStreamSmem, st>>>(p, ntiles);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    const long done_rows = ntiles * R;
    const long rest = p.rows - done_rows;
    if (rest == 0) return cudaSuccess;
    InputsProblem q = p;
    const size_t off = (size_t)done_rows * D;
    q.q_in = static_cast<const T *>(p.q_in) + off;
    q.k_in = static_cast<const T *>(p.k_in) + off;
    q.q_out = static_cast<T *>(p.q_out) + off;
    q.k_out = static_cast<T *>(p.k_out) + off;
    q.z_alpha = p.z_alpha + done_rows; q.z_beta = p.z_beta + done_rows;
    q.z_mu = p.z_mu + done_rows; q.z_eta = p.z_eta + done_rows;
    q.alpha = p.alpha + done_rows; q.beta = p.beta + done_rows;
    q.mu = p.mu + done_rows; q.eta = p.eta + done_rows;
    q.rows = rest;
    const long blocks = (rest + kRowsPerBlock - 1) / kRowsPerBlock;
    prepare_inputs_kernel<D, T, kLoads><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, st>>>(q);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare_inputs(const InputsProblem &p, cudaStream_t st) {
    if (p.D == 128)
        return p.dtype == MDN_BF16 ? launch_t<128, __nv_bfloat16>(p, st) : launch_t<128, float>(p, st);
    return p.dtype == MDN_BF16 ? launch_t<64, __nv_bfloat16>(p, st) : launch_t<64, float>(p, st);
}

}  // namespace mdn
