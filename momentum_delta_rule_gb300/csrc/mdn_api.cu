// C ABI of the MDN library: argument validation, workspace layout, dispatch
// and the device status word.  Declarations and the contract: include/mdn.h.
#include <stdint.h>
#include <atomic>
#include <string.h>

#include "mdn_internal.cuh"

// Device status word (one per device that loads the library).  Kernels with
// bounded waits write MDN_ERR_DEVICE_TIMEOUT here instead of hanging.
__device__ int g_mdn_status;

namespace {

constexpr int kMaxDevices = 64;

// Filled on a device's first call.  Host threads may call concurrently:
// `status` is written before `checked` is published (release) and read only
// after `checked` is seen (acquire).
struct DeviceInfo {
    std::atomic<int> checked;     // 0 = unknown, 1 = supported, -1 = unsupported
    std::atomic<int *> status;    // device address of g_mdn_status
};
DeviceInfo g_dev[kMaxDevices];

bool aligned16(const void *ptr) { return ((uintptr_t)ptr & 15u) == 0; }

// Supported device (compute capability 10.3) and its status-word address.
mdn_status current_device(int **status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MDN_ERR_UNSUPPORTED;
    DeviceInfo &di = g_dev[dev];
    int checked = di.checked.load(std::memory_order_acquire);
    if (checked == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return MDN_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            checked = -1;
        } else {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_mdn_status) != cudaSuccess) {
                cudaGetLastError();
                return MDN_ERR_CUDA;
            }
            di.status.store(static_cast<int *>(addr), std::memory_order_relaxed);
            checked = 1;
        }
        di.checked.store(checked, std::memory_order_release);
    }
    if (checked < 0) return MDN_ERR_UNSUPPORTED;
    *status = di.status.load(std::memory_order_relaxed);
    return MDN_OK;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace head: chunk offsets [n_seq + 1] and the longest-first sequence
// order [n_seq] (both int32), each 256-byte aligned; prepared blocks follow.
size_t meta_bytes(int n_seq) {
    return round256(sizeof(int32_t) * ((size_t)n_seq + 1)) +
           round256(sizeof(int32_t) * ((size_t)n_seq + 1));
}

// fp32 inputs reach the tensor cores as hi / lo bf16 parts of q, k and v:
// six [T_total, H, d] bf16 arrays after the prepared blocks.
size_t split_part_bytes(int T_total, int H, int d) {
    return (((size_t)T_total * H * d * 2) + 255) & ~(size_t)255;
}
size_t split_bytes(int T_total, int H, int d, mdn_dtype dtype) {
    return dtype == MDN_F32 ? 6 * split_part_bytes(T_total, H, d) : 0;
}

// Upper bound on the chunk slots of any split of T_total into n_seq
// sequences: sum ceil(L_s / 64) <= floor(T_total / 64) + n_seq.
long chunk_slots_bound(int n_seq, int T_total) {
    return (long)(T_total / mdn::kChunk) + (long)n_seq;
}

}  // namespace

extern "C" {

int mdn_abi_version(void) { return MDN_ABI_VERSION; }

const char *mdn_status_string(mdn_status status) {
    switch (status) {
        case MDN_OK: return "MDN_OK: success";
        case MDN_ERR_INVALID_ARG: return "MDN_ERR_INVALID_ARG: invalid argument";
        case MDN_ERR_UNSUPPORTED: return "MDN_ERR_UNSUPPORTED: unsupported size, chunk or device";
        case MDN_ERR_CUDA: return "MDN_ERR_CUDA: a CUDA call or kernel launch failed";
        case MDN_ERR_DEVICE_TIMEOUT: return "MDN_ERR_DEVICE_TIMEOUT: a bounded device-side wait expired";
    }
    return "MDN: unknown status";
}

size_t mdn_chunk_fwd_workspace_size(int n_seq, int T_total, int H, int dk,
                                    int dv, mdn_dtype dtype) {
    if (n_seq < 0 || T_total < 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return 0;
    const size_t prep = (size_t)chunk_slots_bound(n_seq, T_total) * (size_t)H *
                        mdn::kPrepBytesMax;
    return round256(meta_bytes(n_seq) + prep) + split_bytes(T_total, H, dk, dtype);
}

}  // extern "C"

namespace mdn {

// Argument checks shared by every chunk-forward entry point (the workspace
// is checked by the caller, since the entry points get it differently), then,
// if `status` is not null, the device check, whose success stores the device
// status word there.
mdn_status chunk_fwd_check(const void *q, const void *k, const void *v, const float *alpha,
                           const float *mu, const float *eta, const float *beta,
                           const float *S0, const float *M0, const void *o, const float *S_T,
                           const float *M_T, const void *vres, const void *S_chunks,
                           const void *M_chunks, const int32_t *cu_seqlens, int n_seq,
                           int B, int T, int H, int dk, int dv, mdn_dtype dtype, int chunk,
                           int **status) {
    // ---- shapes
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || n_seq < 0)
        return MDN_ERR_INVALID_ARG;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return MDN_ERR_INVALID_ARG;
    if (cu_seqlens) {
        if (B != 1) return MDN_ERR_INVALID_ARG;
    } else if (n_seq != B) {
        return MDN_ERR_INVALID_ARG;
    }
    if (chunk != mdn::kChunk) return MDN_ERR_UNSUPPORTED;
    if (dk != dv || (dk != 64 && dk != 128)) return MDN_ERR_UNSUPPORTED;
    const long T_total = (long)B * T;
    if (T_total > 0x7fffffffL / 2) return MDN_ERR_INVALID_ARG;
    if ((long)T_total * H * dk > 0x7fffffffffffL) return MDN_ERR_INVALID_ARG;
    // ---- pointers
    if (T_total > 0 && (!alpha || !mu || !eta)) return MDN_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !o)) return MDN_ERR_INVALID_ARG;
    const void *ptrs16[] = {q, k, v, o, S0, M0, S_T, M_T, vres, S_chunks, M_chunks};
    for (const void *ptr : ptrs16)
        if (ptr && !aligned16(ptr)) return MDN_ERR_INVALID_ARG;
    const void *ptrs4[] = {alpha, mu, eta, beta, cu_seqlens};
    for (const void *ptr : ptrs4)
        if (ptr && ((uintptr_t)ptr & 3u)) return MDN_ERR_INVALID_ARG;
    if ((S_T && S_T != S0 && S0 && (const void *)S_T == (const void *)M0) ||
        (M_T && M_T != M0 && M0 && (const void *)M_T == (const void *)S0))
        return MDN_ERR_INVALID_ARG;
    if (S_T && M_T && S_T == M_T) return MDN_ERR_INVALID_ARG;
    // ---- device
    return status ? current_device(status) : MDN_OK;
}

}  // namespace mdn

namespace {

// Every chunk-forward entry point: validation, workspace carve-up, path
// choice and the launches.  vres (nullable) receives the per-token residuals.
// Long equal-length bf16 sequences whose state pass runs narrow slices (16
// or 32 state columns per CTA, each CTA leaving room on its SM for a prep
// CTA) are walked in time segments: the prep of segment k + 1 runs beside
// the state pass of segment k, which hides all but the first segment's prep.
// Segment k + 1's state pass starts from the states segment k left in S_T,
// M_T, so the path needs both (and no per-token or per-chunk side outputs).
// Segments of 16 chunks, then each twice the previous, the last taking the
// rest (or absorbing a remainder under a quarter segment): a segment's prep, on
// the SM room the state CTAs leave, runs at ~27 prepared blocks per µs,
// against the ~11 per µs the state pass of 16 heads consumes beside it (1.4
// µs per chunk), so the next segment's prep ends before the current state
// pass even at twice its length.
constexpr int kSegFirst = 16;
constexpr int kSegMinChunks = 128;

bool segments_apply(const mdn::ChunkProblem &p, bool packed, bool side_outputs,
                    bool final_states) {
    if (packed || p.dtype != MDN_BF16 || side_outputs || !final_states) return false;
    if ((p.T + mdn::kChunk - 1) / mdn::kChunk < kSegMinChunks) return false;
    const int ns = mdn::chunk_state_slice_width(p);
    return ns == 16 || ns == 32;
}

bool use_segments(const mdn::ChunkProblem &p) {
    return segments_apply(p, p.cu_seqlens != nullptr, p.vres || p.S_chunks, p.S_T && p.M_T);
}

// The end of the segment that starts at chunk c0 (its length `len`), out of
// cps chunks.
int segment_end(int c0, int len, int cps) {
    return cps - (c0 + len) < len / 4 ? cps : c0 + len;
}

int segment_count(int cps) {
    int n = 0;
    for (int c0 = 0, len = kSegFirst; c0 < cps; len *= 2, ++n) c0 = segment_end(c0, len, cps);
    return n;
}

cudaError_t launch_segments(const mdn::ChunkProblem &p, cudaStream_t cs) {
    const int cps = (p.T + mdn::kChunk - 1) / mdn::kChunk;
    cudaError_t err = cudaSuccess;
    int c0 = 0;
    for (int k = 0, len = kSegFirst; c0 < cps && err == cudaSuccess; ++k, len *= 2) {
        const int c1 = segment_end(c0, len, cps);
        const bool last = c1 == cps;
        mdn::ChunkProblem q = p;
        q.seg_c0 = c0;
        q.seg_c1 = c1;
        q.seg_mode = k > 0 ? mdn::kSegPrepFollower : 0;
        err = mdn::launch_chunk_prep_tc(q, cs);
        if (err != cudaSuccess) break;
        if (k > 0) {            // from the states the previous segment left
            q.S0 = p.S_T;
            q.M0 = p.M_T;
        }
        q.seg_mode = (last ? 0 : mdn::kSegStateTrigger) | (k > 0 ? mdn::kSegStateWaitFirst : 0);
        err = mdn::launch_chunk_state_tc(q, cs);
        c0 = c1;
    }
    return err;
}

mdn_status chunk_fwd_impl(
    const void *q, const void *k, const void *v, const float *alpha,
    const float *mu, const float *eta, const float *beta, const float *S0,
    const float *M0, void *o, float *S_T, float *M_T, void *vres,
    void *S_chunks, void *M_chunks,
    const int32_t *cu_seqlens, int n_seq, int B, int T, int H, int dk, int dv,
    mdn_dtype dtype, int chunk, void *workspace, size_t workspace_bytes,
    void *stream, void *const *stage_events, int n_stage_events,
    int *path_out) {
    if (n_stage_events != 0 && n_stage_events != 3) return MDN_ERR_INVALID_ARG;
    if (n_stage_events && !stage_events) return MDN_ERR_INVALID_ARG;
    for (int i = 0; i < n_stage_events; ++i)
        if (!stage_events[i]) return MDN_ERR_INVALID_ARG;
    mdn_status st = mdn::chunk_fwd_check(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T,
                                         vres, S_chunks, M_chunks, cu_seqlens, n_seq, B, T, H,
                                         dk, dv, dtype, chunk, nullptr);
    if (st != MDN_OK) return st;
    const long T_total = (long)B * T;
    const size_t need = mdn_chunk_fwd_workspace_size(n_seq, (int)T_total, H, dk, dv, dtype);
    if (n_seq > 0 && T_total > 0) {
        if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
            return MDN_ERR_INVALID_ARG;
    }

    int *status = nullptr;
    st = current_device(&status);
    if (st != MDN_OK) return st;
    if (n_seq == 0) return MDN_OK;

    mdn::ChunkProblem p;
    memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v;
    p.alpha = alpha; p.mu = mu; p.eta = eta; p.beta = beta;
    p.S0 = S0; p.M0 = M0; p.o = o; p.S_T = S_T; p.M_T = M_T; p.vres = vres;
    p.S_chunks = S_chunks; p.M_chunks = M_chunks;
    // with no tokens every sequence is empty: cu_seqlens is not read
    p.cu_seqlens = T_total > 0 ? cu_seqlens : nullptr;
    p.n_seq = n_seq; p.B = B; p.T = T; p.H = H; p.D = dk;
    p.T_total = (int)T_total;
    p.dtype = dtype;
    p.status = status;
    if (p.cu_seqlens) {
        p.max_chunks = (int)chunk_slots_bound(n_seq, (int)T_total);
    } else {
        p.max_chunks = B * ((T + mdn::kChunk - 1) / mdn::kChunk);
    }
    if (T_total == 0) p.max_chunks = 0;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    p.chunk_offsets = reinterpret_cast<int32_t *>(ws);
    p.seq_order = (p.cu_seqlens && ws)
                      ? reinterpret_cast<int32_t *>(ws + round256(sizeof(int32_t) * ((size_t)n_seq + 1)))
                      : nullptr;
    p.prep = ws ? ws + meta_bytes(n_seq) : nullptr;
    if (p.max_chunks == 0) p.seq_order = nullptr;   // the offsets kernel does not run
    p.prep_stride = mdn::kPrepBytesMax;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
    for (int i = 0; i < n_stage_events; ++i) ev[i] = static_cast<cudaEvent_t>(stage_events[i]);
    // The state pass runs on the tensor cores for every input: bf16 inputs
    // directly (prep on the tensor cores too), fp32 inputs as hi / lo bf16
    // parts with three products per contraction, their T and A_O T from the
    // fp32 prep (an fp32-level error bound needs the fp32 inverse).  With no
    // tokens only the initial states pass through.
    const bool tensor = T_total > 0;
    const bool split = tensor && dtype == MDN_F32;
    if (split) {
        const size_t part = split_part_bytes((int)T_total, H, dk);
        unsigned char *sp = ws + round256(meta_bytes(n_seq) + (size_t)chunk_slots_bound(
                                              n_seq, (int)T_total) * (size_t)H * mdn::kPrepBytesMax);
        p.q_hi = sp; p.q_lo = sp + part; p.k_hi = sp + 2 * part;
        p.k_lo = sp + 3 * part; p.v_hi = sp + 4 * part; p.v_lo = sp + 5 * part;
    }
    const int path = tensor ? MDN_PATH_TENSOR_CORE : MDN_PATH_CUDA_CORE;
    if (path_out) *path_out = path;
    cudaError_t err = cudaSuccess;
    if (ev[0]) err = cudaEventRecord(ev[0], cs);
    if (err == cudaSuccess && p.cu_seqlens && p.max_chunks > 0)
        err = mdn::launch_chunk_offsets(p, cs);
    if (err == cudaSuccess && split) err = mdn::launch_split_inputs(p, cs);
    if (tensor && !ev[1] && use_segments(p)) {
        // (stage events mark the prep and the state pass apart: whole sequences)
        if (err == cudaSuccess) err = launch_segments(p, cs);
    } else {
        if (err == cudaSuccess && tensor)
            err = split ? mdn::launch_chunk_prep_simt(p, cs) : mdn::launch_chunk_prep_tc(p, cs);
        if (err == cudaSuccess && ev[1]) err = cudaEventRecord(ev[1], cs);
        if (err == cudaSuccess)
            err = tensor ? mdn::launch_chunk_state_tc(p, cs) : mdn::launch_states_passthrough(p, cs);
    }
    if (err == cudaSuccess && ev[2]) err = cudaEventRecord(ev[2], cs);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    return MDN_OK;
}

}  // namespace

extern "C" {

mdn_status mdn_chunk_fwd_profiled(
    const void *q, const void *k, const void *v, const float *alpha,
    const float *mu, const float *eta, const float *beta, const float *S0,
    const float *M0, void *o, float *S_T, float *M_T,
    const int32_t *cu_seqlens, int n_seq, int B, int T, int H, int dk, int dv,
    mdn_dtype dtype, int chunk, void *workspace, size_t workspace_bytes,
    void *stream, void *const *stage_events, int n_stage_events,
    int *path_out) {
    return chunk_fwd_impl(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T, nullptr, nullptr, nullptr,
                          cu_seqlens, n_seq, B, T, H, dk, dv, dtype, chunk, workspace,
                          workspace_bytes, stream, stage_events, n_stage_events, path_out);
}

int mdn_chunk_fwd_kernel_count(int n_seq, int B, int T, int H, int dk, int dv, mdn_dtype dtype,
                               int packed, int final_states) {
    if (n_seq <= 0 || B <= 0 || T < 0 || H <= 0 || dk != dv || (dk != 64 && dk != 128) ||
        (dtype != MDN_F32 && dtype != MDN_BF16))
        return 0;
    if ((long)B * T == 0) return 1;                 // the initial states pass through
    mdn::ChunkProblem p;
    memset(&p, 0, sizeof(p));
    p.n_seq = n_seq; p.B = B; p.T = T; p.H = H; p.D = dk; p.dtype = dtype;
    p.T_total = B * T;
    int n = (packed ? 1 : 0) + (dtype == MDN_F32 ? 1 : 0);   // chunk offsets, split inputs
    if (segments_apply(p, packed != 0, false, final_states != 0))
        n += 2 * segment_count((T + mdn::kChunk - 1) / mdn::kChunk);
    else
        n += 2;                                     // prep, state pass
    return n;
}

mdn_status mdn_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *alpha, const float *mu, const float *eta,
                         const float *beta, const float *S0, const float *M0,
                         void *o, float *S_T, float *M_T,
                         const int32_t *cu_seqlens, int n_seq, int B, int T,
                         int H, int dk, int dv, mdn_dtype dtype, int chunk,
                         void *workspace, size_t workspace_bytes, void *stream) {
    return chunk_fwd_impl(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T, nullptr, nullptr, nullptr,
                          cu_seqlens, n_seq, B, T, H, dk, dv, dtype, chunk, workspace,
                          workspace_bytes, stream, nullptr, 0, nullptr);
}

mdn_status mdn_chunk_fwd_vres(const void *q, const void *k, const void *v,
                              const float *alpha, const float *mu, const float *eta,
                              const float *beta, const float *S0, const float *M0,
                              void *o, float *S_T, float *M_T, void *vres,
                              const int32_t *cu_seqlens, int n_seq, int B, int T,
                              int H, int dk, int dv, mdn_dtype dtype, int chunk,
                              void *workspace, size_t workspace_bytes, void *stream) {
    if ((long)B * T > 0 && !vres) return MDN_ERR_INVALID_ARG;
    if (vres && (vres == o || vres == v || vres == q || vres == k)) return MDN_ERR_INVALID_ARG;
    return chunk_fwd_impl(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T, vres, nullptr, nullptr,
                          cu_seqlens, n_seq, B, T, H, dk, dv, dtype, chunk, workspace,
                          workspace_bytes, stream, nullptr, 0, nullptr);
}

size_t mdn_chunk_state_slots(int n_seq, int B, int T, int packed) {
    if (n_seq < 0 || B < 0 || T < 0) return 0;
    const long T_total = (long)B * T;
    if (T_total > 0x7fffffffL) return 0;
    if (packed) return (size_t)chunk_slots_bound(n_seq, (int)T_total);
    return (size_t)B * (size_t)((T + mdn::kChunk - 1) / mdn::kChunk);
}

mdn_status mdn_chunk_fwd_states(const void *q, const void *k, const void *v,
                                const float *alpha, const float *mu, const float *eta,
                                const float *beta, const float *S0, const float *M0,
                                void *o, float *S_T, float *M_T, void *S_chunks,
                                void *M_chunks, const int32_t *cu_seqlens, int n_seq,
                                int B, int T, int H, int dk, int dv, mdn_dtype dtype,
                                int chunk, void *workspace, size_t workspace_bytes,
                                void *stream) {
    if ((long)B * T > 0 && (!S_chunks || !M_chunks)) return MDN_ERR_INVALID_ARG;
    if (S_chunks && S_chunks == M_chunks) return MDN_ERR_INVALID_ARG;
    const void *others[] = {q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T};
    for (const void *ptr : others)
        if (ptr && (ptr == S_chunks || ptr == M_chunks)) return MDN_ERR_INVALID_ARG;
    return chunk_fwd_impl(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T, nullptr,
                          S_chunks, M_chunks, cu_seqlens, n_seq, B, T, H, dk, dv, dtype,
                          chunk, workspace, workspace_bytes, stream, nullptr, 0, nullptr);
}

mdn_status mdn_prepare_inputs(const void *q_in, const void *k_in, const float *z_alpha,
                              const float *z_beta, const float *z_mu, const float *z_eta,
                              void *q_out, void *k_out, float *alpha, float *beta,
                              float *mu, float *eta, int n_tokens, int H, int d,
                              mdn_dtype dtype, float a, float b, float s, float tau,
                              float log_mu_min, float comba_d, void *stream) {
    if (n_tokens < 0 || H <= 0) return MDN_ERR_INVALID_ARG;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return MDN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return MDN_ERR_UNSUPPORTED;
    if (!(a > 0.f) || !(tau > 0.f)) return MDN_ERR_INVALID_ARG;   // also rejects NaN
    const long rows = (long)n_tokens * H;
    if (rows > 0) {
        const void *need[] = {q_in, k_in, z_alpha, z_beta, z_mu, z_eta, q_out, k_out,
                              alpha, beta, mu, eta};
        for (const void *ptr : need)
            if (!ptr) return MDN_ERR_INVALID_ARG;
    }
    const void *ptrs16[] = {q_in, k_in, q_out, k_out};
    for (const void *ptr : ptrs16)
        if (ptr && !aligned16(ptr)) return MDN_ERR_INVALID_ARG;
    const void *ptrs4[] = {z_alpha, z_beta, z_mu, z_eta, alpha, beta, mu, eta};
    for (const void *ptr : ptrs4)
        if (ptr && ((uintptr_t)ptr & 3u)) return MDN_ERR_INVALID_ARG;
    if (q_out && q_out == k_out) return MDN_ERR_INVALID_ARG;
    if ((q_out && q_out == k_in) || (k_out && k_out == q_in)) return MDN_ERR_INVALID_ARG;
    int *status = nullptr;
    mdn_status st = current_device(&status);
    if (st != MDN_OK) return st;
    if (rows == 0) return MDN_OK;
    mdn::InputsProblem p;
    p.q_in = q_in; p.k_in = k_in;
    p.z_alpha = z_alpha; p.z_beta = z_beta; p.z_mu = z_mu; p.z_eta = z_eta;
    p.q_out = q_out; p.k_out = k_out;
    p.alpha = alpha; p.beta = beta; p.mu = mu; p.eta = eta;
    p.rows = rows; p.D = d; p.dtype = dtype;
    p.a = a; p.b = b; p.s = s; p.tau = tau; p.log_mu_min = log_mu_min; p.comba_d = comba_d;
    if (mdn::launch_prepare_inputs(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    return MDN_OK;
}

mdn_status mdn_decode_step(const void *q, const void *k, const void *v,
                           const float *alpha, const float *mu,
                           const float *eta, const float *beta, float *S,
                           float *M, void *o, int N, int H, int dk, int dv,
                           mdn_dtype dtype, void *stream) {
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return MDN_ERR_INVALID_ARG;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return MDN_ERR_INVALID_ARG;
    if (dk != dv || (dk != 64 && dk != 128)) return MDN_ERR_UNSUPPORTED;
    if ((long)N * H > 0x7fffffffL / 4) return MDN_ERR_INVALID_ARG;
    if (N > 0) {
        if (!q || !k || !v || !alpha || !mu || !eta || !S || !M || !o)
            return MDN_ERR_INVALID_ARG;
        const void *ptrs16[] = {S, M};
        for (const void *ptr : ptrs16)
            if (!aligned16(ptr)) return MDN_ERR_INVALID_ARG;
        const uintptr_t emask = dtype == MDN_BF16 ? 1u : 3u;
        const void *ptrs_e[] = {q, k, v, o};
        for (const void *ptr : ptrs_e)
            if ((uintptr_t)ptr & emask) return MDN_ERR_INVALID_ARG;
        const void *ptrs4[] = {alpha, mu, eta, beta};
        for (const void *ptr : ptrs4)
            if (ptr && ((uintptr_t)ptr & 3u)) return MDN_ERR_INVALID_ARG;
        if (S == M) return MDN_ERR_INVALID_ARG;
    }
    int *status = nullptr;
    mdn_status st = current_device(&status);
    if (st != MDN_OK) return st;
    if (N == 0) return MDN_OK;

    mdn::DecodeProblem p;
    p.q = q; p.k = k; p.v = v;
    p.alpha = alpha; p.mu = mu; p.eta = eta; p.beta = beta;
    p.S = S; p.M = M; p.o = o;
    p.N = N; p.H = H; p.D = dk; p.dtype = dtype;
    p.status = status;
    if (mdn::launch_decode(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    return MDN_OK;
}

size_t mdn_chunk_bwd_workspace_size(int n_seq, int T_total, int H, int dk, int dv,
                                    mdn_dtype dtype) {
    if (n_seq < 0 || T_total < 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
    if (dtype != MDN_F32 && dtype != MDN_BF16) return 0;
    // per (chunk slot, head): the gradient block, then the chunk-end adjoints
    // (fp32 inputs: fp32, and the residual adjoints dR; bf16 inputs: bf16
    // operand tiles, and the tensor-core operand block)
    const size_t per = mdn::BwdLayout::kBytes +
                       (dtype == MDN_BF16
                            ? sizeof(__nv_bfloat16) * 2 * (size_t)dk * dv + mdn::BwdChainLayout::kBytes
                            : sizeof(float) * (2 * (size_t)dk * dv + (size_t)mdn::kChunk * dv));
    const size_t slots = (size_t)chunk_slots_bound(n_seq, T_total) * (size_t)H;
    return round256(meta_bytes(n_seq) + slots * per);
}

mdn_status mdn_chunk_bwd(const void *q, const void *k, const void *v, const float *alpha,
                         const float *mu, const float *eta, const float *beta,
                         const void *S_chunks, const void *M_chunks,
                         const void *fwd_workspace, const void *dout,
                         const float *dS_T, const float *dM_T, void *dq, void *dk_out,
                         void *dv_out, float *dalpha, float *dmu, float *deta, float *dbeta,
                         float *dS0, float *dM0, const int32_t *cu_seqlens, int n_seq, int B,
                         int T, int H, int dk, int dv, mdn_dtype dtype, int chunk,
                         void *workspace, size_t workspace_bytes, void *stream) {
    // shapes and the forward's own inputs as mdn_chunk_fwd checks them
    mdn_status st = mdn::chunk_fwd_check(q, k, v, alpha, mu, eta, beta, nullptr, nullptr, dout,
                                         nullptr, nullptr, nullptr, nullptr, nullptr, cu_seqlens,
                                         n_seq, B, T, H, dk, dv, dtype, chunk, nullptr);
    if (st != MDN_OK) return st;
    const long T_total = (long)B * T;
    if (T_total > 0) {
        const void *need[] = {S_chunks, M_chunks, dq, dk_out, dv_out, dalpha, dmu, deta};
        for (const void *ptr : need)
            if (!ptr) return MDN_ERR_INVALID_ARG;
    }
    const void *ptrs16[] = {S_chunks, M_chunks, dS_T, dM_T, dq, dk_out, dv_out, dS0, dM0};
    for (const void *ptr : ptrs16)
        if (ptr && !aligned16(ptr)) return MDN_ERR_INVALID_ARG;
    const void *ptrs4[] = {dalpha, dmu, deta, dbeta};
    for (const void *ptr : ptrs4)
        if (ptr && ((uintptr_t)ptr & 3u)) return MDN_ERR_INVALID_ARG;
    if (fwd_workspace && ((uintptr_t)fwd_workspace & 255u)) return MDN_ERR_INVALID_ARG;
    // no output may be an input or another output
    const void *ins[] = {q, k, v, alpha, mu, eta, beta, S_chunks, M_chunks, dout, dS_T, dM_T,
                         cu_seqlens, fwd_workspace};
    const void *outs[] = {dq, dk_out, dv_out, dalpha, dmu, deta, dbeta, dS0, dM0};
    for (int a = 0; a < 9; ++a) {
        if (!outs[a]) continue;
        for (const void *in : ins)
            if (in == outs[a]) return MDN_ERR_INVALID_ARG;
        for (int b = a + 1; b < 9; ++b)
            if (outs[b] == outs[a]) return MDN_ERR_INVALID_ARG;
    }
    const size_t need = mdn_chunk_bwd_workspace_size(n_seq, (int)T_total, H, dk, dv, dtype);
    if (n_seq > 0 && T_total > 0) {
        if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
            return MDN_ERR_INVALID_ARG;
    }
    int *status = nullptr;
    st = current_device(&status);
    if (st != MDN_OK) return st;
    if (n_seq == 0) return MDN_OK;

    mdn::BwdProblem p;
    memset(&p, 0, sizeof(p));
    mdn::ChunkProblem &L = p.loc;
    L.cu_seqlens = T_total > 0 ? cu_seqlens : nullptr;
    L.n_seq = n_seq; L.B = B; L.T = T; L.H = H; L.D = dk;
    L.T_total = (int)T_total;
    L.dtype = dtype;
    L.status = status;
    L.max_chunks = T_total == 0 ? 0
                 : L.cu_seqlens ? (int)chunk_slots_bound(n_seq, (int)T_total)
                                : B * ((T + mdn::kChunk - 1) / mdn::kChunk);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    L.chunk_offsets = reinterpret_cast<int32_t *>(ws);
    L.seq_order = (L.cu_seqlens && ws && L.max_chunks > 0)
                      ? reinterpret_cast<int32_t *>(ws + round256(sizeof(int32_t) * ((size_t)n_seq + 1)))
                      : nullptr;
    const size_t slots = ws ? (size_t)chunk_slots_bound(n_seq, (int)T_total) * (size_t)H : 0;
    unsigned char *base = ws ? ws + meta_bytes(n_seq) : nullptr;
    p.prep = base;
    p.adj = base ? reinterpret_cast<float *>(base + slots * mdn::BwdLayout::kBytes) : nullptr;
    if (dtype == MDN_BF16) {
        // bf16 inputs run on the tensor cores: the adjoints as bf16 operand
        // tiles, then the operand blocks
        p.tcblk = (p.adj && T_total > 0)
                      ? reinterpret_cast<unsigned char *>(p.adj) +
                            slots * sizeof(__nv_bfloat16) * 2 * (size_t)dk * dv
                      : nullptr;
        // the forward's prepared blocks, laid out as mdn_chunk_fwd lays out
        // its workspace: their [T; A_O T] tiles are the gradient's
        if (fwd_workspace && p.tcblk) {
            p.fwd_tile = static_cast<const unsigned char *>(fwd_workspace) + meta_bytes(n_seq);
            p.fwd_tile_stride = mdn::kPrepBytesMax;
        }
    } else {
        // fp32 inputs keep the fp32 kernels (for the fp32 bound)
        p.dR = p.adj ? p.adj + slots * 2 * (size_t)dk * dv : nullptr;
    }
    p.q = q; p.k = k; p.v = v; p.dout = dout;
    p.alpha = alpha; p.mu = mu; p.eta = eta; p.beta = beta;
    p.S_chunks = S_chunks; p.M_chunks = M_chunks;
    p.dS_T = dS_T; p.dM_T = dM_T;
    p.dq = dq; p.dk = dk_out; p.dv = dv_out;
    p.dalpha = dalpha; p.dmu = dmu; p.deta = deta; p.dbeta = dbeta;
    p.dS0 = dS0; p.dM0 = dM0;
    p.D = dk;
    p.dtype = dtype;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaSuccess;
    if (L.cu_seqlens && L.max_chunks > 0) err = mdn::launch_chunk_offsets(L, cs);
    if (err == cudaSuccess) err = mdn::launch_chunk_bwd(p, cs);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    return MDN_OK;
}

mdn_status mdn_wait_selftest(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 1000000) return MDN_ERR_INVALID_ARG;
    int *status = nullptr;
    mdn_status st = current_device(&status);
    if (st != MDN_OK) return st;
    if (mdn::launch_wait_selftest((uint64_t)limit_us * 1000u, status,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    return MDN_OK;
}

mdn_status mdn_get_device_status(void *stream) {
    int *status = nullptr;
    mdn_status st = current_device(&status);
    if (st != MDN_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    int value = 0;
    const int zero = 0;
    if (cudaMemcpy(&value, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    return value == 0 ? MDN_OK : (mdn_status)value;
}

}  // extern "C"
