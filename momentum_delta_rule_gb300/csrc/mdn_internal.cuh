// Internal declarations shared by the MDN CUDA translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "mdn.h"

namespace mdn {

constexpr int kChunk = 64;  // tokens per chunk (the pages' default C)

// Per-(chunk, head) prepared block written by the prep kernel and read by the
// state-pass kernel.  Matrices are row-major 64 x 64 of `MatT`; vectors fp32.
//   T    = [I + (P Khat^T) . Gamma_shifted]^{-1}
//   AOT  = [(Q Khat^T) . Gamma] T
//   vec  = kVecRows rows of 64 fp32 (see VecRow)
enum VecRow {
    kVecAbar = 0,     // abar_i = prod_{r<=i} alpha_r        (also abar_{i-1} alpha_i)
    kVecBmA = 1,      // b_{i-1} alpha_i  (b_0 = 0)
    kVecB = 2,        // b_i
    kVecGS = 3,       // gamma_{n,i} eta_i      (carry weight of S)
    kVecGM = 4,       // prod_{u=i+1}^{n} mu_u eta_i (carry weight of M)
    kVecScal = 5,     // [0] abar_n, [1] b_n, [2] mubar_n, [3] n (as float)
    kVecRows = 8
};

template <typename MatT>
struct PrepLayout {
    static constexpr size_t kMatBytes = sizeof(MatT) * kChunk * kChunk;
    static constexpr size_t kVecBytes = sizeof(float) * kChunk * kVecRows;
    static constexpr size_t kOffT = 0;
    static constexpr size_t kOffAOT = kMatBytes;
    static constexpr size_t kOffVec = 2 * kMatBytes;
    static constexpr size_t kBytes = 2 * kMatBytes + kVecBytes;
};

// Prepared block of the tensor-core path: T and A_O T in bf16, each 64 rows
// of 128 bytes stored in the 128-byte-swizzled K-major operand layout of
// tcgen05.mma (16-byte chunk c of row r at (r/8)*1024 + (r%8)*128 +
// ((c ^ (r%8)) * 16)), followed by the fp32 vectors.  One bulk copy of the
// whole block into 1024-byte-aligned shared memory yields the MMA operand
// [T; A_O T] directly.
//
// Row order: the 128 operand rows are interleaved in blocks of 16 so that
// every 32-lane TMEM quadrant of the products holds 16 rows of each half:
// T (or K) row i sits at row 32 (i / 16) + i % 16, A_O T (or Q) row i at
// row 32 (i / 16) + 16 + i % 16.  The state pass loads its [K; Q] tiles in
// the same order.
__host__ __device__ constexpr int tc_row(int r) {
    return r < kChunk ? 32 * (r >> 4) + (r & 15) : 32 * ((r - kChunk) >> 4) + 16 + (r & 15);
}

struct PrepLayoutTC {
    static constexpr size_t kOffT = 0;
    static constexpr size_t kOffAOT = 8192;
    static constexpr size_t kOffVec = 16384;
    static constexpr size_t kBytes = 16384 + sizeof(float) * kChunk * kVecRows;
    // fp32 inputs: the operand [T; A_O T] as two bf16 parts, hi = bf16(x)
    // at 0 and lo = bf16(x - hi) at kSplitLo, then the vectors
    static constexpr size_t kSplitLo = 16384;
    static constexpr size_t kSplitVec = 32768;
    static constexpr size_t kSplitBytes = 32768 + sizeof(float) * kChunk * kVecRows;
};

// Largest prepared block of any path (fp32 matrices).
constexpr size_t kPrepBytesMax = PrepLayout<float>::kBytes;

struct ChunkProblem {
    const void *q, *k, *v;
    const float *alpha, *mu, *eta, *beta;
    const float *S0, *M0;
    void *o;
    float *S_T, *M_T;
    void *vres;                  // per-token residuals like v, or nullptr
    void *S_chunks, *M_chunks;   // entry states of every chunk [slot, H, dk, dv] (bf16 for
                                 // bf16 inputs, fp32 for fp32), or nullptr
    const int32_t *cu_seqlens;   // device, or nullptr for equal lengths
    int n_seq, B, T, H, D;       // dk == dv == D
    int T_total;                 // B * T
    int max_chunks;              // prepared-block slots per head
    mdn_dtype dtype;
    int32_t *chunk_offsets;      // [n_seq + 1] in the workspace (varlen only)
    int32_t *seq_order;          // [n_seq] sequences longest first (varlen only), or null
    unsigned char *prep;         // max_chunks * H prepared blocks
    size_t prep_stride;          // bytes per prepared block
    int *status;                 // device status word
    // fp32 inputs on the tensor cores: q, k, v as hi / lo bf16 parts
    // [T_total, H, D] in the workspace (null for bf16 inputs)
    void *q_hi, *q_lo, *k_hi, *k_lo, *v_hi, *v_lo;
    // A time segment of equal-length sequences: chunks [seg_c0, seg_c1) of
    // every sequence (seg_c1 <= seg_c0: the whole sequences), and how the
    // segment's kernels meet their neighbours in the stream (kSeg* bits).
    int seg_c0, seg_c1;
    int seg_mode;
};

// seg_mode bits.  Segment k's state pass lets the next launch (segment
// k + 1's prep) start once all its CTAs run, so that prep fills what the
// state CTAs leave of the SMs; that prep neither lets its own dependent (the
// state pass of segment k + 1) start early nor finishes before segment k's
// state pass has: its last CTA waits for it.  Segment k + 1's state pass
// therefore finds the states segment k left in S_T, M_T complete.
enum SegMode {
    kSegStateTrigger = 1,     // state pass: trigger the dependent launch at start
    kSegStateWaitFirst = 2,   // state pass: wait for the preceding grids before reading S0, M0
    kSegPrepFollower = 4,     // prep: no early trigger; the last CTA waits for the preceding grid
};

__host__ __device__ inline bool is_segment(const ChunkProblem &p) { return p.seg_c1 > p.seg_c0; }

struct DecodeProblem {
    const void *q, *k, *v;
    const float *alpha, *mu, *eta, *beta;
    float *S, *M;
    void *o;
    int N, H, D;
    mdn_dtype dtype;
    int *status;
};

// Launchers (return the first CUDA error, or cudaSuccess).
struct InputsProblem {
    const void *q_in, *k_in;
    const float *z_alpha, *z_beta, *z_mu, *z_eta;
    void *q_out, *k_out;
    float *alpha, *beta, *mu, *eta;
    long rows;                   // tokens x heads
    int D;
    mdn_dtype dtype;
    float a, b, s, tau, log_mu_min, comba_d;
};

// Gradient pass (mdn_chunk_bwd).  `loc` carries the chunk geometry (packed
// offsets, sequence order, status word) for the shared location helpers.
struct BwdProblem {
    ChunkProblem loc;
    const void *q, *k, *v, *dout;
    const float *alpha, *mu, *eta, *beta;
    const void *S_chunks, *M_chunks;   // entry states of every chunk [slot, H, dk, dv],
                                       // in the input precision
    const float *dS_T, *dM_T;          // adjoints of the final states, or nullptr (zero)
    void *dq, *dk, *dv;
    float *dalpha, *dmu, *deta, *dbeta;
    float *dS0, *dM0;
    unsigned char *prep;               // per (slot, head): chunk matrices and vectors
    float *adj;                        // per (slot, head): dS, dM at the chunk's end, fp32
                                       // [2, dk, dv] (fp32 inputs) or bf16 operand tiles
    float *dR;                         // per (slot, head): residual adjoints [64, dv] (fp32 inputs)
    unsigned char *tcblk;              // per (slot, head): the tensor-core chain's operands, or null
    const unsigned char *fwd_tile;     // the forward's prepared blocks (their [T; A_O T] tiles
                                       // serve as the operand blocks' tiles), or null
    size_t fwd_tile_stride;
    int D;
    mdn_dtype dtype;
};

// Per-(slot, head) operand block of the tensor-core gradient kernels (bf16
// inputs): the forward prep's operand tile [T; A_O T] (PrepLayoutTC: bf16,
// 128-byte-swizzled K-major, rows in the tc_row order), then kRows rows of
// 64 fp32 per-token coefficients of the reverse chain, which replace the
// forward's carry vectors there.
struct BwdChainLayout {
    static constexpr size_t kOffTile = 0;
    static constexpr size_t kOffVec = PrepLayoutTC::kOffVec;
    enum { vCS = 0, vCM, vBS, vBM, vQS, vQM, vScal, kRows = 8 };
    static constexpr size_t kBytes = kOffVec + sizeof(float) * kChunk * kRows;
};
static_assert(BwdChainLayout::kBytes == PrepLayoutTC::kBytes, "the forward prep writes the block");

// Per-(slot, head) block of the gradient pass, fp32: five 64 x 64 matrices
// (T, A = (Q Kh^T) . Gamma, X = P Kh^T, Y = Q Kh^T, Gamma), then vector rows.
struct BwdLayout {
    static constexpr int kMat = kChunk * kChunk;
    enum { kT = 0, kA = 1, kX = 2, kY = 3, kG = 4, kMats = 5 };
    enum { vAbar = 0, vB, vAbarM, vBM, vGS, vMuTail, vScal, kRows = 8 };
    static constexpr size_t kBytes = sizeof(float) * ((size_t)kMats * kMat + (size_t)kRows * kChunk);
};

// Shape and pointer checks of the chunk-forward entry points (all but the
// workspace), then, if `status` is not null, the device check, whose success
// stores the device status word there.
mdn_status chunk_fwd_check(const void *q, const void *k, const void *v, const float *alpha,
                           const float *mu, const float *eta, const float *beta,
                           const float *S0, const float *M0, const void *o, const float *S_T,
                           const float *M_T, const void *vres, const void *S_chunks,
                           const void *M_chunks, const int32_t *cu_seqlens, int n_seq,
                           int B, int T, int H, int dk, int dv, mdn_dtype dtype, int chunk,
                           int **status);

cudaError_t launch_prepare_inputs(const InputsProblem &p, cudaStream_t st);
cudaError_t launch_chunk_offsets(const ChunkProblem &p, cudaStream_t st);
cudaError_t launch_chunk_prep_simt(const ChunkProblem &p, cudaStream_t st);
cudaError_t launch_split_inputs(const ChunkProblem &p, cudaStream_t st);
cudaError_t launch_chunk_prep_tc(const ChunkProblem &p, cudaStream_t st);
cudaError_t launch_chunk_state_tc(const ChunkProblem &p, cudaStream_t st);
// The slice width (state columns per CTA) the state pass picks for p.
int chunk_state_slice_width(const ChunkProblem &p);
cudaError_t launch_states_passthrough(const ChunkProblem &p, cudaStream_t st);
cudaError_t launch_decode(const DecodeProblem &p, cudaStream_t st);
cudaError_t launch_wait_selftest(uint64_t limit_ns, int *status, cudaStream_t st);
cudaError_t launch_chunk_bwd(const BwdProblem &p, cudaStream_t st);
cudaError_t launch_bwd_chain_tc(const BwdProblem &p, cudaStream_t st);
cudaError_t launch_bwd_chunk_tc(const BwdProblem &p, cudaStream_t st);

// Multiprocessor count of the current device, cached per device (0 when it
// cannot be read).
inline int device_sm_count() {
    // per device, filled on first use; atomic because host threads driving
    // different streams may launch concurrently
    static std::atomic<int> count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = count[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        count[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

// ---------------------------------------------------------------- device

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Where chunk `gc` (a global chunk slot) lives.  Equal-length batches chunk
// every sequence of T tokens from its own start; packed varlen batches use
// the per-sequence chunk offsets computed on the device.
struct ChunkLoc {
    int seq;     // sequence index
    int t0;      // first token (row of the packed [T_total, H, *] tensors)
    int n;       // tokens in this chunk, 1..64
};

__device__ __forceinline__ bool locate_chunk(const ChunkProblem &p, int gc,
                                             ChunkLoc &loc) {
    if (p.cu_seqlens == nullptr) {
        const int cps = (p.T + kChunk - 1) / kChunk;
        if (cps == 0) return false;
        const int s = gc / cps;
        if (s >= p.n_seq) return false;
        const int c = gc - s * cps;
        loc.seq = s;
        loc.t0 = s * p.T + c * kChunk;
        loc.n = min(kChunk, p.T - c * kChunk);
        return true;
    }
    const int32_t *off = p.chunk_offsets;
    if (gc >= off[p.n_seq]) return false;
    // largest s with off[s] <= gc (empty sequences have off[s] == off[s+1])
    int lo = 0, hi = p.n_seq;     // off[lo] <= gc < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= gc) lo = mid; else hi = mid;
    }
    const int c = gc - off[lo];
    const int start = p.cu_seqlens[lo];
    const int len = p.cu_seqlens[lo + 1] - start;
    loc.seq = lo;
    loc.t0 = start + c * kChunk;
    loc.n = min(kChunk, len - c * kChunk);
    return true;
}

// Chunk-parallel kernels run one CTA per (chunk, head) on a 1-D grid with the
// head varying fastest, so that the heads of a chunk, whose rows of q, k and
// v sit side by side in memory, are resident together and read whole rows.
inline bool chunk_head_grid(int max_chunks, int H, dim3 &grid) {
    const long long n = (long long)max_chunks * H;
    if (n <= 0 || n > 0x7fffffffLL) return false;
    grid = dim3((unsigned)n);
    return true;
}
__device__ __forceinline__ void chunk_head_of_block(int H, int &gc, int &h) {
    const unsigned b = blockIdx.x;
    gc = (int)(b / (unsigned)H);
    h = (int)(b - (unsigned)gc * (unsigned)H);
}

// locate_chunk for a whole CTA at once (every thread calls it; uniform
// result): for packed sequences the containing sequence is the count of
// chunk offsets at or below gc, taken in one round of parallel loads per
// blockDim.x sequences instead of a chain of dependent loads.
__device__ __forceinline__ bool locate_chunk_cta(const ChunkProblem &p, int gc, ChunkLoc &loc) {
    if (p.cu_seqlens == nullptr) return locate_chunk(p, gc, loc);
    const int32_t *off = p.chunk_offsets;
    const int total = off[p.n_seq];
    int lo = 0;
    for (int base = 1; base < p.n_seq; base += blockDim.x) {
        const int s = base + (int)threadIdx.x;
        lo += __syncthreads_count(s < p.n_seq && off[s] <= gc);
    }
    if (gc >= total) return false;
    const int start = p.cu_seqlens[lo];
    const int len = p.cu_seqlens[lo + 1] - start;
    const int c = gc - off[lo];
    loc.seq = lo;
    loc.t0 = start + c * kChunk;
    loc.n = min(kChunk, len - c * kChunk);
    return true;
}

// The state pass walks sequences longest first when an order is given, so the
// longest chains start in the first wave (longest-processing-time order).
__device__ __forceinline__ int ordered_sequence(const ChunkProblem &p, int k) {
    return p.seq_order ? p.seq_order[k] : k;
}

// Token range and chunk-slot base of one sequence.
__device__ __forceinline__ void sequence_range(const ChunkProblem &p, int s,
                                               int &start, int &len,
                                               int &slot0) {
    if (p.cu_seqlens == nullptr) {
        start = s * p.T;
        len = p.T;
        slot0 = s * ((p.T + kChunk - 1) / kChunk);
    } else {
        // Packed sequences exist only with T_total > 0 (the API drops
        // cu_seqlens otherwise), so the chunk offsets have been computed.
        // The sequence keeps at most the chunks its offsets give it: all of
        // them for valid offsets (ceil(len / 64)), none when the offsets
        // kernel rejected cu_seqlens and zeroed them.
        start = p.cu_seqlens[s];
        len = p.cu_seqlens[s + 1] - start;
        slot0 = p.chunk_offsets[s];
        len = max(0, min(len, (p.chunk_offsets[s + 1] - slot0) * kChunk));
    }
}

}  // namespace mdn
