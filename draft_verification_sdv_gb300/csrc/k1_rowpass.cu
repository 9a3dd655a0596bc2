// k1_rowpass.cu -- single-pass online softmax statistics of every logit row.
//
// Temperature softmax of the verifier rows p(.|s, x_<j) and drafter rows
// q_j over the full vocabulary ("SpecDiff-2: Scaling Diffusion Drafter
// Alignment For Faster Speculative Decoding", section 2: the verifier scores
// all positions in parallel; section 5.2: its probabilities are computed once
// and reused by ranking and acceptance).  Each row is read exactly once.
//
// Work decomposition: each row is cut into `chunks` fixed chunks of
// `chunk_vec` 16-byte vectors.  One warp reduces one (row, chunk) item to
// (m, s) = (max l, sum 2^{(l - m) c}), c = log2(e) / T, with a fixed lane
// mapping and a fixed reduction tree, so two rows with the same bytes and the
// same temperature give bit-identical partials whatever their position.  The
// grid holds one CTA per eight items and runs in many waves: the hardware
// hands each freed slot the next CTA, which keeps every SM streaming until
// the end (measured faster than a persistent grid with a static order).
// Row mode, for batches whose rows about fill one wave of four-warp CTAs:
// one CTA per row, its 4 KB blocks dealt to the warps in a fixed interleaved
// order, the warps' (m, s) merged in warp order into one partial per row.
//
// The kernel is HBM-bandwidth bound: per element one 2-byte load, one
// exponential on the special-function unit and a handful of fp32 operations.
#include "sdv_device.cuh"
#include "sdv_plan.h"

namespace sdv {
namespace {

constexpr int kUnroll = 8;   // 16-byte vectors in flight per lane per iteration

// Packed 16-byte vector of -inf values: fills the lanes past a chunk's end.
template <bool BF16>
__device__ __forceinline__ uint4 neg_inf_vec() {
    const uint32_t w = BF16 ? 0xFF80FF80u : 0xFF800000u;
    return make_uint4(w, w, w, w);
}

// The row `row` of the p rows followed by the q rows: its vectors and its
// sequence, or nullptr for a row that is not read (a prefix row that the
// shared one replaces, a row past its sequence's draft length).
__device__ __forceinline__ const uint4* row_source(const RowPassArgs& a, int64_t row, int64_t* seq) {
    const int64_t rows_per_seq_p = static_cast<int64_t>(a.K) * (a.G + 1);
    const int64_t rows_per_seq_q = (a.flags & kFlagSharedQ) ? a.G : static_cast<int64_t>(a.K) * a.G;
    // a sequence with shorter drafts needs no row past its length
    auto draft_len = [&](int64_t b) {
        const int L = a.lens ? __ldg(a.lens + b) : a.G;
        return L < 0 || L > a.G ? a.G : L;            // out of range: K2 reports it
    };
    if (row < a.rows_p) {
        const int64_t b = row / rows_per_seq_p;
        *seq = b;
        const int64_t r = row - b * rows_per_seq_p;
        if ((a.flags & kFlagSharedPrefixRow) && r > a.G && r % (a.G + 1) == 0) return nullptr;
        if (a.lens && r % (a.G + 1) > draft_len(b)) return nullptr;
        return static_cast<const uint4*>(a.p) + row * a.nvec;
    }
    const int64_t b = (row - a.rows_p) / rows_per_seq_q;
    *seq = b;
    if (a.lens && ((row - a.rows_p) - b * rows_per_seq_q) % a.G >= draft_len(b)) return nullptr;
    return static_cast<const uint4*>(a.q) + (row - a.rows_p) * a.nvec;
}

// Add vectors [v0, v1) of a row to a lane's (m, s): lane l takes vectors
// v0 + l, v0 + l + 32, ..., kUnroll of them in flight.
template <bool BF16>
__device__ __forceinline__ void stream_vectors(const uint4* rowv, int64_t v0, int64_t v1, int lane,
                                               float c, float& m, float& s) {
    for (int64_t base = v0 + lane; base < v1; base += 32 * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t idx = base + 32 * u;
            v[u] = idx < v1 ? ld_stream(rowv + idx) : neg_inf_vec<BF16>();
        }
        const float vm = vec_max_n<BF16, kUnroll>(v);
        if (!(vm <= m)) {                 // new maximum (or NaN: poisons s)
            s *= ex2((m - vm) * c);
            m = vm;
        }
        if (m != -INFINITY) {             // all -inf so far: nothing to add
            float t[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) t[u] = vec_exp_sum<BF16>(v[u], m, c);
#pragma unroll
            for (int w = kUnroll / 2; w > 0; w >>= 1)
#pragma unroll
                for (int u = 0; u < w; ++u) t[u] += t[u + w];
            s += t[0];
        }
    }
}

__device__ __forceinline__ void warp_merge(float& m, float& s, float c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        merge_stat(m, s, m2, s2, c);
    }
}

// Item mode: one warp per (row, chunk) item.
template <bool BF16>
__global__ void __launch_bounds__(kRowPassThreads) rowpass_kernel(const RowPassArgs a) {
    // Launched as a programmatic dependent of the previous step's sample
    // kernel, this grid may be resident before that kernel ends: wait for it
    // (and its memory) before reading or writing anything.  A no-op when the
    // launch is an ordinary one.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Then let the select kernel launch: it waits for this grid before it
    // reads any partial, but fetches the step's drafted tokens before that,
    // so it must not start before the work ahead of this grid has finished.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * kRowPassThreads + threadIdx.x) >> 5;
    if (item >= a.items) return;
    const int64_t row = item / a.chunks;
    const int64_t chunk = item - row * a.chunks;
    int64_t b = 0;
    const uint4* rowv = row_source(a, row, &b);
    if (!rowv) return;
    const float T = a.temps ? __ldg(a.temps + b) : a.temperature;
    const float c = kLog2e / T;
    const int64_t v0 = chunk * a.chunk_vec;
    const int64_t v1 = min(v0 + a.chunk_vec, a.nvec);
    float m = -INFINITY, s = 0.0f;
    stream_vectors<BF16>(rowv, v0, v1, lane, c, m, s);
    warp_merge(m, s, c);
    if (lane == 0) a.part[item] = make_float2(m, s);
}

// Row mode: one CTA per row.  The row's 4 KB blocks go to the CTA's warps in
// a fixed interleaved order (warp w takes blocks w, w + 4, ...), each warp
// keeps one (m, s) over its blocks, and the CTA merges its warps' in warp
// order into the row's single partial.
template <bool BF16>
__global__ void __launch_bounds__(kRowModeThreads, kRowModeMinBlocks) rowpass_row_kernel(const RowPassArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int NW = kRowModeThreads / 32;
    __shared__ float2 s_part[NW];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = blockIdx.x;
    int64_t b = 0;
    const uint4* rowv = row_source(a, row, &b);
    if (!rowv) return;                        // the same for the whole CTA
    const float T = a.temps ? __ldg(a.temps + b) : a.temperature;
    const float c = kLog2e / T;
    float m = -INFINITY, s = 0.0f;
    for (int64_t v0 = static_cast<int64_t>(warp) * kRowBlockVec; v0 < a.nvec; v0 += NW * kRowBlockVec)
        stream_vectors<BF16>(rowv, v0, min(v0 + kRowBlockVec, a.nvec), lane, c, m, s);
    warp_merge(m, s, c);
    if (lane == 0) s_part[warp] = make_float2(m, s);
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = s_part[0].x, S = s_part[0].y;
#pragma unroll
        for (int w = 1; w < NW; ++w) merge_stat(M, S, s_part[w].x, s_part[w].y, c);
        a.part[row] = make_float2(M, S);
    }
}

}  // namespace

cudaError_t rowpass_occupancy(bool bf16, int* blocks_per_sm) {
    return bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, rowpass_kernel<true>,
                                                                kRowPassThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      blocks_per_sm, rowpass_kernel<false>, kRowPassThreads, 0);
}

cudaError_t rowpass_row_occupancy(bool bf16, int* blocks_per_sm) {
    return bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, rowpass_row_kernel<true>,
                                                                kRowModeThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, rowpass_row_kernel<false>,
                                                                kRowModeThreads, 0);
}

cudaError_t launch_rowpass(const RowPassArgs& a, bool bf16, cudaStream_t s, bool pdl) {
    const int64_t per_cta = a.row_mode ? 1 : kRowPassThreads / 32;
    const int64_t g = (a.items + per_cta - 1) / per_cta;
    if (g < 1 || g > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if (a.row_mode && a.chunks != 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(g));
    cfg.blockDim = dim3(a.row_mode ? kRowModeThreads : kRowPassThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (a.row_mode)
        return bf16 ? cudaLaunchKernelEx(&cfg, rowpass_row_kernel<true>, a)
                    : cudaLaunchKernelEx(&cfg, rowpass_row_kernel<false>, a);
    if (bf16) return cudaLaunchKernelEx(&cfg, rowpass_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, rowpass_kernel<false>, a);
}

}  // namespace sdv
