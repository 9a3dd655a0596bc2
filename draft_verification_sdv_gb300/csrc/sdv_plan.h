// sdv_plan.h -- launch plan and kernel argument blocks shared by the host
// side of libsdv and its three kernels.  Internal; the public ABI is sdv.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sdv {

// Layout flags of a context (the public SDV_FLAG_* values).
enum : unsigned {
    kFlagSharedQ = 1u,       // q is [B][G][V]: one marginal row per (b, j), shared by all k
    kFlagGreedy = 2u,        // greedy acceptance: no drafter rows at all
    kFlagSharedPrefixRow = 4u,   // the verifier row at j = 0 is (b, 0, 0) for every k
};

// Row index of the verifier row of (b, k, j) within the p buffer.  The row at
// j = 0 sees only the prefix s, so with kFlagSharedPrefixRow the row of draft
// 0 serves every draft (the others are not read).
__host__ __device__ __forceinline__ int64_t p_row_index(unsigned flags, int b, int k, int j, int K,
                                                        int G) {
    const int kk = (flags & kFlagSharedPrefixRow) && j == 0 ? 0 : k;
    return (static_cast<int64_t>(b) * K + kk) * (G + 1) + j;
}

// Row index of the drafter row of (b, k, j) within the q buffer.
__host__ __device__ __forceinline__ int64_t q_row_index(unsigned flags, int b, int k, int j, int K,
                                                        int G) {
    return (flags & kFlagSharedQ) ? static_cast<int64_t>(b) * G + j
                                  : (static_cast<int64_t>(b) * K + k) * G + j;
}

// Bits of the device status word.
enum : unsigned {
    kStatusBadDraft = 1u,    // a draft id outside [0, V)
    kStatusBadRow = 2u,      // a row with NaN / +inf, or only -inf
    kStatusBadTemp = 4u,     // per-sequence temperature not finite and positive
    kStatusTimeout = 8u,     // a bounded device wait gave up
    kStatusBadLength = 16u,  // a draft length outside [kmin, kmax] given to the controller
    kStatusBadStat = 32u,    // supplied drafter-row statistics of another temperature
};

// Adaptive draft length ("DiffuSpec", section 4.3).  A sequence's state is
// [entries in the window (at most W), next ring slot, sum k, sum g, sum a,
// then the W ring entries of k, of g and of a].  One step records (k, g, a)
// -- g clamped to [0, k], a to [0, g] -- evicting the oldest entry of a full
// window, and returns the next draft length: grow by `up` when the window's
// accepted lengths sum to its generated ones and those to its drafted ones,
// hold when only the first holds (generation saturated by EOS), shrink by
// `down` otherwise; clamped to [kmin, kmax].  Shared by the host entry point
// and the device kernel.
constexpr int kAdlMaxWindow = 64;
constexpr int kAdlMaxLength = 1 << 20;
__host__ __device__ inline int adl_state_words(int W) { return 5 + 3 * W; }

__host__ __device__ inline int32_t adl_update(int32_t* st, int W, int kmin, int kmax, int up,
                                              int down, int32_t k, int32_t g, int32_t a) {
    g = g < 0 ? 0 : (g > k ? k : g);
    a = a < 0 ? 0 : (a > g ? g : a);
    int32_t* rk = st + 5;
    int32_t* rg = rk + W;
    int32_t* ra = rg + W;
    int32_t n = st[0], pos = st[1], sk = st[2], sg = st[3], sa = st[4];
    if (n == W) {
        sk -= rk[pos];
        sg -= rg[pos];
        sa -= ra[pos];
    } else {
        ++n;
    }
    rk[pos] = k;
    rg[pos] = g;
    ra[pos] = a;
    sk += k;
    sg += g;
    sa += a;
    st[0] = n;
    st[1] = pos + 1 == W ? 0 : pos + 1;
    st[2] = sk;
    st[3] = sg;
    st[4] = sa;
    int32_t next = k;
    if (sa >= sg && sg >= sk)
        next = k + up;
    else if (sa < sg)
        next = k - down;
    return next < kmin ? kmin : (next > kmax ? kmax : next);
}


// The draw to make for one sequence, decided by the selection and scan.
// mode 0: nothing to draw (data error); 1: residual max(0, p - q) of rows
// (row_p, row_q); 2: bonus draw from row_p alone; 3: greedy replacement, row_p
// with the token zero_id zeroed out.
// The probability of token v of a row is 2^(l_v * c + off) with
// off = -(max * c) - log2(sum 2^{(l - max) c}): one fused multiply-add and
// one exponential per logit.
struct SeqTask {
    int mode;
    int zero_id;
    int64_t row_p;      // row index within the p buffer
    int64_t row_q;      // row index within the q buffer
    float w;            // sampling uniform
    float c;            // log2(e) / T
    float off_p;        // exponent offset of the p row
    float off_q;        // exponent offset of the q row (residual only)
};

// Row pass (K1): rows are split into `chunks` fixed chunks of `chunk_vec`
// 16-byte vectors (the last chunk of a row may be shorter); one warp reduces
// one (row, chunk) item to a partial (max, sum of 2^{(l - max) c}).  Launched
// with one CTA per kRowPassThreads / 32 items.
struct RowPassArgs {
    const void* p;          // [rows_p][V]
    const void* q;          // [rows_q][V]
    float2* part;           // [rows_p + rows_q][chunks]
    const float* temps;     // [B] or nullptr
    float temperature;
    int K, G;
    int chunks;
    unsigned flags;
    int64_t rows_p, rows_total;
    int64_t nvec;           // vectors per row
    int64_t chunk_vec;      // vectors per chunk
    int64_t items;          // rows_total * chunks
    const int32_t* lens = nullptr;   // [B] draft length per sequence (rows past it are skipped)
    // one CTA of kRowModeThreads per row (items = rows, chunks = 1) instead
    // of one warp per item
    int row_mode = 0;
};

// Select / scan (K2): one CTA per sequence.
struct SelectArgs {
    const void* p;
    const void* q;
    const int32_t* drafts;
    const float2* part;
    const float* temps;
    float temperature;
    int B, K, G, V, chunks;
    unsigned flags;
    int64_t rows_p;
    uint32_t seed_lo, seed_hi;
    int32_t* out_sel;
    int32_t* out_len;
    int32_t* out_tok;       // written with -1 here on a data error
    float* out_scores;      // [B][K] or nullptr
    float* out_lse;         // [B][K][2G+1] or nullptr
    SeqTask* tasks;
    unsigned* status;
    const int32_t* lens = nullptr;   // [B] draft length per sequence, or nullptr (= G)
    // lanes that merge one row's chunk partials together: a power of two,
    // at most 32 (select_merge_lanes)
    int merge_lanes = 1;
    // [rows_q] drafter-row statistics {max, sum 2^{(l - max) c}, c, 0} given by
    // the caller (the path search's pruning pass writes them), or nullptr to
    // merge the row pass's partials of the q rows
    const float4* q_stat = nullptr;
};

// Residual / bonus sampling (K3): a cluster of `cluster` CTAs per sequence,
// each staging `slice_vec` vectors of the row(s) in shared memory.
// A bounded wait that gives up (kStatusTimeout) leaves the sequence's three
// outputs at -1.
struct SampleArgs {
    const void* p;
    const void* q;
    const SeqTask* tasks;
    int32_t* out_sel;
    int32_t* out_len;
    int32_t* out_tok;
    unsigned* status;
    int64_t nvec;
    int64_t slice_vec;
    int cluster;
    unsigned hooks = 0;     // kHook* bits (fault-path tests)
};

// Fault-path test hooks (the public SDV_HOOK_* values).
enum : unsigned {
    // the sample kernel arms its barrier for the row copies but issues none,
    // and polls it only kTestPolls times: its bounded wait runs out with no
    // copy in flight, which exercises the timeout path safely
    kHookSampleNoCopy = 1u,
};
constexpr uint32_t kTestPolls = 16;

// Causal-consistency path search (k4_cps.cu): prune kernel over the B*G
// drafter rows, then one warp per sequence for the beam.
constexpr int kCpsMaxBeam = 16;
constexpr int kCpsMaxCand = 16;
constexpr int kCpsMaxGamma = 1024;
struct CpsArgs {
    const void* q;          // [B][G][V]
    const float* temps;     // [B] or nullptr
    float temperature;
    float tau;
    int B, G, mmax, beam, eos_id;
    int64_t nvec;
    int32_t* cand_ids;      // [B][G][mmax]
    float* cand_logp;       // [B][G][mmax]
    float* cand_logit;      // [B][G][mmax] raw logits of the candidates
    int32_t* ncand;         // [B][G]
    int32_t* paths;         // [B][beam][G]
    float* path_logp;       // [B][beam]
    int32_t* npaths;        // [B]
    int32_t* lat_len;       // [B] or nullptr
    float4* row_stat = nullptr;   // [B][G] {max, sum 2^{(l - max) c}, c, 0} or nullptr
};
// Pruning (reads q, temps; writes cand_ids, cand_logp, ncand) and the beam
// (reads and trims the lattice; writes paths, path_logp, npaths, lat_len).
cudaError_t launch_cps_prune(const CpsArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_cps_beam(const CpsArgs& a, cudaStream_t s);

struct AdlArgs {
    int B, W, kmin, kmax, up, down;
    const int32_t* gen_len;   // [B]
    const int32_t* acc_len;   // [B]
    int32_t* k;               // [B] in/out
    int32_t* state;           // [B][adl_state_words(W)]
    int32_t* status;          // or nullptr
};
cudaError_t launch_adl(const AdlArgs& a, cudaStream_t s);

// Launchers (defined next to their kernels).  `bf16` selects the element type
// (bf16 when true, fp32 otherwise).  Each returns the launch's error code.
// All three kernels are launched as programmatic dependents of the kernel
// before them on the stream: they may become resident while it finishes and
// wait (griddepcontrol.wait) for it before touching memory; `pdl` = false
// launches them as ordinary stream-ordered kernels.
cudaError_t launch_rowpass(const RowPassArgs& a, bool bf16, cudaStream_t s, bool pdl);
cudaError_t launch_select(const SelectArgs& a, bool bf16, size_t smem, cudaStream_t s, bool pdl);
cudaError_t launch_sample(const SampleArgs& a, bool bf16, int B, int cluster, size_t smem,
                          cudaStream_t s, bool pdl);
// Per-kernel set-up (shared-memory opt-in): raise the kernels' dynamic
// shared-memory limit on the current device to at least `smem`.
cudaError_t setup_select(size_t smem);
cudaError_t setup_sample(size_t smem);
// The dynamic shared-memory limit of kernel `func` on the current device is
// process-wide state: contexts of different shapes share it.  This raises it
// to `bytes` when it is lower and never lowers it, so that setting up a
// context for a small shape cannot break the launches of one made earlier for
// a larger shape.  Thread-safe (one lock around the per-device record).
cudaError_t raise_smem_limit(const void* func, size_t bytes);

// True when `p` is device (or managed) memory of some device.
inline bool is_device_ptr(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}
// Largest CTAs per sequence of the sampling pass, and how many clusters of
// `cluster` CTAs with `smem` bytes each the device can hold at once (0: none).
int sample_max_cluster();
int sample_active_clusters(bool bf16, int cluster, size_t smem);
// Sequences up to which the sampling pass uses clusters of 16 CTAs (more
// sequences keep 8, so that all clusters of a batch fit the GPU at once).
constexpr int kWideSampleMaxB = 16;
// Resident blocks per SM of the row-pass kernel, in item and in row mode.
cudaError_t rowpass_occupancy(bool bf16, int* blocks_per_sm);
cudaError_t rowpass_row_occupancy(bool bf16, int* blocks_per_sm);

constexpr int kRowPassThreads = 256;

// Row mode: one CTA of four warps per row, the row's 4 KB blocks (kRowBlockVec
// vectors) dealt to the warps in a fixed interleaved order and merged in the
// CTA into one partial per row.  Used when the rows fill between three
// quarters and all of one wave of such CTAs (eight per SM): every row streams
// at once, with no wave turnover, and the select kernel merges one partial
// per row.  On the self-selection shape (1 056 rows of 152 064 logits) item
// mode needs 19 chunks a row to fill its waves.
constexpr int kRowModeThreads = 128;
constexpr int kRowModeMinBlocks = 8;
constexpr int64_t kRowBlockVec = 256;

inline bool plan_row_mode(int64_t rows, int64_t row_slots, int64_t nvec) {
    return row_slots > 0 && rows <= row_slots && 4 * rows >= 3 * row_slots &&
           nvec >= (kRowModeThreads / 32) * kRowBlockVec;
}

// Row-pass chunking.  One warp reduces one (row, chunk) item and the grid is
// one CTA per kRowPassThreads / 32 items, scheduled by the hardware in many
// waves (that balances SMs whose bandwidth differs; a persistent grid with a
// static item order does not).  Chunks target kChunkTargetVec vectors
// (76 KB of bf16), are split further until there are at least
// kMinItemWaves waves of resident warps, but to at most kMaxChunks per row
// (the select kernel merges a row's partials on one thread), stay >= 64
// vectors, and are rounded to 8 vectors (128 bytes).  Chunks are fixed per
// row, so rows with the same bytes give bit-identical partials wherever they
// sit.
constexpr int64_t kChunkTargetVec = 4752;
constexpr int64_t kMinItemWaves = 4;
constexpr int64_t kMaxChunks = 64;

inline void plan_rowpass_chunks(int64_t rows, int64_t nvec, int64_t resident_warps,
                                int64_t max_items, int* chunks, int64_t* chunk_vec) {
    int64_t c = (nvec + kChunkTargetVec - 1) / kChunkTargetVec;
    int64_t want = (kMinItemWaves * resident_warps + rows - 1) / rows;
    if (want > kMaxChunks) want = kMaxChunks;
    if (want > c) c = want;
    const int64_t cmax = nvec >= 64 ? nvec / 64 : 1;
    if (c > cmax) c = cmax;
    if (c < 1) c = 1;
    if (max_items > 0 && rows * c > max_items) c = max_items / rows;
    if (c < 1) c = 1;
    int64_t cv = (nvec + c - 1) / c;
    cv = (cv + 7) / 8 * 8;
    if (cv > nvec) cv = nvec;
    *chunk_vec = cv;
    *chunks = static_cast<int>((nvec + cv - 1) / cv);
}
constexpr int kSelectThreads = 512;

// Dynamic shared memory of the select kernel for K drafts of G tokens: row
// statistics [K][2G+1] float2, ratios [K][G+1] float, then (16-byte
// aligned) the scores [K] float.
inline size_t select_smem_bytes(int K, int G) {
    const size_t head = static_cast<size_t>(K) * (2 * G + 1) * 8 + static_cast<size_t>(K) * (G + 1) * 4;
    return ((head + 15) & ~size_t(15)) + static_cast<size_t>(K) * 4;
}

// Lanes per row merge in the select kernel: the largest power of two up to
// 32, and up to the first power of two at or above the chunk count (lanes
// past the last chunk merge nothing), for which the K * G pairs and K bonus rows
// of a sequence all fit the CTA's threads in one round.  Few rows with many
// chunks each (the latency cases) get whole warps; the large batches keep
// one thread per row.
inline int select_merge_lanes(int K, int G, int chunks) {
    const int64_t items = static_cast<int64_t>(K) * G + K;
    int lanes = 1;
    while (lanes < 32 && lanes < chunks && items * (2 * lanes) <= kSelectThreads) lanes *= 2;
    return lanes;
}

constexpr int kSampleThreads = 512;

}  // namespace sdv
