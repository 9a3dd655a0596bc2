// sdv_static.cu -- sdv_verify_static: the verification step for callers that
// cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a host process whose device
// memory is owned entirely by another allocator (a serving engine's pool), a
// plug-in loaded into such a process, or code that runs where allocation is
// forbidden.  For them this entry point runs the same three kernels as
// sdv_verify_ex (row pass, select/scan, sample), but their scratch -- the
// row-pass partials, the per-sequence tasks and the status word -- lives in
// one file-scope static device array of kStaticScratchBytes, which every GPU
// that loads this library holds until the process exits.  The caller still
// owns and passes every input and output.
//
// Set-up: the first call on a device (with that device current) resolves the
// device address of the array with cudaGetSymbolAddress and raises the
// kernels' shared-memory limits; later calls on that device skip it.  No call
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
//
// Every call shares the one array and leaves its contents behind; the status
// word is cleared at the start of each call and everything else is written
// before it is read.  Calls that overlap on the GPU (two streams, two host
// threads) race on the array and must be serialised by the caller.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/sdv.h"
#include "sdv_plan.h"

using namespace sdv;

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

struct StaticDevice {
    bool ready;
    void* scratch;        // device address of g_static_scratch on this device
    int nsm;
    int rowpass_blocks[2];   // resident row-pass CTAs per SM: [fp32, bf16]
    int row_blocks[2];       // the same in row mode
    int smem_optin;          // largest dynamic shared memory a block may opt into
};

StaticDevice g_devices[kMaxDevices];
std::mutex g_setup_mutex;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Once per device, with that device current.
cudaError_t setup_device(int dev, StaticDevice** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    StaticDevice& d = g_devices[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return e;
        int nsm = 0, optin = 0, bps_f32 = 0, bps_bf16 = 0, rbps_f32 = 0, rbps_bf16 = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = rowpass_occupancy(false, &bps_f32);
        if (e == cudaSuccess) e = rowpass_occupancy(true, &bps_bf16);
        if (e == cudaSuccess) e = rowpass_row_occupancy(false, &rbps_f32);
        if (e == cudaSuccess) e = rowpass_row_occupancy(true, &rbps_bf16);
        if (e != cudaSuccess) return e;
        if (bps_f32 < 1 || bps_bf16 < 1 || optin <= 4096) return cudaErrorInvalidConfiguration;
        // Let both kernels take up to the device's opt-in limit, once: the
        // limit is only ever raised, so launches that ask for less, from here
        // or from any context, are not disturbed.
        e = setup_select(static_cast<size_t>(optin) - 4096);
        if (e == cudaSuccess) e = setup_sample(static_cast<size_t>(optin) - 4096);
        if (e != cudaSuccess) return e;
        d.scratch = ptr;
        d.nsm = nsm;
        d.smem_optin = optin;
        d.rowpass_blocks[0] = bps_f32;
        d.rowpass_blocks[1] = bps_bf16;
        d.row_blocks[0] = rbps_f32;
        d.row_blocks[1] = rbps_bf16;
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

}  // namespace

extern "C" sdv_status sdv_verify_static(int B, int K, int gamma, int V, sdv_dtype dtype,
                                        void* stream, const void* p_logits,
                                        const void* q_logits, const int32_t* drafts,
                                        float temperature, const float* temperature_per_seq,
                                        uint64_t seed, int32_t* out_sel,
                                        int32_t* out_accept_len, int32_t* out_next_token) {
    if (B < 1 || K < 1 || gamma < 1 || V < 1) return SDV_ERR_ARG;
    if (dtype != SDV_BF16 && dtype != SDV_F32) return SDV_ERR_ARG;
    const int64_t elt = dtype == SDV_BF16 ? 2 : 4;
    if ((static_cast<int64_t>(V) * elt) % 16 != 0) return SDV_ERR_ARG;
    if (!p_logits || !q_logits || !drafts || !out_sel || !out_accept_len || !out_next_token)
        return SDV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits)) & 15u)
        return SDV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(drafts) | reinterpret_cast<uintptr_t>(out_sel) |
         reinterpret_cast<uintptr_t>(out_accept_len) | reinterpret_cast<uintptr_t>(out_next_token) |
         reinterpret_cast<uintptr_t>(temperature_per_seq)) & 3u)
        return SDV_ERR_ARG;
    if (!temperature_per_seq && !(std::isfinite(temperature) && temperature > 0.0f))
        return SDV_ERR_ARG;
    // every pointer must be device memory: a host pointer is refused here,
    // before anything is enqueued
    const void* ptrs[7] = {p_logits, q_logits, drafts, out_sel, out_accept_len, out_next_token,
                           temperature_per_seq};
    for (const void* ptr : ptrs)
        if (ptr && !is_device_ptr(ptr)) return SDV_ERR_ARG;

    // Scratch layout in the static array: partials, tasks, status word.
    const int64_t nvec = static_cast<int64_t>(V) * elt / 16;
    const int64_t rows_p = static_cast<int64_t>(B) * K * (gamma + 1);
    const int64_t rows_total = rows_p + static_cast<int64_t>(B) * K * gamma;
    const size_t task_bytes = round_up(static_cast<size_t>(B) * sizeof(SeqTask), 256);
    // Partials (rounded up to 256 bytes), tasks and the status word must fit.
    if (task_bytes + 512 >= kStaticScratchBytes) return SDV_ERR_SCRATCH;
    const int64_t max_items =
        static_cast<int64_t>((kStaticScratchBytes - task_bytes - 512) / sizeof(float2));

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDV_ERR_CUDA;
    StaticDevice* sd = nullptr;
    if (setup_device(dev, &sd) != cudaSuccess) return SDV_ERR_CUDA;

    const int bps = sd->rowpass_blocks[dtype == SDV_BF16 ? 1 : 0];
    const int64_t resident_warps = static_cast<int64_t>(sd->nsm) * bps * (kRowPassThreads / 32);
    if (rows_total > max_items) return SDV_ERR_SCRATCH;
    int chunks = 0;
    int64_t chunk_vec = 0;
    const bool row_mode = plan_row_mode(
        rows_total, static_cast<int64_t>(sd->nsm) * sd->row_blocks[dtype == SDV_BF16 ? 1 : 0], nvec);
    if (row_mode) {
        chunks = 1;
        chunk_vec = nvec;
    } else {
        plan_rowpass_chunks(rows_total, nvec, resident_warps, max_items, &chunks, &chunk_vec);
    }
    const int64_t items = rows_total * chunks;
    if (items > max_items) return SDV_ERR_SCRATCH;
    const size_t part_bytes = round_up(static_cast<size_t>(items) * sizeof(float2), 256);
    unsigned char* base = static_cast<unsigned char*>(sd->scratch);
    float2* part = reinterpret_cast<float2*>(base);
    SeqTask* tasks = reinterpret_cast<SeqTask*>(base + part_bytes);
    unsigned* status = reinterpret_cast<unsigned*>(base + part_bytes + task_bytes);

    int cl = 8;
    while (cl > 1 && cl > nvec) cl >>= 1;
    const int64_t slice_vec = (nvec + cl - 1) / cl;
    const size_t sel_smem = select_smem_bytes(K, gamma);
    const size_t smp_smem = static_cast<size_t>(2) * slice_vec * 16;
    if (sel_smem > static_cast<size_t>(sd->smem_optin) - 4096 ||
        smp_smem > static_cast<size_t>(sd->smem_optin) - 4096)
        return SDV_ERR_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return SDV_ERR_CUDA;

    RowPassArgs ra;
    ra.p = p_logits;
    ra.q = q_logits;
    ra.part = part;
    ra.temps = temperature_per_seq;
    ra.temperature = temperature;
    ra.K = K;
    ra.G = gamma;
    ra.chunks = chunks;
    ra.flags = 0u;
    ra.rows_p = rows_p;
    ra.rows_total = rows_total;
    ra.nvec = nvec;
    ra.chunk_vec = chunk_vec;
    ra.items = items;
    ra.row_mode = row_mode ? 1 : 0;
    if (launch_rowpass(ra, dtype == SDV_BF16, s, true) != cudaSuccess) return SDV_ERR_CUDA;

    SelectArgs sa;
    sa.p = p_logits;
    sa.q = q_logits;
    sa.drafts = drafts;
    sa.part = part;
    sa.temps = temperature_per_seq;
    sa.temperature = temperature;
    sa.B = B;
    sa.K = K;
    sa.G = gamma;
    sa.V = V;
    sa.chunks = chunks;
    sa.merge_lanes = select_merge_lanes(K, gamma, chunks);
    sa.flags = 0u;
    sa.rows_p = rows_p;
    sa.seed_lo = static_cast<uint32_t>(seed & 0xffffffffu);
    sa.seed_hi = static_cast<uint32_t>(seed >> 32);
    sa.out_sel = out_sel;
    sa.out_len = out_accept_len;
    sa.out_tok = out_next_token;
    sa.out_scores = nullptr;
    sa.out_lse = nullptr;
    sa.tasks = tasks;
    sa.status = status;
    if (launch_select(sa, dtype == SDV_BF16, sel_smem, s, true) != cudaSuccess) return SDV_ERR_CUDA;

    SampleArgs ma;
    ma.p = p_logits;
    ma.q = q_logits;
    ma.tasks = tasks;
    ma.out_sel = out_sel;
    ma.out_len = out_accept_len;
    ma.out_tok = out_next_token;
    ma.status = status;
    ma.nvec = nvec;
    ma.slice_vec = slice_vec;
    ma.cluster = cl;
    if (launch_sample(ma, dtype == SDV_BF16, B, cl, smp_smem, s, true) != cudaSuccess) return SDV_ERR_CUDA;
    return SDV_OK;
}
