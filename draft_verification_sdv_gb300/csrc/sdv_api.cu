// sdv_api.cu -- the C ABI of libsdv (declared in include/sdv.h): contexts,
// launch planning, argument checks, the three-kernel step, status reporting.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/sdv.h"
#include "sdv_plan.h"

using namespace sdv;

struct sdv_ctx {
    int B, K, G, V;
    unsigned flags;
    sdv_dtype dtype;
    bool bf16;
    cudaStream_t stream;
    int device;
    int nsm;
    // row pass
    int rp_grid;
    int row_mode;           // row pass: one CTA per row (see plan_row_mode)
    int chunks;
    int64_t nvec, chunk_vec, rows_p, rows_q, rows_total, items;
    // select / sample
    size_t sel_smem;
    int cluster;
    int64_t slice_vec;
    size_t smp_smem;
    // workspace
    void* ws;
    float2* part;
    SeqTask* tasks;
    unsigned* status;
    // device staging of sdv_verify_host (allocated on first use)
    void* hs_p;
    void* hs_q;
    int32_t* hs_drafts;
    float* hs_temps;
    int32_t* hs_out;
    // fault-path test hooks (sdv_set_test_hooks)
    unsigned hooks;
    // kernel timing: 4 events per recorded step
    bool prof_on;
    std::vector<cudaEvent_t> prof_ev;
    int prof_n;
    char err[512];
};

static_assert(SDV_FLAG_SHARED_Q == sdv::kFlagSharedQ && SDV_FLAG_GREEDY == sdv::kFlagGreedy &&
                  SDV_FLAG_SHARED_PREFIX_ROW == sdv::kFlagSharedPrefixRow,
              "public layout flags and kernel flags must agree");
static_assert(SDV_HOOK_SAMPLE_NO_COPY == sdv::kHookSampleNoCopy,
              "public test hooks and kernel hooks must agree");

namespace {

sdv_status fail(sdv_ctx* ctx, sdv_status st, const char* fmt, ...) {
    if (ctx) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(ctx->err, sizeof ctx->err, fmt, ap);
        va_end(ap);
    }
    return st;
}

sdv_status cuda_fail(sdv_ctx* ctx, cudaError_t e, const char* what) {
    return fail(ctx, SDV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t elt_size(sdv_dtype d) { return d == SDV_BF16 ? 2 : 4; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxProfSteps = 65536;

}  // namespace

namespace sdv {

cudaError_t raise_smem_limit(const void* func, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> limit;   // (kernel, device) -> bytes
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t& cur = limit[std::make_pair(func, dev)];
    if (bytes <= cur) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
    if (e == cudaSuccess) cur = bytes;
    return e;
}

}  // namespace sdv

extern "C" {

sdv_status sdv_create(sdv_ctx** out, int B, int K, int gamma, int V, sdv_dtype dtype,
                      void* stream) {
    return sdv_create_ex(out, B, K, gamma, V, dtype, stream, 0u);
}

sdv_status sdv_create_ex(sdv_ctx** out, int B, int K, int gamma, int V, sdv_dtype dtype,
                         void* stream, unsigned flags) {
    if (!out) return SDV_ERR_ARG;
    *out = nullptr;
    if (flags & ~static_cast<unsigned>(SDV_FLAG_SHARED_Q | SDV_FLAG_GREEDY |
                                       SDV_FLAG_SHARED_PREFIX_ROW))
        return SDV_ERR_ARG;
    if ((flags & SDV_FLAG_SHARED_Q) && (flags & SDV_FLAG_GREEDY)) return SDV_ERR_ARG;
    if (B < 1 || K < 1 || gamma < 1 || V < 1) return SDV_ERR_ARG;
    if (dtype != SDV_BF16 && dtype != SDV_F32) return SDV_ERR_ARG;
    const size_t elt = elt_size(dtype);
    if ((static_cast<size_t>(V) * elt) % 16 != 0) return SDV_ERR_ARG;
    if (static_cast<int64_t>(B) * K * (2 * gamma + 1) > (int64_t(1) << 27)) return SDV_ERR_ARG;

    sdv_ctx* ctx = new (std::nothrow) sdv_ctx();
    if (!ctx) return SDV_ERR_OOM;
    ctx->B = B;
    ctx->K = K;
    ctx->G = gamma;
    ctx->V = V;
    ctx->dtype = dtype;
    ctx->flags = flags;
    ctx->bf16 = dtype == SDV_BF16;
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->err[0] = 0;

    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->nsm, cudaDevAttrMultiProcessorCount, ctx->device);
    int bps = 0, rbps = 0;
    if (e == cudaSuccess) e = rowpass_occupancy(ctx->bf16, &bps);
    if (e == cudaSuccess) e = rowpass_row_occupancy(ctx->bf16, &rbps);
    if (e != cudaSuccess || bps < 1) {
        sdv_destroy(ctx);
        return SDV_ERR_CUDA;
    }

    // Row pass plan.
    ctx->nvec = static_cast<int64_t>(V) * static_cast<int64_t>(elt) / 16;
    ctx->rows_p = static_cast<int64_t>(B) * K * (gamma + 1);
    ctx->rows_q = (flags & SDV_FLAG_GREEDY)     ? 0
                  : (flags & SDV_FLAG_SHARED_Q) ? static_cast<int64_t>(B) * gamma
                                                : static_cast<int64_t>(B) * K * gamma;
    ctx->rows_total = ctx->rows_p + ctx->rows_q;
    const int64_t resident_warps = static_cast<int64_t>(ctx->nsm) * bps * (kRowPassThreads / 32);
    ctx->row_mode = plan_row_mode(ctx->rows_total, static_cast<int64_t>(ctx->nsm) * rbps, ctx->nvec);
    if (ctx->row_mode) {
        ctx->chunks = 1;
        ctx->chunk_vec = ctx->nvec;
    } else {
        plan_rowpass_chunks(ctx->rows_total, ctx->nvec, resident_warps, 0, &ctx->chunks, &ctx->chunk_vec);
    }
    ctx->items = ctx->rows_total * ctx->chunks;
    ctx->rp_grid = ctx->row_mode ? static_cast<int>(ctx->items)
                                 : static_cast<int>((ctx->items + (kRowPassThreads / 32) - 1) /
                                                    (kRowPassThreads / 32));

    // Select plan.
    ctx->sel_smem = select_smem_bytes(K, gamma);
    // Sample plan: up to 8 CTAs per sequence (16 for a small batch), each
    // holding a slice of one or two rows in shared memory.
    int cl = B <= kWideSampleMaxB ? sample_max_cluster() : 8;
    while (cl > 1 && cl > ctx->nvec) cl >>= 1;
    ctx->cluster = cl;
    ctx->slice_vec = (ctx->nvec + cl - 1) / cl;
    ctx->smp_smem = static_cast<size_t>(2) * ctx->slice_vec * 16;
    const size_t smem_cap = 200 * 1024;
    if (ctx->sel_smem > smem_cap || ctx->smp_smem > smem_cap) {
        sdv_destroy(ctx);
        return SDV_ERR_ARG;
    }
    e = setup_select(ctx->sel_smem > 0 ? ctx->sel_smem : 16);
    if (e == cudaSuccess) e = setup_sample(ctx->smp_smem);
    if (e == cudaSuccess && ctx->cluster > 8 &&
        sample_active_clusters(ctx->bf16, ctx->cluster, ctx->smp_smem) < 1) {
        // a cluster that wide cannot be scheduled here: the portable 8
        ctx->cluster = 8;
        ctx->slice_vec = (ctx->nvec + 7) / 8;
        ctx->smp_smem = static_cast<size_t>(2) * ctx->slice_vec * 16;
        if (ctx->smp_smem > smem_cap) {
            sdv_destroy(ctx);
            return SDV_ERR_ARG;
        }
        e = setup_sample(ctx->smp_smem);
    }
    if (e != cudaSuccess) {
        sdv_destroy(ctx);
        return SDV_ERR_CUDA;
    }

    // Workspace: partials, tasks, status word.
    const size_t part_bytes = align_up(static_cast<size_t>(ctx->items) * sizeof(float2), 256);
    const size_t task_bytes = align_up(static_cast<size_t>(B) * sizeof(SeqTask), 256);
    const size_t total = part_bytes + task_bytes + 256;
    e = cudaMalloc(&ctx->ws, total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        ctx->ws = nullptr;
        sdv_destroy(ctx);
        return SDV_ERR_OOM;
    }
    char* w = static_cast<char*>(ctx->ws);
    ctx->part = reinterpret_cast<float2*>(w);
    ctx->tasks = reinterpret_cast<SeqTask*>(w + part_bytes);
    ctx->status = reinterpret_cast<unsigned*>(w + part_bytes + task_bytes);
    e = cudaMemsetAsync(ctx->status, 0, sizeof(unsigned), ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) {
        sdv_destroy(ctx);
        return SDV_ERR_CUDA;
    }
    *out = ctx;
    return SDV_OK;
}

namespace {

// Argument checks of a row pass (logits and temperatures).
sdv_status check_rows(sdv_ctx* ctx, const void* p_logits, const void* q_logits, bool need_q,
                      float temperature, const float* temperature_per_seq) {
    if (!p_logits || (need_q && !q_logits)) return fail(ctx, SDV_ERR_ARG, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits)) & 15u)
        return fail(ctx, SDV_ERR_ARG, "logit buffers must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(temperature_per_seq) & 3u)
        return fail(ctx, SDV_ERR_ARG, "int32 / float buffers must be 4-byte aligned");
    if (!temperature_per_seq && !(std::isfinite(temperature) && temperature > 0.0f))
        return fail(ctx, SDV_ERR_ARG, "temperature must be finite and > 0");
    const void* ptrs[3] = {p_logits, q_logits, temperature_per_seq};
    for (const void* p : ptrs)
        if (p && !is_device_ptr(p)) return fail(ctx, SDV_ERR_ARG, "argument is not a device pointer");
    return SDV_OK;
}

// Argument checks of a selection and draw.
sdv_status check_finish(sdv_ctx* ctx, const int32_t* drafts, const int32_t* draft_len,
                        const float* q_row_stat, int32_t* out_sel, int32_t* out_accept_len,
                        int32_t* out_next_token, float* out_scores, float* out_lse) {
    const bool greedy = (ctx->flags & SDV_FLAG_GREEDY) != 0;
    if (!drafts || !out_sel || !out_accept_len || !out_next_token)
        return fail(ctx, SDV_ERR_ARG, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(drafts) | reinterpret_cast<uintptr_t>(out_sel) |
         reinterpret_cast<uintptr_t>(out_accept_len) | reinterpret_cast<uintptr_t>(out_next_token) |
         reinterpret_cast<uintptr_t>(out_scores) | reinterpret_cast<uintptr_t>(out_lse)) & 3u)
        return fail(ctx, SDV_ERR_ARG, "int32 / float buffers must be 4-byte aligned");
    const void* ptrs[6] = {drafts, out_sel, out_accept_len, out_next_token, out_scores, out_lse};
    for (const void* p : ptrs)
        if (p && !is_device_ptr(p)) return fail(ctx, SDV_ERR_ARG, "argument is not a device pointer");
    if (draft_len && ((reinterpret_cast<uintptr_t>(draft_len) & 3u) || !is_device_ptr(draft_len)))
        return fail(ctx, SDV_ERR_ARG, "draft_len must be a 4-byte aligned device pointer");
    if (q_row_stat && greedy)
        return fail(ctx, SDV_ERR_ARG, "greedy acceptance reads no drafter rows: q_row_stat must be null");
    if (q_row_stat &&
        ((reinterpret_cast<uintptr_t>(q_row_stat) & 15u) || !is_device_ptr(q_row_stat)))
        return fail(ctx, SDV_ERR_ARG, "q_row_stat must be a 16-byte aligned device pointer");
    return SDV_OK;
}

// Enqueue the row pass: every verifier row, and the drafter rows when
// `with_q`; rows past a draft length are skipped when `draft_len` is given.
cudaError_t enqueue_rows(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                         const int32_t* draft_len, bool with_q, float temperature,
                         const float* temperature_per_seq, bool pdl) {
    RowPassArgs ra;
    ra.p = p_logits;
    ra.q = q_logits;
    ra.part = ctx->part;
    ra.temps = temperature_per_seq;
    ra.temperature = temperature;
    ra.K = ctx->K;
    ra.G = ctx->G;
    ra.chunks = ctx->chunks;
    ra.flags = ctx->flags;
    ra.rows_p = ctx->rows_p;
    ra.rows_total = ctx->rows_total;
    ra.nvec = ctx->nvec;
    ra.chunk_vec = ctx->chunk_vec;
    // without the drafter rows only the verifier rows are streamed (the q
    // rows come after them in item order)
    ra.items = with_q ? ctx->items : ctx->rows_p * ctx->chunks;
    ra.lens = draft_len;
    ra.row_mode = ctx->row_mode;
    return launch_rowpass(ra, ctx->bf16, ctx->stream, pdl);
}

// Enqueue the selection / scan and the draw on the partials of the row pass.
sdv_status enqueue_finish(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                          const int32_t* drafts, const int32_t* draft_len, const float* q_row_stat,
                          float temperature, const float* temperature_per_seq, uint64_t seed,
                          int32_t* out_sel, int32_t* out_accept_len, int32_t* out_next_token,
                          float* out_scores, float* out_lse, cudaEvent_t* ev) {
    SelectArgs sa;
    sa.p = p_logits;
    sa.q = q_logits;
    sa.drafts = drafts;
    sa.part = ctx->part;
    sa.temps = temperature_per_seq;
    sa.temperature = temperature;
    sa.B = ctx->B;
    sa.K = ctx->K;
    sa.G = ctx->G;
    sa.V = ctx->V;
    sa.chunks = ctx->chunks;
    sa.flags = ctx->flags;
    sa.rows_p = ctx->rows_p;
    sa.seed_lo = static_cast<uint32_t>(seed & 0xffffffffu);
    sa.seed_hi = static_cast<uint32_t>(seed >> 32);
    sa.out_sel = out_sel;
    sa.out_len = out_accept_len;
    sa.out_tok = out_next_token;
    sa.out_scores = out_scores;
    sa.out_lse = out_lse;
    sa.tasks = ctx->tasks;
    sa.status = ctx->status;
    sa.lens = draft_len;
    sa.q_stat = reinterpret_cast<const float4*>(q_row_stat);
    sa.merge_lanes = select_merge_lanes(ctx->K, ctx->G, ctx->chunks);
    cudaError_t e = launch_select(sa, ctx->bf16, ctx->sel_smem, ctx->stream, ev == nullptr);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "select launch");
    if (ev) cudaEventRecord(ev[2], ctx->stream);

    SampleArgs ma;
    ma.p = p_logits;
    ma.q = q_logits;
    ma.tasks = ctx->tasks;
    ma.out_sel = out_sel;
    ma.out_len = out_accept_len;
    ma.out_tok = out_next_token;
    ma.hooks = ctx->hooks;
    ma.status = ctx->status;
    ma.nvec = ctx->nvec;
    ma.slice_vec = ctx->slice_vec;
    ma.cluster = ctx->cluster;
    e = launch_sample(ma, ctx->bf16, ctx->B, ctx->cluster, ctx->smp_smem, ctx->stream, ev == nullptr);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "sample launch");
    if (ev) cudaEventRecord(ev[3], ctx->stream);
    return SDV_OK;
}

sdv_status verify_impl(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                       const int32_t* drafts, const int32_t* draft_len, const float* q_row_stat,
                       float temperature, const float* temperature_per_seq, uint64_t seed,
                       int32_t* out_sel, int32_t* out_accept_len, int32_t* out_next_token,
                       float* out_scores, float* out_lse) {
    if (!ctx) return SDV_ERR_ARG;
    ctx->err[0] = 0;
    const bool greedy = (ctx->flags & SDV_FLAG_GREEDY) != 0;
    sdv_status st = check_rows(ctx, p_logits, q_logits, !greedy, temperature, temperature_per_seq);
    if (st == SDV_OK)
        st = check_finish(ctx, drafts, draft_len, q_row_stat, out_sel, out_accept_len,
                          out_next_token, out_scores, out_lse);
    if (st != SDV_OK) return st;

    cudaEvent_t* ev = nullptr;
    if (ctx->prof_on && ctx->prof_n < kMaxProfSteps) {
        const size_t need = static_cast<size_t>(ctx->prof_n + 1) * 4;
        while (ctx->prof_ev.size() < need) {
            cudaEvent_t x;
            if (cudaEventCreate(&x) != cudaSuccess) return fail(ctx, SDV_ERR_CUDA, "event create");
            ctx->prof_ev.push_back(x);
        }
        ev = &ctx->prof_ev[static_cast<size_t>(ctx->prof_n) * 4];
        ++ctx->prof_n;
    }
    if (ev) cudaEventRecord(ev[0], ctx->stream);
    // with the drafter rows' statistics supplied, only the verifier rows are streamed
    const cudaError_t e = enqueue_rows(ctx, p_logits, q_logits, draft_len, !greedy && !q_row_stat,
                                       temperature, temperature_per_seq, ev == nullptr);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "row pass launch");
    if (ev) cudaEventRecord(ev[1], ctx->stream);
    return enqueue_finish(ctx, p_logits, q_logits, drafts, draft_len, q_row_stat, temperature,
                          temperature_per_seq, seed, out_sel, out_accept_len, out_next_token,
                          out_scores, out_lse, ev);
}

}  // namespace

sdv_status sdv_verify_ex(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                         const int32_t* drafts, float temperature,
                         const float* temperature_per_seq, uint64_t seed, int32_t* out_sel,
                         int32_t* out_accept_len, int32_t* out_next_token, float* out_scores,
                         float* out_lse) {
    return verify_impl(ctx, p_logits, q_logits, drafts, nullptr, nullptr, temperature,
                       temperature_per_seq, seed, out_sel, out_accept_len, out_next_token,
                       out_scores, out_lse);
}

sdv_status sdv_verify_len(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                          const int32_t* drafts, const int32_t* draft_len, float temperature,
                          const float* temperature_per_seq, uint64_t seed, int32_t* out_sel,
                          int32_t* out_accept_len, int32_t* out_next_token, float* out_scores,
                          float* out_lse) {
    if (!draft_len) return ctx ? fail(ctx, SDV_ERR_ARG, "draft_len is null") : SDV_ERR_ARG;
    return verify_impl(ctx, p_logits, q_logits, drafts, draft_len, nullptr, temperature,
                       temperature_per_seq, seed, out_sel, out_accept_len, out_next_token,
                       out_scores, out_lse);
}

sdv_status sdv_verify_qstat(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                            const int32_t* drafts, const int32_t* draft_len,
                            const float* q_row_stat, float temperature,
                            const float* temperature_per_seq, uint64_t seed, int32_t* out_sel,
                            int32_t* out_accept_len, int32_t* out_next_token, float* out_scores,
                            float* out_lse) {
    if (!q_row_stat) return ctx ? fail(ctx, SDV_ERR_ARG, "q_row_stat is null") : SDV_ERR_ARG;
    return verify_impl(ctx, p_logits, q_logits, drafts, draft_len, q_row_stat, temperature,
                       temperature_per_seq, seed, out_sel, out_accept_len, out_next_token,
                       out_scores, out_lse);
}

sdv_status sdv_verify(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                      const int32_t* drafts, float temperature, uint64_t seed, int32_t* out_sel,
                      int32_t* out_accept_len, int32_t* out_next_token) {
    return sdv_verify_ex(ctx, p_logits, q_logits, drafts, temperature, nullptr, seed, out_sel,
                         out_accept_len, out_next_token, nullptr, nullptr);
}

sdv_status sdv_sync(sdv_ctx* ctx) {
    if (!ctx) return SDV_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "stream synchronize");
    unsigned h = 0;
    e = cudaMemcpyAsync(&h, ctx->status, sizeof h, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->status, 0, sizeof(unsigned), ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
    if (h & kStatusTimeout)
        return fail(ctx, SDV_ERR_CUDA, "a bounded device wait gave up (status 0x%x)", h);
    if (h)
        return fail(ctx, SDV_ERR_DEVICE_DATA, "device data error (status 0x%x:%s%s%s%s)", h,
                    (h & kStatusBadDraft) ? " draft id out of range" : "",
                    (h & kStatusBadRow) ? " non-finite or all -inf row" : "",
                    (h & kStatusBadTemp) ? " bad per-sequence temperature" : "",
                    (h & kStatusBadStat) ? " drafter-row statistics of another temperature" : "");
    return SDV_OK;
}

sdv_status sdv_verify_host(sdv_ctx* ctx, const void* p_logits_host, const void* q_logits_host,
                           const int32_t* drafts_host, float temperature,
                           const float* temperature_per_seq_host, uint64_t seed,
                           int32_t* out_sel_host, int32_t* out_accept_len_host,
                           int32_t* out_next_token_host) {
    if (!ctx) return SDV_ERR_ARG;
    const bool greedy = (ctx->flags & SDV_FLAG_GREEDY) != 0;
    if (!p_logits_host || (!q_logits_host && !greedy) || !drafts_host || !out_sel_host ||
        !out_accept_len_host || !out_next_token_host)
        return fail(ctx, SDV_ERR_ARG, "null pointer argument");
    const size_t elt = elt_size(ctx->dtype);
    const size_t pb = static_cast<size_t>(ctx->rows_p) * ctx->V * elt;
    const size_t qb = static_cast<size_t>(ctx->rows_q) * ctx->V * elt;
    const size_t db = static_cast<size_t>(ctx->B) * ctx->K * ctx->G * sizeof(int32_t);
    const size_t B = static_cast<size_t>(ctx->B);
    cudaError_t e = cudaSuccess;
    if (!ctx->hs_p) {
        e = cudaMalloc(&ctx->hs_p, pb);
        if (e == cudaSuccess && qb > 0) e = cudaMalloc(&ctx->hs_q, qb);
        if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&ctx->hs_drafts), db);
        if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&ctx->hs_temps), B * 4);
        if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&ctx->hs_out), 3 * B * 4);
        if (e != cudaSuccess) {
            cudaGetLastError();
            cudaFree(ctx->hs_p);
            cudaFree(ctx->hs_q);
            cudaFree(ctx->hs_drafts);
            cudaFree(ctx->hs_temps);
            cudaFree(ctx->hs_out);
            ctx->hs_p = ctx->hs_q = nullptr;
            ctx->hs_drafts = nullptr;
            ctx->hs_temps = nullptr;
            ctx->hs_out = nullptr;
            return fail(ctx, SDV_ERR_OOM, "device staging allocation failed");
        }
    }
    cudaStream_t s = ctx->stream;
    e = cudaMemcpyAsync(ctx->hs_p, p_logits_host, pb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && qb > 0)
        e = cudaMemcpyAsync(ctx->hs_q, q_logits_host, qb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->hs_drafts, drafts_host, db, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && temperature_per_seq_host)
        e = cudaMemcpyAsync(ctx->hs_temps, temperature_per_seq_host, B * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
    sdv_status st = sdv_verify_ex(ctx, ctx->hs_p, ctx->hs_q, ctx->hs_drafts, temperature,
                                  temperature_per_seq_host ? ctx->hs_temps : nullptr, seed,
                                  ctx->hs_out, ctx->hs_out + B, ctx->hs_out + 2 * B, nullptr,
                                  nullptr);
    if (st != SDV_OK) return st;
    e = cudaMemcpyAsync(out_sel_host, ctx->hs_out, B * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(out_accept_len_host, ctx->hs_out + B, B * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(out_next_token_host, ctx->hs_out + 2 * B, B * 4, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "device-to-host copy");
    return sdv_sync(ctx);
}

const char* sdv_last_error(const sdv_ctx* ctx) { return ctx ? ctx->err : "null context"; }

void sdv_destroy(sdv_ctx* ctx) {
    if (!ctx) return;
    cudaStreamSynchronize(ctx->stream);
    cudaFree(ctx->ws);
    cudaFree(ctx->hs_p);
    cudaFree(ctx->hs_q);
    cudaFree(ctx->hs_drafts);
    cudaFree(ctx->hs_temps);
    cudaFree(ctx->hs_out);
    for (cudaEvent_t x : ctx->prof_ev) cudaEventDestroy(x);
    cudaGetLastError();
    delete ctx;
}

sdv_status sdv_plan(const sdv_ctx* ctx, int* rowpass_ctas, int64_t* chunk_vectors,
                    int* chunks_per_row, int* sample_cluster) {
    if (!ctx) return SDV_ERR_ARG;
    if (rowpass_ctas) *rowpass_ctas = ctx->rp_grid;
    if (chunk_vectors) *chunk_vectors = ctx->chunk_vec;
    if (chunks_per_row) *chunks_per_row = ctx->chunks;
    if (sample_cluster) *sample_cluster = ctx->cluster;
    return SDV_OK;
}

sdv_status sdv_profile_enable(sdv_ctx* ctx, int enable) {
    if (!ctx) return SDV_ERR_ARG;
    ctx->prof_on = enable != 0;
    return SDV_OK;
}

sdv_status sdv_profile_read(sdv_ctx* ctx, float* ms_avg, int* steps) {
    if (!ctx || !ms_avg) return SDV_ERR_ARG;
    double sum[3] = {0.0, 0.0, 0.0};
    const int n = ctx->prof_n;
    for (int i = 0; i < n; ++i) {
        const cudaEvent_t* ev = &ctx->prof_ev[static_cast<size_t>(i) * 4];
        cudaError_t e = cudaEventSynchronize(ev[3]);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "event synchronize");
        for (int k = 0; k < 3; ++k) {
            float ms = 0.0f;
            e = cudaEventElapsedTime(&ms, ev[k], ev[k + 1]);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "event elapsed time");
            sum[k] += ms;
        }
    }
    for (int k = 0; k < 3; ++k) ms_avg[k] = n ? static_cast<float>(sum[k] / n) : 0.0f;
    if (steps) *steps = n;
    ctx->prof_n = 0;
    return SDV_OK;
}

namespace {

// Checks shared by the CPS entry points; q / temps are checked only when
// `with_q`, the beam outputs only when `with_beam`.
sdv_status cps_check(int B, int gamma, int mmax, int beam, bool with_beam, const void* const* ptrs,
                     int nptrs) {
    if (B < 1 || gamma < 1 || gamma > kCpsMaxGamma) return SDV_ERR_ARG;
    if (mmax < 1 || mmax > kCpsMaxCand) return SDV_ERR_ARG;
    if (with_beam && (beam < 1 || beam > kCpsMaxBeam)) return SDV_ERR_ARG;
    for (int i = 0; i < nptrs; ++i)
        if (ptrs[i] && !is_device_ptr(ptrs[i])) return SDV_ERR_ARG;
    return SDV_OK;
}

sdv_status cps_prune_args(int B, int gamma, int V, sdv_dtype dtype, const void* q,
                          float temperature, const float* temps, float tau, int mmax,
                          CpsArgs& a) {
    if (V < 1 || (dtype != SDV_BF16 && dtype != SDV_F32)) return SDV_ERR_ARG;
    const int64_t elt = dtype == SDV_BF16 ? 2 : 4;
    if ((static_cast<int64_t>(V) * elt) % 16 != 0) return SDV_ERR_ARG;
    if (!(tau >= 0.0f && tau <= 1.0f)) return SDV_ERR_ARG;
    if (!temps && !(std::isfinite(temperature) && temperature > 0.0f)) return SDV_ERR_ARG;
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15u)) return SDV_ERR_ARG;
    a.q = q;
    a.temps = temps;
    a.temperature = temperature;
    a.tau = tau;
    a.B = B;
    a.G = gamma;
    a.mmax = mmax;
    a.nvec = static_cast<int64_t>(V) * elt / 16;
    return SDV_OK;
}

}  // namespace

namespace {

sdv_status cps_prune_impl(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                          const void* q_marginals, float temperature,
                          const float* temperature_per_seq, float tau, int mmax,
                          int32_t* out_cand_ids, float* out_cand_logp, float* out_cand_logit,
                          int32_t* out_ncand, float* out_row_stat) {
    if (!out_cand_ids || !out_cand_logp || !out_cand_logit || !out_ncand) return SDV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(out_row_stat) & 15u) return SDV_ERR_ARG;
    const void* ptrs[7] = {q_marginals,    temperature_per_seq, out_cand_ids, out_cand_logp,
                           out_cand_logit, out_ncand,           out_row_stat};
    sdv_status st = cps_check(B, gamma, mmax, 1, false, ptrs, 7);
    if (st != SDV_OK) return st;
    CpsArgs a{};
    st = cps_prune_args(B, gamma, V, dtype, q_marginals, temperature, temperature_per_seq, tau,
                        mmax, a);
    if (st != SDV_OK) return st;
    a.cand_ids = out_cand_ids;
    a.cand_logp = out_cand_logp;
    a.cand_logit = out_cand_logit;
    a.ncand = out_ncand;
    a.row_stat = reinterpret_cast<float4*>(out_row_stat);
    return launch_cps_prune(a, dtype == SDV_BF16, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SDV_OK : SDV_ERR_CUDA;
}

}  // namespace

sdv_status sdv_cps_prune(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                         const void* q_marginals, float temperature,
                         const float* temperature_per_seq, float tau, int mmax,
                         int32_t* out_cand_ids, float* out_cand_logp, float* out_cand_logit,
                         int32_t* out_ncand) {
    return cps_prune_impl(B, gamma, V, dtype, stream, q_marginals, temperature,
                          temperature_per_seq, tau, mmax, out_cand_ids, out_cand_logp,
                          out_cand_logit, out_ncand, nullptr);
}

sdv_status sdv_cps_beam(int B, int gamma, int V, int mmax, int beam, int eos_id, void* stream,
                        int32_t* cand_ids, float* cand_logp, float* cand_logit, int32_t* ncand,
                        int32_t* out_paths, float* out_path_logp, int32_t* out_npaths,
                        int32_t* out_lat_len) {
    if (V < 1 || eos_id >= V) return SDV_ERR_ARG;
    if (!cand_ids || !cand_logp || !cand_logit || !ncand || !out_paths || !out_path_logp ||
        !out_npaths)
        return SDV_ERR_ARG;
    const void* ptrs[8] = {cand_ids,  cand_logp,     cand_logit, ncand,
                           out_paths, out_path_logp, out_npaths, out_lat_len};
    const sdv_status st = cps_check(B, gamma, mmax, beam, true, ptrs, 8);
    if (st != SDV_OK) return st;
    CpsArgs a{};
    a.B = B;
    a.G = gamma;
    a.mmax = mmax;
    a.beam = beam;
    a.eos_id = eos_id;
    a.cand_ids = cand_ids;
    a.cand_logp = cand_logp;
    a.cand_logit = cand_logit;
    a.ncand = ncand;
    a.paths = out_paths;
    a.path_logp = out_path_logp;
    a.npaths = out_npaths;
    a.lat_len = out_lat_len;
    return launch_cps_beam(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SDV_OK
                                                                                : SDV_ERR_CUDA;
}

sdv_status sdv_cps(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                   const void* q_marginals, float temperature, const float* temperature_per_seq,
                   float tau, int mmax, int beam, int eos_id, int32_t* out_cand_ids,
                   float* out_cand_logp, float* out_cand_logit, int32_t* out_ncand,
                   int32_t* out_paths,
                   float* out_path_logp, int32_t* out_npaths, int32_t* out_lat_len) {
    return sdv_cps_ex(B, gamma, V, dtype, stream, q_marginals, temperature, temperature_per_seq,
                      tau, mmax, beam, eos_id, out_cand_ids, out_cand_logp, out_cand_logit,
                      out_ncand, out_paths, out_path_logp, out_npaths, out_lat_len, nullptr);
}

sdv_status sdv_cps_ex(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                      const void* q_marginals, float temperature,
                      const float* temperature_per_seq, float tau, int mmax, int beam,
                      int eos_id, int32_t* out_cand_ids, float* out_cand_logp,
                      float* out_cand_logit, int32_t* out_ncand, int32_t* out_paths,
                      float* out_path_logp, int32_t* out_npaths, int32_t* out_lat_len,
                      float* out_row_stat) {
    // both halves' argument checks run before either launches
    if (V < 1 || eos_id >= V || beam < 1 || beam > kCpsMaxBeam) return SDV_ERR_ARG;
    if (!out_paths || !out_path_logp || !out_npaths) return SDV_ERR_ARG;
    const void* ptrs[4] = {out_paths, out_path_logp, out_npaths, out_lat_len};
    sdv_status st = cps_check(B, gamma, mmax, beam, true, ptrs, 4);
    if (st != SDV_OK) return st;
    st = cps_prune_impl(B, gamma, V, dtype, stream, q_marginals, temperature, temperature_per_seq,
                        tau, mmax, out_cand_ids, out_cand_logp, out_cand_logit, out_ncand,
                        out_row_stat);
    if (st != SDV_OK) return st;
    return sdv_cps_beam(B, gamma, V, mmax, beam, eos_id, stream, out_cand_ids, out_cand_logp,
                        out_cand_logit, out_ncand, out_paths, out_path_logp, out_npaths,
                        out_lat_len);
}

namespace {

bool adl_params_ok(int B, int W, int kmin, int kmax, int up, int down) {
    return B >= 0 && W >= 1 && W <= kAdlMaxWindow && kmin >= 1 && kmax >= kmin &&
           kmax <= kAdlMaxLength && up >= 0 && up <= kAdlMaxLength && down >= 0 &&
           down <= kAdlMaxLength;
}

}  // namespace

int sdv_adl_state_words(int window) {
    return window >= 1 && window <= kAdlMaxWindow ? adl_state_words(window) : -1;
}

sdv_status sdv_adl_step_host(int B, int window, int kmin, int kmax, int up, int down,
                             const int32_t* gen_len, const int32_t* acc_len, int32_t* k,
                             int32_t* state) {
    if (!adl_params_ok(B, window, kmin, kmax, up, down)) return SDV_ERR_ARG;
    if (B > 0 && (!gen_len || !acc_len || !k || !state)) return SDV_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (k[b] < kmin || k[b] > kmax) return SDV_ERR_ARG;     // nothing updated
    const int words = adl_state_words(window);
    for (int b = 0; b < B; ++b)
        k[b] = adl_update(state + static_cast<int64_t>(b) * words, window, kmin, kmax, up, down,
                          k[b], gen_len[b], acc_len[b]);
    return SDV_OK;
}

sdv_status sdv_adl_step(int B, int window, int kmin, int kmax, int up, int down, void* stream,
                        const int32_t* gen_len, const int32_t* acc_len, int32_t* k,
                        int32_t* state, int32_t* status) {
    if (!adl_params_ok(B, window, kmin, kmax, up, down)) return SDV_ERR_ARG;
    if (B == 0) return SDV_OK;
    if (!gen_len || !acc_len || !k || !state) return SDV_ERR_ARG;
    const void* ptrs[5] = {gen_len, acc_len, k, state, status};
    for (const void* p : ptrs)
        if (p && !is_device_ptr(p)) return SDV_ERR_ARG;
    AdlArgs a{B, window, kmin, kmax, up, down, gen_len, acc_len, k, state, status};
    return launch_adl(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SDV_OK : SDV_ERR_CUDA;
}

sdv_status sdv_set_test_hooks(sdv_ctx* ctx, unsigned hooks) {
    if (!ctx) return SDV_ERR_ARG;
    if (hooks & ~static_cast<unsigned>(SDV_HOOK_SAMPLE_NO_COPY))
        return fail(ctx, SDV_ERR_ARG, "unknown test hook bits 0x%x", hooks);
    ctx->hooks = hooks;
    return SDV_OK;
}

sdv_status sdv_set_stream(sdv_ctx* ctx, void* stream) {
    if (!ctx) return SDV_ERR_ARG;
    ctx->stream = static_cast<cudaStream_t>(stream);
    return SDV_OK;
}

}  // extern "C"
