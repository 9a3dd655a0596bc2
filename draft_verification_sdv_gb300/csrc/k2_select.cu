// k2_select.cu -- ratios, expected streaks, self-selection and the
// left-to-right acceptance scan; one CTA per sequence.
//
// Passages: "SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster
// Speculative Decoding", section 2 (accept x when q(x) <= p(x), else with
// probability p/q; the first rejection ends the scan), Figure 2 / section 3
// (position-wise acceptance and the accepted streak), section 5.2 (rank the
// K drafts by a streak-oriented verifier score, verify the best, reuse the
// cached verifier probabilities).  The score is the expected accepted length
// S_k = sum_j prod_{i<=j} min(1, p/q) of draft k; ties go to the lowest k.
//
// Uniforms: Philox4x32-10 with key (seed lo, seed hi), counter (j, b, 0, 0):
// word 0 is the acceptance uniform u_j, word 1 the sampling uniform w_j.
//
// Precision: the log-ratio of a drafted token is formed as
//   ((l_p(x) - m_p) - (l_q(x) - m_q)) * c - log2(S_p / S_q),
// where the bf16 differences are exact in fp32, so that its error scales with
// the log-ratio itself and two identical rows give a ratio of exactly 1.
#include "sdv_device.cuh"
#include "sdv_plan.h"

namespace sdv {
namespace {

constexpr int kBatch = 16;   // chunk partials loaded per round

// Merge the `chunks` partials of two rows in chunk order.  The loads of both
// rows go out together, kBatch at a time, so the merge chains do not wait on
// one load at a time.
__device__ __forceinline__ void merge_rows2(const float2* pa, const float2* pb, int chunks, float c,
                                            float& Ma, float& Sa, float& Mb, float& Sb) {
    Ma = Mb = -INFINITY;
    Sa = Sb = 0.0f;
    for (int i0 = 0; i0 < chunks; i0 += kBatch) {
        float2 va[kBatch], vb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const bool in = i0 + u < chunks;
            va[u] = in ? __ldcg(pa + i0 + u) : make_float2(-INFINITY, 0.0f);
            vb[u] = in ? __ldcg(pb + i0 + u) : make_float2(-INFINITY, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            merge_stat(Ma, Sa, va[u].x, va[u].y, c);
            merge_stat(Mb, Sb, vb[u].x, vb[u].y, c);
        }
    }
}

__device__ __forceinline__ void merge_row(const float2* part, int chunks, float c, float& M,
                                          float& S) {
    float m2, s2;
    merge_rows2(part, part, chunks, c, M, S, m2, s2);
}

// Merge the `chunks` partials of up to two rows (pb may be null) with a group
// of L lanes: lane gl merges chunks gl, gl + L, ... in chunk order, kBatch
// loads of each row in flight, then the lanes combine by a butterfly of
// shuffles (every lane of the warp executes it; L is the same for all).  An
// inactive lane contributes nothing.  With L = 1 this is the plain merge in
// chunk order.
__device__ __forceinline__ void group_merge2(const float2* pa, const float2* pb, int chunks, float c,
                                             int L, int gl, bool active, float& Ma, float& Sa,
                                             float& Mb, float& Sb) {
    Ma = Mb = -INFINITY;
    Sa = Sb = 0.0f;
    if (active) {
        for (int i0 = gl; i0 < chunks; i0 += kBatch * L) {
            float2 va[kBatch], vb[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int ch = i0 + u * L;
                const bool in = ch < chunks;
                va[u] = in ? __ldcg(pa + ch) : make_float2(-INFINITY, 0.0f);
                vb[u] = in && pb ? __ldcg(pb + ch) : make_float2(-INFINITY, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                merge_stat(Ma, Sa, va[u].x, va[u].y, c);
                merge_stat(Mb, Sb, vb[u].x, vb[u].y, c);
            }
        }
    }
    for (int off = L >> 1; off > 0; off >>= 1) {
        const float ma = __shfl_xor_sync(0xffffffffu, Ma, off), sa = __shfl_xor_sync(0xffffffffu, Sa, off);
        const float mb = __shfl_xor_sync(0xffffffffu, Mb, off), sb = __shfl_xor_sync(0xffffffffu, Sb, off);
        merge_stat(Ma, Sa, ma, sa, c);
        merge_stat(Mb, Sb, mb, sb, c);
    }
}

__device__ __forceinline__ bool row_valid(float M, float S) {
    return isfinite(M) && isfinite(S) && S > 0.0f;
}

// Natural-log LSE of l / T from (max, sum of 2^{(l - max) c}).
__device__ __forceinline__ float row_lse(float M, float S, float c) {
    return (M * c + log2f(S)) * kLn2;
}

// The drafter row's statistics of a pair: none under greedy acceptance, the
// caller's when supplied (an entry of another temperature is a data error),
// else those merged from the row pass's partials (left as they are).
__device__ __forceinline__ void pair_q_stat(const SelectArgs& a, bool greedy, int64_t rq, float c,
                                            float& mq, float& sq, unsigned* bad) {
    if (greedy) {
        mq = 0.0f;
        sq = 1.0f;
    } else if (a.q_stat) {
        const float4 st = a.q_stat[rq];
        mq = st.x;
        sq = st.y;
        if (st.z != c) atomicOr(bad, kStatusBadStat);
    }
}

// Acceptance ratio of a drafted token from its two logits and the rows'
// statistics: p(x) under greedy acceptance, else min(1, p/q) in
// exact-difference log form.  A bad row or token id sets its flag; the ratio
// is then 0 and unused.
__device__ __forceinline__ float pair_ratio(bool greedy, bool x_ok, float lp, float lq, float mp,
                                            float sp, float mq, float sq, float c, unsigned* bad) {
    if (!row_valid(mp, sp) || !row_valid(mq, sq)) {
        atomicOr(bad, kStatusBadRow);
        return 0.0f;
    }
    if (!x_ok) {
        atomicOr(bad, kStatusBadDraft);
        return 0.0f;
    }
    if (greedy) {
        const float d = (lp - mp) * c - log2f(sp);
        return d >= 0.0f ? 1.0f : ex2(d);
    }
    if (lq == -INFINITY) return 1.0f;                       // q(x) = 0 <= p(x)
    const float d = ((lp - mp) - (lq - mq)) * c - log2f(sp / sq);
    return d >= 0.0f ? 1.0f : ex2(d);                       // q <= p accepts at once
}

// GROUPED: rows merged by groups of a.merge_lanes lanes (few rows with many
// chunks); otherwise one thread per row, bonus rows on the last threads.
template <bool BF16, bool GROUPED>
__global__ void __launch_bounds__(kSelectThreads) select_kernel(const SelectArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int K = a.K, G = a.G;
    const int KG = K * G;
    // shared memory (select_smem_bytes): merged row statistics (max, sum) of
    // every p row [K][G+1] and q row [K][G], the ratios [K][RS] (an odd row
    // stride, so that the score loop's threads, one per draft, read distinct
    // banks), the scores [K]
    const int RS = G | 1;
    float2* pstat = reinterpret_cast<float2*>(smem_raw);
    float2* qstat = pstat + K * (G + 1);
    float* ratio = reinterpret_cast<float*>(qstat + KG);
    float* score = reinterpret_cast<float*>(
        smem_raw + ((static_cast<size_t>(K) * (2 * G + 1) * 8 + static_cast<size_t>(K) * (G + 1) * 4 +
                     15) & ~size_t(15)));
    __shared__ unsigned s_bad;
    __shared__ int s_len;
    __shared__ int s_sel;

    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const bool greedy = (a.flags & kFlagGreedy) != 0;   // no drafter rows
    const float T = a.temps ? a.temps[b] : a.temperature;
    const float c = kLog2e / T;
    // this sequence's draft length: positions j >= Lg are not read
    const int len_in = a.lens ? a.lens[b] : G;
    const bool len_ok = len_in >= 0 && len_in <= G;
    const int Lg = len_ok ? len_in : 0;
    if (tid == 0) {
        s_bad = (isfinite(T) && T > 0.0f ? 0u : kStatusBadTemp) | (len_ok ? 0u : kStatusBadDraft);
        s_len = Lg;
    }
    __syncthreads();

    const int64_t seq_d = static_cast<int64_t>(b) * K * G;         // first draft of b
    const int nrow = greedy ? G + 1 : 2 * G + 1;        // LSE entries per draft

    if constexpr (!GROUPED) {
        // The drafted token of this thread's first pair and its two logits are
        // inputs of the step, not results of the row pass: fetch them before
        // waiting for the row pass to finish.
        int32_t x0 = 0;
        float lp0 = 0.0f, lq0 = 0.0f;
        if (tid < KG && tid - (tid / G) * G < Lg) {
            const int k = tid / G, j = tid - (tid / G) * G;
            x0 = a.drafts[seq_d + static_cast<int64_t>(k) * G + j];
            if (x0 >= 0 && x0 < a.V) {
                lp0 = load_logit(a.p, p_row_index(a.flags, b, k, j, K, G) * a.V + x0, BF16);
                if (!greedy) lq0 = load_logit(a.q, q_row_index(a.flags, b, k, j, K, G) * a.V + x0, BF16);
            }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // Let the sample kernel launch: it waits for this grid before reading.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

        // Acceptance ratio at every drafted token of every draft.
        for (int idx = tid; idx < KG; idx += kSelectThreads) {
            const int k = idx / G, j = idx - (idx / G) * G;
            if (j >= Lg) {                                    // past this sequence's drafts
                if (a.out_lse) {
                    float* lse = a.out_lse + (static_cast<int64_t>(b) * K + k) * nrow;
                    if (j > Lg) lse[j] = NAN;                 // j == Lg: the bonus row below
                    if (!greedy) lse[G + 1 + j] = NAN;
                }
                continue;
            }
            const int64_t rp = p_row_index(a.flags, b, k, j, K, G);
            const int64_t rq = greedy ? 0 : q_row_index(a.flags, b, k, j, K, G);
            int32_t x = x0;
            float lp = lp0, lq = lq0;
            if (idx != tid) {
                x = a.drafts[seq_d + static_cast<int64_t>(k) * G + j];
                if (x >= 0 && x < a.V) {
                    lp = load_logit(a.p, rp * a.V + x, BF16);
                    if (!greedy) lq = load_logit(a.q, rq * a.V + x, BF16);
                }
            }
            const bool x_ok = x >= 0 && x < a.V;
            float mp, sp, mq = 0.0f, sq = 1.0f;
            const float2* prow_part = a.part + rp * a.chunks;
            if (greedy || a.q_stat)
                merge_row(prow_part, a.chunks, c, mp, sp);
            else
                merge_rows2(prow_part, a.part + (a.rows_p + rq) * a.chunks, a.chunks, c, mp, sp, mq, sq);
            pair_q_stat(a, greedy, rq, c, mq, sq, &s_bad);
            pstat[k * (G + 1) + j] = make_float2(mp, sp);
            qstat[idx] = make_float2(mq, sq);
            if (a.out_lse) {
                float* lse = a.out_lse + (static_cast<int64_t>(b) * K + k) * nrow;
                lse[j] = row_lse(mp, sp, c);
                if (!greedy) lse[G + 1 + j] = row_lse(mq, sq, c);
            }
            ratio[k * RS + j] = pair_ratio(greedy, x_ok, lp, lq, mp, sp, mq, sq, c, &s_bad);
        }
        // The bonus rows (j = Lg, right after the last draft token; G for full
        // drafts): validity and LSE, on the last threads (idle above when K * G
        // leaves them free).
        for (int k = kSelectThreads - 1 - tid; k < K; k += kSelectThreads) {
            const int64_t rp = p_row_index(a.flags, b, k, Lg, K, G);
            float mp, sp;
            merge_row(a.part + rp * a.chunks, a.chunks, c, mp, sp);
            pstat[k * (G + 1) + Lg] = make_float2(mp, sp);
            if (a.out_lse) {
                float* lse = a.out_lse + (static_cast<int64_t>(b) * K + k) * nrow;
                lse[Lg] = row_lse(mp, sp, c);
                if (Lg < G) lse[G] = NAN;
            }
            if (!row_valid(mp, sp)) atomicOr(&s_bad, kStatusBadRow);
        }
        __syncthreads();

    } else {
    // Rows are merged by groups of L lanes (L = a.merge_lanes, a power of two
        // up to 32, the same for every CTA): lane i of a group merges chunks i,
        // i + L, ... in order, then the group combines its lanes by a butterfly.
        // Items are the K * G pairs (p row and q row of a drafted token), then
        // the K bonus rows (p at position Lg).  Every thread runs the same number
        // of rounds, so the butterfly's shuffles see the whole warp.
        const int L = a.merge_lanes;
        const int gid = tid / L, gl = tid & (L - 1);
        const int ngroups = kSelectThreads / L;
        const int nitems = KG + K;

        // The drafted token of this group's first pair and its two logits are
        // inputs of the step, not results of the row pass: fetch them before
        // waiting for the row pass to finish.
        int32_t x0 = 0;
        float lp0 = 0.0f, lq0 = 0.0f;
        if (gl == 0 && gid < KG && gid - (gid / G) * G < Lg) {
            const int k = gid / G, j = gid - (gid / G) * G;
            x0 = a.drafts[seq_d + static_cast<int64_t>(k) * G + j];
            if (x0 >= 0 && x0 < a.V) {
                lp0 = load_logit(a.p, p_row_index(a.flags, b, k, j, K, G) * a.V + x0, BF16);
                if (!greedy) lq0 = load_logit(a.q, q_row_index(a.flags, b, k, j, K, G) * a.V + x0, BF16);
            }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // Let the sample kernel launch: it waits for this grid before reading.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

        for (int base = 0; base < nitems; base += ngroups) {
            const int item = base + gid;
            const bool is_pair = item < KG;
            const bool is_bonus = !is_pair && item < nitems;
            const int k = is_pair ? item / G : item - KG;
            const int j = is_pair ? item - k * G : Lg;
            // a pair past this sequence's drafts reads nothing
            const bool active = is_bonus || (is_pair && j < Lg);
            const int64_t rp = active ? p_row_index(a.flags, b, k, j, K, G) : 0;
            const int64_t rq = is_pair && !greedy ? q_row_index(a.flags, b, k, j, K, G) : 0;
            const bool merge_q = is_pair && !greedy && !a.q_stat;
            float mp, sp, mq, sq;
            group_merge2(a.part + rp * a.chunks, merge_q ? a.part + (a.rows_p + rq) * a.chunks : nullptr,
                         a.chunks, c, L, gl, active, mp, sp, mq, sq);
            if (gl != 0) continue;
            float* lse = a.out_lse ? a.out_lse + (static_cast<int64_t>(b) * K + k) * nrow : nullptr;
            if (is_bonus) {
                // the bonus row (j = Lg, right after the last draft token; G for
                // full drafts): validity and LSE
                pstat[k * (G + 1) + Lg] = make_float2(mp, sp);
                if (lse) {
                    lse[Lg] = row_lse(mp, sp, c);
                    if (Lg < G) lse[G] = NAN;
                }
                if (!row_valid(mp, sp)) atomicOr(&s_bad, kStatusBadRow);
                continue;
            }
            if (!is_pair) continue;
            if (!active) {                                    // past this sequence's drafts
                if (lse) {
                    if (j > Lg) lse[j] = NAN;                 // j == Lg: the bonus row
                    if (!greedy) lse[G + 1 + j] = NAN;
                }
                continue;
            }
            // acceptance ratio at the drafted token
            int32_t x = x0;
            float lp = lp0, lq = lq0;
            if (item != gid) {
                x = a.drafts[seq_d + static_cast<int64_t>(k) * G + j];
                if (x >= 0 && x < a.V) {
                    lp = load_logit(a.p, rp * a.V + x, BF16);
                    if (!greedy) lq = load_logit(a.q, rq * a.V + x, BF16);
                }
            }
            const bool x_ok = x >= 0 && x < a.V;
            pair_q_stat(a, greedy, rq, c, mq, sq, &s_bad);
            pstat[k * (G + 1) + j] = make_float2(mp, sp);
            qstat[item] = make_float2(mq, sq);
            if (lse) {
                lse[j] = row_lse(mp, sp, c);
                if (!greedy) lse[G + 1 + j] = row_lse(mq, sq, c);
            }
            ratio[k * RS + j] = pair_ratio(greedy, x_ok, lp, lq, mp, sp, mq, sq, c, &s_bad);
        }
        __syncthreads();

    }
    if (s_bad) {
        if (tid == 0) {
            a.out_sel[b] = -1;
            a.out_len[b] = -1;
            a.out_tok[b] = -1;
            SeqTask t = {};
            t.mode = 0;
            a.tasks[b] = t;
            atomicOr(a.status, s_bad);
        }
        return;
    }

    // Expected accepted streak of every draft (fp32 prefix products: GB300's
    // fp64 rate is a small fraction of its fp32 rate, and fp32 keeps the
    // score well inside the selection tolerance).
    // One warp per draft: the prefix products of 32 positions at a time by a
    // warp scan, their sum by a butterfly.
    {
        const int lane = tid & 31, warp = tid >> 5;
        for (int k = warp; k < K; k += kSelectThreads / 32) {
            float carry = 1.0f, sc = 0.0f;
            for (int j0 = 0; j0 < Lg; j0 += 32) {
                const bool in = j0 + lane < Lg;
                float pr = in ? ratio[k * RS + j0 + lane] : 1.0f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, pr, off);
                    if (lane >= off) pr *= y;
                }
                pr *= carry;
                float part = in ? pr : 0.0f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
                sc += part;
                carry = __shfl_sync(0xffffffffu, pr, 31);
            }
            if (lane == 0) {
                score[k] = sc;
                if (a.out_scores) a.out_scores[static_cast<int64_t>(b) * K + k] = sc;
            }
        }
    }
    __syncthreads();

    // Self-selection: first draft with the largest expected streak (warp 0:
    // each lane the first maximum of its drafts, then a butterfly that keeps
    // the larger score, on equal scores the lower k).
    if (tid < 32) {
        float best = -INFINITY;
        int bk = K;
        for (int k = tid; k < K; k += 32) {
            const float sc = score[k];
            if (bk == K || sc > best) {
                best = sc;
                bk = k;
            }
        }
        // lanes >= K hold no draft: only the steps below K can change lane 0
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            if (off >= K) continue;
            const float ob = __shfl_xor_sync(0xffffffffu, best, off);
            const int ok = __shfl_xor_sync(0xffffffffu, bk, off);
            if (ok < K && (bk == K || ob > best || (ob == best && ok < bk))) {
                best = ob;
                bk = ok;
            }
        }
        if (tid == 0) s_sel = bk;
    }
    __syncthreads();
    const int sel = s_sel;

    // Left-to-right acceptance of the selected draft: the first rejected j.
    // Thread j also keeps the sampling uniform of position j (up to Lg, the
    // bonus position), so that the thread of the first rejection writes the
    // task without drawing again.
    float my_w = 0.0f;
    for (int j = tid; j <= Lg; j += kSelectThreads) {
        const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u, 0u),
                                      a.seed_lo, a.seed_hi);
        if (j == tid) my_w = uniform24(r.y);
        if (j < Lg) {
            const float u = uniform24(r.x);
            const float aj = ratio[sel * RS + j];
            const bool accepted = (aj >= 1.0f) || (u < aj);
            if (!accepted) atomicMin(&s_len, j);
        }
    }
    __syncthreads();

    const int L = s_len;
    if (tid == (L < kSelectThreads ? L : 0)) {
        a.out_sel[b] = sel;
        a.out_len[b] = L;
        SeqTask t = {};
        if (L < kSelectThreads) {
            t.w = my_w;
        } else {
            const uint4 r = philox4x32_10(
                make_uint4(static_cast<uint32_t>(L), static_cast<uint32_t>(b), 0u, 0u), a.seed_lo,
                a.seed_hi);
            t.w = uniform24(r.y);
        }
        t.c = c;
        t.row_p = p_row_index(a.flags, b, sel, L, K, G);
        const float2 ps = pstat[sel * (G + 1) + L];
        t.off_p = -(ps.x * c) - log2f(ps.y);
        if (L < Lg && greedy) {
            t.mode = 3;                                   // p with the rejected token zeroed
            t.zero_id = a.drafts[seq_d + static_cast<int64_t>(sel) * G + L];
            t.row_q = -1;
        } else if (L < Lg) {
            t.mode = 1;                                   // residual max(0, p - q)
            t.row_q = q_row_index(a.flags, b, sel, L, K, G);
            const float2 qs = qstat[sel * G + L];
            t.off_q = -(qs.x * c) - log2f(qs.y);
        } else {
            t.mode = 2;                                   // bonus token from p at Lg
            t.row_q = -1;
        }
        a.tasks[b] = t;
    }
}

}  // namespace

cudaError_t setup_select(size_t smem) {
    const void* fns[4] = {reinterpret_cast<const void*>(select_kernel<true, false>),
                          reinterpret_cast<const void*>(select_kernel<true, true>),
                          reinterpret_cast<const void*>(select_kernel<false, false>),
                          reinterpret_cast<const void*>(select_kernel<false, true>)};
    for (const void* f : fns) {
        const cudaError_t e = raise_smem_limit(f, smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_select(const SelectArgs& a, bool bf16, size_t smem, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B));
    cfg.blockDim = dim3(kSelectThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const bool grouped = a.merge_lanes > 1;
    if (bf16) return grouped ? cudaLaunchKernelEx(&cfg, select_kernel<true, true>, a)
                             : cudaLaunchKernelEx(&cfg, select_kernel<true, false>, a);
    return grouped ? cudaLaunchKernelEx(&cfg, select_kernel<false, true>, a)
                   : cudaLaunchKernelEx(&cfg, select_kernel<false, false>, a);
}

}  // namespace sdv
