// k3_sample.cu -- the replacement or bonus token: inverse-CDF draw from the
// normalised residual max(0, p - q) of the first rejected position, or from
// p at position gamma + 1 when every draft token was accepted.
//
// Passages: "SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster
// Speculative Decoding", section 2 (at the first rejection the rest of the
// draft is discarded and a replacement is drawn from the normalised residual);
// "DiffuSpec: Unlocking Diffusion Language Models for Speculative Decoding",
// section 3 (the residual replacement keeps the procedure unbiased).  The
// draw returns the first id v whose cumulative weight exceeds w * R, R the
// total weight, w the sampling uniform of that position.  If the residual mass
// is zero (p == q up to rounding) the draw falls back to p.
//
// Only the one or two rows chosen per sequence are re-read.  A cluster of
// `cluster` CTAs (8, or 16 for batches of at most 16 sequences where the
// device can schedule clusters that wide) shares a sequence: each stages its slice of the row(s) in
// shared memory with one bulk (TMA) copy per row, forms the weights on the
// fly, scans them, and the CTAs exchange slice totals through distributed
// shared memory; the CTA whose slice holds the target finds the token.
#include "sdv_device.cuh"
#include "sdv_plan.h"

namespace sdv {
namespace {

constexpr uint32_t kMaxPolls = 1u << 22;   // bounded mbarrier wait
constexpr int kMaxCluster = 16;            // CTAs per sequence (16 is a non-portable cluster size)

// The two halves of a cluster barrier: arrive (no ordering) now, wait later.
// Used to know that every CTA of the cluster has started before writing to
// its shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Write two floats to the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ void st_dsmem_f32x2(float2* local, uint32_t rank, float x, float y) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(x), "f"(y) : "memory");
}

template <bool BF16>
struct Elems {
    static constexpr int kPerVec = BF16 ? 8 : 4;
};

// Element e of a 16-byte vector as fp32.
template <bool BF16>
__device__ __forceinline__ float elem(const uint4& v, int e) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (BF16) return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    else return __uint_as_float(w[e]);
}

// Sampling weights of the elements of vector i of the slice: p, or the
// residual max(0, p - q), each probability 2^(l * c + off) of its row; the
// element at slice position zero_pos (if any) gets weight 0 (greedy
// replacement: the rejected token is excluded).
template <bool BF16>
__device__ __forceinline__ void weights(const uint4* sp, const uint4* sq, int i, bool resid,
                                        int zero_pos, const SeqTask& t,
                                        float (&w)[Elems<BF16>::kPerVec]) {
    constexpr int EPV = Elems<BF16>::kPerVec;
    const uint4 pv = sp[i];
#pragma unroll
    for (int e = 0; e < EPV; ++e)
        w[e] = i * EPV + e == zero_pos ? 0.0f : ex2(fmaf(elem<BF16>(pv, e), t.c, t.off_p));
    if (resid) {
        const uint4 qv = sq[i];
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            w[e] = fmaxf(w[e] - ex2(fmaf(elem<BF16>(qv, e), t.c, t.off_q)), 0.0f);
    }
}

// Sum of the weights of one vector (pairwise tree, fixed order).
template <int N>
__device__ __forceinline__ float tree_sum(const float (&w)[N]) {
    if constexpr (N == 8) return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
    else return (w[0] + w[1]) + (w[2] + w[3]);
}

template <bool BF16>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ float s_incl[kSampleThreads];      // inclusive scan of thread sums
    __shared__ float s_warp[kSampleThreads / 32];
    __shared__ float s_total;                      // read by the whole cluster
    __shared__ float s_ok;                         // 1 if the slice arrived
    __shared__ int s_pick, s_last_thread, s_token;
    // (slice total, slice arrived) of every CTA of the cluster, per pass:
    // each CTA writes its own pair into every CTA's copy
    __shared__ float2 s_tot2[2][kMaxCluster];

    constexpr int EPV = Elems<BF16>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    const int CL = a.cluster;
    const int64_t b = blockIdx.x / CL;
    // Half a cluster barrier now; its wait, long after, tells that every CTA
    // has started, so that the totals may be written into their memory.
    cluster_arrive_relaxed();
    // The next step's row pass, when launched as a programmatic dependent,
    // may become resident now: it waits for this grid before it starts.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // The tasks are written by the select kernel: wait for it to finish.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const SeqTask t = a.tasks[b];
    const int64_t sv0 = static_cast<int64_t>(rank) * a.slice_vec;
    const int64_t sv1 = sv0 + a.slice_vec < a.nvec ? sv0 + a.slice_vec : a.nvec;
    const int nv = sv1 > sv0 ? static_cast<int>(sv1 - sv0) : 0;
    uint4* sp = reinterpret_cast<uint4*>(smem_raw);
    uint4* sq = sp + a.slice_vec;

    if (tid == 0) {
        mbar_init(&bar, 1);
        s_ok = 1.0f;
    }
    __syncthreads();
    if (t.mode != 0 && nv > 0) {
        // test hook: the barrier is armed but no copy is issued, so the wait
        // below runs out after a few polls with nothing in flight
        const bool no_copy = (a.hooks & kHookSampleNoCopy) != 0;
        const uint32_t polls = no_copy ? kTestPolls : kMaxPolls;
        if (tid == 0) {
            const uint32_t bytes = static_cast<uint32_t>(nv) * 16u;
            mbar_arrive_expect_tx(&bar, t.mode == 1 ? 2u * bytes : bytes);
            if (!no_copy) {
                bulk_g2s(sp, static_cast<const uint4*>(a.p) + t.row_p * a.nvec + sv0, bytes, &bar);
                if (t.mode == 1)
                    bulk_g2s(sq, static_cast<const uint4*>(a.q) + t.row_q * a.nvec + sv0, bytes, &bar);
            }
        }
        if (!mbar_wait_bounded(&bar, 0, polls)) {
            // Give the copies a second bounded chance to land before the
            // shared memory is released, and report the timeout.
            mbar_wait_bounded(&bar, 0, polls);
            if (tid == 0) {
                s_ok = 0.0f;
                atomicOr(a.status, kStatusTimeout);
            }
        }
    }
    __syncthreads();
    const bool have_data = (t.mode != 0) && (s_ok != 0.0f);

    // Contiguous vectors [tv0, tv1) of the slice belong to this thread.
    const int vpt = (nv + kSampleThreads - 1) / kSampleThreads;
    const int tv0 = min(tid * vpt, nv), tv1 = min(tv0 + vpt, nv);

    for (int pass = 0; pass < 2; ++pass) {
        const bool resid = (t.mode == 1) && (pass == 0);
        // greedy replacement: the rejected token's position within this slice
        const int zero_pos = (t.mode == 3 && pass == 0)
                                 ? static_cast<int>(static_cast<int64_t>(t.zero_id) - sv0 * EPV)
                                 : -1;
        // Per-vector sums are independent; the thread sum adds them in order.
        float tsum = 0.0f;
        if (have_data)
            for (int i = tv0; i < tv1; ++i) {
                float w[EPV];
                weights<BF16>(sp, sq, i, resid, zero_pos, t, w);
                tsum += tree_sum(w);
            }

        // Block inclusive scan of the thread sums (fixed order).
        float x = tsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        if (tid == 0) {
            s_pick = kSampleThreads;
            s_last_thread = -1;
            s_token = -1;
        }
        __syncthreads();
        if (warp == 0) {
            float wsum = lane < kSampleThreads / 32 ? s_warp[lane] : 0.0f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, wsum, off);
                if (lane >= off) wsum += y;
            }
            if (lane < kSampleThreads / 32) s_warp[lane] = wsum;
        }
        __syncthreads();
        const float incl = x + (warp > 0 ? s_warp[warp - 1] : 0.0f);
        s_incl[tid] = incl;
        if (tid == kSampleThreads - 1) s_total = incl;
        __syncthreads();

        // Slice totals of the whole cluster, in rank order: thread r writes
        // this CTA's (total, arrived) into CTA r; after the barrier every CTA
        // reads its own copy, and no CTA touches another's memory again.
        if (pass == 0) cluster_wait();
        if (tid < CL)
            st_dsmem_f32x2(&s_tot2[pass][rank], static_cast<uint32_t>(tid), s_total, s_ok);
        cluster_sync();
        float R = 0.0f, target_excl = 0.0f;
        bool all_ok = true;
        int owner = -1, last_rank = -1;
        float tot[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            const float2 v = r < CL ? s_tot2[pass][r] : make_float2(0.0f, 1.0f);
            tot[r] = v.x;
            all_ok = all_ok && v.y != 0.0f;
        }
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
            if (r < CL) R += tot[r];
        // Residual mass zero on this row: every CTA sees the same R, so the
        // whole cluster takes the fallback pass to p together.
        if (pass == 0 && (t.mode == 1 || t.mode == 3) && R == 0.0f && all_ok) continue;
        const float target = t.w * R;
        {
            // (loops over the largest cluster, skipping ranks past this one's,
            // so that the totals stay in registers)
            float run = 0.0f;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r) {
                if (r < CL) {
                    const float prev = run;
                    run += tot[r];
                    if (tot[r] > 0.0f) last_rank = r;
                    if (owner < 0 && run > target) {
                        owner = r;
                        target_excl = prev;
                    }
                }
            }
            if (owner < 0 && last_rank >= 0) {         // rounding put the target past the end
                owner = last_rank;
                float run2 = 0.0f;
#pragma unroll
                for (int r = 0; r < kMaxCluster; ++r)
                    if (r < last_rank) run2 += tot[r];
                target_excl = run2;
            }
        }

        if (have_data && all_ok && owner == static_cast<int>(rank)) {
            const float tl = target - target_excl;           // target within this slice
            if (incl > tl) atomicMin(&s_pick, tid);
            if (tsum > 0.0f) atomicMax(&s_last_thread, tid);
            __syncthreads();
            int pick = s_pick;
            if (pick == kSampleThreads) pick = s_last_thread;   // rounding fallback
            if (tid == pick) {
                // Two levels: the vector whose running sum passes the target,
                // then the element inside it.
                const float excl = tid > 0 ? s_incl[tid - 1] : 0.0f;
                const float tt = tl - excl;
                float run = 0.0f;
                int tok = -1, last_pos = -1;
                for (int i = tv0; i < tv1 && tok < 0; ++i) {
                    float w[EPV];
                    weights<BF16>(sp, sq, i, resid, zero_pos, t, w);
                    const float vs = tree_sum(w);
                    if (run + vs > tt) {
                        float r2 = run;
#pragma unroll
                        for (int e = 0; e < EPV; ++e) {
                            r2 += w[e];
                            if (w[e] > 0.0f) last_pos = i * EPV + e;
                            if (tok < 0 && r2 > tt) tok = i * EPV + e;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            if (w[e] > 0.0f) last_pos = i * EPV + e;
                    }
                    run += vs;
                }
                if (tok < 0) tok = last_pos;
                if (tok >= 0) s_token = tok;
            }
            __syncthreads();
            if (tid == 0) {
                int tok = s_token;
                if (tok < 0 && s_last_thread >= 0) {
                    // The picked thread held no mass: take the last id with mass.
                    const int lt = s_last_thread;
                    const int l0 = min(lt * vpt, nv), l1 = min(l0 + vpt, nv);
                    for (int i = l0; i < l1; ++i) {
                        float w[EPV];
                        weights<BF16>(sp, sq, i, resid, zero_pos, t, w);
                        for (int e = 0; e < EPV; ++e)
                            if (w[e] > 0.0f) tok = i * EPV + e;
                    }
                }
                a.out_tok[b] = tok >= 0 ? static_cast<int32_t>(sv0 * EPV + tok) : -1;
            }
        } else if (t.mode != 0 && !all_ok && rank == 0 && tid == 0) {
            // a slice never arrived: no output of this sequence is reported
            a.out_sel[b] = -1;
            a.out_len[b] = -1;
            a.out_tok[b] = -1;
        }
        break;
    }
}

}  // namespace

cudaError_t setup_sample(size_t smem) {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(sample_kernel<true>), smem);
    if (e == cudaSuccess) e = raise_smem_limit(reinterpret_cast<const void*>(sample_kernel<false>), smem);
    // clusters of 16 CTAs (beyond the portable 8) for small batches
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sample_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sample_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

int sample_max_cluster() { return kMaxCluster; }

int sample_active_clusters(bool bf16, int cluster, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    cfg.blockDim = dim3(kSampleThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = bf16 ? cudaOccupancyMaxActiveClusters(&n, sample_kernel<true>, &cfg)
                               : cudaOccupancyMaxActiveClusters(&n, sample_kernel<false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_sample(const SampleArgs& a, bool bf16, int B, int cluster, size_t smem,
                          cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B * cluster));
    cfg.blockDim = dim3(kSampleThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    if (bf16) return cudaLaunchKernelEx(&cfg, sample_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, sample_kernel<false>, a);
}

}  // namespace sdv
