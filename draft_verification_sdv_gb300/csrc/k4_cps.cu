// k4_cps.cu -- causal-consistency path search over drafter marginals
// ("DiffuSpec: Unlocking Diffusion Language Models for Speculative Decoding",
// section 4.2; settings of section 5.3: beam 3, at most 15 candidates, mass
// 0.8).  The causal fluency proxy the page mentions is not specified there, so
// a path is scored by drafter confidence alone: the sum of its per-position
// log-probabilities.
//
// cps_prune_kernel, one CTA per drafter row q[b, j, :]: the row is cut into
// 4 KB chunks and warp w takes chunks w, w + NW, w + 2 NW, ... (eight 16-byte
// loads in flight per lane), keeping the online softmax statistics (max,
// sum 2^{(l - max) c}) and the warp's 16 largest logits (ties to the lower
// id) as one key per lane.  The interleaving spreads a row's first chunks,
// where the best logits often sit, over all its warps; it is fixed, so every
// sum is taken in the same order on every run.  Only a vector holding a
// value at or above a floor the row's 16th best is known to reach enters the
// (rare, warp-uniform) insertion path.  Warp 0 then merges the warps' lists
// and statistics.  The
// kept candidates are the shortest prefix of the row's list, in order of
// probability, whose mass reaches tau, capped at mmax; tokens of probability
// zero are never candidates, and a row with a NaN or +inf logit, or none
// finite, keeps none.  On request it also writes the row's statistics
// {max, sum 2^{(l - max) c}, c}, so that a verification of the same marginals
// need not stream them again.
//
// cps_beam_kernel, one warp per sequence: the lattice ends at the first
// position whose most likely candidate is eos_id (kept alone as the last
// token); a left-to-right beam of width W keeps, at every step, the W best
// prefixes.  A path's score is the sum of its log-probabilities; the
// temperature and the positions' normalisers are common to all paths, so
// prefixes rank by the sum of their raw logits, taken left to right in fp64
// (exact for bf16 logits), with equal sums in lexicographic order of their
// candidate ranks (tracked as each beam's place among the beams).  With a
// separable score this gives the W best paths of the whole lattice.
#include <climits>

#include "sdv_device.cuh"
#include "sdv_plan.h"

namespace sdv {
namespace {

constexpr int kTopK = 16;                  // list length (mmax <= 16)
constexpr int kBeamMaxExp = kCpsMaxBeam * kCpsMaxCand;   // expansions per step

// Order-preserving 32-bit key of a logit (larger value -> larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key32_value(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

__device__ __forceinline__ float key_value(uint64_t key) {
    return key32_value(static_cast<uint32_t>(key >> 32));
}

// Key of (logit, id): value first, then the lower id.  0 = empty slot.
__device__ __forceinline__ uint64_t cand_key(float f, uint32_t id) {
    return (static_cast<uint64_t>(order_key(f)) << 32) | static_cast<uint64_t>(0xffffffffu - id);
}

__device__ __forceinline__ uint32_t key_id(uint64_t key) {
    return 0xffffffffu - static_cast<uint32_t>(key & 0xffffffffu);
}

// The warp's best kTopK keys, one per lane: lane i < kTopK holds the i-th
// largest (0 = empty slot), lanes >= kTopK hold 0.  Inserting a warp-uniform
// key shifts the smaller ones down one lane.
__device__ __forceinline__ uint64_t wlist_insert(uint64_t mine, uint64_t k, int lane) {
    const uint64_t prev = __shfl_up_sync(0xffffffffu, mine, 1);
    if (lane < kTopK && !(mine > k)) mine = (lane == 0 || prev > k) ? k : prev;
    return mine;
}

__device__ __forceinline__ float wlist_threshold(uint64_t mine) {
    const uint64_t last = __shfl_sync(0xffffffffu, mine, kTopK - 1);
    return last ? key_value(last) : -INFINITY;
}

// Logit i of a 16-byte vector (selects, no local memory).
template <bool BF16>
__device__ __forceinline__ float vec_elem(uint32_t x, uint32_t y, uint32_t z, uint32_t w, int i) {
    if constexpr (BF16) {
        const uint32_t wd = i < 4 ? (i < 2 ? x : y) : (i < 6 ? z : w);
        return (i & 1) ? bf16_hi(wd) : bf16_lo(wd);
    } else {
        return __uint_as_float(i < 2 ? (i == 0 ? x : y) : (i == 2 ? z : w));
    }
}

// The list seeded with the 16 largest of the lanes' keys (0 = none): a
// bitonic sort of the 32 keys, descending, of which lanes 0..15 keep theirs.
__device__ __forceinline__ uint64_t wlist_seed(uint64_t key, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xffffffffu, key, j);
            const bool take_max = ((lane & j) == 0) == ((lane & k) == 0);
            const uint64_t hi = key > other ? key : other, lo = key > other ? other : key;
            key = take_max ? hi : lo;
        }
    }
    return lane < kTopK ? key : 0;
}

// Offer the lanes' 16-byte vectors (lane's ids id0 .. id0 + EPV - 1, its
// vector max vmax) to the warp's list.  Only lanes whose vector reaches
// `floor` (a value the warp's 16th best is known to reach) take part: each in
// turn broadcasts its vector, lanes 0 .. EPV-1 take one logit each, and the
// logits that beat the list's last key are inserted.
// With `dedup`, a key already in the list (a seeded one) is not inserted again.
template <bool BF16>
__device__ __noinline__ uint64_t wlist_absorb(uint4 v, uint32_t id0, float vmax, uint64_t mine,
                                              float floor, bool dedup, int lane) {
    constexpr int EPV = BF16 ? 8 : 4;
    uint64_t last = __shfl_sync(0xffffffffu, mine, kTopK - 1);
    unsigned hot = __ballot_sync(0xffffffffu, vmax >= floor && vmax != -INFINITY);
    while (hot) {
        const int src = __ffs(hot) - 1;
        hot &= hot - 1;
        const uint32_t x = __shfl_sync(0xffffffffu, v.x, src);
        const uint32_t y = __shfl_sync(0xffffffffu, v.y, src);
        const uint32_t z = __shfl_sync(0xffffffffu, v.z, src);
        const uint32_t w = __shfl_sync(0xffffffffu, v.w, src);
        const uint32_t base = __shfl_sync(0xffffffffu, id0, src);
        const int i = lane & (EPV - 1);
        const float f = vec_elem<BF16>(x, y, z, w, i);
        const uint64_t key = cand_key(f, base + i);
        // a -inf logit has probability zero and is never a candidate
        unsigned pending = __ballot_sync(
            0xffffffffu, lane < EPV && f != -INFINITY && f >= floor && key > last);
        while (pending) {
            const int l = __ffs(pending) - 1;
            pending &= pending - 1;
            const uint64_t k = __shfl_sync(0xffffffffu, key, l);
            if (k > last && !(dedup && __any_sync(0xffffffffu, mine == k))) {
                mine = wlist_insert(mine, k, lane);
                last = __shfl_sync(0xffffffffu, mine, kTopK - 1);
            }
        }
    }
    return mine;
}

// Sum of 2^{(l - m) c} over the logits of one 16-byte vector, as
// vec_exp_sum computes it, but with each exponent formed by one fused
// multiply-add,
// l * c + nmc with nmc = -(m * c): one instruction fewer per logit than the
// exact-difference form above, at a rounding error of about one unit in the
// last place of |l * c| in the exponent (a relative error near 1e-6 in each
// term for logits of a few tens).
template <bool BF16>
__device__ __forceinline__ float vec_exp_sum_fma(const uint4& v, float c, float nmc) {
    if constexpr (BF16) {
        const float e0 = ex2(fmaf(bf16_lo(v.x), c, nmc)), e1 = ex2(fmaf(bf16_hi(v.x), c, nmc));
        const float e2 = ex2(fmaf(bf16_lo(v.y), c, nmc)), e3 = ex2(fmaf(bf16_hi(v.y), c, nmc));
        const float e4 = ex2(fmaf(bf16_lo(v.z), c, nmc)), e5 = ex2(fmaf(bf16_hi(v.z), c, nmc));
        const float e6 = ex2(fmaf(bf16_lo(v.w), c, nmc)), e7 = ex2(fmaf(bf16_hi(v.w), c, nmc));
        return ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7));
    } else {
        const float e0 = ex2(fmaf(__uint_as_float(v.x), c, nmc));
        const float e1 = ex2(fmaf(__uint_as_float(v.y), c, nmc));
        const float e2 = ex2(fmaf(__uint_as_float(v.z), c, nmc));
        const float e3 = ex2(fmaf(__uint_as_float(v.w), c, nmc));
        return (e0 + e1) + (e2 + e3);
    }
}

constexpr int kHalf = 4;                   // 16-byte vectors per lane in each half-batch
static_assert((kHalf & (kHalf - 1)) == 0, "the pairwise sum tree needs a power of two");

// NaN-propagating max of one 16-byte vector.
template <bool BF16>
__device__ __forceinline__ float vec1_max(const uint4& v) {
    if constexpr (BF16) {
        uint32_t a = v.x, b = v.z;
        asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(v.y));
        asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(b) : "r"(v.w));
        asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(b));
        float r;
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(bf16_lo(a)), "f"(bf16_hi(a)));
        return r;
    } else {
        float r = __uint_as_float(v.x), t = __uint_as_float(v.z);
        asm("max.NaN.f32 %0, %0, %1;" : "+f"(r) : "f"(__uint_as_float(v.y)));
        asm("max.NaN.f32 %0, %0, %1;" : "+f"(t) : "f"(__uint_as_float(v.w)));
        asm("max.NaN.f32 %0, %0, %1;" : "+f"(r) : "f"(t));
        return r;
    }
}

// The 16th largest of the lanes' values (-inf when fewer than 16 are finite):
// at least 16 logits of the batch reach it, so the warp's 16th best does too.
__device__ __forceinline__ float warp_16th(float x, int lane) {
    int rank = 0;
#pragma unroll
    for (int l2 = 0; l2 < 32; ++l2) {
        const float y = __shfl_sync(0xffffffffu, x, l2);
        rank += (y > x) || (y == x && l2 < lane);
    }
    const unsigned at = __ballot_sync(0xffffffffu, rank == kTopK - 1);
    const float t = __shfl_sync(0xffffffffu, x, at ? __ffs(at) - 1 : 0);
    return at && t == t ? t : -INFINITY;
}

// One CTA of NW warps per row; each warp streams a contiguous 1/NW of it.
template <bool BF16, int NW>
__global__ void __launch_bounds__(NW * 32, NW <= 4 ? 7 : (NW <= 8 ? 3 : 2)) cps_prune_kernel(const CpsArgs a) {
    __shared__ uint64_t s_best[NW][kTopK];
    __shared__ float s_m[NW], s_s[NW];
    // the highest list threshold any warp of the row has reached (order key):
    // the row's 16th best is at least that, so every warp may skip below it
    __shared__ unsigned s_floor;
    const int64_t row = blockIdx.x;
    const int b = static_cast<int>(row / a.G);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float T = a.temps ? a.temps[b] : a.temperature;
    const float c = kLog2e / T;
    const uint4* rowv = static_cast<const uint4*>(a.q) + row * a.nvec;
    constexpr int EPV = BF16 ? 8 : 4;
    // The row is cut into chunks of two half-batches (64 * kHalf vectors);
    // warp w takes chunks w, w + NW, ...: a fixed order, so that the row's
    // sums round the same way on every run.
    constexpr int64_t kChunk = 64 * kHalf;
    const int64_t v1 = a.nvec;
    const int nchunks = static_cast<int>((a.nvec + kChunk - 1) / kChunk);

    // No kernel launches as this one's programmatic dependent, but with this
    // trigger back-to-back pruning passes measured 0.060 ms against 0.064 ms.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) s_floor = order_key(-INFINITY);
    __syncthreads();

    uint64_t mine = 0;                // this lane's slot of the warp's list
    float thr = -INFINITY;            // value of the list's last key once full
    float m = -INFINITY, s = 0.0f;
    // One half-batch of kHalf vectors per lane: the softmax statistics, then
    // the candidates when some lane holds a value that may enter the list.
    auto process = [&](const uint4 (&w)[kHalf], int64_t base) {
        const float vm = vec_max_n<BF16, kHalf>(w);
        if (!(vm <= m)) {                 // new maximum (or NaN: poisons s)
            s *= ex2((m - vm) * c);
            m = vm;
        }
        if (m != -INFINITY) {
            const float nmc = -(m * c);
            float t[kHalf];
#pragma unroll
            for (int u = 0; u < kHalf; ++u) t[u] = vec_exp_sum_fma<BF16>(w[u], c, nmc);
#pragma unroll
            for (int h = kHalf / 2; h > 0; h >>= 1)
#pragma unroll
                for (int u = 0; u < h; ++u) t[u] += t[u + h];
            s += t[0];
        }
        const float row_floor = key32_value(*reinterpret_cast<volatile unsigned*>(&s_floor));
        const float gate = thr > row_floor ? thr : row_floor;
        if (!__any_sync(0xffffffffu, vm >= gate && vm != -INFINITY)) return;
        float floor = gate;
        float vmu[kHalf];
#pragma unroll
        for (int u = 0; u < kHalf; ++u) vmu[u] = vec1_max<BF16>(w[u]);
        bool seeded = false;
        if (thr == -INFINITY) {
            if (!__any_sync(0xffffffffu, mine != 0)) {
                // empty list: seed it with the 16 largest lane maxima (each
                // lane's first maximum, the lowest id); the 16th bounds the
                // warp's 16th best from below
                int uu = 0;
#pragma unroll
                for (int u = kHalf - 1; u >= 0; --u) uu = vmu[u] == vm ? u : uu;
                uint4 v = w[0];
#pragma unroll
                for (int u = 1; u < kHalf; ++u) v = u == uu ? w[u] : v;
                int ii = 0;
#pragma unroll
                for (int i = EPV - 1; i >= 0; --i)
                    ii = vec_elem<BF16>(v.x, v.y, v.z, v.w, i) == vm ? i : ii;
                const uint32_t id = static_cast<uint32_t>((base + 32 * uu) * EPV + ii);
                const bool real = vm != -INFINITY && vm == vm;
                const uint64_t key0 = real ? cand_key(vm, id) : 0;
                mine = wlist_seed(key0, lane);
                seeded = true;
                const float t0 = wlist_threshold(mine);
                floor = t0 > floor ? t0 : floor;
                // a lane whose seeded maximum is its only logit at or above
                // the floor has nothing more to offer from that vector
                float m2 = -INFINITY;
#pragma unroll
                for (int i = 0; i < EPV; ++i) {
                    const float e = vec_elem<BF16>(v.x, v.y, v.z, v.w, i);
                    m2 = i != ii && e > m2 ? e : m2;
                }
                const uint64_t last = __shfl_sync(0xffffffffu, mine, kTopK - 1);
                if (real && key0 >= last && !(m2 >= floor)) {
#pragma unroll
                    for (int u = 0; u < kHalf; ++u) vmu[u] = u == uu ? -INFINITY : vmu[u];
                }
            } else {
                // a partly filled list: the 16th largest lane maximum of
                // this batch bounds the warp's 16th best from below
                const float t0 = warp_16th(vm, lane);
                floor = t0 > floor ? t0 : floor;
            }
        }
#pragma unroll
        for (int u = 0; u < kHalf; ++u) {
            if (__any_sync(0xffffffffu, vmu[u] >= floor && vmu[u] != -INFINITY)) {
                const int64_t vec = base + 32 * u;
                mine = wlist_absorb<BF16>(w[u], static_cast<uint32_t>(vec * EPV), vmu[u], mine,
                                          floor, seeded, lane);
                const float t2 = wlist_threshold(mine);
                floor = t2 > floor ? t2 : floor;
            }
        }
        thr = wlist_threshold(mine);
        if (lane == 0 && thr > row_floor) atomicMax(&s_floor, order_key(thr));
    };
    auto load = [&](uint4 (&w)[kHalf], int64_t base) {
#pragma unroll
        for (int u = 0; u < kHalf; ++u) {
            const int64_t idx = base + 32 * u;
            const uint32_t ninf = BF16 ? 0xFF80FF80u : 0xFF800000u;
            w[u] = idx < v1 ? ld_stream(rowv + idx) : make_uint4(ninf, ninf, ninf, ninf);
        }
    };
    // The two half-batches of a chunk in turn: while one is processed the
    // other is in flight, and the next chunk's first half is loaded before
    // the second half of this one is processed, so the loads continue
    // through the candidate work.  Every lane of a warp runs the same
    // iterations (warp-wide votes inside).
    uint4 wa[kHalf], wb[kHalf];
    int chunk = warp;
    int64_t base = chunk * kChunk + lane;
    load(wa, base);
    load(wb, base + 32 * kHalf);
    {
        // A floor for the whole row before any warp builds its list: the
        // 16th largest lane maximum of a warp's first half-batch is a value
        // that 16 logits of the row reach.  The largest of the warps' floors
        // gates every warp from the start.
        const float f = warp_16th(vec_max_n<BF16, kHalf>(wa), lane);
        if (lane == 0 && f != -INFINITY) atomicMax(&s_floor, order_key(f));
    }
    __syncthreads();
    while (chunk < nchunks) {
        const int next = chunk + NW;
        const int64_t nbase = next * kChunk + lane;
        process(wa, base);
        load(wa, nbase);
        process(wb, base + 32 * kHalf);
        load(wb, nbase + 32 * kHalf);
        chunk = next;
        base = nbase;
    }
    // row statistics: warp, then CTA
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        merge_stat(m, s, m2, s2, c);
    }
    if (lane < kTopK) s_best[warp][lane] = mine;
    if (lane == 0) {
        s_m[warp] = m;
        s_s[warp] = s;
    }
    __syncthreads();
    if (warp != 0) return;
    // warp 0 merges the other warps' lists into its own, best keys first
    uint64_t last = __shfl_sync(0xffffffffu, mine, kTopK - 1);
    for (int w2 = 1; w2 < NW; ++w2) {
        for (int i = 0; i < kTopK; ++i) {
            const uint64_t k = s_best[w2][i];          // same address in every lane
            if (k <= last) break;                      // that list is descending
            mine = wlist_insert(mine, k, lane);
            last = __shfl_sync(0xffffffffu, mine, kTopK - 1);
        }
    }
    float M = s_m[0], S = s_s[0];
    for (int w2 = 1; w2 < NW; ++w2) merge_stat(M, S, s_m[w2], s_s[w2], c);
    // the row's softmax statistics, for a verification of these marginals
    // that then need not read the rows again
    if (lane == 0 && a.row_stat) a.row_stat[row] = make_float4(M, S, c, 0.0f);
    // lane r holds the rank-r candidate; the cut is a running sum of masses
    const int mmax = a.mmax;
    const bool ok = isfinite(M) && isfinite(S) && S > 0.0f;
    float pm = 0.0f, lp = -INFINITY;
    if (ok && mine != 0) {
        const float val = key_value(mine);
        lp = ((val - M) * c - log2f(S)) * kLn2;
        pm = ex2((val - M) * c) * (1.0f / S);
    }
    // inclusive running mass in rank order, added one by one in that order
    float run = 0.0f, mine_after = 0.0f;
    for (int r = 0; r < kTopK; ++r) {
        run += __shfl_sync(0xffffffffu, pm, r);
        if (lane == r) mine_after = run;
    }
    // n = first rank whose running mass reaches tau (+1), at most mmax, and
    // only over existing candidates
    const bool stop_here = lane < mmax && mine != 0 && mine_after >= a.tau;
    const unsigned stop_mask = __ballot_sync(0xffffffffu, stop_here);
    const unsigned have_mask = __ballot_sync(0xffffffffu, lane < mmax && mine != 0);
    int n = stop_mask ? __ffs(stop_mask) : __popc(have_mask);
    if (!ok) n = 0;
    int32_t* ids = a.cand_ids + row * mmax;
    float* lpo = a.cand_logp + row * mmax;
    float* lgo = a.cand_logit + row * mmax;
    if (lane < mmax) {
        ids[lane] = lane < n ? static_cast<int32_t>(key_id(mine)) : -1;
        lpo[lane] = lane < n ? lp : -INFINITY;
        lgo[lane] = lane < n ? key_value(mine) : -INFINITY;
    }
    if (lane == 0) a.ncand[row] = n;      // 0 for a row with NaN / +inf / only -inf
}

// ceil(65536 / n) for n = 1..16: (e * kDivMagic[n]) >> 16 == e / n for e < 256.
__constant__ unsigned kDivMagic[17] = {0,    65536, 32768, 21846, 16384, 13108, 10923, 9363, 8192,
                                       7282, 6554,  5958,  5462,  5042,  4682,  4370,  4096};

// An integer with the order of a double (keys here are never NaN and never
// -0: a sum that cancels to zero rounds to +0).  Integer compares keep the
// ranking off the (slow) fp64 pipe.
__device__ __forceinline__ long long ordered_i64(double d) {
    const long long bits = __double_as_longlong(d);
    return bits ^ ((bits >> 63) & 0x7fffffffffffffffLL);
}

// One lattice position as a lane of the beam sees it: the candidate count
// n (1 at an EOS end), the expanded count nw = min(n, W), the divide
// constant for e / nw, and expansion e = lane's parent beam, candidate rank
// and the candidate's raw logit and log-probability.
struct BeamPos {
    int n, nw, par, r;
    unsigned magic;
    float rl, lp;
};

__device__ __forceinline__ BeamPos beam_position(const int* nc_s, const float* rl_s, const float* clp_s,
                                                 int j, int Lc, bool eos_cut, int W, int M, int lane) {
    BeamPos p;
    p.n = eos_cut && j == Lc - 1 ? 1 : nc_s[j];          // EOS is kept alone
    // A parent's expansions come in candidate order (raw logits sorted, ties
    // by id), so only its first W can be among the W best.
    p.nw = p.n < W ? p.n : W;
    // e / nw as a multiply and shift: exact for e < 256 and nw <= 16
    p.magic = kDivMagic[p.nw];
    p.par = static_cast<int>((static_cast<unsigned>(lane) * p.magic) >> 16);
    p.r = lane - p.par * p.nw;
    p.rl = rl_s[j * M + p.r];                            // r < nw <= M
    p.lp = clp_s[j * M + p.r];
    return p;
}

__global__ void __launch_bounds__(32) cps_beam_kernel(const CpsArgs a) {
    // dynamic shared memory: the lattice's log-probabilities [G][M] and raw
    // logits [G][M] (float), counts [G], then the back-pointers [G][W] parent
    // and [G][W] rank, and the final paths' ranks [W][G]
    extern __shared__ __align__(16) unsigned char s_raw[];
    __shared__ double x_key[kBeamMaxExp];      // this step's expansions
    __shared__ long long x_ord[kBeamMaxExp];   // x_key as an order-preserving integer
    __shared__ float x_score[kBeamMaxExp];
    __shared__ int x_lx[kBeamMaxExp];
    __shared__ double b_key[kCpsMaxBeam];      // the beams
    __shared__ float b_score[kCpsMaxBeam];
    __shared__ int b_lex[kCpsMaxBeam];
    __shared__ double n_key[kCpsMaxBeam];      // the beams being chosen
    __shared__ float n_score[kCpsMaxBeam];
    __shared__ int n_lx[kCpsMaxBeam];
    __shared__ int s_src[kCpsMaxBeam];         // beam t's expansion (ranked path)
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    const int G = a.G, W = a.beam, M = a.mmax;
    float* clp_s = reinterpret_cast<float*>(s_raw);
    float* rl_s = clp_s + G * M;
    int* nc_s = reinterpret_cast<int*>(rl_s + G * M);
    unsigned char* bp_parent = reinterpret_cast<unsigned char*>(nc_s + G);
    unsigned char* bp_rank = bp_parent + G * W;
    unsigned char* path_rank = bp_rank + G * W;
    int32_t* cids = a.cand_ids + static_cast<int64_t>(b) * G * M;
    float* clp = a.cand_logp + static_cast<int64_t>(b) * G * M;
    float* crl = a.cand_logit + static_cast<int64_t>(b) * G * M;
    int32_t* nc = a.ncand + static_cast<int64_t>(b) * G;
    if ((G * M) % 4 == 0 &&
        ((reinterpret_cast<uintptr_t>(clp) | reinterpret_cast<uintptr_t>(crl)) & 15u) == 0) {
        const float4* c4 = reinterpret_cast<const float4*>(clp);
        const float4* r4 = reinterpret_cast<const float4*>(crl);
        float4* cs4 = reinterpret_cast<float4*>(clp_s);
        float4* rs4 = reinterpret_cast<float4*>(rl_s);
#pragma unroll 4
        for (int i = lane; i < G * M / 4; i += 32) {
            cs4[i] = c4[i];
            rs4[i] = r4[i];
        }
    } else {
#pragma unroll 4
        for (int i = lane; i < G * M; i += 32) {
            clp_s[i] = clp[i];
            rl_s[i] = crl[i];
        }
    }
    for (int i = lane; i < G; i += 32) nc_s[i] = nc[i];
    __syncwarp();

    // the lattice: cut at the first position whose best candidate is EOS
    int Lc = G;
    bool eos_cut = false;
    if (a.eos_id >= 0) {
        for (int j0 = 0; j0 < G; j0 += 32) {        // lanes test 32 positions at a time
            const int j = j0 + lane;
            const bool hit = j < G && nc_s[j] > 0 && cids[j * M] == a.eos_id;
            const unsigned mask = __ballot_sync(0xffffffffu, hit);
            if (mask) {
                Lc = j0 + __ffs(mask);
                eos_cut = true;
                break;
            }
        }
    }
    bool empty = false;
    for (int j = lane; j < Lc; j += 32) empty |= nc_s[j] == 0;
    empty = __any_sync(0xffffffffu, empty);

    // Beams, lane w holding beam w: order key (sum of raw logits, fp64:
    // exact for bf16 logits, and the same operations as any left-to-right
    // fp64 sum), score (sum of log-probabilities) and place among the beams
    // in lexicographic order of their candidate ranks (the tie rule).
    double bkey = 0.0;
    float bscore = 0.0f;
    int blex = 0;
    int ncur = 1;
    // The per-lane constants of the next position are independent of the
    // beams, so they are read one position ahead of their use.
    BeamPos nxt = {};
    if (Lc > 0 && !empty) nxt = beam_position(nc_s, rl_s, clp_s, 0, Lc, eos_cut, W, M, lane);
    for (int j = 0; j < Lc && !empty; ++j) {
        const BeamPos cur = nxt;
        if (j + 1 < Lc) nxt = beam_position(nc_s, rl_s, clp_s, j + 1, Lc, eos_cut, W, M, lane);
        const int n = cur.n, nw = cur.nw;
        const unsigned magic = cur.magic;
        const int E = ncur * nw;
        const int keep = E < W ? E : W;
        if (E <= 32) {
            // one expansion per lane: e = lane takes candidate cur.r of beam cur.par
            const bool valid = lane < E;
            const double key = __shfl_sync(0xffffffffu, bkey, cur.par) + static_cast<double>(cur.rl);
            const float sc = __shfl_sync(0xffffffffu, bscore, cur.par) + cur.lp;
            // place in lexicographic order of (parent's place, candidate rank): below E
            const int lx = __shfl_sync(0xffffffffu, blex, cur.par) * nw + cur.r;
            const long long ord = ordered_i64(key);
            int src = 0;                       // lane t < keep: the expansion that becomes beam t
            if (keep <= 8) {
                // The kept expansions one at a time, best first: the largest
                // key (its high word, then its low word), ties to the smaller
                // lexicographic place.  Three warp reductions a round.
                const unsigned long long u = static_cast<unsigned long long>(ord) ^ 0x8000000000000000ull;
                const unsigned hi = static_cast<unsigned>(u >> 32), lo = static_cast<unsigned>(u);
                const unsigned tag = (static_cast<unsigned>(lx) << 5) | static_cast<unsigned>(lane);
                bool left = valid;
                for (int t = 0; t < keep; ++t) {
                    const unsigned m1 = __reduce_max_sync(0xffffffffu, left ? hi : 0u);
                    const bool c1 = left && hi == m1;
                    const unsigned m2 = __reduce_max_sync(0xffffffffu, c1 ? lo : 0u);
                    const bool c2 = c1 && lo == m2;
                    const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, c2 ? tag : 0xffffffffu) & 31u);
                    left = left && lane != win;
                    src = lane == t ? win : src;
                }
            } else {
                // every expansion's rank (how many come before it), four
                // sources a round so that their shuffles go out together
                const long long o = valid ? ord : LLONG_MIN;
                int rank = 0;
                for (int s0 = 0; s0 < E; s0 += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s = s0 + u < E ? s0 + u : lane;        // lane itself adds 0
                        const long long o2 = __shfl_sync(0xffffffffu, o, s);
                        const int l2 = __shfl_sync(0xffffffffu, lx, s);
                        rank += (o2 > o) || (o2 == o && l2 < lx);
                    }
                }
                if (valid && rank < keep) s_src[rank] = lane;
                __syncwarp();
                if (lane < keep) src = s_src[lane];
                __syncwarp();
            }
            // beam t takes over its expansion's state; its new place among
            // the kept beams counts the kept places below its own
            const double nkey = __shfl_sync(0xffffffffu, key, src);
            const float nsc = __shfl_sync(0xffffffffu, sc, src);
            const int nlx = __shfl_sync(0xffffffffu, lx, src);
            const unsigned kept = __reduce_or_sync(0xffffffffu, lane < keep ? 1u << nlx : 0u);
            if (lane < keep) {
                const int sp = static_cast<int>((static_cast<unsigned>(src) * magic) >> 16);
                bp_parent[j * W + lane] = static_cast<unsigned char>(sp);
                bp_rank[j * W + lane] = static_cast<unsigned char>(src - sp * nw);
                bkey = nkey;
                bscore = nsc;
                blex = __popc(kept & ((1u << nlx) - 1u));
            }
        } else {
            // more expansions than lanes: through shared memory
            if (lane < ncur) {
                b_key[lane] = bkey;
                b_score[lane] = bscore;
                b_lex[lane] = blex;
            }
            __syncwarp();
            for (int e = lane; e < E; e += 32) {
                const int par = static_cast<int>((e * magic) >> 16), r = e - par * nw;
                const double key = b_key[par] + static_cast<double>(rl_s[j * M + r]);
                x_key[e] = key;
                x_ord[e] = ordered_i64(key);
                x_score[e] = b_score[par] + clp_s[j * M + r];
                x_lx[e] = b_lex[par] * n + r;
            }
            __syncwarp();
            // each expansion's rank: how many expansions come before it (key
            // desc, then lexicographic place asc); the first W are kept
            for (int e = lane; e < E; e += 32) {
                const long long k = x_ord[e];
                const int l = x_lx[e];
                int rank = 0, e2 = 0;
                for (; e2 + 4 <= E; e2 += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const long long k2 = x_ord[e2 + u];
                        rank += (k2 > k) || (k2 == k && x_lx[e2 + u] < l);
                    }
                }
                for (; e2 < E; ++e2) {
                    const long long k2 = x_ord[e2];
                    rank += (k2 > k) || (k2 == k && x_lx[e2] < l);
                }
                if (rank < keep) {
                    const int par = static_cast<int>((e * magic) >> 16);
                    n_key[rank] = x_key[e];
                    n_score[rank] = x_score[e];
                    n_lx[rank] = l;
                    bp_parent[j * W + rank] = static_cast<unsigned char>(par);
                    bp_rank[j * W + rank] = static_cast<unsigned char>(e - par * nw);
                }
            }
            __syncwarp();
            if (lane < keep) {
                const int l = n_lx[lane];
                int pos = 0;
                for (int t = 0; t < keep; ++t) pos += n_lx[t] < l;
                bkey = n_key[lane];
                bscore = n_score[lane];
                blex = pos;
            }
            __syncwarp();
        }
        ncur = keep;
    }
    __syncwarp();
    const int np = empty ? 0 : ncur;
    // back-track the final beams' candidate ranks in shared memory, then
    // gather their ids with independent loads
    if (lane < np) {
        int cur = lane;
        for (int j = Lc - 1; j >= 0; --j) {
            path_rank[lane * G + j] = bp_rank[j * W + cur];
            cur = bp_parent[j * W + cur];
        }
    }
    if (lane < W)
        a.path_logp[static_cast<int64_t>(b) * W + lane] = lane < np ? bscore : -INFINITY;
    __syncwarp();
    int32_t* paths = a.paths + static_cast<int64_t>(b) * W * G;
#pragma unroll 4
    for (int i = lane; i < W * G; i += 32) {
        const int w = i / G, j = i - w * G;
        paths[i] = w < np && j < Lc ? cids[j * M + path_rank[i]] : -1;
    }
    if (lane == 0) {
        a.npaths[b] = np;
        if (a.lat_len) a.lat_len[b] = Lc;
    }
    // the lattice as used: one candidate at an EOS end, none past it
    __syncwarp();
    if (eos_cut) {
        for (int i = lane; i < (G - (Lc - 1)) * M; i += 32) {
            const int j = Lc - 1 + i / M, r = i % M;
            if (j >= Lc || r >= 1) {
                cids[j * M + r] = -1;
                clp[j * M + r] = -INFINITY;
                crl[j * M + r] = -INFINITY;
            }
        }
        for (int j = Lc - 1 + lane; j < G; j += 32) nc[j] = j >= Lc ? 0 : 1;
    }
}

}  // namespace

template <bool BF16>
cudaError_t launch_prune_typed(const CpsArgs& a, cudaStream_t s) {
    // One CTA per row, with more warps per row the fewer the rows (measured
    // on 152064-logit rows: 4 warps from 512 rows up, 8 at 256, 16 at 128
    // and below).  At 4 warps, 7 CTAs fit an SM: 1064 rows in one wave.
    const int64_t rows = static_cast<int64_t>(a.B) * a.G;
    const unsigned grid = static_cast<unsigned>(rows);
    if (rows >= 384)
        cps_prune_kernel<BF16, 4><<<grid, 128, 0, s>>>(a);
    else if (rows >= 128)
        cps_prune_kernel<BF16, 8><<<grid, 256, 0, s>>>(a);
    else
        cps_prune_kernel<BF16, 16><<<grid, 512, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_cps_prune(const CpsArgs& a, bool bf16, cudaStream_t s) {
    return bf16 ? launch_prune_typed<true>(a, s) : launch_prune_typed<false>(a, s);
}

cudaError_t launch_cps_beam(const CpsArgs& a, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(a.G) * a.mmax * 8 + static_cast<size_t>(a.G) * 4 +
                        static_cast<size_t>(3) * a.G * a.beam;
    if (smem > 48 * 1024) {
        const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(cps_beam_kernel), smem);
        if (e != cudaSuccess) return e;
    }
    // An ordinary stream-ordered launch: as a programmatic dependent of the
    // pruning pass the chained pair measured 0.101 ms against 0.083 ms.
    cps_beam_kernel<<<a.B, 32, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sdv
