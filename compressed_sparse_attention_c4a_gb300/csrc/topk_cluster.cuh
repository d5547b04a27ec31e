// The top-k of one row of up to C * THREADS * VPT scores on a cluster of C CTAs, with a lowest-index
// tie-break, as a device function: the decode top-k kernel (topk.cu) runs it once per cluster, and the fused
// top-k + attention kernel (attention.cu) runs it before gathering the selected rows.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2: S_t = TopK(I_{t,:}, k).
//
// CTA rank c holds the part [c THREADS VPT, (c + 1) THREADS VPT) of the row in registers, thread t of it
// the VPT consecutive scores from c THREADS VPT + t VPT.  Decisions (value buckets of the row's range, the
// bucket b* of the k-th largest, direct ranking of a small b* or a radix select of a crowded one, ordered
// compaction with entries equal to the threshold taken lowest index first) are those of the one-CTA
// kernel, with the row's max / min, the bucket histograms, the candidate lists of a small bucket and the
// CTAs' counts exchanged over distributed shared memory; the ordered output is one block scan per CTA plus
// the counts of the CTAs before it (lower CTAs hold lower indices).
#pragma once
#include <cooperative_groups.h>

#include "common.cuh"

namespace dsa {

namespace cg = cooperative_groups;

constexpr int kBins = 2048;
constexpr int kRankMax = 256;  // bucket sizes (cluster-wide) resolved by direct ranking

// Monotone 32-bit key of a score; -0 and +0 compare equal as floats, so they share one key.
__device__ __forceinline__ uint32_t order_key(float f) { return dsa_score_key(f); }

// Block-wide scan and bin selection for a block of THREADS threads (kBins / THREADS bins each).
template <int THREADS>
struct RegScan {
    static constexpr int kWarps = THREADS / 32;
    // Exclusive block scan of two counters; also the totals.  Ends with a barrier.
    static __device__ __forceinline__ void scan2(uint32_t a, uint32_t b, uint32_t* ex_a, uint32_t* ex_b,
                                                 uint32_t* tot_a, uint32_t* tot_b, uint32_t (*wt)[2]) {
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        uint32_t ia = a, ib = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t ta = __shfl_up_sync(0xffffffffu, ia, o), tb = __shfl_up_sync(0xffffffffu, ib, o);
            if (lane >= o) {
                ia += ta;
                ib += tb;
            }
        }
        if (lane == 31) {
            wt[wid][0] = ia;
            wt[wid][1] = ib;
        }
        __syncthreads();
        if (wid == 0) {
            uint32_t wa = lane < kWarps ? wt[lane][0] : 0u, wb = lane < kWarps ? wt[lane][1] : 0u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t ta = __shfl_up_sync(0xffffffffu, wa, o), tb = __shfl_up_sync(0xffffffffu, wb, o);
                if (lane >= o) {
                    wa += ta;
                    wb += tb;
                }
            }
            if (lane < kWarps) {
                wt[lane][0] = wa;
                wt[lane][1] = wb;
            }
        }
        __syncthreads();
        *ex_a = (wid ? wt[wid - 1][0] : 0u) + ia - a;
        *ex_b = (wid ? wt[wid - 1][1] : 0u) + ib - b;
        *tot_a = wt[kWarps - 1][0];
        *tot_b = wt[kWarps - 1][1];
        __syncthreads();
    }
    // The bin (from the top) holding the need-th largest counted element; need drops by the count above.
    static __device__ __forceinline__ uint32_t select(const uint32_t* hist, uint32_t& need, uint32_t (*wt)[2],
                                                      uint32_t* sel) {
        constexpr int BPT = kBins / THREADS;  // bins per thread, in descending order
        const int tid = threadIdx.x;
        uint32_t c[BPT], sum = 0;
#pragma unroll
        for (int e = 0; e < BPT; ++e) {
            c[e] = hist[kBins - 1 - BPT * tid - e];
            sum += c[e];
        }
        uint32_t ex, ex2, tot, tot2;
        scan2(sum, 0u, &ex, &ex2, &tot, &tot2, wt);
#pragma unroll
        for (int e = 0; e < BPT; ++e) {
            if (ex < need && need <= ex + c[e]) {
                sel[0] = (uint32_t)(kBins - 1 - BPT * tid - e);
                sel[1] = ex;
            }
            ex += c[e];
        }
        __syncthreads();
        const uint32_t b = sel[0];
        need -= sel[1];
        __syncthreads();
        return b;
    }
};

// The cluster-wide histogram for a cluster of C CTAs of THREADS threads: every remote bin of a thread is
// requested before any is added (the distributed shared memory loads overlap).  Starts with a cluster barrier
// and ends with a block barrier.
template <int C, int THREADS>
__device__ __forceinline__ const uint32_t* cluster_hist_sum_batched(cg::cluster_group& cluster, uint32_t* hist,
                                                                    uint32_t* hsum) {
    constexpr int BPT = kBins / THREADS;
    cluster.sync();  // every CTA's local histogram is complete
    uint32_t v[C][BPT];
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const uint32_t* rh = cluster.map_shared_rank(hist, c);
#pragma unroll
        for (int e = 0; e < BPT; ++e) v[c][e] = rh[threadIdx.x + e * THREADS];
    }
#pragma unroll
    for (int e = 0; e < BPT; ++e) {
        uint32_t t = 0;
#pragma unroll
        for (int c = 0; c < C; ++c) t += v[c][e];
        hsum[threadIdx.x + e * THREADS] = t;
    }
    __syncthreads();
    return hsum;
}

// Shared memory of topk_row_cluster (any shared-memory region of the CTA that nothing else uses meanwhile).
template <int THREADS, int VPT, int C>
struct TopkRowScratch {
    uint32_t hist[kBins], hsum[kBins];
    uint32_t cand_key[kRankMax], cand_idx[kRankMax];
    uint32_t all_key[kRankMax], all_idx[kRankMax];  // the whole cluster's members of a small bucket
    uint32_t marks[THREADS * VPT / 32];              // ranked winners of a small bucket, by index in this part
    uint32_t wt[32][2];
    uint32_t sel[2];
    uint32_t n_cand;
    uint32_t n_above;       // this CTA's entries above the bucket b* (small-bucket path)
    uint32_t pub[C][2];     // each CTA's (entries above b*, members of b*), written into every CTA of the cluster
    uint32_t sel_cnt[C];    // each CTA's members of b* among the `need` best (small-bucket path)
    float red[2][32];
    float cl_mm[C][2];      // each CTA's (max, min), written into every CTA of the cluster
    uint32_t cl_tot[C][2];  // each CTA's (definite members, entries equal to T)
};

// Row s (n >= 0 valid scores, the same in every CTA: every branch below is cluster-uniform) -> emit(pos,
// index) for each position [0, k) of the ordered output, -1 past the selected entries; each position is
// emitted by exactly one thread of the cluster.  Every thread of every CTA of the cluster calls it.  (Timeline
// builds stamp its phases into slots stamp0 .. stamp0 + 3.)
template <int THREADS, int VPT, int C, class Emit>
__device__ __forceinline__ void topk_row_cluster(cg::cluster_group& cluster, TopkRowScratch<THREADS, VPT, C>& sm,
                                                 const float* __restrict__ s, int n, int k, Emit emit,
                                                 int32_t* status, int stamp0 = 2) {
    static_assert(VPT % 4 == 0 && VPT <= 32, "a thread's run is a multiple of 4 and fits one 32-bit mask");
    using SC = RegScan<THREADS>;
    const int crank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (n <= k) {
        for (int i = crank * THREADS + tid; i < k; i += C * THREADS) emit(i, i < n ? i : -1);
        return;
    }
    // 1. this thread's run of scores; the row's max / min of the finite ones over the cluster
    const int part0 = crank * THREADS * VPT;
        const int i0 = part0 + tid * VPT;
    const int nv = max(0, min(VPT, n - i0));  // valid scores in the run
    float v[VPT];
#pragma unroll
    for (int u = 0; u < VPT; u += 4) {
        if (u + 4 <= nv) {
            const float4 q = *reinterpret_cast<const float4*>(s + i0 + u);
            v[u] = q.x, v[u + 1] = q.y, v[u + 2] = q.z, v[u + 3] = q.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[u + e] = u + e < nv ? s[i0 + u + e] : -INFINITY;
        }
    }
    for (int b = tid; b < kBins; b += THREADS) sm.hist[b] = 0;
    for (int w = tid; w < THREADS * VPT / 32; w += THREADS) sm.marks[w] = 0;
    if (tid == 0) sm.n_cand = 0, sm.n_above = 0;
    if (tid == 0) DSA_STAMP(stamp0);
    float mx = -INFINITY, mn = INFINITY;
#pragma unroll
    for (int u = 0; u < VPT; ++u)
        if (v[u] != -INFINITY) {
            mx = fmaxf(mx, v[u]);
            mn = fminf(mn, v[u]);
        }
    mx = warp_max(mx);
    mn = -warp_max(-mn);
    if (lane == 0) {
        sm.red[0][wid] = mx;
        sm.red[1][wid] = mn;
    }
    __syncthreads();
    if (tid < C) {  // this CTA's (max, min) into slot crank of CTA tid
        float bx = -INFINITY, bn = INFINITY;
        for (int w = 0; w < SC::kWarps; ++w) {
            bx = fmaxf(bx, sm.red[0][w]);
            bn = fminf(bn, sm.red[1][w]);
        }
        float* dst = cluster.map_shared_rank(&sm.cl_mm[0][0], tid);
        dst[2 * crank] = bx;
        dst[2 * crank + 1] = bn;
    }
    cluster.sync();
    mx = -INFINITY;
    mn = INFINITY;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        mx = fmaxf(mx, sm.cl_mm[c][0]);
        mn = fminf(mn, sm.cl_mm[c][1]);
    }
    float scale = (mx != -INFINITY && mx > mn) ? 2046.f / (mx - mn) : 0.f;
    if (!isfinite(scale)) scale = 0.f;  // degenerate range: one bucket, resolved by the radix passes
    // 2. value buckets (as in the one-CTA kernel) and the cluster's histogram
    uint32_t bins[VPT / 2];
#pragma unroll
    for (int u = 0; u < VPT; u += 2) {
        uint32_t b2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float t = fminf(2046.f, (mx - v[u + e]) * scale);
            b2[e] = v[u + e] == -INFINITY ? 0u : 2047u - (__float_as_uint(t + 8388608.f) - 0x4B000000u);
        }
        bins[u / 2] = b2[0] | (b2[1] << 16);
    }
    auto bin_at = [&](int u) -> uint32_t { return (bins[u / 2] >> (16 * (u & 1))) & 0xFFFFu; };
#pragma unroll
    for (int u = 0; u < VPT; ++u)
        if (u < nv && DSA_IDX_OK(bin_at(u), kBins, status)) atomicAdd(&sm.hist[bin_at(u)], 1u);
    const uint32_t* hs = cluster_hist_sum_batched<C, THREADS>(cluster, sm.hist, sm.hsum);
    if (tid == 0) DSA_STAMP(stamp0 + 1);
    uint32_t need = (uint32_t)k;
    const uint32_t bstar = SC::select(hs, need, sm.wt, sm.sel);
    const uint32_t in_bucket = hs[bstar];
    if (tid == 0) DSA_STAMP(stamp0 + 2);
    const bool take_all = in_bucket == need;
    const bool rank_mode = !take_all && in_bucket <= (uint32_t)kRankMax;
#ifdef DSA_TIMELINE
    if (tid == 0 && g_timeline)  // (timeline builds) the bucket's size and which path resolves it
        g_timeline[(unsigned long long)blockIdx.x * 32 + 27] = in_bucket | (take_all ? 1ull << 40 : 0) | (rank_mode ? 1ull << 41 : 0);
#endif
    uint32_t above = 0u, inb = 0u;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const uint32_t b = bin_at(u);
        if (u < nv && b > bstar) above |= 1u << u;
        if (u < nv && b == bstar) inb |= 1u << u;
    }
    // 3a. small bucket: every CTA lists its members; each member counts the better ones (larger score, or
    // equal score and lower index) over all the cluster's lists
    if (rank_mode) {
        const uint32_t cnt = (uint32_t)__popc(inb);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(&sm.n_cand, incl);
        wbase = __shfl_sync(0xffffffffu, wbase, 31);
        uint32_t slot = wbase + incl - cnt;
#pragma unroll
        for (int u = 0; u < VPT; ++u)
            if ((inb >> u) & 1u) {
                if (DSA_IDX_OK(slot, kRankMax, status)) {
                    sm.cand_key[slot] = order_key(v[u]);
                    sm.cand_idx[slot] = (uint32_t)(i0 + u);
                }
                ++slot;
            }
        // this CTA's entries above b* (its definite members), counted now so that the output's offsets need no
        // further exchange: they travel with the list lengths, pushed into every CTA before one cluster barrier
        const uint32_t na_w = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(above));
        if (lane == 0 && na_w) atomicAdd(&sm.n_above, na_w);
        if (tid < C) sm.sel_cnt[tid] = 0;
        __syncthreads();
        if (tid < C) {  // (entries above b*, members of b*) into slot crank of CTA tid
            uint32_t* dst = cluster.map_shared_rank(&sm.pub[0][0], tid);
            dst[2 * crank] = sm.n_above;
            dst[2 * crank + 1] = sm.n_cand;
        }
        cluster.sync();  // every CTA's list and counts are complete
        // the cluster's lists, copied into this CTA's shared memory (at most kRankMax entries in all): a thread's
        // entries of every list are requested before any is stored, so the copy costs one remote round trip
        uint32_t nq[C], base[C], total_c = 0, longest = 0;
#pragma unroll
        for (int q = 0; q < C; ++q) {
            nq[q] = sm.pub[q][1];
            base[q] = total_c;
            total_c += nq[q];
            longest = max(longest, nq[q]);
        }
        for (uint32_t j = tid; j < longest; j += THREADS) {
            uint32_t kq[C], iq[C];
#pragma unroll
            for (int q = 0; q < C; ++q)
                if (j < nq[q]) {
                    kq[q] = cluster.map_shared_rank(sm.cand_key, q)[j];
                    iq[q] = cluster.map_shared_rank(sm.cand_idx, q)[j];
                }
#pragma unroll
            for (int q = 0; q < C; ++q)
                if (j < nq[q] && DSA_IDX_OK(base[q] + j, kRankMax, status)) {
                    sm.all_key[base[q] + j] = kq[q];
                    sm.all_idx[base[q] + j] = iq[q];
                }
        }
        __syncthreads();
        cluster_arrive();  // done reading the other CTAs' lists (waited for before returning)
        // every member of the cluster's lists ranked (larger score, or equal score and lower index, is better):
        // this CTA's winners marked, every CTA's winners counted (the same counts in every CTA)
        const int na = (int)min(total_c, (uint32_t)kRankMax);
        for (int c = tid; c < na; c += THREADS) {
            const uint32_t my_k = sm.all_key[c], my_i = sm.all_idx[c];
            uint32_t better = 0;
            for (int j = 0; j < na; ++j) {
                const uint32_t kj = sm.all_key[j];
                better += (kj > my_k) || (kj == my_k && sm.all_idx[j] < my_i);
            }
            if (better < need) {
                const int src = (int)(my_i / (uint32_t)(THREADS * VPT));  // the CTA whose part holds it
                if (DSA_IDX_OK(src, C, status)) atomicAdd(&sm.sel_cnt[src], 1u);
                const uint32_t li = my_i - (uint32_t)part0;
                if (src == crank && DSA_IDX_OK(li >> 5, THREADS * VPT / 32, status))
                    atomicOr(&sm.marks[li >> 5], 1u << (li & 31));
            }
        }
        __syncthreads();
    }
    // 3b. crowded bucket: radix select on the 32-bit order keys inside b*, with cluster-wide histograms
    uint32_t T = 0u, need_T = 0u;
    if (!take_all && !rank_mode) {
        need_T = need;
        uint32_t prefix = 0u, mask = 0u;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const uint32_t dm = pass == 2 ? 0x3FFu : 0x7FFu;
            cluster.sync();  // the cluster is done reading this CTA's previous histogram
            for (int b = tid; b < kBins; b += THREADS) sm.hist[b] = 0;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const uint32_t key = order_key(v[u]);
                if (((inb >> u) & 1u) && (key & mask) == prefix) atomicAdd(&sm.hist[(key >> sh) & dm], 1u);
            }
            const uint32_t* hp = cluster_hist_sum_batched<C, THREADS>(cluster, sm.hist, sm.hsum);
            const uint32_t dg = SC::select(hp, need_T, sm.wt, sm.sel);
            prefix |= dg << sh;
            mask |= dm << sh;
        }
        T = prefix;
    }
    // 4. ordered compaction: definite members and (lowest index first) entries equal to T, after those of
    // the CTAs before this one
    if (tid == 0) DSA_STAMP(stamp0 + 3);
    uint32_t dmask = above, tmask = 0u;
    if (take_all) dmask |= inb;
    else if (rank_mode) {
        for (uint32_t m = inb; m; m &= m - 1) {
            const int u = __ffs(m) - 1;
            const int li = i0 + u - part0;
            if ((sm.marks[li >> 5] >> (li & 31)) & 1u) dmask |= 1u << u;
        }
    } else {
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const uint32_t key = order_key(v[u]);
            if (((inb >> u) & 1u) && key > T) dmask |= 1u << u;
            if (((inb >> u) & 1u) && key == T) tmask |= 1u << u;
        }
    }
    uint32_t ex_d, ex_t, tot_d, tot_t;
    SC::scan2((uint32_t)__popc(dmask), (uint32_t)__popc(tmask), &ex_d, &ex_t, &tot_d, &tot_t, sm.wt);
    uint32_t off_d = 0, off_t = 0, all_d = 0, all_t = 0;
    if (rank_mode) {  // every CTA's selected count is already known here: above b* plus its winners in b*
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const uint32_t sel = sm.pub[c][0] + sm.sel_cnt[c];
            if (c < crank) off_d += sel;
            all_d += sel;
        }
    } else {
        if (tid < C) {  // this CTA's counts into slot crank of CTA tid
            uint32_t* dst = cluster.map_shared_rank(&sm.cl_tot[0][0], tid);
            dst[2 * crank] = tot_d;
            dst[2 * crank + 1] = tot_t;
        }
        cluster.sync();  // also: no CTA reads another's shared memory after this point
#pragma unroll
        for (int c = 0; c < C; ++c) {
            if (c < crank) {
                off_d += sm.cl_tot[c][0];
                off_t += sm.cl_tot[c][1];
            }
            all_d += sm.cl_tot[c][0];
            all_t += sm.cl_tot[c][1];
        }
    }
    uint32_t tie_rank = off_t + ex_t;
    uint32_t pos = off_d + ex_d + min(tie_rank, need_T);
    for (uint32_t m = dmask | tmask; m; m &= m - 1) {
        const int u = __ffs(m) - 1;
        if ((dmask >> u) & 1u) {
            if (pos < (uint32_t)k) emit((int)pos, i0 + u);
            ++pos;
        } else {
            if (tie_rank < need_T) {
                if (pos < (uint32_t)k) emit((int)pos, i0 + u);
                ++pos;
            }
            ++tie_rank;
        }
    }
    const uint32_t total = all_d + min(all_t, need_T);
    for (int i = (int)total + crank * THREADS + tid; i < k; i += C * THREADS) emit(i, -1);
    if (crank == 0 && tid == 0 && total != (uint32_t)k) report(status, DSA_ERR_DEVICE_FAULT);
    if (rank_mode) cluster_wait();  // no other CTA reads this CTA's lists after this point
}

}  // namespace dsa
