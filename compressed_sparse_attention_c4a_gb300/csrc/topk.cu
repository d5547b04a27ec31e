// dsa_topk: per-query top-k of the indexer scores with a lowest-index tie-break.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2: S_t = TopK(I_{t,:}, k); the
// main attention reads only S_t.  [P2] "DeepSeek V4 稀疏注意力完全解剖" 机制三: k = 512 for c4a.
//
// Rows of up to 16,384 scores: one CTA per row with the row in registers (topk_reg_kernel).  Longer
// rows: one thread-block cluster of C CTAs (512 threads, two CTAs per SM) per row, C = 1 up to 40,960
// scores, else 2 or 4; CTA q handles the q-th of C parts.  Only a 16-bit value bucket per score is kept in
// shared memory, so two rows share an SM and one row's loads overlap the other's arithmetic; exact scores
// are read again (from L2) only where a bucket has to be split.  Partial results are combined through
// distributed shared memory, so every CTA takes the same decisions:
//   1. max M and min m of the finite scores (first read of the part);
//   2. bucket select: bin(v) = 2047 - round(min(2046, (M - v) * 2046 / (M - m))) -- monotone (larger
//      score -> same or larger bin; equal scores share a bin) and even, so the shared-memory histogram
//      has little atomic contention; bins are stored while the histogram is built (second read); the
//      summed histogram gives the bin b* holding the k-th largest score and `need`, the count still
//      missing;
//   3. unless b* holds exactly `need` scores: when it holds at most 256, its members are listed and each
//      counts the better ones (larger score, or equal score and lower index) across the cluster -- the
//      `need` best are marked; otherwise (heavy ties) a radix select over the 32-bit order keys of b*'s
//      scores (digits of 11, 11, 10 bits, histograms summed across the cluster) gives the exact
//      threshold key T and how many entries equal to T are still needed;
//   4. ordered compaction: thread t of CTA q owns a contiguous run of indices; a block scan plus the
//      totals of the lower CTAs give every selected index its slot in increasing index order, and
//      rank entries equal to T by index (the lowest indices win).
#include <cooperative_groups.h>

#include "common.cuh"
#include "topk_cluster.cuh"

namespace cg = cooperative_groups;

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkClusterMax = 4;
constexpr int kPartMax = 40960;  // scores per CTA (rows up to 163,840 with C = 4)
constexpr int kMarkWords = (kPartMax / 32 + 1 + 3) & ~3;  // winner bitmap, padded to 16 bytes

// The cluster-wide histogram: hist itself when the cluster is one CTA, else hsum[b] = the sum of the
// CTAs' hist[b].  Starts and ends with a barrier.
__device__ __forceinline__ const uint32_t* cluster_hist_sum(cg::cluster_group& cluster, int csz, uint32_t* hist,
                                                            uint32_t* hsum) {
    if (csz == 1) {
        __syncthreads();
        return hist;
    }
    cluster.sync();  // every CTA's local histogram is complete
    uint32_t* remote[kTopkClusterMax];
#pragma unroll
    for (int c = 0; c < kTopkClusterMax; ++c) remote[c] = cluster.map_shared_rank(hist, c < csz ? c : 0);
    for (int b = threadIdx.x; b < kBins; b += kTopkThreads) {
        uint32_t v = 0;
#pragma unroll
        for (int c = 0; c < kTopkClusterMax; ++c)
            if (c < csz) v += remote[c][b];
        hsum[b] = v;
    }
    __syncthreads();
    return hsum;
}

// Scores [i, i + 4) of a part as a float4; entries at or past `mq` read as -inf (no access).
__device__ __forceinline__ float4 load_part4(const float* p, int i, int mq) {
    if (i + 4 <= mq) return *reinterpret_cast<const float4*>(p + i);
    float4 q;
    q.x = i < mq ? p[i] : -INFINITY;
    q.y = i + 1 < mq ? p[i + 1] : -INFINITY;
    q.z = i + 2 < mq ? p[i + 2] : -INFINITY;
    q.w = -INFINITY;  // i + 3 >= mq here
    return q;
}

__global__ void __launch_bounds__(kTopkThreads, 2)
    topk_kernel(const float* __restrict__ scores, int ld, const int32_t* __restrict__ n_valid, int k,
                int32_t* __restrict__ idx_out, int32_t* status, int nq, int ahead) {
    using SC = RegScan<kTopkThreads>;
    pdl_wait();
    pdl_launch_dependents();
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) uint32_t smem_topk[];
    uint32_t* hist = smem_topk;                                      // [kBins] this CTA's histogram
    uint32_t* hsum = hist + kBins;                                   // [kBins] cluster-wide histogram (C > 1)
    uint32_t* cand_key = hsum + kBins;                               // [kRankMax] this CTA's members of b*
    uint32_t* cand_idx = cand_key + kRankMax;                        // [kRankMax] their row indices
    uint32_t* marks = cand_idx + kRankMax;                           // [kMarkWords] ranked winners (local index)
    uint16_t* bins = reinterpret_cast<uint16_t*>(marks + kMarkWords);  // [part] bucket of each score
    __shared__ uint32_t n_cand;
    __shared__ uint32_t wt[32][2];
    __shared__ uint32_t sel[2];
    __shared__ float red[2][kTopkThreads / 32];
    __shared__ float red_c[2];
    __shared__ uint32_t totals[2];
    __shared__ uint32_t wcnt[kTopkWarps][2];

    const int csz = (int)cluster.num_blocks();
    // barrier over the cluster, or over the block when the cluster is one CTA
    auto csync = [&]() {
        if (csz > 1) cluster.sync();
        else __syncthreads();
    };
    const int row = blockIdx.x / csz;
    const int qr = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int32_t* out = idx_out + (long long)row * k;
    const int n = n_valid[row];  // the same for the whole cluster: every branch below is cluster-uniform
    if (n < 0 || n > ld) {
        if (qr == 0) {
            if (tid == 0) report(status, DSA_ERR_DEVICE_FAULT);
            for (int i = tid; i < k; i += kTopkThreads) out[i] = -1;
        }
        return;
    }
    if (n <= k) {
        if (qr == 0)
            for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    const int chunk = ((n + csz - 1) / csz + 3) & ~3;  // multiple of 4: aligned float4 loads
    const int base = qr * chunk;
    const int mq = max(0, min(n, base + chunk) - base);  // scores in this CTA's part
    const float* s = scores + (long long)row * ld + base;
    // the row `ahead` rows on (likely the next one this SM slot takes) into L2, in 16 KB pieces
    if (wid == 0 && row + ahead < nq) {
        const int pc = ((ld + csz - 1) / csz + 3) & ~3;  // its part, bounded by the row's width
        const int pb = min(ld, qr * pc), pe = min(ld, pb + pc);
        const char* src = reinterpret_cast<const char*>(scores + (long long)(row + ahead) * ld + pb);
        const int bytes = (pe - pb) * 4;
        for (int off = lane * 16384; off < bytes; off += 32 * 16384)
            prefetch_l2(src + off, (uint32_t)min(16384, bytes - off));
    }

    // 1. max / min of the finite scores of the part (eight float4 loads in flight per thread), then the
    // block's and the cluster's
    float mx = -INFINITY, mn = INFINITY;
    for (int i0 = tid * 4; i0 < mq; i0 += kTopkThreads * 32) {
        float4 q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) q[u] = load_part4(s, i0 + u * kTopkThreads * 4, mq);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float v[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                mx = fmaxf(mx, v[e]);  // -inf never raises the maximum
                mn = fminf(mn, v[e] == -INFINITY ? INFINITY : v[e]);
            }
        }
    }
    for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
    for (int w = tid; w <= (mq >> 5); w += kTopkThreads) marks[w] = 0;
    if (tid == 0) n_cand = 0;
    mx = warp_max(mx);
    mn = -warp_max(-mn);
    if (lane == 0) {
        red[0][wid] = mx;
        red[1][wid] = mn;
    }
    __syncthreads();
    mx = -INFINITY;
    mn = INFINITY;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        mx = fmaxf(mx, red[0][w]);
        mn = fminf(mn, red[1][w]);
    }
    if (csz > 1) {
        if (tid == 0) {
            red_c[0] = mx;
            red_c[1] = mn;
        }
        cluster.sync();
        mx = -INFINITY;
        mn = INFINITY;
        for (int c = 0; c < csz; ++c) {
            const float* rr = cluster.map_shared_rank(red_c, c);
            mx = fmaxf(mx, rr[0]);
            mn = fminf(mn, rr[1]);
        }
    }
    const bool any_finite = mx != -INFINITY;
    float scale = (any_finite && mx > mn) ? 2046.f / (mx - mn) : 0.f;
    if (!isfinite(scale)) scale = 0.f;  // degenerate range: one bucket, resolved by the radix passes
    // bin(v) = 2047 - round(min(2046, (mx - v) * scale)), rounded by adding 2^23 (full-rate arithmetic):
    // monotone (a larger score never lands in a lower bin, equal scores share one); -inf (and NaN
    // products) land in bin 1, the lowest bin of finite scores, where the exact keys order them last.
    // Bin 0 marks the padding past the part.
    auto bin_of = [&](float v) -> uint32_t {
        const float t = fminf(2046.f, (mx - v) * scale);
        return (2047u + 0x4B000000u) - __float_as_uint(t + 8388608.f);
    };

    // 2. second read of the part (from L2): 16-bit bins into shared memory, local histogram, the
    // cluster-wide sum and the bucket of the k-th largest score
    for (int i0 = tid * 4; i0 < mq; i0 += kTopkThreads * 32) {
        float4 q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) q[u] = load_part4(s, i0 + u * kTopkThreads * 4, mq);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * kTopkThreads * 4;
            if (i >= mq) break;
            uint32_t b0 = bin_of(q[u].x), b1 = bin_of(q[u].y), b2 = bin_of(q[u].z), b3 = bin_of(q[u].w);
            if (!(DSA_IDX_OK(b0, kBins, status) && DSA_IDX_OK(b1, kBins, status) && DSA_IDX_OK(b2, kBins, status) &&
                  DSA_IDX_OK(b3, kBins, status)))
                continue;
            if (i + 4 <= mq) {
                atomicAdd(&hist[b0], 1u);
                atomicAdd(&hist[b1], 1u);
                atomicAdd(&hist[b2], 1u);
                atomicAdd(&hist[b3], 1u);
            } else {  // the part's last, partial vector
                b1 = i + 1 < mq ? b1 : 0u;
                b2 = i + 2 < mq ? b2 : 0u;
                b3 = 0u;
                atomicAdd(&hist[b0], 1u);
                if (b1) atomicAdd(&hist[b1], 1u);
                if (b2) atomicAdd(&hist[b2], 1u);
            }
            *reinterpret_cast<uint2*>(bins + i) = make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
        }
    }
    const uint32_t* hs = cluster_hist_sum(cluster, csz, hist, hsum);
    uint32_t need = (uint32_t)k;
    const uint32_t bstar = SC::select(hs, need, wt, sel);
    const uint32_t in_bucket = hs[bstar];
    const bool take_all = in_bucket == need;
    const bool rank_mode = !take_all && in_bucket <= (uint32_t)kRankMax;

    // 3. heavy ties: radix select inside b* (exact scores read again) for the threshold key T and the
    // entries equal to T still needed
    uint32_t T = 0u, need_T = 0u;
    if (!take_all && !rank_mode) {
        need_T = need;
        uint32_t prefix = 0u, mask = 0u;
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const uint32_t dm = pass == 2 ? 0x3FFu : 0x7FFu;
            csync();  // the other CTAs (and the selection) are done reading this CTA's previous histogram
            for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
            __syncthreads();
            for (int i = tid; i < mq; i += kTopkThreads)
                if (bins[i] == bstar) {
                    const uint32_t key = order_key(s[i]);
                    if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
                }
            const uint32_t* hp = cluster_hist_sum(cluster, csz, hist, hsum);
            const uint32_t d = SC::select(hp, need_T, wt, sel);
            prefix |= d << sh;
            mask |= dm << sh;
        }
        T = prefix;
    }

    // 4. warp w owns the contiguous segment [w seg, (w + 1) seg) of the part, lane l its indices
    // l, l + 32, ...; pass one counts what the warp takes (scores above b*, members of b* taken whole,
    // ranked later, or split at T) and lists the members of a small b*
    const int seg = ((mq + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
    const int w0 = min(mq, wid * seg), w1 = min(mq, w0 + seg);
    uint32_t cnt_d = 0, cnt_t = 0;
    for (int i = w0 + lane; i < w1; i += 32) {
        const uint32_t b = bins[i];
        cnt_d += b > bstar;
        if (b == bstar) {  // rare
            if (take_all) {
                ++cnt_d;
            } else if (rank_mode) {
                const uint32_t slot = atomicAdd(&n_cand, 1u);  // at most kRankMax over the cluster
                if (DSA_IDX_OK(slot, kRankMax, status)) {
                    cand_key[slot] = order_key(s[i]);
                    cand_idx[slot] = (uint32_t)(base + i);
                }
            } else {
                const uint32_t key = order_key(s[i]);
                cnt_d += key > T;
                cnt_t += key == T;
            }
        }
    }
    cnt_d = __reduce_add_sync(0xffffffffu, cnt_d);
    cnt_t = __reduce_add_sync(0xffffffffu, cnt_t);
    if (lane == 0) {
        wcnt[wid][0] = cnt_d;
        wcnt[wid][1] = cnt_t;
    }
    // 5. small bucket: each listed member counts the better ones (larger score, or equal score and
    // lower index) across the cluster; the `need` best are marked and counted in their warp
    if (rank_mode) {
        csync();  // every CTA's member list is complete
        if (tid < (int)n_cand) {
            const uint32_t my_k = cand_key[tid], my_i = cand_idx[tid];
            uint32_t better = 0;
#pragma unroll 1
            for (int c = 0; c < csz; ++c) {
                const uint32_t* rk = csz > 1 ? cluster.map_shared_rank(cand_key, c) : cand_key;
                const uint32_t* ri = csz > 1 ? cluster.map_shared_rank(cand_idx, c) : cand_idx;
                const int nc = csz > 1 ? (int)*cluster.map_shared_rank(&n_cand, c) : (int)n_cand;
                for (int j = 0; j < nc; ++j) {
                    const uint32_t kj = rk[j];
                    better += (kj > my_k) || (kj == my_k && ri[j] < my_i);
                }
            }
            if (better < need) {
                const uint32_t li = my_i - (uint32_t)base;
                if (DSA_IDX_OK(li >> 5, kMarkWords, status) && DSA_IDX_OK(li / seg, kTopkWarps, status)) {
                    atomicOr(&marks[li >> 5], 1u << (li & 31));
                    atomicAdd(&wcnt[li / seg][0], 1u);
                }
            }
        }
    }
    __syncthreads();
    // 6. ordered output: warp totals scanned (then the lower CTAs' totals added) give each warp its first
    // slot; pass two walks the segment again in index order, a ballot placing each taken index.
    // Entries equal to T are ranked by index: the lowest `need_T` win.
    if (wid == 0) {
        uint32_t d = lane < kTopkWarps ? wcnt[lane][0] : 0u, t = lane < kTopkWarps ? wcnt[lane][1] : 0u;
        uint32_t id = d, it = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t a = __shfl_up_sync(0xffffffffu, id, o), b = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) {
                id += a;
                it += b;
            }
        }
        if (lane < kTopkWarps) {
            wcnt[lane][0] = id - d;  // exclusive
            wcnt[lane][1] = it - t;
        }
        if (lane == 31) {
            totals[0] = id;
            totals[1] = it;
        }
    }
    __syncthreads();
    uint32_t base_d = 0, base_t = 0, all_d = totals[0], all_t = totals[1];
    if (csz > 1) {
        cluster.sync();
        all_d = all_t = 0;
        for (int c = 0; c < csz; ++c) {
            const uint32_t* tt = cluster.map_shared_rank(totals, c);
            const uint32_t a = tt[0], b = tt[1];
            if (c < qr) {
                base_d += a;
                base_t += b;
            }
            all_d += a;
            all_t += b;
        }
    }
    uint32_t run_d = base_d + wcnt[wid][0], run_t = base_t + wcnt[wid][1];  // taken before this iteration
    const uint32_t lt = (1u << lane) - 1u;
    const bool split = !take_all && !rank_mode;
    for (int i0 = w0; i0 < w1; i0 += 32) {  // warp-uniform trip count
        const int i = i0 + lane;
        bool d = false, t = false;
        if (i < w1) {
            const uint32_t b = bins[i];
            d = b > bstar;
            if (b == bstar) {  // rare
                if (take_all) d = true;
                else if (rank_mode) d = (marks[i >> 5] >> (i & 31)) & 1u;
                else {
                    const uint32_t key = order_key(s[i]);
                    d = key > T;
                    t = key == T;
                }
            }
        }
        const uint32_t bd = __ballot_sync(0xffffffffu, d);
        const uint32_t bt = split ? __ballot_sync(0xffffffffu, t) : 0u;
        if (d | t) {
            const uint32_t nd = run_d + __popc(bd & lt), nt = run_t + __popc(bt & lt);
            if (d) out[nd + min(nt, need_T)] = base + i;
            else if (nt < need_T) out[nd + nt] = base + i;
        }
        run_d += __popc(bd);
        run_t += __popc(bt);
    }
    const uint32_t total = all_d + min(all_t, need_T);
    if (qr == csz - 1) {
        for (int i = (int)total + tid; i < k; i += kTopkThreads) out[i] = -1;
        if (tid == 0 && total != (uint32_t)k) report(status, DSA_ERR_DEVICE_FAULT);
    }
    if (csz > 1) cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// ---------------------------------------------------------------------------------------------
// Rows of up to 16,384 scores: one CTA per row, the row in registers.  Thread t holds the VPT
// consecutive scores [t VPT, t VPT + VPT), so the ordered compaction is one block scan of per-thread
// counts.  Same decisions as above (max / min, value buckets, direct ranking of a small bucket or a
// radix select inside a crowded one), without distributed shared memory or a staged copy of the row.
// ---------------------------------------------------------------------------------------------
template <int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS, 1)
    topk_reg_kernel(const float* __restrict__ scores, int ld, const int32_t* __restrict__ n_valid, int k,
                    int32_t* __restrict__ idx_out, int32_t* status) {
    static_assert(VPT % 4 == 0 && VPT <= 32, "a thread's run is a multiple of 4 and fits one 32-bit mask");
    using SC = RegScan<THREADS>;
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t cand_key[kRankMax], cand_idx[kRankMax];
    __shared__ uint32_t marks[THREADS * VPT / 32];  // ranked winners of a small bucket, by row index
    __shared__ uint32_t wt[32][2];
    __shared__ uint32_t sel[2];
    __shared__ uint32_t n_cand;
    __shared__ float red[2][32];
    if (threadIdx.x == 0) {
        DSA_STAMP_NS(31);
        DSA_STAMP(0);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) DSA_STAMP(1);
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int32_t* out = idx_out + (long long)row * k;
    const int n = n_valid[row];
    if (n < 0 || n > ld) {
        if (tid == 0) report(status, DSA_ERR_DEVICE_FAULT);
        for (int i = tid; i < k; i += THREADS) out[i] = -1;
        return;
    }
    if (n <= k) {
        for (int i = tid; i < k; i += THREADS) out[i] = i < n ? i : -1;
        return;
    }
    // 1. this thread's run of scores; max / min of the finite ones over the row
    const float* s = scores + (long long)row * ld;
    const int i0 = tid * VPT;
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
    for (int b = tid; b < kBins; b += THREADS) hist[b] = 0;
    for (int w = tid; w < THREADS * VPT / 32; w += THREADS) marks[w] = 0;
    if (tid == 0) n_cand = 0;
    if (tid == 0) DSA_STAMP(2);
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
        red[0][wid] = mx;
        red[1][wid] = mn;
    }
    __syncthreads();
    mx = -INFINITY;
    mn = INFINITY;
#pragma unroll
    for (int w = 0; w < SC::kWarps; ++w) {
        mx = fmaxf(mx, red[0][w]);
        mn = fminf(mn, red[1][w]);
    }
    float scale = (mx != -INFINITY && mx > mn) ? 2046.f / (mx - mn) : 0.f;
    if (!isfinite(scale)) scale = 0.f;  // degenerate range: one bucket, resolved by the radix passes
    // 2. value buckets, computed once per score and kept packed (two 16-bit bins per register):
    // bin(v) = 2047 - round((mx - v) * scale) for finite v (the rounding by adding 2^23 keeps it monotone:
    // a larger score never lands in a lower bin, equal scores share one), bin(-inf) = 0
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
        if (u < nv && DSA_IDX_OK(bin_at(u), kBins, status)) atomicAdd(&hist[bin_at(u)], 1u);
    __syncthreads();
    if (tid == 0) DSA_STAMP(3);
    uint32_t need = (uint32_t)k;
    const uint32_t bstar = SC::select(hist, need, wt, sel);
    const uint32_t in_bucket = hist[bstar];
    if (tid == 0) DSA_STAMP(4);
    const bool take_all = in_bucket == need;
    const bool rank_mode = !take_all && in_bucket <= (uint32_t)kRankMax;
    // this thread's scores above b* (always taken) and in b*
    uint32_t above = 0u, inb = 0u;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const uint32_t b = bin_at(u);
        if (u < nv && b > bstar) above |= 1u << u;
        if (u < nv && b == bstar) inb |= 1u << u;
    }
    // 3a. small bucket: its members ranked directly (larger score, or equal score and lower index)
    if (rank_mode) {
        const uint32_t cnt = (uint32_t)__popc(inb);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(&n_cand, incl);
        wbase = __shfl_sync(0xffffffffu, wbase, 31);
        uint32_t slot = wbase + incl - cnt;
#pragma unroll
        for (int u = 0; u < VPT; ++u)  // static indices keep v[] in registers
            if ((inb >> u) & 1u) {
                if (DSA_IDX_OK(slot, kRankMax, status)) {
                    cand_key[slot] = order_key(v[u]);
                    cand_idx[slot] = (uint32_t)(i0 + u);
                }
                ++slot;
            }
        __syncthreads();
        const int nc = (int)n_cand;
        for (int c = tid; c < nc; c += THREADS) {
            const uint32_t my_k = cand_key[c], my_i = cand_idx[c];
            uint32_t better = 0;
            for (int j = 0; j < nc; ++j) {
                const uint32_t kj = cand_key[j];
                better += (kj > my_k) || (kj == my_k && cand_idx[j] < my_i);
            }
            if (better < need && DSA_IDX_OK(my_i >> 5, THREADS * VPT / 32, status))
                atomicOr(&marks[my_i >> 5], 1u << (my_i & 31));
        }
        __syncthreads();
    }
    // 3b. crowded bucket: radix select on the 32-bit order keys inside b* for the threshold key T and
    // the number of entries equal to T still needed
    uint32_t T = 0u, need_T = 0u;
    if (!take_all && !rank_mode) {
        need_T = need;
        uint32_t prefix = 0u, mask = 0u;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const uint32_t dm = pass == 2 ? 0x3FFu : 0x7FFu;
            for (int b = tid; b < kBins; b += THREADS) hist[b] = 0;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const uint32_t key = order_key(v[u]);
                if (((inb >> u) & 1u) && (key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
            }
            __syncthreads();
            const uint32_t dg = SC::select(hist, need_T, wt, sel);
            prefix |= dg << sh;
            mask |= dm << sh;
        }
        T = prefix;
    }
    // 4. ordered compaction: definite members and (lowest-index first) entries equal to T
    if (tid == 0) DSA_STAMP(5);
    uint32_t dmask = above, tmask = 0u;
    if (take_all) dmask |= inb;
    else if (rank_mode) {
        for (uint32_t m = inb; m; m &= m - 1) {
            const int u = __ffs(m) - 1;
            if ((marks[(i0 + u) >> 5] >> ((i0 + u) & 31)) & 1u) dmask |= 1u << u;
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
    SC::scan2((uint32_t)__popc(dmask), (uint32_t)__popc(tmask), &ex_d, &ex_t, &tot_d, &tot_t, wt);
    uint32_t tie_rank = ex_t;
    uint32_t pos = ex_d + min(tie_rank, need_T);
    for (uint32_t m = dmask | tmask; m; m &= m - 1) {
        const int u = __ffs(m) - 1;
        if ((dmask >> u) & 1u) out[pos++] = i0 + u;
        else {
            if (tie_rank < need_T) out[pos++] = i0 + u;
            ++tie_rank;
        }
    }
    const uint32_t total = tot_d + min(tot_t, need_T);
    for (int i = (int)total + tid; i < k; i += THREADS) out[i] = -1;
    if (tid == 0 && total != (uint32_t)k) report(status, DSA_ERR_DEVICE_FAULT);
    if (tid == 0) {
        DSA_STAMP(6);
        DSA_STAMP_NS(30);
    }
}

// ---------------------------------------------------------------------------------------------
// Rows of up to 16,384 scores whose level-1 histogram -- the count of each value of the top 11 bits of the
// scores' keys -- the indexer counted while scoring them (dsa_index_topk).  The same selection as
// topk_reg_kernel, with the key's top 11 bits as the buckets: the max / min reduction and the histogram pass
// drop out, the bucket b* of the k-th largest key comes from the stored counts, and a crowded b* is resolved
// by a radix select over the remaining 21 bits.  The stored counts are cleared for the next call.
// ---------------------------------------------------------------------------------------------
template <int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS, 1)
    topk_hist_kernel(const float* __restrict__ scores, int ld, const int32_t* __restrict__ n_valid, int k,
                     int32_t* __restrict__ idx_out, unsigned* __restrict__ hist, int32_t* status) {
    static_assert(VPT % 4 == 0 && VPT <= 32, "a thread's run is a multiple of 4 and fits one 32-bit mask");
    using SC = RegScan<THREADS>;
    __shared__ uint32_t h[kBins];
    __shared__ uint32_t cand_key[kRankMax], cand_idx[kRankMax];
    __shared__ uint32_t marks[THREADS * VPT / 32];  // ranked winners of a small bucket, by row index
    __shared__ uint32_t wt[32][2];
    __shared__ uint32_t sel[2];
    __shared__ uint32_t n_cand;
    pdl_wait();
    pdl_launch_dependents();
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    int32_t* out = idx_out + (long long)row * k;
    unsigned* gh = hist + (long long)row * kBins;
    for (int b = tid; b < kBins; b += THREADS) {
        h[b] = __ldcg(gh + b);
        gh[b] = 0u;
    }
    const int n = n_valid[row];
    if (n < 0 || n > ld) {
        if (tid == 0) report(status, DSA_ERR_DEVICE_FAULT);
        for (int i = tid; i < k; i += THREADS) out[i] = -1;
        return;
    }
    if (n <= k) {
        for (int i = tid; i < k; i += THREADS) out[i] = i < n ? i : -1;
        return;
    }
    // 1. this thread's run of keys
    const float* s = scores + (long long)row * ld;
    const int i0 = tid * VPT;
    const int nv = max(0, min(VPT, n - i0));  // valid scores in the run
    uint32_t key[VPT];
#pragma unroll
    for (int u = 0; u < VPT; u += 4) {
        if (u + 4 <= nv) {
            const float4 q = *reinterpret_cast<const float4*>(s + i0 + u);
            key[u] = order_key(q.x), key[u + 1] = order_key(q.y), key[u + 2] = order_key(q.z), key[u + 3] = order_key(q.w);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) key[u + e] = u + e < nv ? order_key(s[i0 + u + e]) : 0u;
        }
    }
    for (int w = tid; w < THREADS * VPT / 32; w += THREADS) marks[w] = 0;
    if (tid == 0) n_cand = 0;
    __syncthreads();
    // 2. the bucket (top 11 bits) of the k-th largest key, from the stored counts
    uint32_t need = (uint32_t)k;
    const uint32_t bstar = SC::select(h, need, wt, sel);
    const uint32_t in_bucket = h[bstar];
    const bool take_all = in_bucket == need;
    const bool rank_mode = !take_all && in_bucket <= (uint32_t)kRankMax;
    uint32_t above = 0u, inb = 0u;  // this thread's keys above b* (always taken) and in b*
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const uint32_t b = key[u] >> 21;
        if (u < nv && b > bstar) above |= 1u << u;
        if (u < nv && b == bstar) inb |= 1u << u;
    }
    // 3a. small bucket: its members ranked directly (larger key, or equal key and lower index)
    if (rank_mode) {
        const uint32_t cnt = (uint32_t)__popc(inb);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(&n_cand, incl);
        wbase = __shfl_sync(0xffffffffu, wbase, 31);
        uint32_t slot = wbase + incl - cnt;
#pragma unroll
        for (int u = 0; u < VPT; ++u)
            if ((inb >> u) & 1u) {
                if (DSA_IDX_OK(slot, kRankMax, status)) {
                    cand_key[slot] = key[u];
                    cand_idx[slot] = (uint32_t)(i0 + u);
                }
                ++slot;
            }
        __syncthreads();
        const int nc = (int)n_cand;
        for (int c = tid; c < nc; c += THREADS) {
            const uint32_t my_k = cand_key[c], my_i = cand_idx[c];
            uint32_t better = 0;
            for (int j = 0; j < nc; ++j) {
                const uint32_t kj = cand_key[j];
                better += (kj > my_k) || (kj == my_k && cand_idx[j] < my_i);
            }
            if (better < need && DSA_IDX_OK(my_i >> 5, THREADS * VPT / 32, status))
                atomicOr(&marks[my_i >> 5], 1u << (my_i & 31));
        }
        __syncthreads();
    }
    // 3b. crowded bucket: radix select on the key's remaining bits (11, then 10) inside b* for the threshold key
    // T and the number of keys equal to T still needed
    uint32_t T = 0u, need_T = 0u;
    if (!take_all && !rank_mode) {
        need_T = need;
        uint32_t prefix = bstar << 21, mask = 0xFFE00000u;
#pragma unroll 1
        for (int pass = 1; pass < 3; ++pass) {
            const int sh = pass == 1 ? 10 : 0;
            const uint32_t dm = pass == 1 ? 0x7FFu : 0x3FFu;
            for (int b = tid; b < kBins; b += THREADS) h[b] = 0;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < VPT; ++u)
                if (((inb >> u) & 1u) && (key[u] & mask) == prefix) atomicAdd(&h[(key[u] >> sh) & dm], 1u);
            __syncthreads();
            const uint32_t dg = SC::select(h, need_T, wt, sel);
            prefix |= dg << sh;
            mask |= dm << sh;
        }
        T = prefix;
    }
    // 4. ordered compaction: definite members and (lowest-index first) keys equal to T
    uint32_t dmask = above, tmask = 0u;
    if (take_all) dmask |= inb;
    else if (rank_mode) {
        for (uint32_t m = inb; m; m &= m - 1) {
            const int u = __ffs(m) - 1;
            if ((marks[(i0 + u) >> 5] >> ((i0 + u) & 31)) & 1u) dmask |= 1u << u;
        }
    } else {
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            if (((inb >> u) & 1u) && key[u] > T) dmask |= 1u << u;
            if (((inb >> u) & 1u) && key[u] == T) tmask |= 1u << u;
        }
    }
    uint32_t ex_d, ex_t, tot_d, tot_t;
    SC::scan2((uint32_t)__popc(dmask), (uint32_t)__popc(tmask), &ex_d, &ex_t, &tot_d, &tot_t, wt);
    uint32_t tie_rank = ex_t;
    uint32_t pos = ex_d + min(tie_rank, need_T);
    for (uint32_t m = dmask | tmask; m; m &= m - 1) {
        const int u = __ffs(m) - 1;
        if ((dmask >> u) & 1u) out[pos++] = i0 + u;
        else {
            if (tie_rank < need_T) out[pos++] = i0 + u;
            ++tie_rank;
        }
    }
    const uint32_t total = tot_d + min(tot_t, need_T);
    for (int i = (int)total + tid; i < k; i += THREADS) out[i] = -1;
    if (tid == 0 && total != (uint32_t)k) report(status, DSA_ERR_DEVICE_FAULT);
}

// Rows of up to 16,384 scores over a cluster of C CTAs (few rows: a decode batch), topk_row_cluster.
template <int THREADS, int VPT, int C>
__global__ void __launch_bounds__(THREADS, 1)
    topk_creg_kernel(const float* __restrict__ scores, int ld, const int32_t* __restrict__ n_valid, int k,
                     int32_t* __restrict__ idx_out, int32_t* status) {
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ TopkRowScratch<THREADS, VPT, C> sm;
    if (threadIdx.x == 0) {
        DSA_STAMP_NS(31);
        DSA_STAMP(0);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) DSA_STAMP(1);
    const int row = blockIdx.x / C, tid = threadIdx.x;
    int32_t* out = idx_out + (long long)row * k;
    const int n = n_valid[row];  // the same for every CTA of the cluster
    if (n < 0 || n > ld) {
        if (cluster.block_rank() == 0) {
            if (tid == 0) report(status, DSA_ERR_DEVICE_FAULT);
            for (int i = tid; i < k; i += THREADS) out[i] = -1;
        }
        return;
    }
    topk_row_cluster<THREADS, VPT, C>(cluster, sm, scores + (long long)row * ld, n, k,
                                      [&](int pos, int idx) { out[pos] = idx; }, status);
    if (tid == 0) {
        DSA_STAMP(6);
        DSA_STAMP_NS(30);
    }
}

// Which kernel a call runs: rows of up to 16,384 scores one CTA each with the row in registers (faster
// than a cluster even for few rows); longer rows a cluster of as many CTAs as the row's length needs (a
// part of at most kPartMax scores each), more while the rows leave SMs idle.  Host arithmetic only.
static dsa_status_t topk_plan(int32_t nq, int32_t ld, int32_t k, bool* reg, int* csz, int* chunk) {
    if (nq < 0 || k < 1 || k > 2048 || ld < 0 || (ld & 3)) return DSA_ERR_INVALID_ARG;
    *reg = ld <= 16 * 1024;
    *csz = 1;
    *chunk = ld;
    // short rows: one 1024-thread CTA per row, or, while four CTAs per row fit on the GPU at once, a cluster
    // of four 512-thread CTAs per row (a quarter of the row each)
    if (*reg && (long long)nq * 4 <= 2LL * sm_count()) *csz = 4;
    if (*reg) return DSA_OK;
    const long long slots = 2LL * sm_count();  // CTAs of the cluster kernel resident at once
    int c = ld <= kPartMax ? 1 : (ld <= 2 * kPartMax ? 2 : kTopkClusterMax);
    while (c < kTopkClusterMax && (long long)nq * c * 2 <= slots) c *= 2;
    *csz = c;
    *chunk = ((ld + c - 1) / c + 3) & ~3;
    return *chunk > kPartMax ? DSA_ERR_UNSUPPORTED : DSA_OK;
}

}  // namespace dsa

using namespace dsa;

DSA_TIMELINE_SETTER(dsa_timeline_topk)

extern "C" dsa_status_t dsa_topk_plan(int32_t nq, int32_t ld, int32_t k, int32_t* plan) {
    if (!plan) return DSA_ERR_INVALID_ARG;
    bool reg = false;
    int csz = 1, chunk = 0;
    const dsa_status_t st = topk_plan(nq, ld, k, &reg, &csz, &chunk);
    if (st != DSA_OK) return st;
    plan[0] = reg ? 0 : 1;
    plan[1] = csz;
    plan[2] = reg ? (csz == 4 ? 512 : 1024) : kTopkThreads;
    return DSA_OK;
}

extern "C" dsa_status_t dsa_topk(int32_t nq, const float* scores, int32_t ld, const int32_t* n_valid, int32_t k,
                                 int32_t* idx_out, int32_t* dev_status, void* stream) {
    bool reg = false;
    int csz = 1, chunk = 0;
    const dsa_status_t plan_st = topk_plan(nq, ld, k, &reg, &csz, &chunk);
    if (plan_st == DSA_ERR_INVALID_ARG) return plan_st;
    if (nq == 0) return DSA_OK;
    if (!scores || !n_valid || !idx_out || !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    if (plan_st != DSA_OK) return plan_st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (reg && csz == 4) {
        const cudaError_t e = launch_pdl_cluster(topk_creg_kernel<512, 8, 4>, dim3(nq * 4), dim3(512), 0, st, 4,
                                                 scores, ld, n_valid, k, idx_out, dev_status);
        return e == cudaSuccess ? launch_status() : DSA_ERR_CUDA;
    }
    if (reg) {
        const cudaError_t e = launch_pdl(topk_reg_kernel<1024, 16>, dim3(nq), dim3(1024), 0, st, scores, ld, n_valid,
                                         k, idx_out, dev_status);
        return e == cudaSuccess ? launch_status() : DSA_ERR_CUDA;
    }
    const size_t smem = (size_t)(2 * kBins + 2 * kRankMax + kMarkWords) * sizeof(uint32_t) +
                        ((size_t)chunk * sizeof(uint16_t) + 15) / 16 * 16;
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DSA_ERR_CUDA;
    const int ahead = std::max(1, 2 * sm_count() / csz);  // clusters resident at once (two CTAs per SM)
    if (launch_pdl_cluster(topk_kernel, dim3(nq * csz), dim3(kTopkThreads), smem, st, csz, scores, ld, n_valid, k,
                           idx_out, dev_status, nq, ahead) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_status();
}

extern "C" dsa_status_t dsa_topk_counted(int32_t nq, const float* scores, int32_t ld, const int32_t* n_valid, int32_t k,
                                         int32_t* idx_out, unsigned* counts, int32_t* dev_status, void* stream) {
    if (nq < 0 || k < 1 || k > 2048 || ld < 0 || (ld & 3)) return DSA_ERR_INVALID_ARG;
    if (ld > 16384) return DSA_ERR_UNSUPPORTED;
    if (nq == 0) return DSA_OK;
    if (!scores || !n_valid || !idx_out || !counts || !aligned(scores, 16) || !aligned(counts, 16))
        return DSA_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(topk_hist_kernel<1024, 16>, dim3(nq), dim3(1024), 0, static_cast<cudaStream_t>(stream),
                                     scores, ld, n_valid, k, idx_out, counts, dev_status);
    return e == cudaSuccess ? launch_status() : DSA_ERR_CUDA;
}
