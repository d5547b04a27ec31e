// dsa_topk: per-query top-k of the indexer scores with a lowest-index tie-break.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2: S_t = TopK(I_{t,:}, k); the
// main attention reads only S_t.  [P2] "DeepSeek V4 稀疏注意力完全解剖" 机制三: k = 512 for c4a.
//
// One CTA (1024 threads) per query row.
//   1. The row is read once (coalesced 16-byte loads) into shared memory when it fits (rows up to
//      40,960 entries; longer rows are re-read from L2 in each pass).  Its finite max M and min m are
//      reduced.
//   2. Bucket select: bin(v) = 2047 - floor((M - v) * 2046 / (M - m)) for finite v, bin(-inf) = 0.  The
//      map is monotone (larger score -> same or larger bin; equal scores share a bin) and spreads
//      scores evenly, so one shared-memory histogram pass has little atomic contention.  A suffix
//      scan finds the bin b* holding the k-th largest score and `need`, the count still missing.
//   3. Inside b*: when it holds at most 1024 scores, each candidate is ranked directly against the
//      others (larger score first, lower index first among equals) and the `need` best are marked in
//      a bitmap.  Otherwise (heavy ties) a radix select on the 32-bit order keys of the candidates
//      finds the exact threshold key T and the number of entries equal to T still needed.
//   4. One pass compacts the selection in increasing index order: thread t owns a contiguous run of
//      indices (odd length: bank-conflict-free shared-memory reads) and a block scan gives every
//      selected index its slot; the scan also ranks entries equal to T by index (lowest wins).
#include "common.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;
constexpr int kCandMax = 8192;   // candidate keys kept for the radix path
constexpr int kRankMax = 1024;   // candidates ranked directly (one per thread)
constexpr int kResidentMax = 40960;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of two counters; also returns the totals.
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t* ex_a, uint32_t* ex_b,
                                            uint32_t* tot_a, uint32_t* tot_b, uint32_t (*warp_tot)[2]) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t ta = __shfl_up_sync(0xffffffffu, ia, o), tb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += ta;
            ib += tb;
        }
    }
    if (lane == 31) {
        warp_tot[wid][0] = ia;
        warp_tot[wid][1] = ib;
    }
    __syncthreads();
    if (wid == 0) {
        uint32_t wa = warp_tot[lane][0], wb = warp_tot[lane][1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t ta = __shfl_up_sync(0xffffffffu, wa, o), tb = __shfl_up_sync(0xffffffffu, wb, o);
            if (lane >= o) {
                wa += ta;
                wb += tb;
            }
        }
        warp_tot[lane][0] = wa;
        warp_tot[lane][1] = wb;
    }
    __syncthreads();
    *ex_a = (wid ? warp_tot[wid - 1][0] : 0u) + ia - a;
    *ex_b = (wid ? warp_tot[wid - 1][1] : 0u) + ib - b;
    *tot_a = warp_tot[31][0];
    *tot_b = warp_tot[31][1];
    __syncthreads();
}

// Given a filled histogram, find the bin (scanning from the top) that holds the need-th largest
// remaining element; need is reduced by the count above it.  Returns the bin.
__device__ __forceinline__ uint32_t select_bin(const uint32_t* hist, uint32_t& need, uint32_t (*warp_tot)[2],
                                               uint32_t* sel) {
    const int tid = threadIdx.x;
    const int b_hi = kBins - 1 - 2 * tid, b_lo = b_hi - 1;  // bins in descending order, two per thread
    const uint32_t c_hi = hist[b_hi], c_lo = hist[b_lo];
    uint32_t ex, ex2, tot, tot2;
    block_scan2(c_hi + c_lo, 0u, &ex, &ex2, &tot, &tot2, warp_tot);
    if (ex < need && need <= ex + c_hi) {
        sel[0] = (uint32_t)b_hi;
        sel[1] = ex;
    } else if (ex + c_hi < need && need <= ex + c_hi + c_lo) {
        sel[0] = (uint32_t)b_lo;
        sel[1] = ex + c_hi;
    }
    __syncthreads();
    const uint32_t b = sel[0];
    need -= sel[1];
    __syncthreads();
    return b;
}

__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const float* __restrict__ scores, int ld,
                                                            const int32_t* __restrict__ n_valid, int k,
                                                            int32_t* __restrict__ idx_out, int32_t* status,
                                                            int resident) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ uint32_t smem_topk[];
    uint32_t* hist = smem_topk;                  // [kBins]
    uint32_t* cand_key = hist + kBins;           // [kCandMax]
    uint32_t* cand_idx = cand_key + kCandMax;    // [kRankMax]
    uint32_t* marks = cand_idx + kRankMax;       // [ld / 32 + 1] bitmap of ranked winners
    float* rowv = reinterpret_cast<float*>(marks + (ld >> 5) + 1);  // [ld] the row (resident mode)
    __shared__ uint32_t warp_tot[32][2];
    __shared__ uint32_t sel[2];
    __shared__ uint32_t n_cand;
    __shared__ float red_max[32], red_min[32];

    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int32_t* out = idx_out + (long long)row * k;
    const int n = n_valid[row];
    if (n < 0 || n > ld) {
        if (tid == 0) report(status, DSA_ERR_DEVICE_FAULT);
        for (int i = tid; i < k; i += kTopkThreads) out[i] = -1;
        return;
    }
    if (n <= k) {
        for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    const float* s = scores + (long long)row * ld;
    float mx = -INFINITY, mn = INFINITY;
    if (resident) {
        // up to 4 float4 loads per thread in flight before any is consumed
        for (int i0 = tid * 4; i0 < n; i0 += kTopkThreads * 16) {
            float4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kTopkThreads * 4;
                q[u] = i + 4 <= n ? *reinterpret_cast<const float4*>(s + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kTopkThreads * 4;
                float v[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
                if (i + 4 > n)
                    for (int e = 0; e < 4; ++e) v[e] = i + e < n ? s[i + e] : -INFINITY;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (i + e < n) rowv[i + e] = v[e];
                    if (v[e] != -INFINITY) {
                        mx = fmaxf(mx, v[e]);
                        mn = fminf(mn, v[e]);
                    }
                }
            }
        }
    } else {
        for (int i = tid; i < n; i += kTopkThreads) {
            const float v = __ldg(s + i);
            if (v != -INFINITY) {
                mx = fmaxf(mx, v);
                mn = fminf(mn, v);
            }
        }
    }
    for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
    for (int w = tid; w <= (ld >> 5); w += kTopkThreads) marks[w] = 0;
    if (tid == 0) n_cand = 0;
    mx = warp_max(mx);
    mn = -warp_max(-mn);
    if (lane == 0) {
        red_max[wid] = mx;
        red_min[wid] = mn;
    }
    __syncthreads();
    if (wid == 0) {
        float a = warp_max(red_max[lane]), b = -warp_max(-red_min[lane]);
        if (lane == 0) {
            red_max[0] = a;
            red_min[0] = b;
        }
    }
    __syncthreads();
    mx = red_max[0];
    mn = red_min[0];
    const bool any_finite = mx != -INFINITY;
    float scale = (any_finite && mx > mn) ? 2046.f / (mx - mn) : 0.f;
    if (!isfinite(scale)) scale = 0.f;  // degenerate range: one bucket, resolved by the radix path
    auto val_at = [&](int i) -> float { return resident ? rowv[i] : __ldg(s + i); };
    auto bin_of = [&](float v) -> uint32_t {
        if (v == -INFINITY) return 0u;
        return 2047u - (uint32_t)fminf(2046.f, (mx - v) * scale);
    };

    // 2. value-bucket histogram and the bucket of the k-th largest score
    for (int i = tid; i < n; i += kTopkThreads) atomicAdd(&hist[bin_of(val_at(i))], 1u);
    __syncthreads();
    uint32_t need = (uint32_t)k;
    const uint32_t bstar = select_bin(hist, need, warp_tot, sel);
    const uint32_t in_bucket = hist[bstar];
    const bool take_all = in_bucket == need;
    const bool rank_mode = !take_all && in_bucket <= (uint32_t)kRankMax;
    uint32_t T = 0u, need_T = 0u;  // radix path: threshold key and entries equal to it still needed

    // 3. resolve the bucket
    if (!take_all) {
        const bool keep = in_bucket <= (uint32_t)kCandMax;
        if (rank_mode || keep) {
            for (int i = tid; i < n; i += kTopkThreads) {
                const float v = val_at(i);
                const bool take = bin_of(v) == bstar;
                const unsigned active = __activemask();
                const unsigned ballot = __ballot_sync(active, take);
                if (ballot) {
                    const int leader = __ffs(ballot) - 1;
                    uint32_t base = 0;
                    if (lane == leader) base = atomicAdd(&n_cand, (uint32_t)__popc(ballot));
                    base = __shfl_sync(active, base, leader);
                    if (take) {
                        const uint32_t slot = base + __popc(ballot & ((1u << lane) - 1u));
                        cand_key[slot] = order_key(v);
                        if (rank_mode) cand_idx[slot] = (uint32_t)i;
                    }
                }
            }
            __syncthreads();
        }
        if (rank_mode) {
            const int nc = (int)n_cand;
            if (tid < nc) {
                const uint32_t my_k = cand_key[tid], my_i = cand_idx[tid];
                uint32_t better = 0;
                for (int j = 0; j < nc; ++j) {
                    const uint32_t kj = cand_key[j];
                    better += (kj > my_k) || (kj == my_k && cand_idx[j] < my_i);
                }
                if (better < need) atomicOr(&marks[my_i >> 5], 1u << (my_i & 31));
            }
            __syncthreads();
        } else {
            // radix select on the order keys of the bucket's entries: digits of 11, 11 and 10 bits
            uint32_t prefix = 0u, mask = 0u;
            need_T = need;
            for (int pass = 0; pass < 3; ++pass) {
                const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
                const uint32_t dm = pass == 2 ? 0x3FFu : 0x7FFu;
                for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
                __syncthreads();
                if (keep) {
                    const int nc = (int)n_cand;
                    for (int i = tid; i < nc; i += kTopkThreads) {
                        const uint32_t key = cand_key[i];
                        if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
                    }
                } else {
                    for (int i = tid; i < n; i += kTopkThreads) {
                        const float v = val_at(i);
                        const uint32_t key = order_key(v);
                        if (bin_of(v) == bstar && (key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
                    }
                }
                __syncthreads();
                const uint32_t d = select_bin(hist, need_T, warp_tot, sel);
                prefix |= d << sh;
                mask |= dm << sh;
            }
            T = prefix;
        }
    }

    // 4. ordered compaction: definite winners, plus entries equal to T ranked by index (radix path)
    int run = (n + kTopkThreads - 1) / kTopkThreads;  // <= 64 (ld <= 65,536)
    if (resident) run |= 1;                              // odd: conflict-free strided smem reads (<= 41)
    const int lo = min(n, tid * run), hi = min(n, lo + run);
    auto classify = [&](int i, bool* def, bool* tie) {
        const float v = val_at(i);
        const uint32_t b = bin_of(v);
        *def = false;
        *tie = false;
        if (b > bstar) *def = true;
        else if (b == bstar) {
            if (take_all) *def = true;
            else if (rank_mode) *def = (marks[i >> 5] >> (i & 31)) & 1u;
            else {
                const uint32_t key = order_key(v);
                *def = key > T;
                *tie = key == T;
            }
        }
    };
    // a thread's run is at most 64 entries (rows up to 65,535 scores), so its classification fits two
    // 64-bit masks: computed once, used for the counts and again for the writes
    unsigned long long mdef = 0ull, mtie = 0ull;
    for (int i = lo; i < hi; ++i) {
        bool d, t;
        classify(i, &d, &t);
        mdef |= (unsigned long long)d << (i - lo);
        mtie |= (unsigned long long)t << (i - lo);
    }
    const uint32_t cd = __popcll(mdef), ct = __popcll(mtie);
    uint32_t ex_d, ex_t, tot_d, tot_t;
    block_scan2(cd, ct, &ex_d, &ex_t, &tot_d, &tot_t, warp_tot);
    uint32_t tie_rank = ex_t;
    uint32_t pos = ex_d + min(ex_t, need_T);
    for (unsigned long long m = mdef | mtie; m; m &= m - 1) {
        const int b = __ffsll((long long)m) - 1;
        if ((mdef >> b) & 1ull) {
            out[pos++] = lo + b;
        } else {
            if (tie_rank < need_T) out[pos++] = lo + b;
            ++tie_rank;
        }
    }
    const uint32_t total = tot_d + min(tot_t, need_T);
    for (int i = (int)total + tid; i < k; i += kTopkThreads) out[i] = -1;
    if (tid == 0 && total != (uint32_t)k) report(status, DSA_ERR_DEVICE_FAULT);
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_topk(int32_t nq, const float* scores, int32_t ld, const int32_t* n_valid, int32_t k,
                                 int32_t* idx_out, int32_t* dev_status, void* stream) {
    if (nq < 0 || k < 1 || k > 2048 || ld < 0 || (ld & 3)) return DSA_ERR_INVALID_ARG;
    if (nq == 0) return DSA_OK;
    if (!scores || !n_valid || !idx_out || !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    if (ld > 64 * kTopkThreads) return DSA_ERR_UNSUPPORTED;  // a thread's run must fit a 64-bit mask
    const int resident = ld <= kResidentMax ? 1 : 0;
    const size_t words = (size_t)kBins + kCandMax + kRankMax + (ld >> 5) + 1 + (resident ? ld : 0);
    const size_t smem = words * sizeof(uint32_t);
    if (smem > 227 * 1024) return DSA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DSA_ERR_CUDA;
    if (launch_pdl(topk_kernel, dim3(nq), dim3(kTopkThreads), smem, static_cast<cudaStream_t>(stream), scores, ld,
                   n_valid, k, idx_out, dev_status, resident) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_status();
}
