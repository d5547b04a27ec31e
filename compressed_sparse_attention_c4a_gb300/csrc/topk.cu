// dsa_topk: per-query top-k of the indexer scores with a lowest-index tie-break.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2: S_t = TopK(I_{t,:}, k); the
// main attention reads only S_t.  [P2] "DeepSeek V4 稀疏注意力完全解剖" 机制三: k = 512 for c4a.
//
// One CTA (1024 threads) per query row; scores become order-preserving uint32 keys.
//   1. The row is read once (coalesced, 16-byte loads) into shared memory when it fits (rows up to
//      40,960 entries; longer rows are re-read from L2 in each pass).
//   2. Radix select of the k-th largest key: an 11-bit histogram over the row picks the bucket that
//      holds it; the keys of that bucket (typically a few hundred) are gathered into a candidate
//      list and the remaining 11 + 10 bits are resolved on the candidates only.  The select stops
//      early as soon as a bucket holds exactly the elements still needed.
//   3. One pass compacts the selection in increasing index order: thread t owns a contiguous run
//      of indices (of odd length, so shared-memory reads are bank-conflict free), and one block
//      scan both ranks tied keys by index (lowest indices win) and gives every selected index
//      its output slot.
#include "common.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;
constexpr int kCandMax = 8192;
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

// Histogram increment aggregated over the warp's lanes that hit the same bin (scores cluster in a
// few exponent buckets, so plain shared-memory atomics would serialise).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin) {
    const unsigned active = __activemask();
    const unsigned peers = __match_any_sync(active, bin);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// Append `key` to a shared list when `take`, one atomic per warp.
__device__ __forceinline__ void list_append(uint32_t* list, uint32_t* count, bool take, uint32_t key) {
    const unsigned active = __activemask();
    const unsigned ballot = __ballot_sync(active, take);
    if (!ballot) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(ballot) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(count, (uint32_t)__popc(ballot));
    base = __shfl_sync(active, base, leader);
    if (take) list[base + __popc(ballot & ((1u << lane) - 1u))] = key;
}

struct SelectState {
    uint32_t prefix, mask, need;
};

// Given a filled histogram of one digit, find the bucket holding the need-th largest remaining key.
// Returns true when that bucket holds exactly the keys still needed (select finished).
__device__ __forceinline__ bool select_bucket(const uint32_t* hist, int shift, uint32_t dmask, SelectState& st,
                                              uint32_t (*warp_tot)[2], uint32_t* sel) {
    const int tid = threadIdx.x;
    const int b_hi = kBins - 1 - 2 * tid, b_lo = b_hi - 1;  // bins in descending order, two per thread
    const uint32_t c_hi = hist[b_hi], c_lo = hist[b_lo];
    uint32_t ex, ex2, tot, tot2;
    block_scan2(c_hi + c_lo, 0u, &ex, &ex2, &tot, &tot2, warp_tot);
    if (ex < st.need && st.need <= ex + c_hi) {
        sel[0] = (uint32_t)b_hi;
        sel[1] = ex;
    } else if (ex + c_hi < st.need && st.need <= ex + c_hi + c_lo) {
        sel[0] = (uint32_t)b_lo;
        sel[1] = ex + c_hi;
    }
    __syncthreads();
    const uint32_t b = sel[0];
    st.need -= sel[1];
    st.prefix |= b << shift;
    st.mask |= dmask << shift;
    const bool done = hist[b] == st.need;
    __syncthreads();
    return done;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int ld,
                                                            const int32_t* __restrict__ n_valid, int k,
                                                            int32_t* __restrict__ idx_out, int32_t* status,
                                                            int resident) {
    extern __shared__ uint32_t smem_topk[];
    uint32_t* hist = smem_topk;              // [kBins]
    uint32_t* cand = hist + kBins;           // [kCandMax] keys of the selected bucket
    uint32_t* rowk = cand + kCandMax;        // [ld] order keys of the row (resident mode)
    __shared__ uint32_t warp_tot[32][2];
    __shared__ uint32_t sel[2];
    __shared__ uint32_t n_cand;

    const int row = blockIdx.x;
    const int tid = threadIdx.x;
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
    if (resident) {
        for (int i = tid * 4; i < n; i += kTopkThreads * 4) {
            if (i + 4 <= n) {
                const float4 q = *reinterpret_cast<const float4*>(s + i);
                rowk[i] = order_key(q.x);
                rowk[i + 1] = order_key(q.y);
                rowk[i + 2] = order_key(q.z);
                rowk[i + 3] = order_key(q.w);
            } else {
                for (int u = i; u < n; ++u) rowk[u] = order_key(s[u]);
            }
        }
    }
    auto key_at = [&](int i) -> uint32_t { return resident ? rowk[i] : order_key(__ldg(s + i)); };
    for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
    if (tid == 0) n_cand = 0;
    __syncthreads();

    // digit 1: bits 31..21 over the whole row
    for (int i = tid; i < n; i += kTopkThreads) hist_add(hist, key_at(i) >> 21);
    __syncthreads();
    SelectState st{0u, 0u, (uint32_t)k};
    bool done = select_bucket(hist, 21, 0x7FFu, st, warp_tot, sel);
    if (!done) {
        const uint32_t bucket = hist[st.prefix >> 21];
        const bool use_cand = bucket <= (uint32_t)kCandMax;
        if (use_cand) {
            for (int i = tid; i < n; i += kTopkThreads) {
                const uint32_t key = key_at(i);
                list_append(cand, &n_cand, (key & st.mask) == st.prefix, key);
            }
        }
        for (int pass = 0; pass < 2 && !done; ++pass) {
            const int sh = pass == 0 ? 10 : 0;
            const uint32_t dm = pass == 0 ? 0x7FFu : 0x3FFu;
            __syncthreads();
            for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
            __syncthreads();
            if (use_cand) {
                const int nc = (int)n_cand;
                for (int i = tid; i < nc; i += kTopkThreads) {
                    const uint32_t key = cand[i];
                    if ((key & st.mask) == st.prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
                }
            } else {
                for (int i = tid; i < n; i += kTopkThreads) {
                    const uint32_t key = key_at(i);
                    if ((key & st.mask) == st.prefix) hist_add(hist, (key >> sh) & dm);
                }
            }
            __syncthreads();
            done = select_bucket(hist, sh, dm, st, warp_tot, sel);
        }
    }
    // keys above the final bucket are all taken; inside it, all of it (done) or the `need` lowest indices
    const bool take_all = done;
    const uint32_t bucket_hi = st.prefix | ~st.mask;
    int run = (n + kTopkThreads - 1) / kTopkThreads;
    run |= 1;  // odd run length: conflict-free strided shared-memory reads
    const int lo = min(n, tid * run), hi = min(n, lo + run);
    uint32_t gt = 0, eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = key_at(i);
        if (key > bucket_hi) ++gt;
        else if ((key & st.mask) == st.prefix) ++eq;
    }
    uint32_t ex_gt, ex_eq, tot_gt, tot_eq;
    block_scan2(gt, eq, &ex_gt, &ex_eq, &tot_gt, &tot_eq, warp_tot);
    uint32_t eq_rank = ex_eq;
    uint32_t pos = ex_gt + (take_all ? ex_eq : min(ex_eq, st.need));
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = key_at(i);
        if (key > bucket_hi) {
            out[pos++] = i;
        } else if ((key & st.mask) == st.prefix) {
            if (take_all || eq_rank < st.need) out[pos++] = i;
            ++eq_rank;
        }
    }
    const uint32_t total = tot_gt + (take_all ? tot_eq : min(tot_eq, st.need));
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
    const int resident = ld <= kResidentMax ? 1 : 0;
    const size_t smem = (size_t)(kBins + kCandMax + (resident ? ld : 0)) * sizeof(uint32_t);
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DSA_ERR_CUDA;
    topk_kernel<<<nq, kTopkThreads, smem, static_cast<cudaStream_t>(stream)>>>(scores, ld, n_valid, k, idx_out,
                                                                                 dev_status, resident);
    return launch_status();
}
