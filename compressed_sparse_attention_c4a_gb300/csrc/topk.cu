// dsa_topk: per-query top-k of the indexer scores with a lowest-index tie-break.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2: S_t = TopK(I_{t,:}, k); the
// main attention reads only S_t.  [P2] "DeepSeek V4 稀疏注意力完全解剖" 机制三: k = 512 for c4a.
//
// One CTA (1024 threads) per query row.  Scores become order-preserving uint32 keys.  A radix
// select finds the k-th largest key with digit passes of 11, 11 and 10 bits (shared-memory
// histograms), stopping early once the selected bucket holds exactly the elements still needed.
// A final pass compacts the selection in increasing index order: thread t owns a contiguous run
// of indices, so one block-wide scan both ranks tied elements by index (the lowest-index ones
// win) and gives each selected index its output slot.
#include "common.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block scan of two counters at once; returns the exclusive prefixes and the totals.
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
        warp_tot[lane][0] = wa;  // inclusive over warps
        warp_tot[lane][1] = wb;
    }
    __syncthreads();
    const uint32_t base_a = wid ? warp_tot[wid - 1][0] : 0u, base_b = wid ? warp_tot[wid - 1][1] : 0u;
    *ex_a = base_a + ia - a;
    *ex_b = base_b + ib - b;
    *tot_a = warp_tot[31][0];
    *tot_b = warp_tot[31][1];
    __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int ld,
                                                            const int32_t* __restrict__ n_valid, int k,
                                                            int32_t* __restrict__ idx_out, int32_t* status) {
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t warp_tot[32][2];
    __shared__ uint32_t sel_bin, sel_above;
    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    int32_t* out = idx_out + (long long)row * k;
    int n = n_valid[row];
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
    // contiguous run per thread, a multiple of 4 so float4 loads stay aligned (ld % 4 == 0)
    int run = (n + kTopkThreads - 1) / kTopkThreads;
    run = (run + 3) & ~3;
    const int lo = min(n, tid * run), hi = min(n, lo + run);

    uint32_t prefix = 0, mask = 0;  // selected high bits so far
    uint32_t need = (uint32_t)k;    // elements still to take from inside the current bucket
    bool take_all = false;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
        __syncthreads();
        for (int i = lo; i < hi; i += 4) {
            float v[4];
            if (i + 4 <= hi) {
                float4 q = *reinterpret_cast<const float4*>(s + i);
                v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
            } else {
                for (int u = 0; u < 4; ++u) v[u] = (i + u < hi) ? s[i + u] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i + u >= hi) break;
                const uint32_t key = order_key(v[u]);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dmask], 1u);
            }
        }
        __syncthreads();
        // bins in descending order: thread t sums bins 2047-2t and 2046-2t
        const int b_hi = kBins - 1 - 2 * tid, b_lo = b_hi - 1;
        const uint32_t c_hi = hist[b_hi], c_lo = hist[b_lo];
        uint32_t ex, ex_unused, tot, tot_unused;
        block_scan2(c_hi + c_lo, 0u, &ex, &ex_unused, &tot, &tot_unused, warp_tot);
        // bucket b holds the need-th largest remaining element when above(b) < need <= above(b) + hist[b]
        if (ex < need && need <= ex + c_hi) {
            sel_bin = (uint32_t)b_hi;
            sel_above = ex;
        } else if (ex + c_hi < need && need <= ex + c_hi + c_lo) {
            sel_bin = (uint32_t)b_lo;
            sel_above = ex + c_hi;
        }
        __syncthreads();
        const uint32_t b = sel_bin;
        need -= sel_above;
        prefix |= b << sh;
        mask |= dmask << sh;
        if (hist[b] == need) {
            take_all = true;
            __syncthreads();
            break;
        }
        __syncthreads();
    }
    // selection: key above the bucket, or inside it (all of it, or the `need` lowest indices)
    const uint32_t bucket_hi = prefix | ~mask;
    uint32_t gt = 0, eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = order_key(s[i]);
        if (key > bucket_hi) ++gt;
        else if ((key & mask) == prefix) ++eq;
    }
    uint32_t ex_gt, ex_eq, tot_gt, tot_eq;
    block_scan2(gt, eq, &ex_gt, &ex_eq, &tot_gt, &tot_eq, warp_tot);
    uint32_t eq_rank = ex_eq;
    uint32_t pos = ex_gt + (take_all ? ex_eq : min(ex_eq, need));
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = order_key(s[i]);
        if (key > bucket_hi) {
            out[pos++] = i;
        } else if ((key & mask) == prefix) {
            if (take_all || eq_rank < need) out[pos++] = i;
            ++eq_rank;
        }
    }
    const uint32_t total = tot_gt + (take_all ? tot_eq : min(tot_eq, need));
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
    topk_kernel<<<nq, kTopkThreads, 0, static_cast<cudaStream_t>(stream)>>>(scores, ld, n_valid, k, idx_out,
                                                                              dev_status);
    return launch_status();
}
