// dsa_index_scores: lightning-indexer scores on the 5th-generation tensor cores.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.1: a light scorer with few heads that
// can run in FP8 gives I_{t,s} for every history entry; [P2] "DeepSeek V4 稀疏注意力完全解剖" 机制三:
// it scores every compressed token so that the top-K can be chosen.  Score used here:
//     I(m, i) = sum_h w_h * max(0, sq_h * sk_i * <q8_h, k8_i>)   for i < n_vis(m), else -inf.
//
// Tile: 128 consecutive entries of one request (two 64-entry pages of the paged fp8 key pool) x
// N = (queries of the group) * heads columns.  TMA copies each page (a 64 x dim box, 128B or 64B
// swizzle) and the group's query codes into shared memory; one thread issues
// tcgen05.mma.kind::f8f6f4 (M = 128, N, K = 32 per instruction, fp32 accumulation in TMEM); four
// warps read their 32 TMEM lanes (one entry each) and apply the per-entry scale, ReLU, per-head
// weight and causal mask, writing coalesced score rows.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "common.cuh"

namespace dsa {

constexpr int kIdxThreads = 128;
constexpr int kTileEntries = 128;
constexpr int kPage = 64;  // c4a entries per 256-position block

struct IdxArgs {
    int nq, heads, q_group, n_cols, tmem_cols, ld;
    const float* q_scale;
    const float* w;
    const int32_t* q_pos;
    const int32_t* q_req;
    const float* key_scale;
    int num_blocks;
    dsa_block_table_t bt;
    float* scores;
    int32_t* n_visible;
    int32_t* status;
};

// ---- tcgen05 wrappers -------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand whose rows are `row_bytes` (64 or 128) long,
// stored in the matching swizzle (8-row atoms, atoms 8 * row_bytes apart).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, int row_bytes) {
    const uint64_t layout = row_bytes == 128 ? 2ull : 4ull;  // 128B or 64B swizzle
    const uint64_t sbo = (uint64_t)(8 * row_bytes) >> 4;
    return (uint64_t)((addr >> 4) & 0x3FFF) | (1ull << 16) | (sbo << 32) | (1ull << 46) | (layout << 61);
}

// Instruction descriptor: D fp32, A and B e4m3, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f8(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTileEntries >> 4) << 24);
}

template <int DIM>
__global__ void __launch_bounds__(kIdxThreads) index_kernel(const __grid_constant__ CUtensorMap kmap,
                                                            const __grid_constant__ CUtensorMap qmap, IdxArgs a) {
    constexpr int kA = kTileEntries * DIM;  // bytes of the key tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kA;                                  // n_cols rows x DIM (1024-aligned: kA is)
    float* s_kscale = reinterpret_cast<float*>(sB + a.n_cols * DIM);
    float* s_sq = s_kscale + kTileEntries;
    float* s_w = s_sq + 256;
    int* s_nvis = reinterpret_cast<int*>(s_w + 256);
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_nvis + 64);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2);
    int* s_page_ok = reinterpret_cast<int*>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = blockIdx.y, tile = blockIdx.x;
    const int q0 = grp * a.q_group;
    const int nqg = min(a.q_group, a.nq - q0);
    const int r = a.q_req[q0];

    // group visibility (every thread computes the same values)
    int max_vis = 0;
    bool mixed = false;
    for (int j = 0; j < nqg; ++j) {
        const int m = a.q_pos[q0 + j];
        max_vis = max(max_vis, m < 0 ? 0 : entries_formed((long long)m + 1, 8, 4));
        mixed |= a.q_req[q0 + j] != r;
    }
    if (mixed || r < 0 || r >= a.bt.batch) {
        if (tid == 0 && tile == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
        return;
    }
    if (tile == 0 && tid < nqg && a.n_visible) {
        const int m = a.q_pos[q0 + tid];
        a.n_visible[q0 + tid] = m < 0 ? 0 : entries_formed((long long)m + 1, 8, 4);
    }
    const int e0 = tile * kTileEntries;
    if (e0 >= max_vis) return;

    if (tid < nqg) {
        const int m = a.q_pos[q0 + tid];
        s_nvis[tid] = m < 0 ? 0 : entries_formed((long long)m + 1, 8, 4);
    }
    for (int c = tid; c < a.n_cols; c += kIdxThreads) {
        const int j = c / a.heads;
        const bool ok = j < nqg;
        s_sq[c] = ok ? a.q_scale[(long long)q0 * a.heads + c] : 0.f;
        s_w[c] = ok ? a.w[(long long)q0 * a.heads + c] : 0.f;
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(s_tmem, a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    bool ok = true;
    if (tid == 0) {
        uint32_t bytes = (uint32_t)a.n_cols * DIM;
        int blk[2];
        for (int pi = 0; pi < 2; ++pi) {
            const int lp = 2 * tile + pi;  // logical block
            blk[pi] = -1;
            s_page_ok[pi] = 0;
            if (lp * kPage >= max_vis) continue;
            const int b = lp < a.bt.max_blocks ? a.bt.table[(long long)r * a.bt.max_blocks + lp] : -1;
            if (b < 0 || b >= a.num_blocks) {
                report(a.status, DSA_ERR_DEVICE_FAULT);
                continue;
            }
            blk[pi] = b;
            s_page_ok[pi] = 1;
            bytes += kPage * DIM + kPage * 4;
        }
        mbar_arrive_expect_tx(&bars[0], bytes);
        for (int pi = 0; pi < 2; ++pi) {
            if (blk[pi] < 0) continue;
            tma_load_2d(sA + pi * kPage * DIM, &kmap, 0, blk[pi] * kPage, &bars[0]);
            bulk_g2s(s_kscale + pi * kPage, a.key_scale + (long long)blk[pi] * kPage, kPage * 4, &bars[0]);
        }
        tma_load_2d(sB, &qmap, 0, q0 * a.heads, &bars[0]);
    }
    __syncthreads();
    ok = mbar_wait_bounded(&bars[0], 0, kWaitLimitNs);
    ok = __syncthreads_and(ok);   // block-uniform: tcgen05.ld below is warp-collective
    if (!ok && tid == 0) {
        report(a.status, DSA_ERR_TIMEOUT);
        mbar_wait_bounded(&bars[0], 0, kWaitLimitNs);  // give copies still in flight a last chance to land
    }
    if (ok && tid == 0) {
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
        const uint32_t idesc = idesc_f8(a.n_cols);
#pragma unroll
        for (int ks = 0; ks < DIM / 32; ++ks)
            mma_f8(tmem, smem_desc(a_addr + ks * 32, DIM), smem_desc(b_addr + ks * 32, DIM), idesc, ks > 0);
        mma_commit(&bars[1]);
    }
    bool mma_ok = ok ? mbar_wait_bounded(&bars[1], 0, kWaitLimitNs) : false;
    mma_ok = __syncthreads_and(mma_ok);
    if (ok && !mma_ok && tid == 0) report(a.status, DSA_ERR_TIMEOUT);
    ok = mma_ok;
    tc_fence_after();

    // epilogue: thread <-> TMEM lane <-> entry
    const int row = warp * 32 + lane;
    const int e = e0 + row;
    const bool page_ok = s_page_ok[row / kPage] != 0;
    const float sk = page_ok ? s_kscale[row] : 0.f;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float acc_q = 0.f;
    for (int c0 = 0; c0 < a.n_cols; c0 += 16) {
        float v[16];
        if (ok) tmem_ld16(lane_base + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (ok) acc_q += s_w[c] * fmaxf(0.f, s_sq[c] * sk * v[i]);
            if ((c + 1) % a.heads == 0) {
                const int j = c / a.heads;
                if (j < nqg && e < a.ld) {
                    const bool vis = ok && page_ok && e < s_nvis[j];
                    a.scores[(long long)(q0 + j) * a.ld + e] = vis ? acc_q : -INFINITY;
                }
                acc_q = 0.f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

static bool make_map(CUtensorMap* map, const void* base, uint64_t rows, int dim, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)dim, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)dim};
    cuuint32_t box[2] = {(cuuint32_t)dim, (cuuint32_t)box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estride,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

template <int DIM>
static dsa_status_t launch_index(const CUtensorMap& kmap, const CUtensorMap& qmap, const IdxArgs& a, int tiles,
                                 int groups, cudaStream_t st) {
    const int need = 1024 + kTileEntries * DIM + a.n_cols * DIM + (kTileEntries + 256 + 256 + 64) * 4 + 64;
    // at most 512 / tmem_cols resident CTAs per SM, so that every tcgen05.alloc is satisfied at once
    const int per_sm = 512 / a.tmem_cols;
    const int cap = 232448 / per_sm - 1024;
    const int smem = per_sm >= 16 ? need : (need > cap ? need : cap);
    if (cudaFuncSetAttribute(index_kernel<DIM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSA_ERR_CUDA;
    index_kernel<DIM><<<dim3(tiles, groups), kIdxThreads, smem, st>>>(kmap, qmap, a);
    return launch_status();
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_index_scores(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8,
                                         const float* q_scale, const float* w, const int32_t* q_pos,
                                         const int32_t* q_req, int32_t q_group, const dsa_pool_t* keys,
                                         const dsa_block_table_t* bt, float* scores, int32_t ld, int32_t* n_visible,
                                         int32_t* dev_status, void* stream) {
    if (nq < 0 || ld < 0 || (ld & 3)) return DSA_ERR_INVALID_ARG;
    if (nq == 0) return DSA_OK;
    if (heads != 4 && heads != 8 && heads != 16) return DSA_ERR_UNSUPPORTED;
    if (dim != 64 && dim != 128) return DSA_ERR_UNSUPPORTED;
    if (q_group < 1 || q_group * heads > 256) return DSA_ERR_INVALID_ARG;
    if (!q8 || !q_scale || !w || !q_pos || !q_req || !scores || !keys || !bt || !bt->table || bt->max_blocks <= 0)
        return DSA_ERR_INVALID_ARG;
    if (!pool_ok(keys) || keys->dtype != DSA_FP8_E4M3 || keys->dim != dim || keys->rows_per_block != kPage)
        return DSA_ERR_INVALID_ARG;
    if (!aligned(q8, 16)) return DSA_ERR_INVALID_ARG;
    const int n_cols = ((q_group * heads + 15) / 16) * 16;  // M = 128 needs N % 16 == 0
    IdxArgs a{};
    a.nq = nq;
    a.heads = heads;
    a.q_group = q_group;
    a.n_cols = n_cols;
    a.tmem_cols = n_cols <= 32 ? 32 : (n_cols <= 64 ? 64 : (n_cols <= 128 ? 128 : 256));
    a.ld = ld;
    a.q_scale = q_scale;
    a.w = w;
    a.q_pos = q_pos;
    a.q_req = q_req;
    a.key_scale = keys->scale;
    a.num_blocks = keys->num_blocks;
    a.bt = *bt;
    a.scores = scores;
    a.n_visible = n_visible;
    a.status = dev_status;
    CUtensorMap kmap, qmap;
    if (!make_map(&kmap, keys->data, (uint64_t)keys->num_blocks * kPage, dim, kPage)) return DSA_ERR_CUDA;
    if (!make_map(&qmap, q8, (uint64_t)nq * heads, dim, n_cols)) return DSA_ERR_CUDA;
    const int tiles = (ld + kTileEntries - 1) / kTileEntries;
    const int groups = (nq + q_group - 1) / q_group;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return dim == 128 ? launch_index<128>(kmap, qmap, a, tiles, groups, st)
                      : launch_index<64>(kmap, qmap, a, tiles, groups, st);
}
