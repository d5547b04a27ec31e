// dsa_index_scores: lightning-indexer scores on the 5th-generation tensor cores.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.1: a light scorer with few heads that
// can run in FP8 gives I_{t,s} for every history entry; [P2] "DeepSeek V4 稀疏注意力完全解剖" 机制三:
// it scores every compressed token so that the top-K can be chosen.  Score used here:
//     I(m, i) = sum_h w_h * max(0, sq_h * sk_i * <q8_h, k8_i>)   for i < n_vis(m), else -inf.
//
// Tile: 128 consecutive entries of one request (two 64-entry pages of the paged fp8 key pool) x
// N = (queries of the group) * heads columns.  TMA copies each page (a 64 x dim box, 128B or 64B
// swizzle) into a stage; the group's query codes, head weights and query scales go into one of two
// group buffers only when the group changes (a CTA's items are consecutive tiles of few groups).  One
// thread issues tcgen05.mma.kind::f8f6f4 (M = 128, N, K = 32 per instruction, fp32 accumulation in
// TMEM); the epilogue warps read their 32 TMEM lanes (one entry each) over a slice of the columns, apply
// the entry's key scale, ReLU, the per-head weights (folded with the query scales once per group) and
// the causal mask, writing coalesced score rows.  Every wait is bounded.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>

#include "common.cuh"

namespace dsa {

// warp 0: TMA producer, warp 1: MMA issuer, then EW epilogue warps: 4 for narrow groups (N <= 128, two
// tiles per item, two CTAs per SM), 12 for wide ones (N up to 256, one tile per item, one CTA per SM), so
// that the epilogue keeps pace with the tensor cores.  Epilogue warp w reads TMEM lanes 32 * (w % 4) ..
// + 31 (the quadrant its warp id allows) and column slice (w - 2) / 4 of EW / 4 slices.  Registers: a
// sub-partition holds 16K of them and at most 3 (narrow, two CTAs) or 4 (wide) of the CTA's warps.
template <int TPI>
__host__ __device__ constexpr int epi_warps() { return TPI == 2 ? 4 : 12; }
template <int TPI>
__host__ __device__ constexpr int idx_threads() { return 64 + 32 * epi_warps<TPI>(); }
// columns of one epilogue slice, at most: 16-column chunks of N split over EW / 4 slices
template <int TPI>
__host__ __device__ constexpr int slice_cols() { return TPI == 2 ? 128 : 96; }
constexpr int kTileEntries = 128;
constexpr int kPage = 64;         // c4a entries per 256-position block
constexpr int kChunkItems = 32;   // items resolved together (one per producer lane)

struct IdxArgs {
    int nq, heads, q_group, n_cols, tmem_cols, ld;
    int n_groups, items, stages, stage_bytes, n_acc;  // items per group; n_acc: TMEM accumulators (2 or 4)
    int gbuf_bytes;                                   // one group buffer: query codes, head weights, query scales
    long long total_items;
    const float* q_scale;
    const float* w;
    const int32_t* q_pos;
    const int32_t* q_req;
    const int32_t* fresh_pos;   // [batch] first raw position the preceding kernel may still compress, or NULL
    unsigned* work;             // [2] item counter and finished-CTA counter (dynamic split), or NULL (static)
    const float* key_scale;
    int num_blocks;
    dsa_block_table_t bt;
    float* scores;
    int32_t* n_visible;
    int32_t* status;
    unsigned long long wait_ns;  // limit of every bounded wait
    int withhold;                // test hook: the producer issues no copy and posts no stage
    unsigned* hist;              // fused top-k: [nq][2048] counts of the top 11 bits of each row's score keys, or NULL
    int key_e2m1;                // keys are fp4 e2m1 codes (else e4m3)
};

// Shared-memory matrix descriptor of a K-major operand whose rows are `row_bytes` (64 or 128) long,
// stored in the matching swizzle (8-row atoms, atoms 8 * row_bytes apart).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, int row_bytes) {
    const uint64_t layout = row_bytes == 128 ? 2ull : 4ull;  // 128B or 64B swizzle
    const uint64_t sbo = (uint64_t)(8 * row_bytes) >> 4;
    return (uint64_t)((addr >> 4) & 0x3FFF) | (1ull << 16) | (sbo << 32) | (1ull << 46) | (layout << 61);
}

// Instruction descriptor of kind::f8f6f4: D fp32, A (keys) e4m3 or e2m1 (A type field 0 or 5), B (queries)
// e4m3, both K-major, M = 128, N = n.  e2m1 keys sit in shared memory one code per byte (the TMA's unpacking
// format), so the operand layout and descriptors are those of e4m3 keys.
__device__ __forceinline__ uint32_t idesc_f8(int n, bool a_e2m1) {
    return (1u << 4) | ((a_e2m1 ? 5u : 0u) << 7) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTileEntries >> 4) << 24);
}

// c4a entries visible to the query at position m: those whose last raw token 4i + 7 <= m.
__device__ __forceinline__ int visible_at(int m) { return m < 7 ? 0 : ((m - 7) >> 2) + 1; }

__device__ __forceinline__ int visible_of(const IdxArgs& a, int q) { return visible_at(a.q_pos[q]); }
// Entries complete before raw position p, which a compressor that starts at position p cannot write: n_vis(p - 1).
__device__ __forceinline__ int entries_complete_before(int p) { return p < 1 ? 0 : visible_at(p - 1); }

// Item = `tpi` consecutive 128-entry tiles of one query group (tpi = 1 or 2).  Its request, visibility
// and the physical blocks of its 64-entry pages, resolved by one producer lane.
struct ItemInfo {
    int valid, g, t, r, max_vis, want;  // want: bit p set when page p holds visible entries
    int fresh;                          // 1: a loaded page holds entries the preceding kernel may write
    int blk[4];
};

// Request and visible-entry bound of query group g (r = -1 if the group mixes requests or names a
// request beyond the table).
__device__ __forceinline__ void group_of(const IdxArgs& a, int g, int* r, int* max_vis) {
    const int q0 = g * a.q_group;
    const int nqg = min(a.q_group, a.nq - q0);
    int rr = a.q_req[q0], mv = 0;
    for (int j = 0; j < nqg; ++j) {
        mv = max(mv, visible_of(a, q0 + j));
        if (a.q_req[q0 + j] != rr) rr = -1;
    }
    if (rr >= a.bt.batch) rr = -1;
    *r = rr;
    *max_vis = mv;
}

// Item (g, t): tile t of group g; `valid` = 0 marks "no item".  The group's request and visible-entry
// bound come from the producer's shared-memory table (filled once per CTA).
template <int TPI>
__device__ __forceinline__ ItemInfo item_info(const IdxArgs& a, int valid, int g, int t, const int* grp_r,
                                              const int* grp_mv) {
    ItemInfo x{0, g, t, -1, 0, 0, 1, {-1, -1, -1, -1}};
    if (!valid || !DSA_IDX_OK(g, a.n_groups, a.status)) return x;
    x.r = grp_r[g];
    x.max_vis = grp_mv[g];
    if (x.r < 0 || t * TPI * kTileEntries >= x.max_vis) return x;
    x.valid = 1;
    if (a.fresh_pos) {  // the loaded pages end at the page holding the item's last visible entry
        const int end = (min(x.max_vis, (t + 1) * TPI * kTileEntries) + kPage - 1) / kPage * kPage;
        x.fresh = end > entries_complete_before(__ldg(a.fresh_pos + x.r)) ? 1 : 0;
    }
    // no branch on the loaded table entries: the loads stay in flight until the item is used
#pragma unroll
    for (int pi = 0; pi < 2 * TPI; ++pi) {
        const int lp = 2 * TPI * t + pi;
        const bool want = lp * kPage < x.max_vis;
        const bool in_table = want && lp < a.bt.max_blocks;
        x.blk[pi] = in_table ? a.bt.table[(long long)x.r * a.bt.max_blocks + lp] : -1;
        x.want |= want ? (1 << pi) : 0;
    }
    return x;
}

__device__ __forceinline__ ItemInfo shfl_item(const ItemInfo& x, int src) {
    ItemInfo y;
    y.valid = __shfl_sync(0xffffffffu, x.valid, src);
    y.g = __shfl_sync(0xffffffffu, x.g, src);
    y.t = __shfl_sync(0xffffffffu, x.t, src);
    y.r = __shfl_sync(0xffffffffu, x.r, src);
    y.max_vis = __shfl_sync(0xffffffffu, x.max_vis, src);
    y.want = __shfl_sync(0xffffffffu, x.want, src);
    y.fresh = __shfl_sync(0xffffffffu, x.fresh, src);
#pragma unroll
    for (int p = 0; p < 4; ++p) y.blk[p] = __shfl_sync(0xffffffffu, x.blk[p], src);
    return y;
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            report(status, DSA_ERR_TIMEOUT);
            return false;
        }
    }
}

// Shared memory: S stages of key tiles [TPI][128][DIM] (swizzled; TMA, completing on full[s]), released by
// the tensor cores' completion (tcgen05.commit on empty[s]) as soon as the MMAs that read them are done;
// item slots (4 for two-tile items, 8 for one-tile items) of StageMeta and fp32 entry scales [TPI * 128]
// (cp.async, 16 bytes per producer lane and tile, completing on ifull[k]), released by the epilogue
// (sempty[k]); NA TMEM accumulators (tfull[b] / tempty[b]).  So the epilogue may trail the copies by a few
// items without holding key tiles.
// Group buffer: query tile [n_cols][DIM] (swizzled), head weights [n_cols], query scales [n_cols], visible
// entries of each query of the group [64] (written by the producer lanes before the buffer's barrier is
// armed).  Only the producer walks the work list; it describes each item in its slot (or posts a terminal
// item), so the MMA and epilogue roles never touch global metadata.
struct StageMeta {
    int terminal;  // 1: no more items for this CTA
    int gb;        // group buffer holding the item's query codes, weights and query scales
    int blk[4];    // physical block of each 64-entry page, -1 if not loaded (key tiles in stage n mod S)
    int nq;        // queries in the group
    int q0;        // first query of the group
    int e0;        // first entry of the tile
};

__host__ __device__ constexpr int meta_bytes() { return ((int)sizeof(StageMeta) + 15) / 16 * 16; }

// Bytes of one item slot: StageMeta + the item's fp32 entry scales.
template <int TPI>
__host__ __device__ constexpr int item_slot_bytes() { return meta_bytes() + TPI * kTileEntries * 4; }
template <int TPI>
__host__ __device__ constexpr int item_slots() { return TPI == 2 ? 4 : 8; }

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// Two fp32 lanes in one 64-bit register, and their fused multiply-add (fma.rn.f32x2: each lane rounds as
// a scalar fmaf would).
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void fma_f32x2(unsigned long long& acc, unsigned long long a, unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ float sum_f32x2(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}

__host__ __device__ constexpr int gbuf_nvis_offset(int n_cols, int dim) { return n_cols * dim + 2 * n_cols * 4; }

// Level-1 histogram of the fused top-k ([P1] §4.2: S_t = TopK(I_t, k)): each visible entry's score is counted
// by the top 11 bits of its order key (dsa_score_key), the first digit of the top-k's radix select.
constexpr int kSelBins = 2048;

template <int DIM, int HEADS, int TPI, bool N16>
__global__ void __maxnreg__(TPI == 2 ? 168 : 128) index_kernel(const __grid_constant__ CUtensorMap kmap,
                                                            const __grid_constant__ CUtensorMap qmap, IdxArgs a) {
    constexpr int kItem = TPI * kTileEntries;  // entries per item
    constexpr int kPages = 2 * TPI;
    constexpr int EW = epi_warps<TPI>(), NSL = EW / 4, kSlice = slice_cols<TPI>();
    constexpr int kThreads = idx_threads<TPI>();
    constexpr int kBatch = TPI == 2 ? 4 : 2;  // 16-column TMEM loads in flight per wait (register budget)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = a.stages, NA = a.n_acc;
    uint8_t* gbase = smem + (size_t)S * a.stage_bytes;  // two group buffers
    constexpr int NK = item_slots<TPI>();
    uint8_t* slots = gbase + 2 * a.gbuf_bytes;          // [NK] item slots: StageMeta + entry scales
    float* s_fold = reinterpret_cast<float*>(slots + NK * item_slot_bytes<TPI>());  // [EW][kSlice]: w_h * sq_h per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(s_fold + EW * kSlice);
    uint64_t* empty = full + S;
    uint64_t* ifull = empty + S;    // [NK] item slot written (meta + scales)
    uint64_t* sempty = ifull + 8;   // [NK] item slot released by the epilogue
    uint64_t* tfull = sempty + 8;   // [NA]
    uint64_t* tempty = tfull + 4;   // [NA] accumulator released by the epilogue
    uint64_t* gfull = tempty + 4;  // [2] group buffer loaded
    uint64_t* gempty = gfull + 2;  // [2] group buffer released by the epilogue warps
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(gempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(s_tmem + 1);
    int* grp_prefix = reinterpret_cast<int*>(s_tmem + 2);  // [n_groups + 1] valid tiles before each group
    int* grp_r = grp_prefix + a.n_groups + 1;            // [n_groups] request of each group (-1: invalid)
    int* grp_mv = grp_r + a.n_groups;                    // [n_groups] visible-entry bound of each group

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto slot_meta = [&](int b) { return reinterpret_cast<StageMeta*>(slots + (size_t)b * item_slot_bytes<TPI>()); };
    auto slot_scale = [&](int b) { return reinterpret_cast<float*>(slots + (size_t)b * item_slot_bytes<TPI>() + meta_bytes()); };

    if (tid == 0) {
        DSA_STAMP_NS(31);
        DSA_STAMP(0);
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);   // the producer's lane 0, with the TMA bytes
            mbar_init(&empty[i], 1);  // the MMAs that read the stage are complete (tcgen05.commit)
        }
        for (int k = 0; k < NK; ++k) {
            mbar_init(&ifull[k], 1 + 32);  // the producer's lane 0 (meta written) + 32 scale copies
            mbar_init(&sempty[k], EW * 32);
        }
        for (int b = 0; b < NA; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], EW * 32);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&gfull[b], 1);
            // released by the epilogue warps (and, for decode-shaped groups, whose epilogue keeps the group's
            // values in registers and lets go at once, by the tensor cores' completion of the group's last MMA)
            mbar_init(&gempty[b], N16 ? EW + 1 : EW);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(s_tmem, a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    if (tid == 0) DSA_STAMP(1);
    // Programmatic dependent launch: the producer resolves its first items (query positions and requests,
    // the block table: inputs no preceding kernel of the layer writes) while the preceding kernel (the
    // compressor, which writes keys) finishes.  Without fresh_pos, key copies and every global write come
    // after the wait; with it, pages wholly below entry n_vis(fresh_pos[r] - 1) are copied and scored before
    // it and the producer waits before its first fresh page (and before the CTA ends in any case).
    const bool early = a.fresh_pos != nullptr;
    if (warp != 0) {
        if (!early) {
            pdl_wait();
            pdl_launch_dependents();
        }
        // visible-entry count of every query (grid-strided over the non-producer threads)
        if (a.n_visible)
            for (int q = blockIdx.x * (kThreads - 32) + tid - 32; q < a.nq; q += gridDim.x * (kThreads - 32))
                a.n_visible[q] = visible_of(a, q);
    }

    if (warp == 0) {
        // ---- producer warp ---------------------------------------------------------------------------
        // Valid tiles per group -> prefix sums in shared memory; this CTA takes an equal contiguous
        // share [lo, hi) of all valid (group, tile) items.  Lanes resolve items kChunkItems at a time
        // (the next batch is prefetched while the current one is issued); lane 0 issues the copies.
        int* pre = grp_prefix;
        long long carry = 0;
        bool bad_group = false;  // reported after the wait
        for (int g0 = 0; g0 < a.n_groups; g0 += 32) {
            const int g = g0 + lane;
            int cnt = 0;
            if (g < a.n_groups) {
                int r, mv;
                group_of(a, g, &r, &mv);
                grp_r[g] = r;
                grp_mv[g] = mv;
                if (r < 0) bad_group = true;
                else cnt = min((mv + kItem - 1) / kItem, a.items);
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (g < a.n_groups) pre[g] = (int)(carry + incl - cnt);
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) pre[a.n_groups] = (int)carry;
        __syncwarp();
        const long long V = carry;
        // static split: an equal contiguous share [lo, hi).  With a work counter (a.work): a contiguous run of
        // half a fair share first, then runs of consecutive items taken from the counter (two requests in
        // flight from the start, read when the static run ends), so that a CTA that starts late takes less
        const bool dyn = a.work != nullptr;
        const long long R = dyn ? V / (2 * gridDim.x) : 0;         // static run per CTA (dynamic split)
        const long long base_dyn = R * gridDim.x;                   // first item of the shared remainder
        const int G = dyn ? (int)max(1ll, min((long long)kChunkItems, (V - base_dyn) / gridDim.x)) : kChunkItems;
        const long long lo = dyn ? R * blockIdx.x : V * blockIdx.x / gridDim.x;
        const long long hi = dyn ? R * (blockIdx.x + 1) : V * (blockIdx.x + 1) / gridDim.x;
        auto grab = [&]() -> long long {  // lane 0 issues the atomic; the value is read (shuffled) later
            long long v = 0;
            if (lane == 0) v = (long long)atomicAdd(a.work, (unsigned)G);
            return v;
        };
        // item index -> (group, tile) by binary search over the prefix
        auto locate = [&](long long idx, int* g, int* t) {
            int l = 0, h = a.n_groups - 1;
            while (l < h) {
                const int mid = (l + h + 1) >> 1;
                if (pre[mid] <= idx) l = mid;
                else h = mid - 1;
            }
            *g = l;
            *t = (int)(idx - pre[l]);
        };
        auto resolve = [&](long long base, long long end) {  // items [base, end), at most 32
            const long long idx = base + lane;
            int g = 0, t = 0;
            const int valid = lane < kChunkItems && idx < end;
            if (valid) locate(idx, &g, &t);
            return item_info<TPI>(a, valid, g, t, grp_r, grp_mv);
        };
        // with at most one query group per request (decode) every key page is read once: it leaves L2 first;
        // groups that share a request's pages (prefill) keep the default policy, so the pages stay for the next
        const uint64_t key_policy = a.n_groups <= a.bt.batch ? l2_evict_first() : l2_evict_normal();
        int n = 0, ps = 0, pphase = 0;  // items issued; stage index and its phase parity
        int pb = 0, pbph = 0;           // item slot index and its phase parity
        int cur_g = -1, gb = 1, guse[2] = {0, 0};  // group in the current buffer, buffer index, loads per buffer
        bool alive = true;
        if (lane == 0) DSA_STAMP(2);
        long long ahead1 = dyn ? grab() : 0, ahead2 = dyn ? grab() : 0;  // lane 0: the next two runs, in flight
        long long base = lo, run_end = hi;  // the current run: [base, run_end)
        auto next_run = [&](long long* b, long long* e) {  // a run from the counter (empty past the last item)
            *b = base_dyn + __shfl_sync(0xffffffffu, ahead1, 0);
            *e = min(*b + G, V);
            ahead1 = ahead2;
            ahead2 = grab();
        };
        if (dyn && base >= run_end) next_run(&base, &run_end);
        ItemInfo cur = resolve(base, run_end);
        bool waited = !early;
        if (!early) {
            pdl_wait();  // keys may come from the preceding kernel
            pdl_launch_dependents();
        }
        if (bad_group) report(a.status, DSA_ERR_DEVICE_FAULT);
        // (test hook) withhold: no copy is issued and no stage posted, so every consumer wait runs out
        while (base < run_end && alive && !a.withhold) {
            long long nb = base + kChunkItems, ne = run_end;  // the next chunk of this run, or the next run
            if (nb >= run_end) {
                if (dyn) next_run(&nb, &ne);
                else ne = nb;
            }
            const ItemInfo nxt = resolve(nb, ne);
            for (int u = 0; u < kChunkItems; ++u) {
                ItemInfo it = shfl_item(cur, u);
                if (!it.valid) continue;
                if (it.fresh && !waited) {  // warp-uniform: this item's pages may still be being written
                    pdl_wait();
                    pdl_launch_dependents();
                    waited = true;
                }
                // a visible page whose table entry is unmapped or outside the pool: a device fault, not loaded
                bool bad = false;
#pragma unroll
                for (int p = 0; p < kPages; ++p) {
                    const bool w = (it.want >> p) & 1;
                    const bool b = w && (it.blk[p] < 0 || it.blk[p] >= a.num_blocks);
                    bad |= b;
                    if (b || !w) it.blk[p] = -1;
                }
                if (bad && lane == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
                const int q0 = it.g * a.q_group;
                const int nqg = min(a.q_group, a.nq - q0);
                if (it.g != cur_g) {  // warp-uniform
                    // a new group: its query codes, weights, query scales and per-query visible entries into
                    // the other buffer, once the epilogue has let go of that buffer's previous group
                    gb ^= 1;
                    bool ok = true;
                    if (lane == 0 && guse[gb] > 0) ok = wait_or_abort(&gempty[gb], (guse[gb] - 1) & 1, abort_flag, a.status, a.wait_ns);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        alive = false;
                    } else {
                        uint8_t* gp = gbase + (size_t)gb * a.gbuf_bytes;
                        int* gnv = reinterpret_cast<int*>(gp + gbuf_nvis_offset(a.n_cols, DIM));
                        for (int j = lane; j < nqg; j += 32) gnv[j] = a.q_group == 1 ? it.max_vis : visible_of(a, q0 + j);
                        __syncwarp();
                        if (lane == 0) {  // release: the lanes' writes above are ordered before the arrival
                            mbar_arrive_expect_tx(&gfull[gb], (uint32_t)a.n_cols * DIM + 2u * nqg * HEADS * 4u);
                            tma_load_2d(gp, &qmap, 0, q0 * HEADS, &gfull[gb]);
                            bulk_g2s(gp + a.n_cols * DIM, a.w + (long long)q0 * HEADS, nqg * HEADS * 4, &gfull[gb]);
                            bulk_g2s(gp + a.n_cols * DIM + a.n_cols * 4, a.q_scale + (long long)q0 * HEADS,
                                     nqg * HEADS * 4, &gfull[gb]);
                        }
                        ++guse[gb];
                        cur_g = it.g;
                    }
                }
                const int s = ps, b = pb;
                bool go = false;
                if (lane == 0 && alive) {  // the stage's previous MMAs done, the slot's previous item scored
                    go = wait_or_abort(&empty[s], pphase ^ 1, abort_flag, a.status, a.wait_ns) &&
                         wait_or_abort(&sempty[b], pbph ^ 1, abort_flag, a.status, a.wait_ns);
                    alive = go;
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (lane == 0) DSA_TRACE(n, 0);
                uint8_t* st = smem + (size_t)s * a.stage_bytes;
                if (go) {  // the entry scales: 16 lanes per page, zero-filled where a page is absent
                    float* sc = slot_scale(b);
#pragma unroll
                    for (int i = 0; i < TPI; ++i) {
                        const int pg = 2 * i + (lane >> 4);
                        const int bp = (lane >> 4) ? it.blk[2 * i + 1] : it.blk[2 * i];
                        const float* src = bp >= 0 ? a.key_scale + (long long)bp * kPage + (lane & 15) * 4 : a.key_scale;
                        cp_async16_nc(smem_u32(sc + pg * kPage + (lane & 15) * 4), src, bp >= 0 ? 16u : 0u);
                    }
                    cp_async_arrive_noinc(&ifull[b]);
                }
                if (lane == 0 && go) {
                    StageMeta* meta = slot_meta(b);
                    meta->terminal = 0;
                    meta->gb = gb;
                    // a page's copy completes its global bytes on the barrier: 64 rows of DIM e4m3 codes, or of
                    // DIM / 2 bytes of packed e2m1 codes (which land unpacked, one code per byte, in shared memory)
                    const uint32_t page_bytes = a.key_e2m1 ? kPage * DIM / 2 : kPage * DIM;
                    uint32_t bytes = 0;
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        meta->blk[p] = p < kPages ? it.blk[p] : -1;
                        if (p < kPages && it.blk[p] >= 0) bytes += page_bytes;
                    }
                    meta->nq = nqg;
                    meta->q0 = q0;
                    meta->e0 = it.t * kItem;
                    mbar_arrive(&ifull[b]);                  // release: the meta writes above are visible
                    mbar_arrive_expect_tx(&full[s], bytes);
                }
                __syncwarp();
                if (n == 0 && lane == 0) DSA_STAMP(3);
                if (go && lane < kPages) {  // one page per lane
                    int bp = it.blk[0];
#pragma unroll
                    for (int p = 1; p < kPages; ++p)
                        if (lane == p) bp = it.blk[p];
                    if (bp >= 0) tma_load_2d_hint(st + lane * kPage * DIM, &kmap, 0, bp * kPage, &full[s], key_policy);
                }
                alive = __shfl_sync(0xffffffffu, alive, 0);
                if (!alive) break;
                ++n;
                if (++ps == S) {
                    ps = 0;
                    pphase ^= 1;
                }
                if (++pb == NK) {
                    pb = 0;
                    pbph ^= 1;
                }
            }
            cur = nxt;
            base = nb;
            run_end = ne;
        }
        if (lane == 0) DSA_STAMP(4);
        if (!waited) {  // the kernel ends after the preceding kernel, whatever it read
            pdl_wait();
            pdl_launch_dependents();
            if (lane == 0) DSA_STAMP(17);
        }
        if (!a.withhold) {  // terminal item: consumers stop here (no bytes; 33 slot arrivals, 1 stage arrival)
            const int s = ps, b = pb;
            bool go = false;
            if (lane == 0 && alive) {
                go = wait_or_abort(&empty[s], pphase ^ 1, abort_flag, a.status, a.wait_ns) &&
                     wait_or_abort(&sempty[b], pbph ^ 1, abort_flag, a.status, a.wait_ns);
                if (go) slot_meta(b)->terminal = 1;
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (go) {
                mbar_arrive(&ifull[b]);
                if (lane == 0) {
                    mbar_arrive(&ifull[b]);
                    mbar_arrive(&full[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer: D[entry][q*heads + h] = <k8_entry, q8_(q,h)>, accumulated over dim; the warp
        // waits, one elected lane issues --------------------------------------------------------------
        const uint32_t idesc = idesc_f8(a.n_cols, a.key_e2m1 != 0);
        int prev_gb = -1, muse[2] = {0, 0};
        int s = 0, sph = 0, b = 0, bph = 0;  // stage / accumulator index and phase parity
        int k = 0, kph = 0;                  // item slot index and phase parity
        for (int n = 0;; ++n) {
            bool ok = wait_or_abort(&full[s], sph, abort_flag, a.status, a.wait_ns);
            ok = ok && wait_or_abort(&ifull[k], kph, abort_flag, a.status, a.wait_ns);
            ok = ok && wait_or_abort(&tempty[b], bph ^ 1, abort_flag, a.status, a.wait_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) DSA_TRACE(n, 1);
            if (slot_meta(k)->terminal) {
                if (lane == 0) mbar_arrive(&tfull[b]);
                break;
            }
            const int gbi = slot_meta(k)->gb;
            if (gbi != prev_gb) {  // the first item of a group: its buffer's load
                // decode-shaped groups: the previous group's buffer is free once its MMAs are complete
                if constexpr (N16)
                    if (prev_gb >= 0) mma_commit_elect(&gempty[prev_gb]);
                prev_gb = gbi;
                ++muse[gbi];
                ok = wait_or_abort(&gfull[gbi], (muse[gbi] - 1) & 1, abort_flag, a.status, a.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (lane == 0) DSA_TRACE(n, 6);
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + (size_t)s * a.stage_bytes);
            const uint32_t b_addr = smem_u32(gbase + (size_t)gbi * a.gbuf_bytes);
#pragma unroll
            for (int tt = 0; tt < TPI; ++tt)
#pragma unroll
                for (int ks = 0; ks < DIM / 32; ++ks)
                    mma_f8_elect(tmem + (b * TPI + tt) * a.n_cols, smem_desc(a_addr + tt * kTileEntries * DIM + ks * 32, DIM),
                                 smem_desc(b_addr + ks * 32, DIM), idesc, ks > 0 ? 1u : 0u);
            mma_commit_elect(&tfull[b]);
            mma_commit_elect(&empty[s]);  // the key tiles are free once these MMAs are done
            if (lane == 0) DSA_TRACE(n, 2);
            if (n == 0 && lane == 0) DSA_STAMP(5);
            if (++s == S) {
                s = 0;
                sph ^= 1;
            }
            if (++b == NA) {
                b = 0;
                bph ^= 1;
            }
            if (++k == NK) {
                k = 0;
                kph ^= 1;
            }
        }
    } else if constexpr (N16) {
        // ---- epilogue of decode-shaped groups (q_group * heads <= 16: one 16-column chunk): both tiles of an
        // item come out of TMEM under one wait, the group's folded weights stay in registers, and each entry's
        // score is a short sum over its query's heads ------------------------------------------------------
        constexpr int QPC = 16 / HEADS;  // queries per 16-column chunk
        const int quad = warp & 3;       // TMEM lanes this warp may access (EW == 4)
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        float u[16];              // w_c * sq_c of the group's columns (0 past its queries)
        float wr[16], sqr[16];    // w_c and sq_c (the literal formula of a group with a negative query scale)
        int nv[QPC];  // visible entries of each query of the group
        bool q_neg = false;
        int nqg = 0, q0 = 0;
        int prev_gb = -1, euse[2] = {0, 0};
        int b = 0, bph = 0;  // accumulator index and phase parity
        int k = 0, kph = 0;  // item slot index and phase parity
        for (int n = 0;; ++n) {
            bool ok = wait_or_abort(&ifull[k], kph, abort_flag, a.status, a.wait_ns);  // completed: orders the meta
            if (!__all_sync(0xffffffffu, ok)) break;
            const StageMeta* meta = slot_meta(k);
            if (meta->terminal) break;
            const int gbi = meta->gb;
            const bool new_group = gbi != prev_gb;
            if (new_group) {  // the group's values come into registers below, and the buffer is let go there
                prev_gb = gbi;
                ++euse[gbi];
                ok = wait_or_abort(&gfull[gbi], (euse[gbi] - 1) & 1, abort_flag, a.status, a.wait_ns);
            }
            if (tid == 64) DSA_TRACE(n, 5);
            ok = ok && wait_or_abort(&tfull[b], bph, abort_flag, a.status, a.wait_ns);
            if (!__all_sync(0xffffffffu, ok)) break;  // warp-uniform: tcgen05.ld is warp-collective
            if (tid == 64) DSA_TRACE(n, 3);
            tc_fence_after();
            float v0[16], v1[16];
            tmem_ld_nowait<16>(lane_base + (b * 2) * 16, v0);
            tmem_ld_nowait<16>(lane_base + (b * 2 + 1) * 16, v1);
            // while the loads are in flight: the group's weights, the entries' scales and pages
            if (new_group) {
                const uint8_t* gp = gbase + (size_t)gbi * a.gbuf_bytes;
                const float* sw = reinterpret_cast<const float*>(gp + 16 * DIM);
                const float* ssq = sw + 16;
                const int* gnv = reinterpret_cast<const int*>(gp + gbuf_nvis_offset(16, DIM));
                nqg = meta->nq;
                q0 = meta->q0;
                bool neg = false;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const bool live = c < nqg * HEADS;  // columns past the group's queries hold stale values
                    wr[c] = live ? sw[c] : 0.f;
                    sqr[c] = live ? ssq[c] : 0.f;
                    u[c] = wr[c] * sqr[c];
                    neg |= live && ssq[c] < 0.f;
                }
                q_neg = neg;
#pragma unroll
                for (int j = 0; j < QPC; ++j) nv[j] = j < nqg ? gnv[j] : 0;
                __syncwarp();
                if (lane == 0) mbar_arrive(&gempty[gbi]);  // this warp no longer reads the buffer
                if (tid == 64) DSA_TRACE(n, 7);
            }
            const float* sc = slot_scale(k);
            const int e0 = meta->e0;
            const bool ok0 = meta->blk[row / kPage] >= 0, ok1 = meta->blk[(kTileEntries + row) / kPage] >= 0;
            const float sk0 = ok0 ? sc[row] : 0.f, sk1 = ok1 ? sc[kTileEntries + row] : 0.f;
            tmem_wait_ld();
            tmem_regs_after_wait<16>(v0);
            tmem_regs_after_wait<16>(v1);
            auto emit = [&](const float (&x)[16], float sk, bool page_ok, int e) {
#pragma unroll
                for (int j = 0; j < QPC; ++j) {
                    if (j >= nqg) break;
                    float a0 = 0.f, a1 = 0.f;
                    if (!q_neg) {  // sk * sum_h u_h * (sk >= 0 ? max(x, 0) : min(x, 0)), two chains
#pragma unroll
                        for (int h = 0; h < HEADS; h += 2) {
                            const float x0 = x[j * HEADS + h], x1 = x[j * HEADS + h + 1];
                            a0 = fmaf(u[j * HEADS + h], sk >= 0.f ? fmaxf(x0, 0.f) : fminf(x0, 0.f), a0);
                            a1 = fmaf(u[j * HEADS + h + 1], sk >= 0.f ? fmaxf(x1, 0.f) : fminf(x1, 0.f), a1);
                        }
                        a0 = (a0 + a1) * sk;
                    } else {  // a negative query scale: the literal w_h * max(0, sq_h * sk * x_h)
#pragma unroll
                        for (int h = 0; h < HEADS; ++h) {
                            const int c = j * HEADS + h;
                            a0 = fmaf(wr[c], fmaxf(0.f, sqr[c] * sk * x[c]), a0);
                        }
                    }
                    if (e < a.ld) {
                        const bool vis = e < nv[j];
                        const float sv = (page_ok && vis) ? a0 : -INFINITY;
                        a.scores[(long long)(q0 + j) * a.ld + e] = sv;
                        // fused top-k: each visible entry's score also counted in its row's level-1 histogram
                        if (a.hist && vis)
                            atomicAdd(a.hist + (long long)(q0 + j) * kSelBins + (dsa_score_key(sv) >> 21), 1u);
                    }
                }
            };
            emit(v0, sk0, ok0, e0 + row);
            if (tid == 64) DSA_TRACE(n, 8);
            emit(v1, sk1, ok1, e0 + kTileEntries + row);
            tc_fence_before();
            if (tid == 64) DSA_TRACE(n, 4);
            mbar_arrive(&tempty[b]);
            mbar_arrive(&sempty[k]);
            if (tid == 64) {
                if (n == 0) DSA_STAMP(6);
                DSA_STAMP(7);
            }
            if (++b == NA) {
                b = 0;
                bph ^= 1;
            }
            if (++k == NK) {
                k = 0;
                kph ^= 1;
            }
        }
    } else {
        // ---- epilogue: TMEM lane <-> entry, one column slice per warp ----------------------------------
        // Per group the warp folds its columns' head weight and query scale, u_c = w_c * sq_c.  With
        // every sq_c >= 0:  w_c * max(0, sq_c * sk * x) = sk * u_c * (sk >= 0 ? max(x, 0) : min(x, 0)),
        // two instructions a column; a group with a negative query scale takes the literal formula.
        const int quad = warp & 3;  // TMEM lanes this warp may access
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const int nch = a.n_cols / 16, sl = (warp - 2) >> 2;
        const int ch_lo = sl * nch / NSL, ch_hi = (sl + 1) * nch / NSL;  // this warp's 16-column chunks
        float* fold = s_fold + (warp - 2) * kSlice;
        bool q_neg = false;
        int g_vis = 0;  // fewest visible entries over the group's queries
        int prev_gb = -1, euse[2] = {0, 0};
        int b = 0, bph = 0;  // accumulator index and phase parity
        int k = 0, kph = 0;  // item slot index and phase parity
        for (int n = 0;; ++n) {
            bool ok = wait_or_abort(&ifull[k], kph, abort_flag, a.status, a.wait_ns);  // completed: orders the meta
            if (!__all_sync(0xffffffffu, ok)) break;
            const StageMeta* meta = slot_meta(k);
            if (meta->terminal) break;

            const int gbi = meta->gb, nqg = meta->nq, q0 = meta->q0;
            const bool new_group = gbi != prev_gb;
            if (new_group) {  // this warp is done with the previous group's buffer
                if (prev_gb >= 0 && lane == 0) mbar_arrive(&gempty[prev_gb]);
                prev_gb = gbi;
                ++euse[gbi];
                ok = wait_or_abort(&gfull[gbi], (euse[gbi] - 1) & 1, abort_flag, a.status, a.wait_ns);
            }
            if (tid == 64) DSA_TRACE(n, 5);
            ok = ok && wait_or_abort(&tfull[b], bph, abort_flag, a.status, a.wait_ns);
            if (!__all_sync(0xffffffffu, ok)) break;  // warp-uniform: tcgen05.ld is warp-collective
            if (tid == 64) DSA_TRACE(n, 3);
            tc_fence_after();
            const uint8_t* gp = gbase + (size_t)gbi * a.gbuf_bytes;
            const float* sw = reinterpret_cast<const float*>(gp + a.n_cols * DIM);
            const float* ssq = sw + a.n_cols;
            const int* gnv = reinterpret_cast<const int*>(gp + gbuf_nvis_offset(a.n_cols, DIM));
            if (new_group) {
                bool neg = false;
                for (int c = ch_lo * 16 + lane; c < ch_hi * 16; c += 32) {
                    const bool live = c < nqg * HEADS;  // columns past the group's queries hold stale values
                    fold[c - ch_lo * 16] = live ? sw[c] * ssq[c] : 0.f;
                    neg |= live && ssq[c] < 0.f;
                }
                q_neg = __any_sync(0xffffffffu, neg);
                int vmin = INT_MAX;
                for (int j = lane; j < nqg; j += 32) vmin = min(vmin, gnv[j]);
                g_vis = __reduce_min_sync(0xffffffffu, vmin);
                __syncwarp();
                if (tid == 64) DSA_TRACE(n, 7);
            }
            // every entry of the item present and visible to every query of the group: unmasked stores
            bool clean = meta->e0 + kItem <= min(g_vis, a.ld);
#pragma unroll
            for (int p = 0; p < kPages; ++p) clean = clean && meta->blk[p] >= 0;
            const float* sscale = slot_scale(k);
#pragma unroll
            for (int tt = 0; tt < TPI; ++tt) {
                const int er = tt * kTileEntries + row;  // entry of the item
                const bool page_ok = meta->blk[er / kPage] >= 0;
                const float sk = page_ok ? sscale[er] : 0.f;
                const int e = meta->e0 + er;
                const bool e_ok = e < a.ld;
                float* out = a.scores + (long long)q0 * a.ld + e;
                const uint32_t tbase = lane_base + (b * TPI + tt) * a.n_cols;
                for (int cb = ch_lo; cb < ch_hi; cb += kBatch) {  // kBatch chunks per TMEM wait
                    // the loads and the wait are warp-collective: warp-uniform control flow only
                    float v[kBatch][16];
#pragma unroll
                    for (int k = 0; k < kBatch; ++k)
                        if (cb + k < ch_hi) tmem_ld_nowait<16>(tbase + (cb + k) * 16, v[k]);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) tmem_regs_after_wait<16>(v[k]);
                    // register arithmetic and stores only (lanes may take different sides of the branches):
                    // kNeg: the entry's key scale is negative, so min(x, 0) survives the ReLU; kLit: the group
                    // holds a negative query scale and takes the literal formula.  Each query's head sum runs
                    // as two independent chains and no branch separates the queries of a chunk; only the
                    // stores are predicated.
                    auto emit = [&](auto neg_tag, auto lit_tag, auto clean_tag) {
                        constexpr bool kNeg = decltype(neg_tag)::value, kLit = decltype(lit_tag)::value;
                        constexpr bool kClean = decltype(clean_tag)::value;
#pragma unroll
                        for (int k = 0; k < kBatch; ++k) {
                            if (cb + k >= ch_hi) break;  // warp-uniform
                            float acc[16 / HEADS];
#pragma unroll
                            for (int jj = 0; jj < 16 / HEADS; ++jj) {
                                const float* x = v[k] + jj * HEADS;
                                const int c0 = (cb + k) * 16 + jj * HEADS;  // first column of query jj
                                float a0 = 0.f, a1 = 0.f;
                                if constexpr (!kLit) {  // even and odd heads in the two lanes of one register
                                    const float4* u4 = reinterpret_cast<const float4*>(fold + c0 - ch_lo * 16);
                                    unsigned long long a2 = 0ull;
#pragma unroll
                                    for (int h4 = 0; h4 < HEADS / 4; ++h4) {
                                        const float4 u = u4[h4];
                                        const float* xh = x + 4 * h4;
                                        auto relu = [&](float t) { return kNeg ? fminf(t, 0.f) : fmaxf(t, 0.f); };
                                        fma_f32x2(a2, pack_f32x2(u.x, u.y), pack_f32x2(relu(xh[0]), relu(xh[1])));
                                        fma_f32x2(a2, pack_f32x2(u.z, u.w), pack_f32x2(relu(xh[2]), relu(xh[3])));
                                    }
                                    acc[jj] = sum_f32x2(a2) * sk;
                                } else {
#pragma unroll
                                    for (int h = 0; h < HEADS; h += 2) {
                                        a0 = fmaf(sw[c0 + h], fmaxf(0.f, ssq[c0 + h] * sk * x[h]), a0);
                                        a1 = fmaf(sw[c0 + h + 1], fmaxf(0.f, ssq[c0 + h + 1] * sk * x[h + 1]), a1);
                                    }
                                    acc[jj] = a0 + a1;
                                }
                            }
#pragma unroll
                            for (int jj = 0; jj < 16 / HEADS; ++jj) {
                                const int j = (cb + k) * (16 / HEADS) + jj;  // query of the group
                                // fused top-k: each visible entry's score also counted in its row's level-1 histogram
                                if constexpr (kClean) {
                                    if (j < nqg) {
                                        out[(long long)j * a.ld] = acc[jj];
                                        if (a.hist) atomicAdd(a.hist + (long long)(q0 + j) * kSelBins + (dsa_score_key(acc[jj]) >> 21), 1u);
                                    }
                                } else if (e_ok && j < nqg) {
                                    const float sv = (page_ok && e < gnv[j]) ? acc[jj] : -INFINITY;
                                    out[(long long)j * a.ld] = sv;
                                    if (a.hist && e < gnv[j])
                                        atomicAdd(a.hist + (long long)(q0 + j) * kSelBins + (dsa_score_key(sv) >> 21), 1u);
                                }
                            }
                        }
                    };
                    if (q_neg) emit(BoolTag<false>{}, BoolTag<true>{}, BoolTag<false>{});
                    else if (sk < 0.f) {
                        if (clean) emit(BoolTag<true>{}, BoolTag<false>{}, BoolTag<true>{});
                        else emit(BoolTag<true>{}, BoolTag<false>{}, BoolTag<false>{});
                    } else if (clean) {
                        emit(BoolTag<false>{}, BoolTag<false>{}, BoolTag<true>{});
                    } else {
                        emit(BoolTag<false>{}, BoolTag<false>{}, BoolTag<false>{});
                    }
                    __syncwarp();  // reconverge before the next collective load
                }
                if (tid == 64 && tt == 0) DSA_TRACE(n, 8);
            }
            tc_fence_before();
            if (tid == 64) DSA_TRACE(n, 4);
            mbar_arrive(&tempty[b]);
            mbar_arrive(&sempty[k]);
            if (tid == 64) {
                if (n == 0) DSA_STAMP(6);
                DSA_STAMP(7);
            }
            if (++b == NA) {
                b = 0;
                bph ^= 1;
            }
            if (++k == NK) {
                k = 0;
                kph ^= 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        DSA_STAMP(8);
        DSA_STAMP_NS(30);
        if (a.work) {  // every CTA has taken its last run: the last to finish leaves the counters zero
            __threadfence();
            if (atomicAdd(a.work + 1, 1u) == gridDim.x - 1) {
                atomicExch(a.work, 0u);
                atomicExch(a.work + 1, 0u);
            }
        }
    }
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

}  // namespace dsa
DSA_TIMELINE_SETTER(dsa_timeline_index)
namespace dsa {

// Tensor map of [rows][dim] 8-bit codes (or, e2m1, packed 4-bit codes unpacked to one per byte in shared
// memory: 16 codes of 8 bytes into 16 bytes) in boxes of box_rows rows, swizzled as the MMA operand wants.
static bool make_map(CUtensorMap* map, const void* base, uint64_t rows, int dim, int box_rows, bool e2m1 = false) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)dim, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)(e2m1 ? dim / 2 : dim)};
    cuuint32_t box[2] = {(cuuint32_t)dim, (cuuint32_t)box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult res = fn(map, e2m1 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                      const_cast<void*>(base), gdim, gstride, box, estride,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

template <int DIM, int HEADS, int TPI, bool N16>
static dsa_status_t launch_index(const CUtensorMap& kmap, const CUtensorMap& qmap, IdxArgs a, cudaStream_t st) {
    // stage = TPI key tiles; two group buffers of query codes + weights + query scales + per-query visible
    // entries; the item slots of metadata + entry scales
    a.stage_bytes = TPI * kTileEntries * DIM;  // a multiple of 1024 (the swizzle atom's alignment)
    a.gbuf_bytes = (gbuf_nvis_offset(a.n_cols, DIM) + 64 * 4 + 1023) / 1024 * 1024;
    a.items = (a.items + TPI - 1) / TPI;  // tiles -> items per group
    // alignment slack + group buffers + item slots + the epilogue warps' folded weights + barriers and flags
    // + the per-group prefix of valid items, requests and visible-entry bounds
    const int extra = 1024 + 2 * a.gbuf_bytes + item_slots<TPI>() * item_slot_bytes<TPI>() +
                      epi_warps<TPI>() * slice_cols<TPI>() * 4 + 448 + ((3 * a.n_groups + 1) * 4 + 15) / 16 * 16;
    // an SM holds 228 KB of shared memory, 1 KB of it reserved per resident CTA
    constexpr int kSmemPerSm = 228 * 1024, kReservedPerCta = 1024;
    const int two_cta_budget = kSmemPerSm / 2 - kReservedPerCta;
    const int ctas_per_sm = extra + 3 * a.stage_bytes <= two_cta_budget && 2 * a.tmem_cols <= 512 ? 2 : 1;
    const int budget = ctas_per_sm == 2 ? two_cta_budget : 227 * 1024;
    a.stages = max(2, min(8, (budget - extra) / a.stage_bytes));
    const int smem = extra + a.stages * a.stage_bytes;
    if (cudaFuncSetAttribute(index_kernel<DIM, HEADS, TPI, N16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return DSA_ERR_CUDA;
    a.total_items = (long long)a.items * a.n_groups;
    // Two CTAs per SM fill the GPU only if every SM is free: the compressor that the indexer follows (launched
    // programmatically, so still running on some SMs) leaves room for one indexer CTA there, and the CTAs that
    // did not fit started a compressor's duration late with a full static share (measured on the decode batch:
    // 16 of 304).  A fifth of the SMs' second slots is left out: every CTA starts at once, each with a share
    // a few percent larger (decode step 44.7 -> 43.6 us; leaving out 0, 8, 16, 24, 32 slots measured 44.7, 44.3,
    // 43.7, 43.9, 43.6 us).
    const long long slots = ctas_per_sm == 2 ? 2LL * sm_count() - sm_count() / 5 : (long long)sm_count();
    const long long grid = std::min<long long>(a.total_items, slots);
    if (launch_pdl(index_kernel<DIM, HEADS, TPI, N16>, dim3((unsigned)std::max<long long>(grid, 1)), dim3(idx_threads<TPI>()), smem,
                   st, kmap, qmap, a) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_status();
}

template <int DIM, int HEADS>
static dsa_status_t launch_index_tpi(const CUtensorMap& kmap, const CUtensorMap& qmap, const IdxArgs& a,
                                     cudaStream_t st) {
    if (a.n_cols == 16) return launch_index<DIM, HEADS, 2, true>(kmap, qmap, a, st);  // decode-shaped groups
    return a.n_cols <= 128 ? launch_index<DIM, HEADS, 2, false>(kmap, qmap, a, st)
                           : launch_index<DIM, HEADS, 1, false>(kmap, qmap, a, st);
}

template <int DIM>
static dsa_status_t launch_index_heads(const CUtensorMap& kmap, const CUtensorMap& qmap, const IdxArgs& a,
                                       cudaStream_t st) {
    switch (a.heads) {
        case 4: return launch_index_tpi<DIM, 4>(kmap, qmap, a, st);
        case 8: return launch_index_tpi<DIM, 8>(kmap, qmap, a, st);
        default: return launch_index_tpi<DIM, 16>(kmap, qmap, a, st);
    }
}

}  // namespace dsa

using namespace dsa;

static dsa_status_t index_scores(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8, const float* q_scale,
                                 const float* w, const int32_t* q_pos, const int32_t* q_req, int32_t q_group,
                                 const dsa_pool_t* keys, const dsa_block_table_t* bt, float* scores, int32_t ld,
                                 int32_t* n_visible, const int32_t* fresh_pos, uint32_t* work, int32_t* dev_status,
                                 void* stream, uint64_t wait_ns, int withhold, unsigned* hist = nullptr) {
    if (nq < 0 || ld < 0 || (ld & 3)) return DSA_ERR_INVALID_ARG;
    if (nq == 0) return DSA_OK;
    if (heads != 4 && heads != 8 && heads != 16) return DSA_ERR_UNSUPPORTED;
    if (dim != 64 && dim != 128) return DSA_ERR_UNSUPPORTED;
    if (q_group < 1 || q_group * heads > 256) return DSA_ERR_INVALID_ARG;
    if (!q8 || !q_scale || !w || !q_pos || !q_req || !scores || !keys || !bt || !bt->table || bt->max_blocks <= 0)
        return DSA_ERR_INVALID_ARG;
    if (!pool_ok(keys) || keys->dim != dim || keys->rows_per_block != kPage) return DSA_ERR_INVALID_ARG;
    if (keys->dtype == DSA_BF16 || (keys->dtype == DSA_FP4_E2M1 && dim != 128)) return DSA_ERR_UNSUPPORTED;
    if (!aligned(q8, 16) || !aligned(q_scale, 16) || !aligned(w, 16) || !aligned(work, 8)) return DSA_ERR_INVALID_ARG;
    if (q_group > 64) return DSA_ERR_INVALID_ARG;
    if ((nq + q_group - 1) / q_group > 4096) return DSA_ERR_UNSUPPORTED;  // per-group tables live in smem
    const int n_cols = ((q_group * heads + 15) / 16) * 16;  // M = 128 needs N % 16 == 0
    IdxArgs a{};
    a.nq = nq;
    a.heads = heads;
    a.q_group = q_group;
    a.n_cols = n_cols;
    const int tpi = n_cols <= 128 ? 2 : 1;  // 128-entry tiles per item (a stage)
    a.n_acc = tpi * n_cols <= 128 ? 4 : 2;  // TMEM accumulators in flight (at most 512 columns)
    a.tmem_cols = 32;
    while (a.tmem_cols < a.n_acc * tpi * n_cols) a.tmem_cols *= 2;
    a.ld = ld;
    a.q_scale = q_scale;
    a.w = w;
    a.q_pos = q_pos;
    a.q_req = q_req;
    a.fresh_pos = fresh_pos;
    a.work = work;
    a.key_scale = keys->scale;
    a.num_blocks = keys->num_blocks;
    a.bt = *bt;
    a.scores = scores;
    a.n_visible = n_visible;
    a.status = dev_status;
    a.wait_ns = wait_ns;
    a.withhold = withhold;
    a.hist = hist;
    a.key_e2m1 = keys->dtype == DSA_FP4_E2M1;
    CUtensorMap kmap, qmap;
    if (!make_map(&kmap, keys->data, (uint64_t)keys->num_blocks * kPage, dim, kPage, a.key_e2m1 != 0))
        return DSA_ERR_CUDA;
    if (!make_map(&qmap, q8, (uint64_t)nq * heads, dim, n_cols)) return DSA_ERR_CUDA;
    a.items = (ld + kTileEntries - 1) / kTileEntries;  // tiles per group; items once the launch picks TPI
    a.n_groups = (nq + q_group - 1) / q_group;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return dim == 128 ? launch_index_heads<128>(kmap, qmap, a, st) : launch_index_heads<64>(kmap, qmap, a, st);
}

extern "C" dsa_status_t dsa_index_scores(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8,
                                         const float* q_scale, const float* w, const int32_t* q_pos,
                                         const int32_t* q_req, int32_t q_group, const dsa_pool_t* keys,
                                         const dsa_block_table_t* bt, float* scores, int32_t ld, int32_t* n_visible,
                                         const int32_t* fresh_pos, uint32_t* work, int32_t* dev_status, void* stream) {
    return index_scores(nq, heads, dim, q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, ld, n_visible,
                        fresh_pos, work, dev_status, stream, kWaitLimitNs, 0);
}

// Test hook of the bounded waits: the same launch with a caller-chosen wait limit and the copy-issuing warp
// withholding every copy, so that the consumers' waits run out while nothing is in flight.
extern "C" dsa_status_t dsa_debug_index_scores_stalled(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8,
                                                       const float* q_scale, const float* w, const int32_t* q_pos,
                                                       const int32_t* q_req, int32_t q_group, const dsa_pool_t* keys,
                                                       const dsa_block_table_t* bt, float* scores, int32_t ld,
                                                       int32_t* n_visible, uint64_t wait_limit_ns, int32_t* dev_status,
                                                       void* stream) {
    if (wait_limit_ns == 0 || wait_limit_ns > kWaitLimitNs) return DSA_ERR_INVALID_ARG;
    return index_scores(nq, heads, dim, q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, ld, n_visible,
                        nullptr, nullptr, dev_status, stream, wait_limit_ns, 1);
}

// Fused indexer + top-k: the indexer counts each row's level-1 histogram while scoring (rows of up to 16,384
// entries), then the top-k of every row starts its radix select from it (dsa_topk_counted, topk.cu).  The
// counts are zero-filled by the caller before the first call and cleared again by the top-k of every call that
// completes.
// Workspace of dsa_index_topk: the level-1 counts [nq][2048], then the indexer's work counters [2].
static size_t counts_bytes(int32_t nq) { return ((size_t)nq * kSelBins * 4 + 255) / 256 * 256; }
extern "C" size_t dsa_index_topk_workspace_size(int32_t nq) { return nq > 0 ? counts_bytes(nq) + 256 : 0; }

extern "C" dsa_status_t dsa_index_scores_counted(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8,
                                                 const float* q_scale, const float* w, const int32_t* q_pos,
                                                 const int32_t* q_req, int32_t q_group, const dsa_pool_t* keys,
                                                 const dsa_block_table_t* bt, float* scores, int32_t ld,
                                                 int32_t* n_visible, const int32_t* fresh_pos, uint32_t* work,
                                                 unsigned* counts, int32_t* dev_status, void* stream) {
    if (nq < 0) return DSA_ERR_INVALID_ARG;
    if (nq == 0) return DSA_OK;
    if (!counts || !aligned(counts, 16) || ld > 16384) return DSA_ERR_INVALID_ARG;
    return index_scores(nq, heads, dim, q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, ld, n_visible,
                        fresh_pos, work, dev_status, stream, kWaitLimitNs, 0, counts);
}

extern "C" dsa_status_t dsa_index_topk(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8, const float* q_scale,
                                       const float* w, const int32_t* q_pos, const int32_t* q_req, int32_t q_group,
                                       const dsa_pool_t* keys, const dsa_block_table_t* bt, float* scores, int32_t ld,
                                       int32_t* n_visible, const int32_t* fresh_pos, int32_t k, int32_t* idx_out,
                                       void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (nq < 0) return DSA_ERR_INVALID_ARG;
    if (nq == 0) return DSA_OK;
    if (k < 1 || k > 2048 || !idx_out || !n_visible || !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < dsa_index_topk_workspace_size(nq)) return DSA_ERR_INVALID_ARG;
    unsigned* counts = static_cast<unsigned*>(workspace);
    uint32_t* work = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + counts_bytes(nq));
    if (ld > 16384) {  // rows the counted top-k does not hold: the plain indexer and top-k
        const dsa_status_t r = dsa_index_scores(nq, heads, dim, q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores,
                                                ld, n_visible, fresh_pos, work, dev_status, stream);
        return r != DSA_OK ? r : dsa_topk(nq, scores, ld, n_visible, k, idx_out, dev_status, stream);
    }
    const dsa_status_t r = dsa_index_scores_counted(nq, heads, dim, q8, q_scale, w, q_pos, q_req, q_group, keys, bt,
                                                    scores, ld, n_visible, fresh_pos, work, counts, dev_status, stream);
    return r != DSA_OK ? r : dsa_topk_counted(nq, scores, ld, n_visible, k, idx_out, counts, dev_status, stream);
}
