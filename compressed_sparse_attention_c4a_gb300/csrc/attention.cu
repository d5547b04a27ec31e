// dsa_sparse_attn_decode / dsa_sparse_attn_prefill: MQA attention over gathered top-k compressed
// entries plus the sliding window, K = V, with the inverse-RoPE epilogue fused into the store.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2-4.3: the main attention reads only
// the top-k entries, MQA-style (one latent entry serves every head); §5.3 and [P2] "DeepSeek V4
// 稀疏注意力完全解剖" 机制四: a 128-token window of uncompressed tokens is seen alongside; [P2] 机制一:
// K and V are one stored row; [P2] 深潜 (Inverse RoPE): out = R_m^-1 sum_j p_j k_j; [P2] 融合点 2:
// the inverse rotation is fused with the output store.
//
// Work split: see attn_cl_kernel below (a cluster of CTAs per query row, 32-key sub-tiles, tcgen05 MMAs
// with TMEM accumulators, on-chip merge).  When one cluster per row cannot fill the GPU, a row's keys are
// split over several clusters; each writes an unnormalised partial (O, max, the two sums) and
// attn_combine_kernel merges them and applies the inverse rotation.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "topk_cluster.cuh"

namespace dsa {

constexpr int kD = 512;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
    int rows, heads, hg_count, nsplit, cps;   // cps = 32-key sub-tiles per split
    const uint16_t* q;
    const int32_t* q_pos;
    const int32_t* q_req;                     // NULL: row r belongs to request r
    int kind_w, kind_s;
    const int32_t* topk;                      // NULL: every visible entry
    int k;
    dsa_pool_t main;
    dsa_block_table_t main_bt;
    dsa_pool_t swa;
    dsa_block_table_t swa_bt;
    int window;
    float scale_log2;                         // sm_scale * log2(e)
    RopeTable rope;
    uint16_t* out;                            // bf16 output, or NULL with out8
    uint8_t* out8;                            // e4m3 output [rows][heads][512] (with out_scale), or NULL
    float* out_scale;                         // [rows][heads][4]: amax / 448 of each 128-dim block
    float* lse;
    float* ws_o;                              // [rows][nsplit][heads][512]
    float* ws_ml;                             // [rows][nsplit][heads][4]: M, L (bf16 P), E (fp32 P), 0
    const float* scores;                      // fused top-k: indexer scores [rows][score_ld]
    int score_ld;
    const int32_t* n_valid;                   // fused top-k: [rows] valid scores of a row
    int32_t* topk_out;                        // fused top-k: the selected entries [rows][k]
    int32_t* status;
};

// ---- PTX wrappers ---------------------------------------------------------------------
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src), "r"(src_bytes),
                 "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)float_to_bf16(lo) | ((uint32_t)float_to_bf16(hi) << 16);
}
// {lo, hi} -> bf16x2 in one conversion (round to nearest even, as pack_bf16), lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// 2^x on the special-function unit (PTX ex2.approx.ftz: a few ulp, 2^-inf = 0); for softmax
// probabilities, which enter the product rounded to bf16.
__device__ __forceinline__ float ex2_sfu(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge split partials of one (row, head): 128 threads x 4 dims; inverse RoPE; bf16 store.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int row = blockIdx.x / a.heads, head = blockIdx.x % a.heads;
    const int tid = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < a.nsplit; ++sp)
        M = fmaxf(M, a.ws_ml[(((long long)row * a.nsplit + sp) * a.heads + head) * 4]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float Ls = 0.f, Es = 0.f;
    bool fault = false;
    for (int sp = 0; sp < a.nsplit; ++sp)
        fault |= a.ws_ml[(((long long)row * a.nsplit + sp) * a.heads + head) * 4 + 3] != 0.f;
    for (int sp = 0; sp < a.nsplit && !fault; ++sp) {
        const long long b = ((long long)row * a.nsplit + sp) * a.heads + head;
        const float ms = a.ws_ml[b * 4], ls = a.ws_ml[b * 4 + 1], es = a.ws_ml[b * 4 + 2];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        Ls += f * ls;
        Es += f * es;
        const float4 v = *reinterpret_cast<const float4*>(a.ws_o + b * kD + tid * 4);
        acc[0] += f * v.x;
        acc[1] += f * v.y;
        acc[2] += f * v.z;
        acc[3] += f * v.w;
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] *= inv;
    const int first = kD - a.rope.rope_dim;
    const int m = a.q_pos[row];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
        const int col = tid * 4 + e;
        if (col >= first) {
            float cs, sn;
            rope_cos_sin(m, a.rope, (col - first) >> 1, &cs, &sn);
            const float x0 = acc[e], x1 = acc[e + 1];
            acc[e] = x0 * cs + x1 * sn;
            acc[e + 1] = -x0 * sn + x1 * cs;
        }
    }
    if (a.out8) {  // e4m3 with one scale per 128-dim block: a warp holds one block
        float am = fmaxf(fmaxf(fabsf(acc[0]), fabsf(acc[1])), fmaxf(fabsf(acc[2]), fabsf(acc[3])));
        am = warp_max(am);
        const float sc = am > 0.f ? am / 448.f : 1.f;
        uint32_t c = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) c |= (uint32_t)float_to_e4m3(acc[e] / sc) << (8 * e);
        *reinterpret_cast<uint32_t*>(a.out8 + ((long long)row * a.heads + head) * kD + tid * 4) = c;
        if ((tid & 31) == 0) a.out_scale[((long long)row * a.heads + head) * 4 + tid / 32] = sc;
    } else {
        uint16_t* dst = a.out + ((long long)row * a.heads + head) * kD + tid * 4;
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
    }
    if (a.lse && tid == 0)
        a.lse[(long long)row * a.heads + head] = Es > 0.f ? (M + log2f(Es)) / kLog2e : -INFINITY;
}

// ---------------------------------------------------------------------------------------------
// bf16 rows on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// Work split.  A row's keys (top-k entries, then window positions) form 32-key sub-tiles.  One
// cluster of CL CTAs (CL = 1, 2 or 4, chosen at launch) serves one (query row, group of NH <= 64 heads,
// key split); CTA c of the cluster takes the split's sub-tiles c, c + CL, c + 2 CL, ...  Each CTA keeps
// its partial softmax state on chip, and the cluster merges the CL partials through distributed
// shared memory, so a split-K workspace in global memory is needed only when one cluster per row is
// not enough to fill the GPU (several splits per row, merged by attn_combine_kernel).
//
// Inside a CTA (512 threads), warp-specialised and pipelined over four 32 KB key stages (a stage is
// gathered again as soon as its sub-tile's P V is done, so up to three gathers run ahead of the math):
//   warps 4 + MW .. 15 gather (MW MMA warps below: 2 for bf16 rows, 4 for e4m3 rows): resolve keys a round
//              (one sub-tile per gather warp) ahead (top-k index -> block table ->
//              physical row, tables cached in shared memory) and copy
//              the rows into a stage with cp.async, 128B-swizzled, laid out [64-dim chunk][32 keys]
//              [128 B]; e4m3 rows are converted to bf16 on the way, their scales kept beside the stage.
//              Decode rows are gathered with an evict-first L2 policy (each serves one query row).
//              No L2 prefetch of rows ahead of their copy: measured, it cost more (the prefetches queue
//              in front of the copies that are needed first) than the early arrival saved;
//   warps 4 .. 3 + MW issue the MMAs, one elected lane each (an MMA's issue costs the issuing warp about
//              49 cycles at these shapes, so MW warps issue MW times as fast as one, up to the tensor pipe's
//              own rate at M = 64); warp 4 also loads the query rows (TMA, one 64-dim box per lane):
//              S   = Q K^T   : M = 64 (heads), N = 32 keys, K = 512 split in MW parts, warp 4 + q summing
//                              dims (512 / MW) q .. into its own accumulator (TMEM lanes = heads,
//                              columns = keys); the softmax adds the MW partial sums;
//              O^T += V^T P^T: M = 128 dims per MMA (the stage read MN-major, K = V), N = NH heads,
//                              K = 32 keys; four 128-dim accumulators, 4 / MW tiles per MMA warp;
//              S of sub-tile i + 1 is issued before O^T of sub-tile i, so it overlaps the softmax;
//   warps 0-3  softmax, one thread per head (lanes 0-15 of each quadrant hold the M = 64 rows): the
//              32 logits of a sub-tile are a row of TMEM, so max and sum are thread-local; P is
//              written as the head's row of the P^T operand (two buffers).  The running maximum is
//              lazy: it moves (and O^T is rescaled in TMEM) only when a sub-tile's maximum exceeds it
//              by more than 2^8, so exp2(s - m) <= 2^8 stays exact in fp32 and rescales are rare.
// Merge (tile t of the 4 128-dim tiles of O^T belongs to CTA t mod CL): as soon as its own products are
// done, each CTA writes the tiles other CTAs own, unscaled, as bf16 into its idle query rows, and sends
// (m, l, e) per head to every CTA of the cluster; after one cluster barrier it pushes those tiles into
// the owners' idle key stages (bulk copies).  The owner weighs each CTA's partial by 2^(m_c - M) (M the
// cluster maximum), divides by L and applies R_m^-1 (pairs of dims sit in neighbouring lanes) before the
// bf16 store, or writes an fp32 partial with (M, L) when the row has several splits.
// ---------------------------------------------------------------------------------------------
constexpr int kClKeys = 32;                 // keys per sub-tile
constexpr int kClStages = 4;                // key stages in flight (a stage is free again after its P V)
constexpr int kClThreads = 512;             // 16 warps: 4 softmax, MW issuing MMAs, the rest gathering
// Warp roles for MW MMA-issuing warps (4 .. 3 + MW); the gather warps follow.  bf16 rows take MW = 2 (the
// gather, ten warps strong, sets the pace); e4m3 rows, half the bytes, MW = 4 (the MMA issue sets it).
template <int MW>
struct ClRoles {
    static constexpr int kMma = MW;
    static constexpr int kFirstGather = 4 + MW;
    static constexpr int kGatherWarps = 16 - kFirstGather;
    static constexpr int kGatherThreads = 32 * kGatherWarps;
    static constexpr int kRound = kGatherThreads / kClKeys;  // sub-tiles resolved per round
    static constexpr int kRing = 2 * kRound;                 // resolved sub-tiles kept
};
constexpr int kClRingMax = ClRoles<2>::kRing;
constexpr int kClStage = kClKeys * kD * 2;
static_assert(kClKeys == 32, "one 32-bit key mask and 32 S columns per sub-tile");
static_assert(kClThreads == 512, "16 warps");
constexpr float kLazyLog2 = 8.f;            // the running maximum moves when exceeded by more than this
constexpr int kBtCache = 1024;              // main block tables up to this many blocks are cached in shared memory
constexpr int kFusedK = 512;                // the fused top-k + attention kernel: k up to this
constexpr int kFusedVpt = 8;                // ... scores per thread: rows up to 4 * 512 * 8 = 16,384 entries

template <int NH>
struct ClSmem {
    static constexpr int kQ = 64 * kD * 2;                          // [8][64 rows][128 B]
    static constexpr int kP = NH * 64 * 2;                          // [NH rows][128 B]: keys 0 .. 31 of 64 used
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQ;                        // key stages; received tiles
    static constexpr int kOffP = kOffK + kClStages * kClStage;      // two P^T buffers; output staging at the end
    static constexpr int kOffRow = kOffP + 2 * kP;                  // int [ring][32]: physical rows (-1 masked)
    static constexpr int kOffPool = kOffRow + kClRingMax * kClKeys * 4;  // uint8 [ring][32]: 1 main, 2 window
    static constexpr int kOffKsc = kOffPool + kClRingMax * kClKeys;    // float [stages + 2][32]: e4m3 row scales
    static constexpr int kOffMask = kOffKsc + (kClStages + 2) * kClKeys * 4;  // uint32 [stages]: valid keys of a stage
    static constexpr int kOffAlpha = kOffMask + (kClStages * 4 + 15) / 16 * 16;  // float [2][NH]
    static constexpr int kOffVote = kOffAlpha + 2 * NH * 4;         // int [2][4]
    static constexpr int kOffOwn = kOffVote + 32;                   // float m[NH], l[NH], e[NH] of this CTA
    static constexpr int kOffStat = kOffOwn + 3 * NH * 4;           // float [4 ranks][NH][4]: (m, l, e, fault)
    static constexpr int kOffFac = kOffStat + 4 * NH * 16;          // float f[4 ranks][NH], 1/L, M, L, E [NH]
    static constexpr int kOffBt = kOffFac + 8 * NH * 4;             // int [kBtCache]: the request's main block table
    static constexpr int kOffSwb = kOffBt + kBtCache * 4;           // int [8]: window-pool blocks from that of wlo
    static constexpr int kOffFault = kOffSwb + 32;                  // int: a key of this CTA hit a device fault
    static constexpr int kOffRope = kOffFault + 16;                 // float [32][2]: cos, sin of each pair's angle at m
    static constexpr int kBars = 2 * kClStages + 8;
    static constexpr int kOffBar = kOffRope + 256;                  // kBars mbarriers, TMEM address
    static constexpr int kOffTopk = kOffBar + kBars * 8 + 16;       // int [kFusedK]: the row's top-k (fused)
    static constexpr int kBytes = kOffTopk + kFusedK * 4;
    static constexpr int kAlloc = kBytes + 1024;                    // + alignment slack
    static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
    static_assert(kOffKsc % 16 == 0, "the row scales are read as float4");
    // every region starts on a 16-byte boundary (float4 reads, 8-byte mbarriers), whatever the stage count
    static_assert(kOffAlpha % 16 == 0 && kOffVote % 16 == 0 && kOffOwn % 16 == 0 && kOffStat % 16 == 0 &&
                      kOffFac % 16 == 0 && kOffBt % 16 == 0 && kOffSwb % 16 == 0 && kOffFault % 16 == 0 &&
                      kOffRope % 16 == 0 && kOffBar % 16 == 0 && kOffTopk % 16 == 0,
                  "shared-memory regions 16-byte aligned");
    static constexpr int kTile = 128 * NH * 2;                      // one exchanged 128-dim O tile: [NH / 4][128] x 4 bf16
    static_assert(3 * kTile <= kQ, "the sent tiles fit in the query rows");
    static_assert(6 * kTile <= kQ + kClStages * kClStage, "the received tiles fit after them");
    static_assert(NH * 128 * 2 <= 2 * kP, "an output tile must fit in the P^T buffers");
    static constexpr int kTmemCols = 512;  // S: [2 buffers][4 parts][32 keys]; O^T: [4 tiles][NH heads]
};

// Byte offset of element (row r, element e) in a tile of 128B-swizzled atoms whose rows are 128 bytes
// (64 bf16) long: atoms of 8 rows are 1024 bytes apart, 64-element chunks `chunk_stride` apart.
__device__ __forceinline__ uint32_t sw128_offset(int r, int e, int chunk_stride) {
    const int c = e >> 6, in = e & 63;
    return (uint32_t)(c * chunk_stride + (r >> 3) * 1024 + (r & 7) * 128 + ((((in >> 3) ^ (r & 7))) << 4) +
                      ((in & 7) << 1));
}

// Keys of a row for the tensor-core kernel: [0, n_comp) compressed slots, [n_comp, ncp) padding up to a
// multiple of 4, [ncp, ncp + window count) window positions.

template <int NH, bool FP8, bool FUSED>
__global__ void __launch_bounds__(kClThreads, 1)
    attn_cl_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap, AttnArgs a) {
    using L = ClSmem<NH>;
    using Ro = ClRoles<FP8 ? 4 : 2>;
    // bf16 key stages: four for bf16 rows; three for e4m3 rows, whose codes land in a ring of two raw slots
    // (16 KB each, the fourth stage's space) and are widened into a stage once its previous product is done
    constexpr int NS = FP8 ? kClStages - 1 : kClStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem + L::kOffQ), sK = smem_u32(smem + L::kOffK), sP = smem_u32(smem + L::kOffP);
    int* s_row = reinterpret_cast<int*>(smem + L::kOffRow);
    uint8_t* s_pool = smem + L::kOffPool;
    float* s_ksc = reinterpret_cast<float*>(smem + L::kOffKsc);
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + L::kOffMask);
    float* s_alpha = reinterpret_cast<float*>(smem + L::kOffAlpha);
    int* s_vote = reinterpret_cast<int*>(smem + L::kOffVote);
    float* s_own = reinterpret_cast<float*>(smem + L::kOffOwn);
    float* s_stat = reinterpret_cast<float*>(smem + L::kOffStat);
    float* s_fac = reinterpret_cast<float*>(smem + L::kOffFac);  // [4][NH]: weight of each CTA's partial
    float* s_inv = s_fac + 4 * NH;
    float* s_M = s_inv + NH;
    float* s_L = s_M + NH;
    float* s_E = s_L + NH;
    // sub-tile i: key stage i % NS; S columns, P^T buffer and softmax scratch i & 1
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);  // [stages] stage gathered (gather threads)
    uint64_t* sfull = full + kClStages;                                 // [2] S in TMEM (both MMA warps' commits)
    uint64_t* pfull = sfull + 2;                                        // [2] P^T written (4 warps)
    uint64_t* pvdone = pfull + 2;                                       // [stages] O^T += V^T P^T done (2 commits)
    uint64_t* qfull = pvdone + kClStages;                               // query rows loaded
    uint64_t* xfull = qfull + 1;                                        // [3] each received tile slot loaded
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(xfull + 3);
    volatile int* s_fault = reinterpret_cast<volatile int*>(smem + L::kOffFault);
    float* s_rc = reinterpret_cast<float*>(smem + L::kOffRope);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int crank = (int)cluster_ctarank(), csize = (int)cluster_nctarank();
    const int cid = blockIdx.x / csize;
    const int split = cid % a.nsplit;
    const int hg = (cid / a.nsplit) % a.hg_count;
    const int row = cid / (a.nsplit * a.hg_count);
    if (tid == 0) {
        DSA_STAMP_NS(31);
        DSA_STAMP(0);
        for (int b = 0; b < kClStages; ++b) {
            mbar_init(&full[b], Ro::kGatherThreads);
            mbar_init(&pvdone[b], Ro::kMma);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sfull[b], Ro::kMma);
            mbar_init(&pfull[b], 4);
        }
        mbar_init(qfull, 1);
        for (int b = 0; b < 3; ++b) mbar_init(&xfull[b], 1);
        *s_fault = 0;
        fence_barrier_init();
    }
    if constexpr (NH < 64)  // the S product reads 64 query rows: rows NH.. are zero
        for (int i = tid; i < 8 * (64 - NH) * 8; i += kClThreads) {
            const int c = i / ((64 - NH) * 8), rr = NH + (i / 8) % (64 - NH), u = i % 8;
            *reinterpret_cast<uint4*>(smem + L::kOffQ + c * 8192 + rr * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
    fence_proxy_async_smem();
    if (warp == 0) tmem_alloc(s_tmem, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tS = tmem, tO = tmem + 2 * Ro::kMma * kClKeys;  // S: [2 buffers][MW parts][32]; O^T: [4][NH]
    if (tid == 0) DSA_STAMP(1);
    if (csize > 1) cluster_arrive_relaxed();  // phase 0: this CTA has started (waited on before DSMEM use)

    // The row's position, request and block tables, and the query rows: inputs that no kernel of the layer
    // step writes, read while the preceding kernel (the top-k) finishes.  Top-k indices, cache rows and
    // every output come after the programmatic-dependent-launch wait.
    const int r = a.q_req ? a.q_req[row] : row;
    // the gather threads' share of the request's main block table (when it has at most kBtCache blocks): its
    // loads, which need only the request, are in flight with the position's and are stored in shared memory
    // later (after the wait, unless the kernel selects its own top-k first)
    const bool bt_cached = a.main_bt.max_blocks <= kBtCache;
    constexpr int kBtPer = (kBtCache + Ro::kGatherThreads - 1) / Ro::kGatherThreads;
    int btv[kBtPer];
    if (warp >= Ro::kFirstGather) {
        const bool r_in = bt_cached && r >= 0 && r < a.main_bt.batch;
#pragma unroll
        for (int u = 0; u < kBtPer; ++u) {
            const int b = tid - 32 * Ro::kFirstGather + u * Ro::kGatherThreads;
            btv[u] = r_in && b < a.main_bt.max_blocks ? __ldg(a.main_bt.table + (long long)r * a.main_bt.max_blocks + b) : -1;
        }
    }
    const int m = a.q_pos[row];
    const bool row_ok = r >= 0 && r < a.main_bt.batch && r < a.swa_bt.batch && m >= 0;
    if (!row_ok && tid == 0) *s_fault = 1;
    const int n_vis = row_ok ? entries_formed((long long)m + 1, a.kind_w, a.kind_s) : 0;
    const int n_comp = (FUSED || a.topk) ? a.k : n_vis;
    const int ncp = (n_comp + 3) & ~3;
    const int wlo = max(0, m - a.window + 1);
    const int n_keys = row_ok ? ncp + (m - wlo + 1) : 0;
    const int n_sub = (n_keys + kClKeys - 1) / kClKeys;
    const int g_lo = split * a.cps, g_hi = min(n_sub, g_lo + a.cps);
    const int n_mine = g_hi > g_lo + crank ? (g_hi - g_lo - crank + csize - 1) / csize : 0;
    int* s_bt = reinterpret_cast<int*>(smem + L::kOffBt);
    int* s_swb = reinterpret_cast<int*>(smem + L::kOffSwb);
    if (warp == 0 && lane < a.rope.rope_dim / 2) {  // R_m^-1 of the output: cos and sin of each pair's angle at m
        float c = 1.f, sn = 0.f;
        if (row_ok) rope_cos_sin(m, a.rope, lane, &c, &sn);
        s_rc[2 * lane] = c;
        s_rc[2 * lane + 1] = sn;
    }
    if (warp == 4 && n_mine > 0) {  // the query rows, one 64-dim box per lane
        if (lane == 0) mbar_expect_tx(qfull, NH * kD * 2);
        __syncwarp();
        if (lane < kD / 64) tma_load_2d(smem + L::kOffQ + lane * 8192, &qmap, lane * 64, row * a.heads + hg * NH, qfull);
        __syncwarp();
        if (lane == 0) mbar_arrive(qfull);
    }
    const int gt = tid - 32 * Ro::kFirstGather, gw = warp - Ro::kFirstGather;
    // the cached tables: the main block table (above) and the window pool's blocks of positions wlo .. m; a
    // key then resolves with one global load (its top-k index) at most.  Published by the caller's barrier.
    int swbv = -1;
    if (warp >= Ro::kFirstGather && gt < 8 && n_mine > 0) {
        const int lb = wlo / kBlockPositions + gt;
        if (row_ok && lb <= m / kBlockPositions && lb < a.swa_bt.max_blocks)
            swbv = __ldg(a.swa_bt.table + (long long)r * a.swa_bt.max_blocks + lb);
    }
    auto store_tables = [&]() {
        if (bt_cached)
#pragma unroll
            for (int u = 0; u < kBtPer; ++u) {
                const int b = gt + u * Ro::kGatherThreads;
                if (b < a.main_bt.max_blocks) s_bt[b] = btv[u];
            }
        if (gt < 8) s_swb[gt] = swbv;
    };
    if constexpr (FUSED) {
        if (warp >= Ro::kFirstGather && n_mine > 0) {
            store_tables();
            named_bar_sync(1, Ro::kGatherThreads);  // cached tables visible to every gather thread
        }
    }
    pdl_wait();  // global memory the preceding kernel writes, and every output, only below
    pdl_launch_dependents();
    if (tid == 0) DSA_STAMP(2);
    if (!row_ok && tid == 0 && crank == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
    int* s_topk = reinterpret_cast<int*>(smem + L::kOffTopk);
    if constexpr (FUSED) {
        // The row's top-k of the indexer scores on this cluster (one cluster of four CTAs per row), every
        // selected entry written into each CTA's s_topk (and topk_out); its scratch is the key stages, idle
        // until the gather below.  Its first cluster barrier completes phase 0 (every CTA has started).
        cg::cluster_group cluster = cg::this_cluster();
        cluster_wait();
        auto& ts = *reinterpret_cast<TopkRowScratch<kClThreads, kFusedVpt, 4>*>(smem + L::kOffK);
        int32_t* tout = a.topk_out + (long long)row * a.k;
        auto emit = [&](int pos, int idx) {
#pragma unroll
            for (int c = 0; c < 4; ++c) *cluster.map_shared_rank(s_topk + pos, c) = idx;
            tout[pos] = idx;
        };
        const int nv_row = a.n_valid[row];  // the same in every CTA of the cluster
        if (nv_row < 0 || nv_row > a.score_ld) {
            if (tid == 0 && crank == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
            for (int i = crank * kClThreads + tid; i < a.k; i += 4 * kClThreads) emit(i, -1);
        } else {
            topk_row_cluster<kClThreads, kFusedVpt, 4>(cluster, ts, a.scores + (long long)row * a.score_ld, nv_row,
                                                       a.k, emit, a.status, 23);
        }
        cluster.sync();  // every CTA's s_topk complete; the scratch (key stages) no longer read by a peer
    }
    bool ok = true;

    if (warp >= Ro::kFirstGather) {
        // ---- gather warps: resolve keys a round ahead, copy with cp.async ----------------------------
        // decode rows (one query row per request): a gathered row serves this query row only and leaves L2 first;
        // prefill rows of one request share their keys, which keep the default policy
        const uint64_t row_policy = a.q_req ? l2_evict_normal() : l2_evict_first();
        // sub-tiles [R * Ro::kRound, (R + 1) * Ro::kRound): thread -> sub-tile R * Ro::kRound + gt / 32, key gt % 32.
        // Step 1: the key's top-k index (or entry / window position), no dependent load.
        auto key_id = [&](int R, int* id) -> int {  // returns j (the key's index in the row), -1 if none
            const int i = R * Ro::kRound + gt / kClKeys;
            if (gt >= Ro::kRound * kClKeys || i >= n_mine) return -1;
            const int j = (g_lo + crank + csize * i) * kClKeys + gt % kClKeys;
            *id = -1;
            if (j < n_keys && j < n_comp) *id = FUSED ? s_topk[j] : (a.topk ? __ldg(a.topk + (long long)row * a.k + j) : j);
            return j;
        };
        // Step 2: index -> physical row through the cached tables (or global memory), ring slot.
        auto finish_key = [&](int R, int j, int id) {
            const int i = R * Ro::kRound + gt / kClKeys;
            if (j < 0) return;
            int v = -1, pool = 1;
            if (j < ncp) {
                if (j < n_comp && id >= 0) {
                    if (id >= n_vis) {
                        report(a.status, DSA_ERR_DEVICE_FAULT);
                        *s_fault = 1;
                    } else {
                        const int epb = a.main.rows_per_block;
                        const int lb = id / epb;
                        const int pb = lb < a.main_bt.max_blocks && (!bt_cached || DSA_IDX_OK(lb, kBtCache, a.status))
                                           ? (bt_cached ? s_bt[lb] : __ldg(a.main_bt.table + (long long)r * a.main_bt.max_blocks + lb))
                                           : -1;
                        if (pb < 0 || pb >= a.main.num_blocks) {
                            report(a.status, DSA_ERR_DEVICE_FAULT);
                            *s_fault = 1;
                        } else {
                            v = pb * epb + (id - lb * epb);
                        }
                    }
                }
            } else if (j < n_keys) {
                pool = 2;
                const int pos = wlo + (j - ncp);
                const int lb = pos / kBlockPositions;
                const int sb = lb - wlo / kBlockPositions;  // the window (<= 1024 positions) spans <= 5 blocks
                const int pb = DSA_IDX_OK(sb, 8, a.status) ? s_swb[sb] : -1;
                if (pb < 0 || pb >= a.swa.num_blocks) {
                    report(a.status, DSA_ERR_DEVICE_FAULT);
                    *s_fault = 1;
                } else {
                    v = pb * kBlockPositions + (pos - lb * kBlockPositions);
                }
            }
            s_row[(i % Ro::kRing) * kClKeys + gt % kClKeys] = v;
            s_pool[(i % Ro::kRing) * kClKeys + gt % kClKeys] = (uint8_t)pool;
        };
        auto resolve_round = [&](int R) {
            int id = -1;
            const int j = key_id(R, &id);
            finish_key(R, j, id);
        };
        // e4m3 rows of sub-tile j (landed in raw slot j & 1) -> bf16 in key stage j % NS, exactly (e4m3 -> fp16 ->
        // fp32 -> bf16 loses nothing), with the rows' scales and the stage's key mask, once the stage's previous
        // product (sub-tile j - NS) is done; then the stage is reported full.  Called by all gather threads
        // alike, after each has waited for its own copies of sub-tile j.
        auto widen_fp8 = [&](int j) {
            constexpr int kRowsPerWarp = (kClKeys + Ro::kGatherWarps - 1) / Ro::kGatherWarps;
            const int st = j % NS;
            const uint32_t stage = sK + st * kClStage;
            const uint8_t* raw = smem + L::kOffK + NS * kClStage + (j & 1) * (kClStage / 2);
            named_bar_sync(1, Ro::kGatherThreads);  // every thread's copies of the sub-tile have landed
            if (j >= NS) ok = ok && mbar_wait_bounded(&pvdone[st], ((j - NS) / NS) & 1, kWaitLimitNs);
            if (gt < kClKeys) {  // the first gather warp (whole): the stage's row scales and key mask
                if (ok) s_ksc[st * kClKeys + gt] = s_ksc[(kClStages + (j & 1)) * kClKeys + gt];
                const uint32_t bits = __ballot_sync(0xffffffffu, s_row[(j % Ro::kRing) * kClKeys + gt] >= 0);
                if (ok && lane == 0) s_mask[st] = bits;
            }
#pragma unroll
            for (int u = 0; u < kRowsPerWarp; ++u) {
                const int kk = gw + u * Ro::kGatherWarps;
                if (ok && kk < kClKeys) {
                    const uint4 code = *reinterpret_cast<const uint4*>(raw + kk * kD + lane * 16);
                    const uint32_t w4[4] = {code.x, code.y, code.z, code.w};
                    uint32_t bf[8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
#pragma unroll
                        for (int hlf = 0; hlf < 2; ++hlf) {
                            const __half2_raw h2 =
                                __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w4[q] >> (16 * hlf)), __NV_E4M3);
                            const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&h2));
                            bf[2 * q + hlf] = pack_bf16(f2.x, f2.y);
                        }
                    }
                    const int d0 = 16 * lane;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + sw128_offset(kk, d0, kClKeys * 128)),
                                 "r"(bf[0]), "r"(bf[1]), "r"(bf[2]), "r"(bf[3])
                                 : "memory");
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + sw128_offset(kk, d0 + 8, kClKeys * 128)),
                                 "r"(bf[4]), "r"(bf[5]), "r"(bf[6]), "r"(bf[7])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();  // the bf16 rows -> visible to the tensor core (async proxy)
            mbar_arrive(&full[st]);
            if (gt == 0) DSA_TRACE(j, 1);
        };
        if constexpr (FUSED) {
            if (n_mine > 0) resolve_round(0);
        } else if (n_mine > 0) {
            // the first round's top-k indices requested before the cached tables are stored, so that both
            // loads' latencies overlap (a CTA that starts after the top-k has ended waits for neither alone)
            int id0 = -1;
            const int j0 = key_id(0, &id0);
            store_tables();
            named_bar_sync(1, Ro::kGatherThreads);  // cached tables visible to every gather thread
            finish_key(0, j0, id0);
        }
        int sig = 0;  // first sub-tile whose stage this thread has not yet reported full
        if constexpr (!FP8) {
            for (int i = 0; i < n_mine; ++i) {
                const int s = i % NS;
                if (i >= NS) {
                    // before waiting for a stage, report every sub-tile issued so far (never hold landed rows back)
                    if (sig < i) {
                        cp_async_wait_all();
                        for (; sig < i; ++sig) {
                            fence_proxy_async_smem();  // cp.async writes -> visible to the tensor core (async proxy)
                            mbar_arrive(&full[sig % NS]);
                            if (gt == 0) DSA_TRACE(sig, 1);
                        }
                    }
                    // the stage's previous sub-tile has been multiplied into O^T
                    ok = ok && mbar_wait_bounded(&pvdone[s], ((i - NS) / NS) & 1, kWaitLimitNs);
                }
                named_bar_sync(1, Ro::kGatherThreads);  // sub-tile i's rows are visible; earlier gathers are done
                const int* rows = s_row + (i % Ro::kRing) * kClKeys;
                const uint8_t* pools = s_pool + (i % Ro::kRing) * kClKeys;
                if (gt < kClKeys) {  // the first gather warp: the stage's key mask for the softmax
                    const uint32_t bits = __ballot_sync(0xffffffffu, rows[gt] >= 0);
                    if (lane == 0) s_mask[s] = bits;
                }
                if (ok) {
                    const uint32_t stage = sK + s * kClStage;
#pragma unroll 1
                    for (int kk = gw; kk < kClKeys; kk += Ro::kGatherWarps) {
                        const int rr = rows[kk];
                        const uint8_t* base = pools[kk] == 2 ? static_cast<const uint8_t*>(a.swa.data)
                                                             : static_cast<const uint8_t*>(a.main.data);
                        const uint8_t* src = rr >= 0 ? base + (long long)rr * (2 * kD) : base;
#pragma unroll
                        for (int piece = lane; piece < kD / 8; piece += 32)
                            cp_async16_hint(stage + sw128_offset(kk, piece * 8, kClKeys * 128), src + piece * 16,
                                            rr >= 0 ? 16u : 0u, row_policy);
                    }
                }
                cp_async_commit();
                if (gt == 0) DSA_TRACE(i, 0);
                if (i == 0 && gt == 0) DSA_STAMP(3);
                // the next round of keys once this one's second sub-tile is under way, so its rows are known
                // before they are copied (ring slots of sub-tiles < i are free by now)
                if (i % Ro::kRound == 2) resolve_round(i / Ro::kRound + 1);
                // a thread keeps up to two sub-tiles of copies in flight: with two outstanding, the older is
                // reported once its group has landed (a third in flight was measured slower: the copies of
                // the sub-tile the MMAs wait for share the memory pipe with those of one more)
                if (i - sig >= 1) {
                    cp_async_wait_group<1>();
                    fence_proxy_async_smem();
                    mbar_arrive(&full[sig % NS]);
                    if (gt == 0) DSA_TRACE(sig, 1);
                    ++sig;
                }
            }
            if (sig < n_mine) {  // the sub-tiles not yet reported
                cp_async_wait_all();
                for (; sig < n_mine; ++sig) {
                    fence_proxy_async_smem();
                    mbar_arrive(&full[sig % NS]);
                    if (gt == 0) DSA_TRACE(sig, 1);
                }
            }
        } else {
            // e4m3 rows: sub-tile i's codes are copied as they are into raw slot i & 1 (row kk at 512 kk, lane
            // l the codes of dims 16 l .. 16 l + 15; the row scales into the slot's scale row) as soon as the
            // slot's previous sub-tile has been widened, without waiting for a key stage; each landed sub-tile
            // is then widened into its stage (widen_fp8), so two sub-tiles of copies stay in flight
            constexpr int kRowsPerWarp = (kClKeys + Ro::kGatherWarps - 1) / Ro::kGatherWarps;
            for (int i = 0; i < n_mine; ++i) {
                if (i - sig >= 2) {  // raw slot i & 1 still holds sub-tile i - 2: widen it first
                    cp_async_wait_group<1>();
                    widen_fp8(sig++);
                }
                named_bar_sync(1, Ro::kGatherThreads);  // sub-tile i's rows are visible; raw slot i & 1 is free
                const int* rows = s_row + (i % Ro::kRing) * kClKeys;
                const uint8_t* pools = s_pool + (i % Ro::kRing) * kClKeys;
                if (ok) {
                    const uint32_t raw = sK + NS * kClStage + (i & 1) * (kClStage / 2);
                    float* ksc = s_ksc + (kClStages + (i & 1)) * kClKeys;
#pragma unroll
                    for (int u = 0; u < kRowsPerWarp; ++u) {
                        const int kk = gw + u * Ro::kGatherWarps;
                        if (kk < kClKeys) {
                            const int rr = rows[kk];
                            const dsa_pool_t& pl = pools[kk] == 2 ? a.swa : a.main;
                            const uint8_t* src = static_cast<const uint8_t*>(pl.data) + (rr >= 0 ? (long long)rr * kD : 0);
                            cp_async16_hint(raw + kk * kD + lane * 16, src + lane * 16, rr >= 0 ? 16u : 0u, row_policy);
                            if (lane == 0)
                                cp_async4(smem_u32(ksc + kk), rr >= 0 ? pl.scale + rr : pl.scale, rr >= 0 ? 4u : 0u);
                        }
                    }
                }
                cp_async_commit();
                if (gt == 0) DSA_TRACE(i, 0);
                if (i == 0 && gt == 0) DSA_STAMP(3);
                if (i % Ro::kRound == 2) resolve_round(i / Ro::kRound + 1);
                if (i - sig >= 1) {  // the older of the two sub-tiles in flight, once landed
                    cp_async_wait_group<1>();
                    widen_fp8(sig++);
                }
            }
            if (sig < n_mine) {
                cp_async_wait_all();
                for (; sig < n_mine; ++sig) widen_fp8(sig);
            }
        }
        if (!ok) report(a.status, DSA_ERR_TIMEOUT);
    } else if (warp >= 4) {
        // ---- MMA issue: two warps, each waiting whole and issuing from one elected lane --------------
        // S of sub-tile i + 1 goes first when its keys are in (it overlaps the softmax of sub-tile i), but
        // the product of sub-tile i never waits behind a gather that has not arrived.
        const int part = warp - 4;  // this warp's 512 / MW dims of S and its 4 / MW 128-dim tiles of O^T
        const uint32_t idesc_s = idesc_bf16(kClKeys, 0, 64), idesc_o = idesc_bf16(NH, 1, 128);
        const uint64_t dq = sw128_desc(sQ, 16, 1024);
        if (n_mine > 0) ok = mbar_wait_bounded(qfull, 0, kWaitLimitNs);
        auto issue_s = [&](int i) {  // this warp's 512 / MW dims into its own accumulator
            const int s = i % NS;
            tc_fence_after();
            const uint64_t dk = sw128_desc(sK + s * kClStage, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / (16 * Ro::kMma); ++k) {  // 64-dim chunks: 64 query rows / 32 key rows apart
                const int ks = part * (kD / (16 * Ro::kMma)) + k;
                const uint64_t oq = (uint64_t)((((ks >> 2) * (64 * 128)) + (ks & 3) * 32) >> 4);
                const uint64_t ok_ = (uint64_t)((((ks >> 2) * (kClKeys * 128)) + (ks & 3) * 32) >> 4);
                mma_bf16_ss_elect(tS + ((i & 1) * Ro::kMma + part) * kClKeys, dq + oq, dk + ok_, idesc_s, k > 0 ? 1u : 0u);
            }
            mma_commit_elect(&sfull[i & 1]);
        };
        auto issue_pv = [&](int i) {  // this warp's 128-dim tiles
            const int s = i % NS;
            tc_fence_after();
            const uint64_t dv = sw128_desc(sK + s * kClStage, kClKeys * 128, 1024);
            const uint64_t dp = sw128_desc(sP + (i & 1) * L::kP, 16, 1024);
#pragma unroll
            for (int mt = part * (4 / Ro::kMma); mt < (part + 1) * (4 / Ro::kMma); ++mt)
#pragma unroll
                for (int ks = 0; ks < kClKeys / 16; ++ks)
                    mma_bf16_ss_elect(tO + mt * NH,
                                      dv + (uint64_t)(((2 * mt) * (kClKeys * 128) + (2 * ks) * 1024) >> 4),
                                      dp + (uint64_t)((ks * 32) >> 4), idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
            mma_commit_elect(&pvdone[s]);
        };
        int next_s = 0;  // next sub-tile whose S is to be issued
        ok = __all_sync(0xffffffffu, ok);
        for (int i = 0; i < n_mine && ok; ++i) {
            // S for every sub-tile <= i whose keys are in; then P V of sub-tile i, issuing the next S
            // meanwhile if its keys arrive first
            const uint64_t t0 = global_ns();
            bool pv_done = false;
            while (ok && !pv_done) {
                if (next_s < n_mine && next_s <= i + 1 &&
                    __all_sync(0xffffffffu, mbar_try_wait(&full[next_s % NS], (next_s / NS) & 1))) {
                    issue_s(next_s);
                    if (tid == 128) DSA_TRACE(next_s, 2);
                    if (next_s == 0 && tid == 128) DSA_STAMP(4);
                    ++next_s;
                    continue;
                }
                if (next_s > i && __all_sync(0xffffffffu, mbar_try_wait(&pfull[i & 1], (i >> 1) & 1))) {
                    issue_pv(i);
                    if (tid == 128) DSA_TRACE(i, 5);
                    if (i == n_mine - 1 && tid == 128) DSA_STAMP(6);
                    pv_done = true;
                    continue;
                }
                if (global_ns() - t0 > kWaitLimitNs) ok = false;
                ok = __all_sync(0xffffffffu, ok);
            }
        }
        if (!ok && lane == 0) report(a.status, DSA_ERR_TIMEOUT);
    } else {
        // ---- softmax warps: thread = head (lanes 0-15 of the quadrant) --------------------------
        const int h = warp * 16 + lane;
        const bool hthread = lane < 16 && h < NH;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        // l: sum of the probabilities as rounded into P^T (the output's normaliser, so a one-hot row stays
        // exact); e: sum of the fp32 probabilities (the log-sum-exp)
        float m_run = -INFINITY, l_run = 0.f, e_run = 0.f;
        for (int i = 0; i < n_mine; ++i) {
            const int st = i % NS, s = i & 1;  // key stage; S columns, P^T buffer and scratch
            ok = ok && mbar_wait_bounded(&full[st], (i / NS) & 1, kWaitLimitNs);  // the stage's key mask
            ok = ok && mbar_wait_bounded(&sfull[s], (i >> 1) & 1, kWaitLimitNs);
            if (i >= 2)  // P^T buffer free: the product of sub-tile i - 2 is done
                ok = ok && mbar_wait_bounded(&pvdone[(i - 2) % NS], ((i - 2) / NS) & 1, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (tid == 0) DSA_TRACE(i, 3);
            float sv[kClKeys];
            float alpha = 1.f;
            bool resc = false;
            if (ok) {
                tc_fence_after();
                float sh[kClKeys];  // a further partial sum of the logits
                // the MW partial products summed in order: ((p0 + p1) + p2) + ...
                tmem_ld_nowait<16>(tS + (s * Ro::kMma) * kClKeys + lane_off, *reinterpret_cast<float(*)[16]>(sv));
                tmem_ld_nowait<16>(tS + (s * Ro::kMma) * kClKeys + lane_off + 16, *reinterpret_cast<float(*)[16]>(sv + 16));
#pragma unroll 1
                for (int pp = 1; pp < Ro::kMma; ++pp) {
                    tmem_ld_nowait<16>(tS + (s * Ro::kMma + pp) * kClKeys + lane_off, *reinterpret_cast<float(*)[16]>(sh));
                    tmem_ld_nowait<16>(tS + (s * Ro::kMma + pp) * kClKeys + lane_off + 16,
                                       *reinterpret_cast<float(*)[16]>(sh + 16));
                    tmem_wait_ld();
                    tmem_regs_after_wait<16>(*reinterpret_cast<float(*)[16]>(sv));
                    tmem_regs_after_wait<16>(*reinterpret_cast<float(*)[16]>(sv + 16));
                    tmem_regs_after_wait<16>(*reinterpret_cast<float(*)[16]>(sh));
                    tmem_regs_after_wait<16>(*reinterpret_cast<float(*)[16]>(sh + 16));
#pragma unroll
                    for (int j = 0; j < kClKeys; ++j) sv[j] += sh[j];
                }
                const uint32_t vm = s_mask[st];
                float mx = -INFINITY;
                if (!FP8 && vm == 0xFFFFFFFFu) {  // every key of the stage present (the same for all threads)
#pragma unroll
                    for (int j = 0; j < kClKeys; ++j) {
                        sv[j] *= a.scale_log2;
                        mx = fmaxf(mx, sv[j]);
                    }
                } else {
                    const float4* k4 = reinterpret_cast<const float4*>(s_ksc + st * kClKeys);  // e4m3 row scales
#pragma unroll
                    for (int j4 = 0; j4 < kClKeys; j4 += 4) {
                        float4 ks = make_float4(1.f, 1.f, 1.f, 1.f);
                        if constexpr (FP8) ks = k4[j4 / 4];
                        const float kv[4] = {ks.x, ks.y, ks.z, ks.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = j4 + e;
                            const float ls = FP8 ? a.scale_log2 * kv[e] : a.scale_log2;  // e4m3: times the row scale
                            sv[j] = ((vm >> j) & 1) ? sv[j] * ls : -INFINITY;
                            mx = fmaxf(mx, sv[j]);
                        }
                    }
                }
                if (mx > m_run + kLazyLog2) {  // also the first finite maximum (m_run = -inf)
                    alpha = exp2f(m_run - mx);
                    resc = i > 0;
                    m_run = mx;
                }
                const float mr = m_run == -INFINITY ? 0.f : m_run;  // all keys so far masked: p = 0
                const uint32_t prow = sP + s * L::kP + (h >> 3) * 1024 + (h & 7) * 128;
                float sum = 0.f, esum = 0.f;
#pragma unroll
                for (int c = 0; c < kClKeys / 8; ++c) {
                    uint32_t w[4];
                    float kc[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
                    if constexpr (FP8) {  // the eight row scales of this chunk
                        const float4* k4 = reinterpret_cast<const float4*>(s_ksc + st * kClKeys + 8 * c);
                        const float4 ka = k4[0], kb = k4[1];
                        kc[0] = ka.x, kc[1] = ka.y, kc[2] = ka.z, kc[3] = ka.w, kc[4] = kb.x, kc[5] = kb.y, kc[6] = kb.z,
                        kc[7] = kb.w;
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = ex2_sfu(sv[8 * c + 2 * e] - mr), p1 = ex2_sfu(sv[8 * c + 2 * e + 1] - mr);
                        esum += p0 + p1;
                        if constexpr (FP8) {  // the probability that multiplies the codes carries the row scale
                            sum += p0 + p1;
                            w[e] = bf16x2_rn(p0 * kc[2 * e], p1 * kc[2 * e + 1]);
                        } else {
                            w[e] = bf16x2_rn(p0, p1);
                            sum += __uint_as_float(w[e] << 16) + __uint_as_float(w[e] & 0xFFFF0000u);
                        }
                    }
                    if (hthread)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + ((c ^ (h & 7)) << 4)),
                                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                     : "memory");
                }
                l_run = l_run * alpha + sum;
                e_run = e_run * alpha + esum;
            }
            if (hthread) s_alpha[s * NH + h] = alpha;
            const bool any = __any_sync(0xffffffffu, resc && hthread);
            if (lane == 0) s_vote[s * 4 + warp] = any ? 1 : 0;
            named_bar_sync(2, 128);
            if (s_vote[s * 4] | s_vote[s * 4 + 1] | s_vote[s * 4 + 2] | s_vote[s * 4 + 3]) {
                // a head's maximum moved: O^T (after the previous sub-tile's product) times alpha per head
                ok = ok && mbar_wait_bounded(&pvdone[(i - 1) % NS], ((i - 1) / NS) & 1, kWaitLimitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
                        for (int c0 = 0; c0 < NH; c0 += 16) {
                            float v[16];
                            tmem_ld16(tO + mt * NH + lane_off + c0, v);
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] *= s_alpha[s * NH + c0 + e];
                            tmem_st16(tO + mt * NH + lane_off + c0, v);
                        }
                    }
                    tmem_wait_st();
                }
            }
            fence_proxy_async_smem();  // P^T stores -> async proxy
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pfull[s]);
            if (tid == 0) DSA_TRACE(i, 4);
            if (i == 0 && tid == 0) DSA_STAMP(5);
        }
        if (n_mine > 0) {  // the last product must be complete before O^T is read
            ok = ok && mbar_wait_bounded(&pvdone[(n_mine - 1) % NS], ((n_mine - 1) / NS) & 1, kWaitLimitNs);
            tc_fence_after();
        }
        if (tid == 0) DSA_STAMP(7);
        if (hthread) {
            s_own[h] = m_run;
            s_own[NH + h] = l_run;
            s_own[2 * NH + h] = e_run;
        }
        if (!ok) report(a.status, DSA_ERR_TIMEOUT);
    }

    // ---- merge across the cluster ---------------------------------------------------------------
    tc_fence_before();
    const bool all_ok = __syncthreads_and(ok);  // O^T complete (the softmax warps waited for it); s_own set
    tc_fence_after();
    if (tid == 0) DSA_STAMP(8);
    const bool have = n_mine > 0 && all_ok;
    constexpr int G = NH / 4;                    // heads per finishing thread (a TMEM load of G columns)
    const int quad = warp & 3, quarter = warp >> 2;
    const int d = quad * 32 + lane, h0 = quarter * G;  // thread: dim d of a 128-dim tile, heads h0 .. h0 + G
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int tiles_per = 4 / csize;
    auto tmem_cols = [&](int t, float (&v)[G]) {
        if constexpr (G == 16) tmem_ld16(tO + t * NH + lane_off + h0, v);
        else if constexpr (G == 8) tmem_ld8(tO + t * NH + lane_off + h0, v);
        else tmem_ld4(tO + t * NH + lane_off + h0, v);
    };
    auto tmem_cols_nowait = [&](int t, float (&v)[G]) { tmem_ld_nowait<G>(tO + t * NH + lane_off + h0, v); };
    // Tiles this CTA sends sit at [0, 3 tiles) of shared memory (the query rows, idle now), the tiles it
    // receives at [3, 6 tiles) (query rows and key stages); each as [NH / 4 head quads][128 dims] x 4 bf16.
    uint8_t* xout = smem + L::kOffQ;
    uint8_t* xin = smem + L::kOffQ + 3 * L::kTile;
    if (csize > 1) {
        // 1. the tiles other CTAs own, unscaled (the owner applies this CTA's factor), staged as bf16; only
        // this CTA's own accumulators are needed, so no CTA waits for another here
        float v[4][G];  // static register indices; the sent tiles' columns in flight together
        if (have) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (t % csize != crank) tmem_cols_nowait(t, v[t]);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 4; ++t) tmem_regs_after_wait<G>(v[t]);
        }
        if (tid == 0) DSA_STAMP(15);
        int sl = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (t % csize == crank) continue;
#pragma unroll
            for (int q4 = 0; q4 < G / 4; ++q4)
                *reinterpret_cast<uint2*>(xout + sl * L::kTile + ((h0 / 4 + q4) * 128 + d) * 8) =
                    have ? make_uint2(bf16x2_rn(v[t][4 * q4], v[t][4 * q4 + 1]), bf16x2_rn(v[t][4 * q4 + 2], v[t][4 * q4 + 3]))
                         : make_uint2(0u, 0u);
            ++sl;
        }
        if (tid == 0) DSA_STAMP(16);
        fence_proxy_async_smem();  // staged tiles -> async proxy (the bulk copies after the cluster barrier)
    }
    if (tid == 0) DSA_STAMP(9);
    // 2. (m, l, e, fault) per head to every CTA of the cluster
    if constexpr (!FUSED)
        if (csize > 1) cluster_wait();  // phase 0: every CTA of the cluster has started (fused: waited above)
    if (tid == 0) DSA_STAMP(17);
    if (csize > 1 && tid == 0)  // before any peer can push (pushes follow phase 1)
        for (int b = 0; b < (csize - 1) * tiles_per; ++b) mbar_arrive_expect_tx(&xfull[b], (uint32_t)L::kTile);
    const float fo = *s_fault ? 1.f : 0.f;  // this CTA met a device fault: the whole row is written as zeros
    for (int h = tid; h < NH; h += kClThreads) {
        const uint32_t dst = smem_u32(s_stat + (crank * NH + h) * 4);
        const float mo = have ? s_own[h] : -INFINITY, lo = have ? s_own[NH + h] : 0.f,
                    eo = have ? s_own[2 * NH + h] : 0.f;
        if (csize == 1)
            *reinterpret_cast<float4*>(s_stat + h * 4) = make_float4(mo, lo, eo, fo);
        else
            for (int q = 0; q < csize; ++q)
                st_cluster_v4(mapa_shared(dst, (uint32_t)q), mo, lo, eo, fo);
    }
    if (tid == 0) DSA_STAMP(18);
    if (csize > 1) {
        cluster_arrive();  // phase 1: statistics delivered, sent tiles staged, every CTA's products complete
        cluster_wait();
    } else {
        __syncthreads();  // one CTA: the statistics in its own shared memory, its products complete
    }
    if (tid == 0) DSA_STAMP(10);
    // 3. push: one bulk copy per sent tile, all from lane 0 of the last warp (the first warps compute the
    // factors meanwhile), the next CTA's tiles first, then the one after: every owner receives one CTA's tiles at
    // a time, each tile signalling its own slot, so the owner adds the first arrivals while the rest stream in
    const bool pusher = csize > 1 && warp == 15 && lane == 0;
    if (pusher) {
        for (int k = 1; k < csize; ++k) {
            const int o = (crank + k) % csize;
            for (int t = 0, sl = 0; t < 4; ++t) {
                if (t % csize == crank) continue;
                if (t % csize == o) {
                    const int slot = ((crank - o - 1 + csize) % csize) * tiles_per + t / csize;  // in the owner's xin
                    bulk_s2cluster(mapa_shared(smem_u32(xin + slot * L::kTile), (uint32_t)o),
                                   smem_u32(xout + sl * L::kTile), L::kTile,
                                   mapa_shared(smem_u32(&xfull[slot]), (uint32_t)o));
                }
                ++sl;
            }
        }
        bulk_commit();
    }
    // 4. per head: the cluster maximum M, each CTA's weight 2^(m_c - M), 1 / L; one thread per (head, CTA),
    // the four of a head in neighbouring lanes
    if (tid < NH * 4) {
        const int h = tid >> 2, qq = tid & 3;
        const bool in = qq < csize;
        const float4 st = in ? *reinterpret_cast<const float4*>(s_stat + (qq * NH + h) * 4)
                             : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        float M = fmaxf(st.x, __shfl_xor_sync(0xffffffffu, st.x, 1));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
        int fault = st.w != 0.f;
        fault |= __shfl_xor_sync(0xffffffffu, fault, 1);
        fault |= __shfl_xor_sync(0xffffffffu, fault, 2);
        const float fq = (st.x == -INFINITY || fault) ? 0.f : exp2f(st.x - M);
        float Ls = fq != 0.f ? st.y * fq : 0.f, Es = fq != 0.f ? st.z * fq : 0.f;
        Ls += __shfl_xor_sync(0xffffffffu, Ls, 1);
        Es += __shfl_xor_sync(0xffffffffu, Es, 1);
        Ls += __shfl_xor_sync(0xffffffffu, Ls, 2);
        Es += __shfl_xor_sync(0xffffffffu, Es, 2);
        if (in) s_fac[qq * NH + h] = fq;
        if (qq == 0) {
            s_inv[h] = Ls > 0.f ? 1.f / Ls : 0.f;
            s_M[h] = fault ? -INFINITY : M;
            s_L[h] = Ls;
            s_E[h] = Es;
            if (h == 0) s_vote[0] = fault;  // (the softmax votes are done) the row's fault flag for the partials
        }
    }
    if (tid == 0) DSA_STAMP(19);
    if (csize > 1) {
        // the factors reach every thread; the pushing warp (15, still issuing its copies one after another)
        // joins through a barrier of its own with the factor threads, so that the others need not wait for it
        static_assert(kClThreads == 512, "warps 0-14 and warp 15");
        if (tid < NH * 4) named_bar_arrive(4, NH * 4 + 32);
        if (warp == 15) {
            __syncwarp();  // lane 0 has issued the pushes
            named_bar_sync(4, NH * 4 + 32);
        } else {
            named_bar_sync(3, kClThreads - 32);
        }
    } else {
        __syncthreads();
    }
    if (tid == 0) DSA_STAMP(11);
    // this CTA's first owned tile leaves TMEM while the other CTAs' tiles are still arriving
    float v_first[G];
    if (have) tmem_cols(crank, v_first);
    if (tid == 0) DSA_STAMP(12);
    // ---- owner: finish each owned tile; bf16 output staged as [NH][128] in the P^T buffers and stored
    // with 16-byte writes, or fp32 split partials ------------------------------------------------------
    float inv[G], fown[G];
#pragma unroll
    for (int e = 0; e < G; e += 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(s_inv + h0 + e);
        const float4 a4 = *reinterpret_cast<const float4*>(s_fac + crank * NH + h0 + e);
        inv[e] = b4.x, inv[e + 1] = b4.y, inv[e + 2] = b4.z, inv[e + 3] = b4.w;
        fown[e] = a4.x, fown[e + 1] = a4.y, fown[e + 2] = a4.z, fown[e + 3] = a4.w;
    }
    // output staging: two buffers of [NH][128] bf16 (the P^T buffers, and key stages 2-3, idle by now), each
    // stored by one TMA box
    uint8_t* const ob0 = smem + L::kOffP;
    uint8_t* const ob1 = smem + L::kOffK + 2 * kClStage;
    const int firstd = kD - a.rope.rope_dim;
    const bool odd = lane & 1;
    float v_next[G];  // the next owned tile's columns, loaded from TMEM while this one is finished and stored
#pragma unroll 1
    for (int j = 0; j < tiles_per; ++j) {
        const int t = crank + csize * j;
        const int D = t * 128 + d;
        float v[G];
        if (have) {
            if (j == 0) {
#pragma unroll
                for (int e = 0; e < G; ++e) v[e] = v_first[e];
            } else {
                tmem_wait_ld();
                tmem_regs_after_wait<G>(v_next);
#pragma unroll
                for (int e = 0; e < G; ++e) v[e] = v_next[e];
            }
            if (j + 1 < tiles_per) tmem_cols_nowait(t + csize, v_next);
        }
        if (tid == 0 && j == 0) DSA_STAMP(20);
#pragma unroll
        for (int e = 0; e < G; ++e) v[e] = have ? v[e] * fown[e] : 0.f;
        // received tiles in the order they arrive: slot si holds CTA crank + 1 + si's, and CTA crank - 1 (the
        // last si) sends to this CTA first
#pragma unroll
        for (int sr = 0; sr < 3; ++sr) {
            const int si = csize - 2 - sr;
            if (si >= 0) {
                const int src = (crank + 1 + si) % csize;
                const float* fsrc = s_fac + src * NH + h0;
                const uint8_t* p = xin + (si * tiles_per + j) * L::kTile;
                const bool landed = mbar_wait_bounded(&xfull[si * tiles_per + j], 0, kWaitLimitNs);
                if (!landed && tid == 0) report(a.status, DSA_ERR_TIMEOUT);
                ok = ok && landed;
#pragma unroll
                for (int q4 = 0; q4 < G / 4; ++q4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(p + ((h0 / 4 + q4) * 128 + d) * 8);
                    const float4 f4 = *reinterpret_cast<const float4*>(fsrc + 4 * q4);
                    v[4 * q4] = fmaf(f4.x, __uint_as_float(w.x << 16), v[4 * q4]);
                    v[4 * q4 + 1] = fmaf(f4.y, __uint_as_float(w.x & 0xFFFF0000u), v[4 * q4 + 1]);
                    v[4 * q4 + 2] = fmaf(f4.z, __uint_as_float(w.y << 16), v[4 * q4 + 2]);
                    v[4 * q4 + 3] = fmaf(f4.w, __uint_as_float(w.y & 0xFFFF0000u), v[4 * q4 + 3]);
                }
            }
        }
        if (a.nsplit == 1) {
            if (j >= 2) {  // this buffer's previous box has been read out
                if (tid == 0) bulk_wait_read<1>();
                __syncthreads();
            }
            uint8_t* const obuf = (j & 1) ? ob1 : ob0;
            uint32_t* o32 = reinterpret_cast<uint32_t*>(obuf);
            const int De = D & ~1;  // the pair's even dim
            float rc = 1.f, rs = 0.f;
            if (De >= firstd) {
                rc = s_rc[De - firstd];
                rs = s_rc[De - firstd + 1];
            }
            // neighbouring lanes swap one value per pair of heads: the even lane then holds dims (De, De + 1) of
            // head 2p, the odd lane those of head 2p + 1; each rotates its pair by R_m^-1 and stores it packed
            float rr[G];
#pragma unroll
            for (int pp = 0; pp < G / 2; ++pp) {
                const float x0 = v[2 * pp] * inv[2 * pp], x1 = v[2 * pp + 1] * inv[2 * pp + 1];
                const float recv = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
                const float lo = odd ? recv : x0, hi = odd ? x1 : recv;
                rr[2 * pp] = lo * rc + hi * rs;
                rr[2 * pp + 1] = hi * rc - lo * rs;
            }
            if (!a.out8) {
#pragma unroll
                for (int pp = 0; pp < G / 2; ++pp)
                    o32[(h0 + 2 * pp + (odd ? 1 : 0)) * 64 + (d >> 1)] = bf16x2_rn(rr[2 * pp], rr[2 * pp + 1]);
            } else {
                // e4m3 ([P2] 融合点 2: the inverse rotation and the fp8 quantisation in one pass): each head's 128
                // dims of this tile share a scale amax / 448; the amax of a head is reduced over the lanes of its
                // parity, then over the quarter's four warps in shared memory (the statistics slots, free now)
                unsigned* s_amax = reinterpret_cast<unsigned*>(s_own);
                if (tid < NH) s_amax[tid] = 0u;
                __syncthreads();
#pragma unroll
                for (int pp = 0; pp < G / 2; ++pp) {
                    float am = fmaxf(fabsf(rr[2 * pp]), fabsf(rr[2 * pp + 1]));
#pragma unroll
                    for (int o = 2; o < 32; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
                    if (lane < 2) atomicMax(&s_amax[h0 + 2 * pp + lane], __float_as_uint(am));
                }
                __syncthreads();
                uint16_t* o16 = reinterpret_cast<uint16_t*>(obuf);  // [NH][128] e4m3 codes
#pragma unroll
                for (int pp = 0; pp < G / 2; ++pp) {
                    const int hh = h0 + 2 * pp + (odd ? 1 : 0);
                    const float am = __uint_as_float(s_amax[hh]);
                    const float sc = am > 0.f ? am / 448.f : 1.f;
                    o16[hh * 64 + (d >> 1)] =
                        (uint16_t)(float_to_e4m3(rr[2 * pp] / sc) | ((uint32_t)float_to_e4m3(rr[2 * pp + 1] / sc) << 8));
                }
                if (tid < NH) {
                    const float am = __uint_as_float(s_amax[tid]);
                    a.out_scale[((long long)row * a.heads + hg * NH + tid) * 4 + t] = am > 0.f ? am / 448.f : 1.f;
                }
            }
            if (tid == 0 && j == 0) DSA_STAMP(21);
            fence_proxy_async_smem();  // staged output -> async proxy (the TMA store)
            __syncthreads();
            if (tid == 0 && j == 0) DSA_STAMP(22);
            if (tid == 0) {  // NH rows of 128 dims -> out[row][hg * NH .. + NH][t * 128 .. + 128]
                tma_store_2d(&omap, a.out8 ? t * 128 : t * 128, row * a.heads + hg * NH, obuf);
                bulk_commit();
            }
        } else {
            const long long base0 = ((long long)row * a.nsplit + split) * a.heads + hg * NH + h0;
#pragma unroll
            for (int e = 0; e < G; ++e) a.ws_o[(base0 + e) * kD + D] = v[e];
        }
    }
    if (crank == 0) {
        for (int h = tid; h < NH; h += kClThreads) {
            const float Ls = s_L[h], M = s_M[h], Es = s_E[h];
            if (a.nsplit == 1) {
                if (a.lse) a.lse[(long long)row * a.heads + hg * NH + h] = Es > 0.f ? (M + log2f(Es)) / kLog2e : -INFINITY;
            } else {
                const long long b = ((long long)row * a.nsplit + split) * a.heads + hg * NH + h;
                a.ws_ml[b * 4 + 0] = Ls > 0.f ? M : -INFINITY;
                a.ws_ml[b * 4 + 1] = Ls;
                a.ws_ml[b * 4 + 2] = Es;
                a.ws_ml[b * 4 + 3] = s_vote[0] ? 1.f : 0.f;  // a faulted split zeroes the row in the combine
            }
        }
    }
    if (tid == 0) DSA_STAMP(13);
    if (pusher || tid == 0) bulk_wait_all();  // this CTA's shared memory is no longer read by its copies / stores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        DSA_STAMP(14);
        DSA_STAMP_NS(30);
    }
    if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// Split plans, shared by the workspace query and the launch (both row formats run on the tcgen05
// kernel): one cluster of `cl` CTAs per (row, head group, split) over 32-key sub-tiles: clusters of 4
// while four CTAs per row still fit on the GPU at once, then 2, then 1; a row splits further only when
// its clusters leave SMs idle, and never below two sub-tiles per CTA.
struct SplitPlan {
    int hg, hg_count, nsplit, cps, cl;
};

static SplitPlan plan_cluster(int rows, int heads, int max_keys) {
    SplitPlan p;
    p.hg = heads >= 64 ? 64 : heads;
    p.hg_count = heads / p.hg;
    const int n_sub = max(1, (max_keys + kClKeys - 1) / kClKeys);
    const long long units = (long long)rows * p.hg_count;
    const long long sms = sm_count();
    int cl = units * 4 <= sms ? 4 : (units * 2 <= sms ? 2 : 1);
    while (cl > 1 && cl > n_sub) cl >>= 1;
    long long ns = units * cl >= sms ? 1 : sms / (units * cl);
    ns = std::max(1ll, std::min(ns, (long long)((n_sub + 2 * cl - 1) / (2 * cl))));
    p.cl = cl;
    p.cps = (int)((n_sub + ns - 1) / ns);
    p.nsplit = (n_sub + p.cps - 1) / p.cps;
    return p;
}

static SplitPlan plan_for(int rows, int heads, int max_keys, int dtype) {
    (void)dtype;  // both row formats run on the cluster kernel
    return plan_cluster(rows, heads, max_keys);
}

// Workspace: split partials [rows][nsplit][heads][512] + (m, l) [rows][nsplit][heads][2] when a row's keys
// are split over several clusters (the CTAs of one cluster merge on chip).
static size_t workspace_bytes_for(int rows, const SplitPlan& p, int heads) {
    if (p.nsplit <= 1) return 0;
    return (size_t)rows * p.nsplit * heads * (kD + 4) * sizeof(float);
}

// Workspace that covers either row format (the size query does not know the pool's format).
static size_t workspace_bytes_any(int rows, int heads, int max_keys) {
    return std::max(workspace_bytes_for(rows, plan_for(rows, heads, max_keys, DSA_BF16), heads),
                    workspace_bytes_for(rows, plan_for(rows, heads, max_keys, DSA_FP8_E4M3), heads));
}

// Tensor map of a [rows][512] bf16 matrix with boxes of 64 columns x box_rows rows, 128B-swizzled.
static bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t rows, int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the [rows][512] bf16 output for boxes of 128 columns x box_rows rows, unswizzled (the staging
// layout [box_rows][128]).
static bool make_out_map(CUtensorMap* map, void* base, uint64_t rows, int box_rows, bool e4m3) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const int es = e4m3 ? 1 : 2;
    cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)kD * es};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estride[2] = {1, 1};
    return fn(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NH, bool FP8, bool FUSED = false>
static dsa_status_t launch_attn_cl(const AttnArgs& a, int cl, cudaStream_t st) {
    using L = ClSmem<NH>;
    CUtensorMap qmap, omap;
    if (!make_bf16_map(&qmap, a.q, (uint64_t)a.rows * a.heads, NH)) return DSA_ERR_CUDA;
    if (!make_out_map(&omap, a.out8 ? static_cast<void*>(a.out8) : static_cast<void*>(a.out), (uint64_t)a.rows * a.heads,
                      NH, a.out8 != nullptr))
        return DSA_ERR_CUDA;
    if (cudaFuncSetAttribute(attn_cl_kernel<NH, FP8, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) !=
        cudaSuccess)
        return DSA_ERR_CUDA;
    const long long grid = (long long)a.rows * a.hg_count * a.nsplit * cl;
    cudaError_t e = launch_pdl_cluster(attn_cl_kernel<NH, FP8, FUSED>, dim3((unsigned)grid), dim3(kClThreads), L::kAlloc, st, cl,
                                       qmap, omap, a);
    if (e == cudaSuccess && a.nsplit > 1)
        e = launch_pdl(attn_combine_kernel, dim3(a.rows * a.heads), dim3(128), 0, st, a);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    return launch_status();
}

// The indexer scores a fused call selects from (the kernel's top-k phase), and whether a plan allows it: one
// cluster of four CTAs per row holding all 64 heads, no key split, rows of at most 16,384 scores, k <= 512.
struct FusedTopk {
    const float* scores;
    int32_t ld;
    const int32_t* n_valid;
};

static bool fusable(const SplitPlan& p, int heads, int ld, int k) {
    return heads == 64 && p.hg_count == 1 && p.cl == 4 && p.nsplit == 1 && ld <= 4 * kClThreads * kFusedVpt &&
           k <= kFusedK;
}

static dsa_status_t sparse_attn(int32_t rows, int32_t heads, const void* q, const int32_t* q_pos,
                                const int32_t* q_req, int32_t kind, const int32_t* topk, int32_t k,
                                const dsa_pool_t* main, const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                const dsa_rope_t* rope, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream, uint8_t* out8 = nullptr,
                                float* out_scale = nullptr, const FusedTopk* fz = nullptr) {
    if (rows < 0) return DSA_ERR_INVALID_ARG;
    if (rows == 0) return DSA_OK;
    if (kind != DSA_C4A && kind != DSA_C128A) return DSA_ERR_INVALID_ARG;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return DSA_ERR_UNSUPPORTED;
    void* const dst = out8 ? static_cast<void*>(out8) : out;
    if (!q || !q_pos || !dst || !rope || !aligned(q, 16) || !aligned(dst, 16)) return DSA_ERR_INVALID_ARG;
    if (out8 && (!out_scale || !aligned(out_scale, 16))) return DSA_ERR_INVALID_ARG;
    if (topk && (k < 1 || k > 2048)) return DSA_ERR_INVALID_ARG;
    if (window < 1 || window > 1024 || !(sm_scale > 0.f)) return DSA_ERR_INVALID_ARG;
    if (!pool_ok(main) || !pool_ok(swa) || !main_bt || !main_bt->table || !swa_bt || !swa_bt->table)
        return DSA_ERR_INVALID_ARG;
    if (main->dim != kD || swa->dim != kD) return DSA_ERR_UNSUPPORTED;
    if (main->dtype != swa->dtype || main->dtype == DSA_FP4_E2M1) return DSA_ERR_UNSUPPORTED;
    if ((long long)main->num_blocks * main->rows_per_block > 0x7fffffffll ||
        (long long)swa->num_blocks * swa->rows_per_block > 0x7fffffffll)
        return DSA_ERR_UNSUPPORTED;  // rows are addressed with 32-bit indices
    if (main->rows_per_block != kBlockPositions / stride_of(kind) || swa->rows_per_block != kBlockPositions)
        return DSA_ERR_INVALID_ARG;
    if (rope->rope_dim < 0 || rope->rope_dim > 64 || (rope->rope_dim & 1) || !(rope->theta > 0.0))
        return DSA_ERR_INVALID_ARG;
    const int max_comp = topk ? k : main_bt->max_blocks * main->rows_per_block;
    const int max_keys = max_comp + window;
    const SplitPlan p = plan_for(rows, heads, max_keys, main->dtype);
    const size_t need = workspace_bytes_for(rows, p, heads);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256))) return DSA_ERR_INVALID_ARG;

    AttnArgs a{};
    a.rows = rows;
    a.heads = heads;
    a.hg_count = p.hg_count;
    a.nsplit = p.nsplit;
    a.cps = p.cps;
    a.q = static_cast<const uint16_t*>(q);
    a.q_pos = q_pos;
    a.q_req = q_req;
    a.kind_w = window_of(kind);
    a.kind_s = stride_of(kind);
    a.topk = topk;
    a.k = topk ? k : 0;
    a.main = *main;
    a.main_bt = *main_bt;
    a.swa = *swa;
    a.swa_bt = *swa_bt;
    a.window = window;
    a.scale_log2 = sm_scale * kLog2e;
    a.rope = make_rope_table(rope->rope_dim, rope->theta);
    a.out = out8 ? nullptr : static_cast<uint16_t*>(out);
    a.out8 = out8;
    a.out_scale = out_scale;
    a.lse = lse;
    if (p.nsplit > 1) {
        a.ws_o = static_cast<float*>(workspace);
        a.ws_ml = a.ws_o + (size_t)rows * p.nsplit * heads * kD;
    }

    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool fp8 = main->dtype == DSA_FP8_E4M3;
    if (fz) {  // topk is the output of the kernel's own top-k phase
        if (!fusable(p, heads, fz->ld, k)) return DSA_ERR_UNSUPPORTED;
        a.topk = nullptr;
        a.topk_out = const_cast<int32_t*>(topk);
        a.scores = fz->scores;
        a.score_ld = fz->ld;
        a.n_valid = fz->n_valid;
        return fp8 ? launch_attn_cl<64, true, true>(a, p.cl, st) : launch_attn_cl<64, false, true>(a, p.cl, st);
    }
    if (!fp8) {
        switch (p.hg) {
            case 16: return launch_attn_cl<16, false>(a, p.cl, st);
            case 32: return launch_attn_cl<32, false>(a, p.cl, st);
            default: return launch_attn_cl<64, false>(a, p.cl, st);
        }
    }
    switch (p.hg) {
        case 16: return launch_attn_cl<16, true>(a, p.cl, st);
        case 32: return launch_attn_cl<32, true>(a, p.cl, st);
        default: return launch_attn_cl<64, true>(a, p.cl, st);
    }
}

}  // namespace dsa

using namespace dsa;

DSA_TIMELINE_SETTER(dsa_timeline_attention)

extern "C" size_t dsa_attn_workspace_size(int32_t nq, int32_t heads, int32_t max_keys) {
    if (nq <= 0 || heads <= 0 || max_keys <= 0) return 0;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return 0;
    return workspace_bytes_any(nq, heads, max_keys);
}

extern "C" dsa_status_t dsa_attn_plan(int32_t nq, int32_t heads, int32_t max_keys, int32_t dtype, int32_t* plan) {
    if (!plan || nq <= 0 || max_keys <= 0) return DSA_ERR_INVALID_ARG;
    if (dtype == DSA_FP4_E2M1) return DSA_ERR_UNSUPPORTED;  // e2m1 holds indexer keys only
    if (dtype != DSA_BF16 && dtype != DSA_FP8_E4M3) return DSA_ERR_INVALID_ARG;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return DSA_ERR_UNSUPPORTED;
    const SplitPlan p = plan_for(nq, heads, max_keys, dtype);
    plan[0] = p.hg;
    plan[1] = p.cl;
    plan[2] = p.nsplit;
    plan[3] = p.nsplit > 1 ? 2 : 1;
    return DSA_OK;
}

extern "C" dsa_status_t dsa_sparse_attn_decode(int32_t batch, int32_t heads, const void* q, const int32_t* q_pos,
                                               int32_t kind, const int32_t* topk, int32_t k, const dsa_pool_t* main,
                                               const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                               const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                               const dsa_rope_t* rope, void* out, float* lse, void* workspace,
                                               size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return sparse_attn(batch, heads, q, q_pos, nullptr, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale,
                       rope, out, lse, workspace, workspace_bytes, dev_status, stream);
}

extern "C" dsa_status_t dsa_topk_sparse_attn_decode(
    int32_t batch, int32_t heads, const void* q, const int32_t* q_pos, int32_t kind, const float* scores, int32_t ld,
    const int32_t* n_visible, int32_t k, int32_t* topk_out, const dsa_pool_t* main, const dsa_block_table_t* main_bt,
    const dsa_pool_t* swa, const dsa_block_table_t* swa_bt, int32_t window, float sm_scale, const dsa_rope_t* rope,
    void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (batch < 0) return DSA_ERR_INVALID_ARG;
    if (batch == 0) return DSA_OK;
    if (!scores || !n_visible || !topk_out || k < 1 || k > 2048 || ld < 0 || (ld & 3) || !aligned(scores, 16) ||
        !main)
        return DSA_ERR_INVALID_ARG;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return DSA_ERR_UNSUPPORTED;
    if (window < 1 || window > 1024) return DSA_ERR_INVALID_ARG;
    const SplitPlan p = plan_for(batch, heads, k + window, main->dtype);
    if (!fusable(p, heads, ld, k)) {  // two launches: the top-k, then the attention over its output
        const dsa_status_t e = dsa_topk(batch, scores, ld, n_visible, k, topk_out, dev_status, stream);
        if (e != DSA_OK) return e;
        return sparse_attn(batch, heads, q, q_pos, nullptr, kind, topk_out, k, main, main_bt, swa, swa_bt, window,
                           sm_scale, rope, out, lse, workspace, workspace_bytes, dev_status, stream);
    }
    const FusedTopk fz{scores, ld, n_visible};
    return sparse_attn(batch, heads, q, q_pos, nullptr, kind, topk_out, k, main, main_bt, swa, swa_bt, window, sm_scale,
                       rope, out, lse, workspace, workspace_bytes, dev_status, stream, nullptr, nullptr, &fz);
}

extern "C" dsa_status_t dsa_sparse_attn_q8(int32_t nq, int32_t heads, const void* q, const int32_t* q_pos,
                                           const int32_t* q_req, int32_t kind, const int32_t* topk, int32_t k,
                                           const dsa_pool_t* main, const dsa_block_table_t* main_bt,
                                           const dsa_pool_t* swa, const dsa_block_table_t* swa_bt, int32_t window,
                                           float sm_scale, const dsa_rope_t* rope, uint8_t* out, float* out_scale,
                                           float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                           void* stream) {
    return sparse_attn(nq, heads, q, q_pos, q_req, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale, rope,
                       nullptr, lse, workspace, workspace_bytes, dev_status, stream, out, out_scale);
}

extern "C" dsa_status_t dsa_sparse_attn_prefill(int32_t nq, int32_t heads, const void* q, const int32_t* q_pos,
                                                const int32_t* q_req, int32_t kind, const int32_t* topk, int32_t k,
                                                const dsa_pool_t* main, const dsa_block_table_t* main_bt,
                                                const dsa_pool_t* swa, const dsa_block_table_t* swa_bt,
                                                int32_t window, float sm_scale, const dsa_rope_t* rope, void* out,
                                                float* lse, void* workspace, size_t workspace_bytes,
                                                int32_t* dev_status, void* stream) {
    if (!q_req) return DSA_ERR_INVALID_ARG;
    return sparse_attn(nq, heads, q, q_pos, q_req, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale, rope,
                       out, lse, workspace, workspace_bytes, dev_status, stream);
}

// ---------------------------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving loop that forbids cudaMalloc on its
// hot path (an allocation can synchronise the device and stall every stream), a host that owns all
// device memory through its own arena and exposes no allocator, or a plugin that only receives the
// input and output pointers.  For them this entry point keeps the split-K partials in a fixed array
// that is part of the library image (a file-scope __device__ array): every GPU that loads the library
// holds these bytes until the process exits.  All calls share the one array, so calls that may
// overlap on the GPU (different streams, or different host threads on one device) race on it and
// must be serialised by the caller.  Every partial a call reads was written earlier in the same call,
// so no part of the array has to start at zero.
// ---------------------------------------------------------------------------------------------
namespace dsa {

constexpr size_t kStaticScratchBytes = 32u << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mutex;
static void* g_scratch_addr[kMaxDevices];
static CUcontext g_scratch_ctx[kMaxDevices];

// The calling thread's current driver context (the one the array's device copy belongs to), through the
// runtime's driver entry point (no libcuda link dependency); NULL if it cannot be queried.
static CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the array in the current device's current context.  In host code `g_attn_scratch`
// names a host-side stand-in, not device memory, so the address is looked up (with that device current)
// and cached per device together with the context it belongs to; a different context on the same device
// (after cudaDeviceReset, or a caller-created context) looks it up again.
static void* static_scratch(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = DSA_ERR_CUDA;
        return nullptr;
    }
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
            *status = DSA_ERR_CUDA;
            return nullptr;
        }
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context();  // the runtime makes a primary context current if none was
    }
    *status = DSA_OK;
    return g_scratch_addr[dev];
}

}  // namespace dsa

extern "C" size_t dsa_attn_static_scratch_bytes(void) { return dsa::kStaticScratchBytes; }

extern "C" dsa_status_t dsa_sparse_attn_decode_static(int32_t batch, int32_t heads, const void* q,
                                                      const int32_t* q_pos, int32_t kind, const int32_t* topk,
                                                      int32_t k, const dsa_pool_t* main,
                                                      const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                                      const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                                      const dsa_rope_t* rope, void* out, float* lse,
                                                      int32_t* dev_status, void* stream) {
    if (batch < 0 || !main || !main_bt || window < 1) return DSA_ERR_INVALID_ARG;
    if (batch == 0) return DSA_OK;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return DSA_ERR_UNSUPPORTED;
    const int max_comp = topk ? k : main_bt->max_blocks * main->rows_per_block;
    const size_t need = workspace_bytes_any(batch, heads, max_comp + window);
    if (need > kStaticScratchBytes) return DSA_ERR_UNSUPPORTED;  // beyond the fixed scratch: use the workspace call
    int st = DSA_OK;
    void* scratch = need > 0 ? static_scratch(&st) : nullptr;
    if (st != DSA_OK) return st;
    return sparse_attn(batch, heads, q, q_pos, nullptr, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale,
                       rope, out, lse, scratch, need > 0 ? kStaticScratchBytes : 0, dev_status, stream);
}
