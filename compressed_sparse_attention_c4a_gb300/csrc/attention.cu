// dsa_sparse_attn_decode / dsa_sparse_attn_prefill: MQA attention over gathered top-k compressed
// entries plus the sliding window, K = V, with the inverse-RoPE epilogue fused into the store.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §4.2-4.3: the main attention reads only
// the top-k entries, MQA-style (one latent entry serves every head); §5.3 and [P2] "DeepSeek V4
// 稀疏注意力完全解剖" 机制四: a 128-token window of uncompressed tokens is seen alongside; [P2] 机制一:
// K and V are one stored row; [P2] 深潜 (Inverse RoPE): out = R_m^-1 sum_j p_j k_j; [P2] 融合点 2:
// the inverse rotation is fused with the output store.
//
// Work split.  One CTA per (query row, group of HG heads, key split).  Keys are processed in chunks
// of 64 rows gathered through the block tables into shared memory (double buffered, cp.async);
// each chunk is used twice from the same tile: as K for S = Q K^T and as V for O += P V, both on
// the tensor cores (bf16 mma, fp32 accumulation).  Softmax is online (base-2, fp32).  When a row's
// keys are split over several CTAs, each writes an unnormalised partial (O, max, sum) and a
// combine kernel merges them and applies the inverse rotation.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace dsa {

constexpr int kD = 512;
constexpr int kChunk = 64;                    // keys per chunk
constexpr int kRowStride = kD * 2 + 16;       // bf16 row + 16 B pad: conflict-free ldmatrix
constexpr int kPStride = kChunk * 2 + 16;     // P tile row stride (bytes)
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
    int rows, heads, hg_count, nsplit, cps;   // cps = chunks per split
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
    uint16_t* out;
    float* lse;
    float* ws_o;                              // [rows][nsplit][heads][512]
    float* ws_ml;                             // [rows][nsplit][heads][2]
    int32_t* status;
};

// ---- PTX wrappers ---------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)float_to_bf16(lo) | ((uint32_t)float_to_bf16(hi) << 16);
}

// Key j of a row: compressed slot j < n_comp, else window position.  Returns the physical row
// (in the pool chosen by *use_swa), or -1 for a masked key; reports faults.
__device__ __forceinline__ long long resolve_key(const AttnArgs& a, int row, int r, int m, int n_vis, int n_comp,
                                                 int wlo, int j, bool* use_swa) {
    if (j < n_comp) {
        *use_swa = false;
        int id = a.topk ? __ldg(a.topk + (long long)row * a.k + j) : j;
        if (id < 0) return -1;
        if (id >= n_vis) {
            report(a.status, DSA_ERR_DEVICE_FAULT);
            return -1;
        }
        long long p = physical_row(a.main_bt, r, id, a.main.rows_per_block, a.main.num_blocks);
        if (p < 0) report(a.status, DSA_ERR_DEVICE_FAULT);
        return p;
    }
    *use_swa = true;
    const long long pos = (long long)wlo + (j - n_comp);
    long long p = physical_row(a.swa_bt, r, pos, kBlockPositions, a.swa.num_blocks);
    if (p < 0) report(a.status, DSA_ERR_DEVICE_FAULT);
    return p;
}

template <int HG, bool FP8>
struct AttnSmem {
    static constexpr int kQ = HG * kRowStride;
    static constexpr int kK = kChunk * kRowStride;              // one bf16 tile
    static constexpr int kNumK = FP8 ? 1 : 2;                   // bf16 tiles
    static constexpr int kK8 = FP8 ? kChunk * kD : 0;           // fp8 staging tile
    static constexpr int kP = HG * kPStride;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQ;
    static constexpr int kOffK8 = kOffK + kNumK * kK;
    static constexpr int kOffP = kOffK8 + 2 * kK8;
    static constexpr int kOffMeta = kOffP + kP;                 // long long rows[3][64]
    static constexpr int kOffFlags = kOffMeta + 3 * kChunk * 8; // int8: 0 masked, 1 main, 2 swa
    static constexpr int kOffScale = kOffFlags + 3 * kChunk;    // float[2][64]
    static constexpr int kOffStats = kOffScale + 2 * kChunk * 4;// float rowmax[HG][8], rowsum[HG][8]
    static constexpr int kOffML = kOffStats + 2 * HG * 8 * 4;   // float m[HG], l[HG]
    static constexpr int kBytes = kOffML + 2 * HG * 4;
};

template <int HG, bool FP8>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(AttnArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    using L = AttnSmem<HG, FP8>;
    constexpr int MT = HG / 16;        // 16-head m-tiles
    constexpr int WPM = 8 / MT;        // warps per m-tile
    constexpr int KW = kChunk / WPM;   // keys per warp in S = Q K^T
    constexpr int NT = KW / 8;         // n-tiles per warp in S
    constexpr int DW = kD / WPM;       // output dims per warp in O += P V
    constexpr int ON = DW / 8;         // n-tiles per warp in O

    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    long long* meta_row = reinterpret_cast<long long*>(smem + L::kOffMeta);
    int8_t* meta_flag = reinterpret_cast<int8_t*>(smem + L::kOffFlags);
    float* key_scale = reinterpret_cast<float*>(smem + L::kOffScale);
    float* row_max = reinterpret_cast<float*>(smem + L::kOffStats);
    float* row_sum = row_max + HG * 8;
    float* sm_m = reinterpret_cast<float*>(smem + L::kOffML);
    float* sm_l = sm_m + HG;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int mt = warp / WPM, wk = warp % WPM;

    const int split = blockIdx.x % a.nsplit;
    const int hg = (blockIdx.x / a.nsplit) % a.hg_count;
    const int row = blockIdx.x / (a.nsplit * a.hg_count);
    const int r = a.q_req ? a.q_req[row] : row;
    const int m = a.q_pos[row];
    const bool row_ok = r >= 0 && r < a.main_bt.batch && r < a.swa_bt.batch && m >= 0;
    if (!row_ok && tid == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
    const int n_vis = row_ok ? entries_formed((long long)m + 1, a.kind_w, a.kind_s) : 0;
    const int n_comp = a.topk ? a.k : n_vis;
    const int wlo = max(0, m - a.window + 1);
    const int n_keys = row_ok ? n_comp + (m - wlo + 1) : 0;
    const int key_lo = split * a.cps * kChunk;
    const int key_hi = min(n_keys, key_lo + a.cps * kChunk);
    const int n_chunks = key_hi > key_lo ? (key_hi - key_lo + kChunk - 1) / kChunk : 0;

    for (int i = tid; i < HG; i += kThreads) {
        sm_m[i] = -INFINITY;
        sm_l[i] = 0.f;
    }
    // key metadata of chunks 0 and 1
    auto resolve_chunk = [&](int c, int jj) {
        const int j = key_lo + c * kChunk + jj;
        long long p = -1;
        bool sw = false;
        if (j < key_hi) p = resolve_key(a, row, r, m, n_vis, n_comp, wlo, j, &sw);
        meta_row[(c % 3) * kChunk + jj] = p;
        meta_flag[(c % 3) * kChunk + jj] = p < 0 ? 0 : (sw ? 2 : 1);
    };
    if (tid < kChunk) {
        if (n_chunks > 0) resolve_chunk(0, tid);
    } else if (tid < 2 * kChunk) {
        if (n_chunks > 1) resolve_chunk(1, tid - kChunk);
    }
    __syncthreads();

    const int row_bytes = FP8 ? kD : 2 * kD;
    auto issue_chunk = [&](int c) {
        // warp w gathers keys 8w .. 8w+7 of the chunk; each key row is one contiguous copy
        const int mb = (c % 3) * kChunk;
        const int buf = c & 1;
        const uint32_t dst0 = FP8 ? sbase + L::kOffK8 + buf * L::kK8 : sbase + L::kOffK + buf * L::kK;
        const int dst_stride = FP8 ? kD : kRowStride;
        for (int kk = warp * 8; kk < warp * 8 + 8; ++kk) {
            const int flag = meta_flag[mb + kk];
            const long long prow = meta_row[mb + kk];
            const uint8_t* base = flag == 2 ? static_cast<const uint8_t*>(a.swa.data)
                                            : static_cast<const uint8_t*>(a.main.data);
            const uint8_t* src = flag ? base + prow * row_bytes : base;
            for (int piece = lane; piece < row_bytes / 16; piece += 32)
                cp_async16(dst0 + kk * dst_stride + piece * 16, src + piece * 16, flag ? 16u : 0u);
            if (FP8 && lane == 0)
                key_scale[buf * kChunk + kk] =
                    flag == 2 ? a.swa.scale[prow] : (flag == 1 ? a.main.scale[prow] : 0.f);
        }
    };
    // Q rows of this head group
    {
        const uint16_t* qsrc = a.q + ((long long)row * a.heads + (long long)hg * HG) * kD;
        for (int i = tid; i < HG * (kD / 8); i += kThreads) {
            const int h = i / (kD / 8), piece = i % (kD / 8);
            cp_async16(sbase + L::kOffQ + h * kRowStride + piece * 16, qsrc + (long long)h * kD + piece * 8,
                       row_ok ? 16u : 0u);
        }
    }
    if (n_chunks > 0) issue_chunk(0);
    cp_async_commit();

    float o[ON][4];
#pragma unroll
    for (int i = 0; i < ON; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    const uint32_t sQ = sbase + L::kOffQ;
    const uint32_t sP = sbase + L::kOffP;
    for (int c = 0; c < n_chunks; ++c) {
        cp_async_wait_all();
        __syncthreads();
        if (c + 1 < n_chunks) issue_chunk(c + 1);
        cp_async_commit();
        if (c + 2 < n_chunks && tid < kChunk) resolve_chunk(c + 2, tid);
        const int buf = c & 1;
        uint32_t sK;
        if constexpr (FP8) {
            // exact e4m3 -> bf16 conversion of the staged codes into the single bf16 tile
            const uint8_t* src = smem + L::kOffK8 + buf * L::kK8;
            uint8_t* dst = smem + L::kOffK;
            for (int i = tid; i < kChunk * kD / 4; i += kThreads) {
                const int kk = i / (kD / 4), e4 = (i % (kD / 4)) * 4;
                const uint32_t cw = *reinterpret_cast<const uint32_t*>(src + kk * kD + e4);
                uint2 v;
                v.x = pack_bf16(e4m3_to_float(cw & 0xff), e4m3_to_float((cw >> 8) & 0xff));
                v.y = pack_bf16(e4m3_to_float((cw >> 16) & 0xff), e4m3_to_float(cw >> 24));
                *reinterpret_cast<uint2*>(dst + kk * kRowStride + e4 * 2) = v;
            }
            __syncthreads();
            sK = sbase + L::kOffK;
        } else {
            sK = sbase + L::kOffK + buf * L::kK;
        }
        const int mb = (c % 3) * kChunk;

        // ---- S = Q K^T for heads [16 mt, 16 mt + 16) x keys [KW wk, KW wk + KW) ----------
        float s[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        const uint32_t qa = sQ + (mt * 16 + (lane & 15)) * kRowStride + (lane >> 4) * 16;
#pragma unroll 4
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(qa + ks * 32, a0, a1, a2, a3);
            if constexpr (NT == 1) {
                uint32_t b0, b1;
                const uint32_t kb = sK + (wk * KW + (lane & 7)) * kRowStride + ((lane >> 3) & 1) * 16 + ks * 32;
                ldsm_x2(kb, b0, b1);
                mma_bf16(s[0], a0, a1, a2, a3, b0, b1);
            } else {
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int key = wk * KW + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    ldsm_x4(sK + key * kRowStride + ((lane >> 3) & 1) * 16 + ks * 32, b0, b1, b2, b3);
                    mma_bf16(s[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_bf16(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        // ---- scale, mask, chunk row max ----------------------------------------------------
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = wk * KW + nt * 8 + 2 * t4 + e;
                float f = a.scale_log2;
                if constexpr (FP8) f *= key_scale[buf * kChunk + key];
                const bool valid = meta_flag[mb + key] != 0;
                s[nt][e] = valid ? s[nt][e] * f : -INFINITY;
                s[nt][2 + e] = valid ? s[nt][2 + e] * f : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][e]);
                mx1 = fmaxf(mx1, s[nt][2 + e]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const int h0 = mt * 16 + g, h1 = h0 + 8;
        if (t4 == 0) {
            row_max[h0 * 8 + wk] = mx0;
            row_max[h1 * 8 + wk] = mx1;
        }
        __syncthreads();
        float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
        for (int i = 0; i < WPM; ++i) {
            cm0 = fmaxf(cm0, row_max[h0 * 8 + i]);
            cm1 = fmaxf(cm1, row_max[h1 * 8 + i]);
        }
        const float mo0 = sm_m[h0], mo1 = sm_m[h1];
        const float mn0 = fmaxf(mo0, cm0), mn1 = fmaxf(mo1, cm1);
        // ---- P = exp2(S - m_new), row sums, P (times the fp8 row scale) to shared memory ----
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int key = wk * KW + nt * 8 + 2 * t4;
            float p0 = mn0 == -INFINITY ? 0.f : exp2f(s[nt][0] - mn0);
            float p1 = mn0 == -INFINITY ? 0.f : exp2f(s[nt][1] - mn0);
            float p2 = mn1 == -INFINITY ? 0.f : exp2f(s[nt][2] - mn1);
            float p3 = mn1 == -INFINITY ? 0.f : exp2f(s[nt][3] - mn1);
            ps0 += p0 + p1;
            ps1 += p2 + p3;
            if constexpr (FP8) {
                const float k0 = key_scale[buf * kChunk + key], k1 = key_scale[buf * kChunk + key + 1];
                p0 *= k0; p1 *= k1; p2 *= k0; p3 *= k1;
            }
            *reinterpret_cast<uint32_t*>(smem + L::kOffP + h0 * kPStride + key * 2) = pack_bf16(p0, p1);
            *reinterpret_cast<uint32_t*>(smem + L::kOffP + h1 * kPStride + key * 2) = pack_bf16(p2, p3);
        }
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
        if (t4 == 0) {
            row_sum[h0 * 8 + wk] = ps0;
            row_sum[h1 * 8 + wk] = ps1;
        }
        __syncthreads();
        float cs0 = 0.f, cs1 = 0.f;
#pragma unroll
        for (int i = 0; i < WPM; ++i) {
            cs0 += row_sum[h0 * 8 + i];
            cs1 += row_sum[h1 * 8 + i];
        }
        const float al0 = mo0 == -INFINITY ? 0.f : exp2f(mo0 - mn0);
        const float al1 = mo1 == -INFINITY ? 0.f : exp2f(mo1 - mn1);
        if (wk == 0 && t4 == 0) {
            sm_m[h0] = mn0;
            sm_m[h1] = mn1;
            sm_l[h0] = sm_l[h0] * al0 + cs0;
            sm_l[h1] = sm_l[h1] * al1 + cs1;
        }
#pragma unroll
        for (int i = 0; i < ON; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al0;
            o[i][2] *= al1;
            o[i][3] *= al1;
        }
        // ---- O += P V, dims [DW wk, DW wk + DW) -------------------------------------------
        const uint32_t pa = sP + (mt * 16 + (lane & 15)) * kPStride + (lane >> 4) * 16;
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(pa + ks * 32, a0, a1, a2, a3);
            const uint32_t vb = sK + (ks * 16 + (lane & 15)) * kRowStride + (lane >> 4) * 16 + wk * DW * 2;
#pragma unroll
            for (int np = 0; np < ON / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vb + np * 32, b0, b1, b2, b3);
                mma_bf16(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    __syncthreads();

    // ---- epilogue ----------------------------------------------------------------------------
    const int h0 = mt * 16 + g, h1 = h0 + 8;
    const float m0 = sm_m[h0], m1 = sm_m[h1], l0 = sm_l[h0], l1 = sm_l[h1];
    const int head0 = hg * HG + h0, head1 = hg * HG + h1;
    if (a.nsplit == 1) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        uint16_t* out0 = a.out + ((long long)row * a.heads + head0) * kD;
        uint16_t* out1 = a.out + ((long long)row * a.heads + head1) * kD;
        const int first = kD - a.rope.rope_dim;
#pragma unroll
        for (int nt = 0; nt < ON; ++nt) {
            const int col = wk * DW + nt * 8 + 2 * t4;
            float x0 = o[nt][0] * i0, x1 = o[nt][1] * i0, y0 = o[nt][2] * i1, y1 = o[nt][3] * i1;
            if (col >= first) {
                float cs, sn;
                rope_cos_sin(m, a.rope.inv_freq[(col - first) >> 1], &cs, &sn);
                // R_m^-1: rotation by -angle
                const float u0 = x0 * cs + x1 * sn, u1 = -x0 * sn + x1 * cs;
                const float v0 = y0 * cs + y1 * sn, v1 = -y0 * sn + y1 * cs;
                x0 = u0; x1 = u1; y0 = v0; y1 = v1;
            }
            *reinterpret_cast<uint32_t*>(out0 + col) = pack_bf16(x0, x1);
            *reinterpret_cast<uint32_t*>(out1 + col) = pack_bf16(y0, y1);
        }
        if (a.lse && wk == 0 && t4 == 0) {
            a.lse[(long long)row * a.heads + head0] = l0 > 0.f ? (m0 + log2f(l0)) / kLog2e : -INFINITY;
            a.lse[(long long)row * a.heads + head1] = l1 > 0.f ? (m1 + log2f(l1)) / kLog2e : -INFINITY;
        }
    } else {
        const long long base0 = ((long long)row * a.nsplit + split) * a.heads;
        float* wo0 = a.ws_o + (base0 + head0) * kD;
        float* wo1 = a.ws_o + (base0 + head1) * kD;
#pragma unroll
        for (int nt = 0; nt < ON; ++nt) {
            const int col = wk * DW + nt * 8 + 2 * t4;
            *reinterpret_cast<float2*>(wo0 + col) = make_float2(o[nt][0], o[nt][1]);
            *reinterpret_cast<float2*>(wo1 + col) = make_float2(o[nt][2], o[nt][3]);
        }
        if (wk == 0 && t4 == 0) {
            a.ws_ml[(base0 + head0) * 2 + 0] = m0;
            a.ws_ml[(base0 + head0) * 2 + 1] = l0;
            a.ws_ml[(base0 + head1) * 2 + 0] = m1;
            a.ws_ml[(base0 + head1) * 2 + 1] = l1;
        }
    }
}

// Merge split partials of one (row, head): 128 threads x 4 dims; inverse RoPE; bf16 store.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int row = blockIdx.x / a.heads, head = blockIdx.x % a.heads;
    const int tid = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < a.nsplit; ++sp)
        M = fmaxf(M, a.ws_ml[(((long long)row * a.nsplit + sp) * a.heads + head) * 2]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float Ls = 0.f;
    for (int sp = 0; sp < a.nsplit; ++sp) {
        const long long b = ((long long)row * a.nsplit + sp) * a.heads + head;
        const float ms = a.ws_ml[b * 2], ls = a.ws_ml[b * 2 + 1];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        Ls += f * ls;
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
            rope_cos_sin(m, a.rope.inv_freq[(col - first) >> 1], &cs, &sn);
            const float x0 = acc[e], x1 = acc[e + 1];
            acc[e] = x0 * cs + x1 * sn;
            acc[e + 1] = -x0 * sn + x1 * cs;
        }
    }
    uint16_t* dst = a.out + ((long long)row * a.heads + head) * kD + tid * 4;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
    if (a.lse && tid == 0)
        a.lse[(long long)row * a.heads + head] = Ls > 0.f ? (M + log2f(Ls)) / kLog2e : -INFINITY;
}

// ---------------------------------------------------------------------------------------------
// bf16 rows on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// One CTA (4 warps) per (query row, group of NH heads, key split); a split is a run of 128-key
// tiles.  For each tile the 128 key rows are gathered through the block tables into shared memory
// in 128B-swizzled 8-row x 128-byte atoms, laid out [64-dim chunk][8-key group][8 keys][128 B].
// That one copy serves both products (K = V):
//   S^T = K Q^T   : A = K tile, K-major (M = 128 keys, K = 512 dims), B = Q (N = NH heads, K-major),
//                   accumulated in TMEM columns [0, NH): lane = key, column = head;
//   O^T += V^T P^T: A = the same tile read MN-major (M = 128 dims per MMA, K = 16 keys),
//                   B = P^T (N = NH heads, K = keys, K-major), four 128-dim tiles in TMEM columns
//                   [NH, 5 NH): lane = dim, column = head.
// Softmax runs per head over TMEM lanes: each thread holds one key's NH logits; per-head max and sum
// are warp shuffle reductions plus a 4-warp combine in shared memory (online across tiles, with O^T
// rescaled in TMEM when a head's max grows).  The epilogue reads O^T (lane = dim), applies 1/l and
// R_m^-1 (pairs of dims sit in neighbouring lanes) and stores bf16, or writes split-K partials.
// ---------------------------------------------------------------------------------------------
constexpr int kTcKeys = 128;
constexpr int kTcThreads = 256;  // 8 warps: two per TMEM lane quadrant

template <int NH>
struct TcSmem {
    static constexpr int kQ = NH * kD * 2;          // [8][NH][128 B]
    static constexpr int kK = kTcKeys * kD * 2;     // [8][128][128 B]
    static constexpr int kP = NH * kTcKeys * 2;     // [2][NH][128 B]
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQ;
    static constexpr int kOffP = kOffK + kK;
    static constexpr int kOffMeta = kOffP + kP;                  // long long [128]
    static constexpr int kOffFlag = kOffMeta + kTcKeys * 8;      // int [128]
    static constexpr int kOffRed = kOffFlag + kTcKeys * 4;       // float [4][NH] x 2
    static constexpr int kOffStat = kOffRed + 2 * 4 * NH * 4;    // float m[NH], l[NH], mnew[NH], alpha[NH]
    static constexpr int kOffBar = kOffStat + 4 * NH * 4;        // mbarrier, tmem address
    static constexpr int kBytes = kOffBar + 64;
    static constexpr int kAlloc = kBytes + 1024;                 // + alignment slack
    static constexpr int kTmemCols = 5 * NH <= 128 ? 128 : (5 * NH <= 256 ? 256 : 512);
};

// Byte offset of element (row r, element e) in a tile of 128B-swizzled atoms whose rows are 128 bytes
// (64 bf16) long: atoms of 8 rows are 1024 bytes apart, 64-element chunks `chunk_stride` apart.
__device__ __forceinline__ uint32_t sw128_offset(int r, int e, int chunk_stride) {
    const int c = e >> 6, in = e & 63;
    return (uint32_t)(c * chunk_stride + (r >> 3) * 1024 + (r & 7) * 128 + ((((in >> 3) ^ (r & 7))) << 4) +
                      ((in & 7) << 1));
}

// Reduce N values per lane across the 32 lanes of a warp, transposed: after log2(32) exchange steps
// lane l holds the reduction (over all lanes) of value index l * N / 32 (N <= 32), using N - 1
// shuffles instead of 5 N.  `op` is max or add.
template <int N, typename Op>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], Op op) {
    const int lane = threadIdx.x & 31;
    int n = N;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (i < n / 2) {
                    const float send = upper ? v[i] : v[i + n / 2];
                    const float keep = upper ? v[i + n / 2] : v[i];
                    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, o));
                }
            }
            n >>= 1;
        } else {
            v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
        }
    }
    return v[0];
}

template <int NH>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(AttnArgs a) {
    using L = TcSmem<NH>;
    constexpr int HH = NH / 2;  // heads per warp in the softmax (the two warps of a quadrant split them)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem + L::kOffQ), sK = smem_u32(smem + L::kOffK), sP = smem_u32(smem + L::kOffP);
    long long* meta_row = reinterpret_cast<long long*>(smem + L::kOffMeta);
    int* meta_flag = reinterpret_cast<int*>(smem + L::kOffFlag);
    float* red_a = reinterpret_cast<float*>(smem + L::kOffRed);
    float* red_b = red_a + 4 * NH;
    float* st_m = reinterpret_cast<float*>(smem + L::kOffStat);
    float* st_l = st_m + NH;
    float* st_mnew = st_l + NH;
    float* st_alpha = st_mnew + NH;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 1);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2;  // TMEM lanes 32 quad .. ; heads / dim tiles of this half
    const int split = blockIdx.x % a.nsplit;
    const int hg = (blockIdx.x / a.nsplit) % a.hg_count;
    const int row = blockIdx.x / (a.nsplit * a.hg_count);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(s_tmem, L::kTmemCols);
    for (int h = tid; h < NH; h += kTcThreads) {
        st_m[h] = -INFINITY;
        st_l[h] = 0.f;
    }
    pdl_wait();  // on-chip set-up above; global memory only below
    pdl_launch_dependents();
    const int r = a.q_req ? a.q_req[row] : row;
    const int m = a.q_pos[row];
    const bool row_ok = r >= 0 && r < a.main_bt.batch && r < a.swa_bt.batch && m >= 0;
    if (!row_ok && tid == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
    const int n_vis = row_ok ? entries_formed((long long)m + 1, a.kind_w, a.kind_s) : 0;
    const int n_comp = a.topk ? a.k : n_vis;
    const int wlo = max(0, m - a.window + 1);
    const int n_keys = row_ok ? n_comp + (m - wlo + 1) : 0;
    const int key_lo = split * a.cps * kTcKeys;
    const int key_hi = min(n_keys, key_lo + a.cps * kTcKeys);
    // Q rows of this head group -> B operand layout
    {
        const uint16_t* qsrc = a.q + ((long long)row * a.heads + (long long)hg * NH) * kD;
        for (int i = tid; i < NH * (kD / 8); i += kTcThreads) {
            const int h = i / (kD / 8), e = (i % (kD / 8)) * 8;
            cp_async16(sQ + sw128_offset(h, e, NH * 128), qsrc + (long long)h * kD + e, row_ok ? 16u : 0u);
        }
        cp_async_commit();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tS = tmem, tO = tmem + NH;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t idesc_s = idesc_bf16(NH, 0), idesc_o = idesc_bf16(NH, 1);
    const int h0 = half * HH;  // this warp's heads in the softmax: [h0, h0 + HH)
    auto fmax_op = [](float x, float y) { return fmaxf(x, y); };
    auto add_op = [](float x, float y) { return x + y; };

    // key resolution (top-k index -> block table -> physical row) of the next tile runs one tile
    // ahead, so its dependent global loads overlap the current tile's copies, MMAs and softmax
    long long nxt_row = -1;
    int nxt_flag = 0;
    auto resolve_tile = [&](int kt) {
        if (tid < kTcKeys) {
            const int j = kt + tid;
            long long p = -1;
            bool sw = false;
            if (j < key_hi) p = resolve_key(a, row, r, m, n_vis, n_comp, wlo, j, &sw);
            nxt_row = p;
            nxt_flag = p < 0 ? 0 : (sw ? 2 : 1);
        }
    };
    resolve_tile(key_lo);

    uint32_t phase = 0;
    bool ok = true, first = true;
    for (int kt = key_lo; kt < key_hi && ok; kt += kTcKeys) {
        // publish the tile's resolved keys (thread j <-> key kt + j), then gather rows warp by warp
        if (tid < kTcKeys) {
            meta_row[tid] = nxt_row;
            meta_flag[tid] = nxt_flag;
        }
        __syncthreads();
        for (int kk = warp; kk < kTcKeys; kk += kTcThreads / 32) {
            const int flag = meta_flag[kk];
            const uint8_t* base = flag == 2 ? static_cast<const uint8_t*>(a.swa.data)
                                            : static_cast<const uint8_t*>(a.main.data);
            const uint8_t* src = flag ? base + meta_row[kk] * (2 * kD) : base;
            for (int piece = lane; piece < kD / 8; piece += 32)
                cp_async16(sK + sw128_offset(kk, piece * 8, kTcKeys * 128), src + piece * 16, flag ? 16u : 0u);
        }
        cp_async_commit();
        if (kt + kTcKeys < key_hi) resolve_tile(kt + kTcKeys);
        cp_async_wait_all();
        fence_proxy_async_smem();  // cp.async writes -> visible to the tensor core (async proxy)
        __syncthreads();

        // S^T = K Q^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll 4
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t koff = (ks >> 2) * (kTcKeys * 128) + (ks & 3) * 32;
                const uint32_t qoff = (ks >> 2) * (NH * 128) + (ks & 3) * 32;
                mma_bf16_ss(tS, sw128_desc(sK + koff, 16, 1024), sw128_desc(sQ + qoff, 16, 1024), idesc_s, ks > 0);
            }
            mma_commit(bar);
        }
        ok = mbar_wait_bounded(bar, phase, kWaitLimitNs);
        phase ^= 1;
        ok = __syncthreads_and(ok);
        if (!ok) {
            if (tid == 0) report(a.status, DSA_ERR_TIMEOUT);
            break;
        }
        tc_fence_after();

        // softmax over this tile's keys, per head: thread = key (quadrant lane), HH heads of this half
        const int key = quad * 32 + lane;
        const bool valid = meta_flag[key] != 0;
        float sv[HH], tmp[HH];
#pragma unroll
        for (int c0 = 0; c0 < HH; c0 += 16) {
            float v[16];
            tmem_ld16(tS + lane_off + h0 + c0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (c0 + i < HH) sv[c0 + i] = valid ? v[i] * a.scale_log2 : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < HH; ++i) tmp[i] = sv[i];
        {
            const float w = transpose_reduce<HH>(tmp, fmax_op);  // head h0 + lane * HH / 32
            if ((lane & (32 / HH - 1)) == 0) red_a[quad * NH + h0 + lane * HH / 32] = w;
        }
        __syncthreads();
        for (int h = tid; h < NH; h += kTcThreads) {
            const float mo = st_m[h];
            const float mt = fmaxf(fmaxf(red_a[h], red_a[NH + h]), fmaxf(red_a[2 * NH + h], red_a[3 * NH + h]));
            const float mn = fmaxf(mo, mt);
            st_mnew[h] = mn;
            st_alpha[h] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
        }
        __syncthreads();
        // P^T (bf16) for the PV product, per-head partial sums
#pragma unroll
        for (int i = 0; i < HH; ++i) {
            const int h = h0 + i;
            const float mn = st_mnew[h];
            const float p = mn == -INFINITY ? 0.f : exp2f(sv[i] - mn);
            sv[i] = p;
            *reinterpret_cast<uint16_t*>(smem + L::kOffP + sw128_offset(h, key, NH * 128)) = float_to_bf16(p);
        }
        {
            const float w = transpose_reduce<HH>(sv, add_op);
            if ((lane & (32 / HH - 1)) == 0) red_b[quad * NH + h0 + lane * HH / 32] = w;
        }
        __syncthreads();
        bool grew = false;
        for (int h = tid; h < NH; h += kTcThreads) {
            const float sum = red_b[h] + red_b[NH + h] + red_b[2 * NH + h] + red_b[3 * NH + h];
            st_l[h] = st_l[h] * st_alpha[h] + sum;
            grew |= st_alpha[h] != 1.f;
            st_m[h] = st_mnew[h];
        }
        grew = __syncthreads_or(grew);
        // rescale the running O^T where a head's max grew (lane = dim, column = head); each half of
        // the warps owns two of the four 128-dim tiles
        if (!first && grew) {
#pragma unroll 1
            for (int mt = 2 * half; mt < 2 * half + 2; ++mt) {
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 16) {
                    float v[16];
                    tmem_ld16(tO + mt * NH + lane_off + c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= st_alpha[c0 + i];
                    tmem_st16(tO + mt * NH + lane_off + c0, v);
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();  // P^T stores -> async proxy
        tc_fence_before();
        __syncthreads();

        // O^T += V^T P^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll 1
            for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
                for (int ks = 0; ks < kTcKeys / 16; ++ks) {
                    const uint32_t voff = (2 * mt) * (kTcKeys * 128) + (2 * ks) * 1024;
                    const uint32_t poff = (ks >> 2) * (NH * 128) + (ks & 3) * 32;
                    mma_bf16_ss(tO + mt * NH, sw128_desc(sK + voff, kTcKeys * 128, 1024),
                                sw128_desc(sP + poff, 16, 1024), idesc_o, (first && ks == 0) ? 0u : 1u);
                }
            }
            mma_commit(bar);
        }
        ok = mbar_wait_bounded(bar, phase, kWaitLimitNs);
        phase ^= 1;
        ok = __syncthreads_and(ok);
        if (!ok && tid == 0) report(a.status, DSA_ERR_TIMEOUT);
        tc_fence_after();
        first = false;
    }

    // ---- epilogue: thread = dim of a 128-dim tile of O^T; each half of the warps owns two tiles -----
    __syncthreads();
    const bool have = !first && ok;
    if (a.nsplit == 1) {
        const int rd = a.rope.rope_dim, firstd = kD - rd;
#pragma unroll 1
        for (int mt = 2 * half; mt < 2 * half + 2; ++mt) {
            const int d = mt * 128 + quad * 32 + lane;
            float cs = 1.f, sn = 0.f;
            if (d >= firstd) rope_cos_sin(m, a.rope.inv_freq[(d - firstd) >> 1], &cs, &sn);
#pragma unroll
            for (int c0 = 0; c0 < NH; c0 += 16) {
                float v[16];
                if (have) tmem_ld16(tO + mt * NH + lane_off + c0, v);
                else
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int h = c0 + i;
                    const float l = st_l[h];
                    const float x = l > 0.f ? v[i] / l : 0.f;
                    const float y = __shfl_xor_sync(0xffffffffu, x, 1);  // the pair partner's value
                    float o = x;
                    if (d >= firstd) o = (d & 1) ? (-y * sn + x * cs) : (x * cs + y * sn);  // R_m^-1
                    const float o_hi = __shfl_xor_sync(0xffffffffu, o, 1);
                    if ((d & 1) == 0)  // even lane stores the (d, d + 1) pair
                        *reinterpret_cast<uint32_t*>(a.out + ((long long)row * a.heads + hg * NH + h) * kD + d) =
                            (uint32_t)float_to_bf16(o) | ((uint32_t)float_to_bf16(o_hi) << 16);
                }
            }
        }
        if (a.lse)
            for (int h = tid; h < NH; h += kTcThreads) {
                const float l = st_l[h];
                a.lse[(long long)row * a.heads + hg * NH + h] = l > 0.f ? (st_m[h] + log2f(l)) / kLog2e : -INFINITY;
            }
    } else {
        const long long base0 = ((long long)row * a.nsplit + split) * a.heads + hg * NH;
#pragma unroll 1
        for (int mt = 2 * half; mt < 2 * half + 2; ++mt) {
            const int d = mt * 128 + quad * 32 + lane;
#pragma unroll
            for (int c0 = 0; c0 < NH; c0 += 16) {
                float v[16];
                if (have) tmem_ld16(tO + mt * NH + lane_off + c0, v);
                else
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) a.ws_o[(base0 + c0 + i) * kD + d] = v[i];
            }
        }
        for (int h = tid; h < NH; h += kTcThreads) {
            a.ws_ml[(base0 + h) * 2 + 0] = st_m[h];
            a.ws_ml[(base0 + h) * 2 + 1] = st_l[h];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// Split plan shared by the workspace query and the launch.
struct SplitPlan {
    int hg, hg_count, nsplit, cps;
};

static SplitPlan plan_splits(int rows, int heads, int max_keys, int chunk) {
    SplitPlan p;
    p.hg = heads >= 64 ? 64 : heads;
    p.hg_count = heads / p.hg;
    const int n_chunks = max(1, (max_keys + chunk - 1) / chunk);
    const long long units = (long long)rows * p.hg_count;
    const int sms = sm_count();
    int ns = units >= sms ? 1 : (int)(sms / units);
    ns = max(1, min(ns, n_chunks));
    p.cps = (n_chunks + ns - 1) / ns;
    p.nsplit = (n_chunks + p.cps - 1) / p.cps;
    return p;
}

static size_t workspace_bytes_for(int rows, const SplitPlan& p, int heads) {
    if (p.nsplit <= 1) return 0;
    return (size_t)rows * p.nsplit * heads * (kD + 2) * sizeof(float);
}

// Keys per split unit: 128-key tiles on the tensor-core path (bf16 rows), 64-key chunks for e4m3 rows.
static int chunk_for(int dtype) { return dtype == DSA_BF16 ? kTcKeys : kChunk; }

// Workspace that covers either row format (the size query does not know the pool's format).
static size_t workspace_bytes_any(int rows, int heads, int max_keys) {
    return std::max(workspace_bytes_for(rows, plan_splits(rows, heads, max_keys, kTcKeys), heads),
                    workspace_bytes_for(rows, plan_splits(rows, heads, max_keys, kChunk), heads));
}

template <int NH>
static dsa_status_t launch_attn_tc(const AttnArgs& a, cudaStream_t st) {
    using L = TcSmem<NH>;
    if (cudaFuncSetAttribute(attn_tc_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) !=
        cudaSuccess)
        return DSA_ERR_CUDA;
    const long long grid = (long long)a.rows * a.hg_count * a.nsplit;
    cudaError_t e = launch_pdl(attn_tc_kernel<NH>, dim3((unsigned)grid), dim3(kTcThreads), L::kAlloc, st, a);
    if (e == cudaSuccess && a.nsplit > 1)
        e = launch_pdl(attn_combine_kernel, dim3(a.rows * a.heads), dim3(128), 0, st, a);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    return launch_status();
}

template <int HG, bool FP8>
static dsa_status_t launch_attn(const AttnArgs& a, cudaStream_t st) {
    using L = AttnSmem<HG, FP8>;
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HG, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    const long long grid = (long long)a.rows * a.hg_count * a.nsplit;
    e = launch_pdl(attn_kernel<HG, FP8>, dim3((unsigned)grid), dim3(kThreads), L::kBytes, st, a);
    if (e == cudaSuccess && a.nsplit > 1)
        e = launch_pdl(attn_combine_kernel, dim3(a.rows * a.heads), dim3(128), 0, st, a);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    return launch_status();
}

static dsa_status_t sparse_attn(int32_t rows, int32_t heads, const void* q, const int32_t* q_pos,
                                const int32_t* q_req, int32_t kind, const int32_t* topk, int32_t k,
                                const dsa_pool_t* main, const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                const dsa_rope_t* rope, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (rows < 0) return DSA_ERR_INVALID_ARG;
    if (rows == 0) return DSA_OK;
    if (kind != DSA_C4A && kind != DSA_C128A) return DSA_ERR_INVALID_ARG;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return DSA_ERR_UNSUPPORTED;
    if (!q || !q_pos || !out || !rope || !aligned(q, 16) || !aligned(out, 16)) return DSA_ERR_INVALID_ARG;
    if (topk && (k < 1 || k > 2048)) return DSA_ERR_INVALID_ARG;
    if (window < 1 || window > 1024 || !(sm_scale > 0.f)) return DSA_ERR_INVALID_ARG;
    if (!pool_ok(main) || !pool_ok(swa) || !main_bt || !main_bt->table || !swa_bt || !swa_bt->table)
        return DSA_ERR_INVALID_ARG;
    if (main->dim != kD || swa->dim != kD) return DSA_ERR_UNSUPPORTED;
    if (main->dtype != swa->dtype) return DSA_ERR_UNSUPPORTED;
    if (main->rows_per_block != kBlockPositions / stride_of(kind) || swa->rows_per_block != kBlockPositions)
        return DSA_ERR_INVALID_ARG;
    if (rope->rope_dim < 0 || rope->rope_dim > 64 || (rope->rope_dim & 1) || !(rope->theta > 0.0))
        return DSA_ERR_INVALID_ARG;
    const int max_comp = topk ? k : main_bt->max_blocks * main->rows_per_block;
    const int max_keys = max_comp + window;
    const SplitPlan p = plan_splits(rows, heads, max_keys, chunk_for(main->dtype));
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
    a.out = static_cast<uint16_t*>(out);
    a.lse = lse;
    if (need > 0) {
        a.ws_o = static_cast<float*>(workspace);
        a.ws_ml = a.ws_o + (size_t)rows * p.nsplit * heads * kD;
    }
    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool fp8 = main->dtype == DSA_FP8_E4M3;
    if (!fp8) {
        switch (p.hg) {
            case 16: return launch_attn_tc<16>(a, st);
            case 32: return launch_attn_tc<32>(a, st);
            default: return launch_attn_tc<64>(a, st);
        }
    }
    switch (p.hg) {
        case 16: return fp8 ? launch_attn<16, true>(a, st) : launch_attn<16, false>(a, st);
        case 32: return fp8 ? launch_attn<32, true>(a, st) : launch_attn<32, false>(a, st);
        default: return fp8 ? launch_attn<64, true>(a, st) : launch_attn<64, false>(a, st);
    }
}

}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_attn_workspace_size(int32_t nq, int32_t heads, int32_t max_keys) {
    if (nq <= 0 || heads <= 0 || max_keys <= 0) return 0;
    if (heads != 16 && heads != 32 && heads != 64 && heads != 128) return 0;
    return workspace_bytes_any(nq, heads, max_keys);
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

// Device address of the array on the current device.  In host code `g_attn_scratch` names a
// host-side stand-in, not device memory, so the address is looked up once per device (with that
// device current) and cached.
static void* static_scratch(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = DSA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
            *status = DSA_ERR_CUDA;
            return nullptr;
        }
        g_scratch_addr[dev] = p;
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
