// dsa_compress: c4a / c128a compressor + RMSNorm + RoPE + paged insert, SWA insert and the
// rolling residual, in one streaming pass.
//
// [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §5.2 and [P2] "DeepSeek V4
// 稀疏注意力完全解剖" 机制二: a compressed token is a weighted sum of w raw tokens taken at
// stride s (c4a: 8 / 4, c128a: 128 / 128).  [P2] 融合点 1: the sum, RMSNorm, RoPE and the
// cache insert are one kernel that reads each raw token once and writes each entry once.
// [P2] 设计 2: the last w raw tokens are kept as a per-request rolling residual.
//
// Work split: one warp per emitted entry or per new token; a warp owns a whole row, each lane
// DIM/32 consecutive elements, so every row load and store is one coalesced transaction set.
// Raw tokens of an entry that are shared with its neighbour (c4a overlap) are re-read from L2.
#include "common.cuh"

namespace dsa {


struct CompressArgs {
    int w, s, batch, dim;
    const int32_t* cu_new;
    const int32_t* start_pos;
    const uint16_t* x_new;
    const float* logit_new;
    uint16_t* state_x;
    float* state_logit;
    const int32_t* state_slot;
    int num_slots;
    const float* gamma;
    float eps;
    RopeTable rope;
    dsa_pool_t out;
    dsa_block_table_t out_bt;
    dsa_pool_t swa;
    dsa_block_table_t swa_bt;
    int has_swa;
    int entry_items;  // warps per request reserved for entries
    int token_items;  // warps per request reserved for new tokens
    int fuse_ring;    // token warps also update the rolling state (at most one new token per request)
    int gate_pc;      // per-channel gate: logits [n][dim] and rolling logits [slots][w][dim]
    int nsub;         // warps per entry (kSplit for the c128a window with a scalar gate, else 1)
    int req_items;    // warps per request: entry_items * nsub + token_items, rounded up to whole CTAs
    int32_t* status;
};

template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t* row, int lane, float (&v)[E]) {
    const uint16_t* p = row + lane * E;
    if constexpr (E == 16) {
        uint4 a = *reinterpret_cast<const uint4*>(p);
        uint4 b = *reinterpret_cast<const uint4*>(p + 8);
        uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v[2 * k] = __uint_as_float(u[k] << 16);
            v[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
        }
    } else if constexpr (E == 4) {
        uint2 a = *reinterpret_cast<const uint2*>(p);
        v[0] = __uint_as_float(a.x << 16);
        v[1] = __uint_as_float(a.x & 0xffff0000u);
        v[2] = __uint_as_float(a.y << 16);
        v[3] = __uint_as_float(a.y & 0xffff0000u);
    } else {
        static_assert(E == 2, "row width");
        uint32_t a = *reinterpret_cast<const uint32_t*>(p);
        v[0] = __uint_as_float(a << 16);
        v[1] = __uint_as_float(a & 0xffff0000u);
    }
}

template <int E>
__device__ __forceinline__ void copy_bf16(uint16_t* dst, const uint16_t* src, int lane) {
    if constexpr (E == 16) {
        reinterpret_cast<uint4*>(dst + lane * E)[0] = reinterpret_cast<const uint4*>(src + lane * E)[0];
        reinterpret_cast<uint4*>(dst + lane * E)[1] = reinterpret_cast<const uint4*>(src + lane * E)[1];
    } else if constexpr (E == 4) {
        *reinterpret_cast<uint2*>(dst + lane * E) = *reinterpret_cast<const uint2*>(src + lane * E);
    } else {
        *reinterpret_cast<uint32_t*>(dst + lane * E) = *reinterpret_cast<const uint32_t*>(src + lane * E);
    }
}

template <int E>
__device__ __forceinline__ void load_f32(const float* row, int lane, float (&v)[E]) {
    const float* p = row + lane * E;
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int k = 0; k < E; k += 4) {
            const float4 t = *reinterpret_cast<const float4*>(p + k);
            v[k] = t.x, v[k + 1] = t.y, v[k + 2] = t.z, v[k + 3] = t.w;
        }
    } else {
        static_assert(E == 2, "row width");
        const float2 t = *reinterpret_cast<const float2*>(p);
        v[0] = t.x, v[1] = t.y;
    }
}

template <int E>
__device__ __forceinline__ void copy_f32(float* dst, const float* src, int lane) {
    float v[E];
    load_f32<E>(src, lane, v);
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int k = 0; k < E; k += 4)
            *reinterpret_cast<float4*>(dst + lane * E + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
    } else {
        *reinterpret_cast<float2*>(dst + lane * E) = make_float2(v[0], v[1]);
    }
}

// Store one row (the warp's E values per lane) into a pool row: bf16, e4m3 + amax/448 scale, or e2m1 + amax/6.
template <int E>
__device__ __forceinline__ void store_row(const dsa_pool_t& pool, long long prow, int lane, const float (&v)[E]) {
    if (pool.dtype == DSA_BF16) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(pool.data) + prow * (E * 32) + lane * E;
        uint32_t u[E / 2];
#pragma unroll
        for (int k = 0; k < E / 2; ++k)
            u[k] = (uint32_t)float_to_bf16(v[2 * k]) | ((uint32_t)float_to_bf16(v[2 * k + 1]) << 16);
        if constexpr (E == 16) {
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(u[0], u[1], u[2], u[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(u[4], u[5], u[6], u[7]);
        } else if constexpr (E == 4) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(u[0], u[1]);
        } else {
            *reinterpret_cast<uint32_t*>(dst) = u[0];
        }
    } else if (pool.dtype == DSA_FP4_E2M1) {  // e2m1 codes, two per byte, scale amax / 6
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(v[k]));
        amax = warp_max(amax);
        const float scale = amax > 0.f ? amax / 6.f : 1.f;
        uint8_t* dst = reinterpret_cast<uint8_t*>(pool.data) + prow * (E * 16) + lane * (E / 2);
        uint32_t c[(E / 2 + 3) / 4] = {};  // the lane's E/2 code bytes, little-endian in words
#pragma unroll
        for (int k = 0; k < E / 2; ++k)
            c[k / 4] |= (uint32_t)float2_to_e2m1x2(v[2 * k] / scale, v[2 * k + 1] / scale) << (8 * (k % 4));
        if constexpr (E == 16) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(c[0], c[1]);
        } else if constexpr (E == 4) {
            *reinterpret_cast<uint16_t*>(dst) = (uint16_t)c[0];
        } else {
            *dst = (uint8_t)c[0];
        }
        if (lane == 0) pool.scale[prow] = scale;
    } else {
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(v[k]));
        amax = warp_max(amax);
        const float scale = amax > 0.f ? amax / 448.f : 1.f;
        uint8_t* dst = reinterpret_cast<uint8_t*>(pool.data) + prow * (E * 32) + lane * E;
        uint32_t c[(E + 3) / 4] = {};  // the lane's E codes, little-endian in words
#pragma unroll
        for (int k = 0; k < E; ++k) c[k / 4] |= (uint32_t)float_to_e4m3(v[k] / scale) << (8 * (k % 4));
        if constexpr (E == 16) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
        } else if constexpr (E == 4) {
            *reinterpret_cast<uint32_t*>(dst) = c[0];
        } else {
            *reinterpret_cast<uint16_t*>(dst) = (uint16_t)c[0];
        }
        if (lane == 0) pool.scale[prow] = scale;
    }
}

// Rotate the lane's pairs that fall in the last rope_dim dims by R_pos.
template <int E>
__device__ __forceinline__ void rope_row(float (&v)[E], int lane, int dim, const RopeTable& rt, long long pos) {
    const int first = dim - rt.rope_dim;
#pragma unroll
    for (int k = 0; k < E; k += 2) {
        const int d = lane * E + k;
        if (d >= first) {
            float c, s;
            rope_cos_sin(pos, rt, (d - first) >> 1, &c, &s);
            const float x0 = v[k], x1 = v[k + 1];
            v[k] = x0 * c - x1 * s;
            v[k + 1] = x0 * s + x1 * c;
        }
    }
}

// One warp's item of one job: an entry (item < entry_items) or a new token.  The request's schedule
// (cu_new, start_pos, state_slot), the destination rows' block-table entries and the norm weights are read
// before waiting for the preceding kernel in the stream; raw tokens, logits and the rolling state after it.
// Every thread reaches the wait exactly once.
// Warps per entry of a 128-token window (c128a, scalar gate): eight warps of one CTA each sum 16 of the rows,
// warp 0 adds the partial sums in shared memory.
constexpr int kSplit = 8;

template <int DIM, int W>
__device__ __forceinline__ void compress_item(const CompressArgs& a, int item, int r, int lane, int sub = 0,
                                              float* part = nullptr) {
    constexpr int E = DIM / 32;
    constexpr int w = W;
    const int s = a.s;
    const int cu0 = __ldg(a.cu_new + r);
    const int n = __ldg(a.cu_new + r + 1) - cu0;
    const long long start = __ldg(a.start_pos + r);
    const long long end = start + n;
    const int slot = __ldg(a.state_slot + r);
    const bool bad_req = n < 0 || start < 0 || slot < 0 || slot >= a.num_slots;
    // this warp's work: entry i (is_entry) or new token j
    const bool is_entry = item < a.entry_items;
    long long i = -1, prow = -1;
    int j = -1;
    float gam[E];
    if (!bad_req && is_entry) {
        // entries whose last raw token s*i + w - 1 lies in [start, end)
        const long long lo_num = start - w + 1;
        const long long i_lo = lo_num <= 0 ? 0 : (lo_num + s - 1) / s;
        const long long i_hi = end >= w ? (end - w) / s : -1;
        i = i_lo + item;
        if (i > i_hi) i = -1;
        else prow = physical_row(a.out_bt, r, i, a.out.rows_per_block, a.out.num_blocks);
#pragma unroll
        for (int k = 0; k < E; ++k) gam[k] = a.gamma ? __ldg(a.gamma + lane * E + k) : 1.f;
    } else if (!bad_req) {
        j = item - a.entry_items;
        if (j >= n || j >= a.token_items) j = -1;
        else if (a.has_swa) prow = physical_row(a.swa_bt, r, start + j, kBlockPositions, a.swa.num_blocks);
    }
    // No L2 prefetch of the window's rows before the wait: measured without it, the smallest decode step
    // was about 1 us faster and no other workload slower.
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) DSA_STAMP(1);
    if (bad_req) {
        if (item == 0 && lane == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
        return;
    }

    if (is_entry) {
        if (i < 0) return;
        const long long base = (long long)s * i;
        auto logit_at = [&](long long p) -> float {
            return p < start ? a.state_logit[(long long)slot * w + (p % w)] : a.logit_new[cu0 + (p - start)];
        };
        auto row_at = [&](long long p) -> const uint16_t* {
            return p < start ? a.state_x + ((long long)slot * w + (p % w)) * DIM
                             : a.x_new + (long long)(cu0 + (p - start)) * DIM;
        };
        float acc[E];
        if (a.gate_pc) {
            // per-channel gate: for each of the lane's channels an online softmax over the window (running
            // maximum, denominator and weighted sum), RC window rows of values and logits in flight at a time
            auto zrow_at = [&](long long p) -> const float* {
                return p < start ? a.state_logit + ((long long)slot * w + (p % w)) * DIM
                                 : a.logit_new + (long long)(cu0 + (p - start)) * DIM;
            };
            constexpr int RC = E >= 16 ? 2 : (W < 8 ? W : 8);
            float m[E], den[E];
#pragma unroll
            for (int k = 0; k < E; ++k) m[k] = -INFINITY, den[k] = 0.f, acc[k] = 0.f;
#pragma unroll 1
            for (int j0 = 0; j0 < W; j0 += RC) {
                float xv[RC][E], zv[RC][E];
#pragma unroll
                for (int u = 0; u < RC; ++u) {
                    load_bf16<E>(row_at(base + j0 + u), lane, xv[u]);
                    load_f32<E>(zrow_at(base + j0 + u), lane, zv[u]);
                }
#pragma unroll
                for (int u = 0; u < RC; ++u)
#pragma unroll
                    for (int k = 0; k < E; ++k) {
                        const float mn = fmaxf(m[k], zv[u][k]);
                        const float sc = expf(m[k] - mn), e = expf(zv[u][k] - mn);
                        den[k] = fmaf(den[k], sc, e);
                        acc[k] = fmaf(acc[k], sc, e * xv[u][k]);
                        m[k] = mn;
                    }
            }
#pragma unroll
            for (int k = 0; k < E; ++k) acc[k] /= den[k];
        } else {
        // gate g_j = softmax_j(z_{s i + j}): lane l holds the logits of window tokens l, l + 32, ...
        constexpr int LPL = (W + 31) / 32;  // logits per lane
        constexpr int RB = W < 8 ? W : 8;   // window rows in flight at a time
        float z[LPL];
        float x[RB][E];
#pragma unroll
        for (int u = 0; u < RB; ++u) load_bf16<E>(row_at(base + u), lane, x[u]);  // with the logits
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < LPL; ++u) {
            const int jj = lane + 32 * u;
            z[u] = jj < W ? logit_at(base + jj) : -INFINITY;
            mx = fmaxf(mx, z[u]);
        }
        mx = warp_max(mx);
        if (lane == 0 && threadIdx.x < 64) DSA_STAMP(2 + 4 * (threadIdx.x >> 5));
        float den = 0.f;
#pragma unroll
        for (int u = 0; u < LPL; ++u) {
            z[u] = (lane + 32 * u) < W ? expf(z[u] - mx) : 0.f;
            den += z[u];
        }
        den = warp_sum(den);
        const float inv_den = 1.f / den;
#pragma unroll
        for (int k = 0; k < E; ++k) acc[k] = 0.f;
        // this warp's window rows (a 128-token window may be split over kSplit warps)
        const int j_lo = W == 128 ? sub * (W / a.nsub) : 0, j_hi = W == 128 ? j_lo + W / a.nsub : W;
        if (j_lo > 0) {
#pragma unroll
            for (int u = 0; u < RB; ++u) load_bf16<E>(row_at(base + j_lo + u), lane, x[u]);
        }
#pragma unroll 1
        for (int j0 = j_lo; j0 < j_hi; j0 += RB) {
            if (j0 > j_lo) {
#pragma unroll
                for (int u = 0; u < RB; ++u) load_bf16<E>(row_at(base + j0 + u), lane, x[u]);
            }
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int jj = j0 + u;
                const float g = __shfl_sync(0xffffffffu, z[jj / 32 < LPL ? jj / 32 : 0], jj & 31) * inv_den;
#pragma unroll
                for (int k = 0; k < E; ++k) acc[k] = fmaf(g, x[u][k], acc[k]);
            }
        }
        if (W == 128 && a.nsub > 1) {  // the CTA's warps are this entry's: warp 0 adds their partial sums
#pragma unroll
            for (int k = 0; k < E; ++k) part[sub * DIM + lane * E + k] = acc[k];
            __syncthreads();
            if (sub != 0) return;
#pragma unroll
            for (int k = 0; k < E; ++k) {
                float t = 0.f;
                for (int q = 0; q < a.nsub; ++q) t += part[q * DIM + lane * E + k];
                acc[k] = t;
            }
        }
        }
        if (lane == 0 && threadIdx.x < 64) DSA_STAMP(3 + 4 * (threadIdx.x >> 5));
        // RMSNorm
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k) ss = fmaf(acc[k], acc[k], ss);
        ss = warp_sum(ss);
        const float rs = rsqrtf(ss / (float)DIM + a.eps);
#pragma unroll
        for (int k = 0; k < E; ++k) acc[k] *= rs * gam[k];
        // RoPE at the last covered position
        rope_row<E>(acc, lane, DIM, a.rope, base + w - 1);
        if (prow < 0) {
            if (lane == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
            return;
        }
        store_row<E>(a.out, prow, lane, acc);
        if (lane == 0 && threadIdx.x < 64) DSA_STAMP(4 + 4 * (threadIdx.x >> 5));
        return;
    }

    if (j < 0) return;
    const long long p = start + j;
    const uint16_t* xrow = a.x_new + (long long)(cu0 + j) * DIM;
    if (a.has_swa) {
        float v[E];
        load_bf16<E>(xrow, lane, v);
        rope_row<E>(v, lane, DIM, a.rope, p);
        if (lane == 0 && threadIdx.x < 64) DSA_STAMP(3 + 4 * (threadIdx.x >> 5));
        if (prow < 0) {
            if (lane == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
        } else {
            store_row<E>(a.swa, prow, lane, v);
        }
    }
    if (a.fuse_ring && j >= n - w) {
        const long long ring = (long long)slot * w + (p % w);
        copy_bf16<E>(a.state_x + ring * DIM, xrow, lane);
        if (a.gate_pc) copy_f32<E>(a.state_logit + ring * DIM, a.logit_new + (long long)(cu0 + j) * DIM, lane);
        else if (lane == 0) a.state_logit[ring] = a.logit_new[cu0 + j];
    }
    if (lane == 0 && threadIdx.x < 64) DSA_STAMP(4 + 4 * (threadIdx.x >> 5));
}

constexpr int kMaxJobs = 4;

// The query job of a launch: each (query, head) row of the raw queries RMS-normalised and rotated at the
// query's position ([P2] 融合点 3: the Q-norm beside the key RoPE and insert).
struct QueryArgs {
    int nq, heads, dim;
    const uint16_t* q_raw;
    uint16_t* q_out;
    const int32_t* q_pos;
    const float* gamma;
    float eps;
    RopeTable rope;
    int32_t* status;
};

// The jobs of one launch: the caches of one layer that compress the same tokens of the same requests
// (main cache with its window insert, indexer cache), each its own rows, norm, RoPE and pool, and optionally
// the layer's queries.  Job k takes CTAs [cta_off[k], cta_off[k + 1]); the query job is job n_jobs.
struct CompressJobs {
    CompressArgs job[kMaxJobs];
    QueryArgs query;
    int n_jobs, has_query;
    int cta_off[kMaxJobs + 2];
};

// One warp's (query, head) row: q / sqrt(mean(q^2) + eps) * gamma, then R_m on the last rope_dim dims, as
// bf16.  The position is read before waiting for the preceding kernel, the raw row after it.
template <int DIM>
__device__ __forceinline__ void query_item(const QueryArgs& a, long long wi, int lane) {
    constexpr int E = DIM / 32;
    const long long q = wi / a.heads;
    const bool live = q < a.nq;
    const int m = live ? __ldg(a.q_pos + q) : 0;
    float gam[E];
#pragma unroll
    for (int k = 0; k < E; ++k) gam[k] = a.gamma ? __ldg(a.gamma + lane * E + k) : 1.f;
    pdl_wait();
    pdl_launch_dependents();
    if (!live) return;
    if (m < 0) {
        if (lane == 0) report(a.status, DSA_ERR_DEVICE_FAULT);
        return;
    }
    float v[E];
    load_bf16<E>(a.q_raw + wi * DIM, lane, v);
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) ss = fmaf(v[k], v[k], ss);
    ss = warp_sum(ss);
    const float rs = rsqrtf(ss / (float)DIM + a.eps);
#pragma unroll
    for (int k = 0; k < E; ++k) v[k] *= rs * gam[k];
    rope_row<E>(v, lane, DIM, a.rope, m);
    uint16_t* dst = a.q_out + wi * DIM + lane * E;
#pragma unroll
    for (int k = 0; k < E; k += 8) {
        uint4 u;
        u.x = (uint32_t)float_to_bf16(v[k]) | ((uint32_t)float_to_bf16(v[k + 1]) << 16);
        u.y = E > k + 2 ? ((uint32_t)float_to_bf16(v[k + 2]) | ((uint32_t)float_to_bf16(v[k + 3]) << 16)) : 0u;
        u.z = E > k + 4 ? ((uint32_t)float_to_bf16(v[k + 4]) | ((uint32_t)float_to_bf16(v[k + 5]) << 16)) : 0u;
        u.w = E > k + 6 ? ((uint32_t)float_to_bf16(v[k + 6]) | ((uint32_t)float_to_bf16(v[k + 7]) << 16)) : 0u;
        if constexpr (E >= 8) *reinterpret_cast<uint4*>(dst + k) = u;
        else if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(u.x, u.y);
        else *reinterpret_cast<uint32_t*>(dst) = u.x;
    }
}

// Grid: the CTAs of every job side by side along x (job k from cta_off[k]), so the caches of a layer (and its
// queries) are processed in one launch ([P2] 融合点 3: independent per-token work of one layer dispatched by
// warp and block index in one kernel).  The (request, item) pairs of a job are dealt to consecutive warps, so
// a decode batch (two items per request) fills few CTAs and leaves the other SMs to the kernel that follows.
template <int W>
__global__ void __launch_bounds__(256) compress_kernel(const __grid_constant__ CompressJobs js) {
    if (threadIdx.x == 0) {
        DSA_STAMP_NS(31);
        DSA_STAMP(0);
    }
    int k = 0;
    while (k < js.n_jobs + js.has_query - 1 && (int)blockIdx.x >= js.cta_off[k + 1]) ++k;
    const int lane = threadIdx.x & 31;
    const long long wi = (long long)(blockIdx.x - js.cta_off[k]) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (k == js.n_jobs) {  // the query job
        switch (js.query.dim) {
            case 64: query_item<64>(js.query, wi, lane); break;
            case 128: query_item<128>(js.query, wi, lane); break;
            default: query_item<512>(js.query, wi, lane); break;
        }
        return;
    }
    const CompressArgs& a = js.job[k];
    const int per_req = a.req_items;
    const int r = (int)(wi / per_req), it = (int)(wi - (long long)r * per_req);
    // items [0, entry_items * nsub) are entries (nsub consecutive warps each, one CTA when nsub > 1), then tokens
    const int split_items = a.entry_items * a.nsub;
    const int item = it < split_items ? it / a.nsub : a.entry_items + (it - split_items);
    const int sub = it < split_items ? it % a.nsub : 0;
    if (r >= a.batch || (it >= split_items && it - split_items >= a.token_items)) {  // no work
        pdl_wait();
        pdl_launch_dependents();
        if (lane == 0) DSA_STAMP_NS(30);
        return;
    }
    float* part = nullptr;
    if constexpr (W == 128) {
        __shared__ float s_part[kSplit * 512];  // the partial window sums of a split entry
        part = s_part;
    }
    switch (a.dim) {
        case 64: compress_item<64, W>(a, item, r, lane, sub, part); break;
        case 128: compress_item<128, W>(a, item, r, lane, sub, part); break;
        default: compress_item<512, W>(a, item, r, lane, sub, part); break;
    }
    if (lane == 0) DSA_STAMP_NS(30);  // (timeline builds) the last warp to finish sets the CTA's end
}

// Rolling-state update after a multi-token append: slot p % w <- token p for the last w new tokens.
template <int DIM>
__device__ __forceinline__ void ring_update_item(const CompressArgs& a, int item, int r, int lane) {
    constexpr int E = DIM / 32;
    const int cu0 = a.cu_new[r];
    const int n = a.cu_new[r + 1] - cu0;
    const int slot = a.state_slot[r];
    if (item >= a.w || n <= 0 || slot < 0 || slot >= a.num_slots) return;
    const int j = n - a.w + item;  // new-token index
    if (j < 0) return;
    const long long p = (long long)a.start_pos[r] + j;
    const long long ring = (long long)slot * a.w + (p % a.w);
    copy_bf16<E>(a.state_x + ring * DIM, a.x_new + (long long)(cu0 + j) * DIM, lane);
    if (a.gate_pc) copy_f32<E>(a.state_logit + ring * DIM, a.logit_new + (long long)(cu0 + j) * DIM, lane);
    else if (lane == 0) a.state_logit[ring] = a.logit_new[cu0 + j];
}

__global__ void __launch_bounds__(256) ring_update_kernel(const __grid_constant__ CompressJobs js) {
    pdl_wait();
    pdl_launch_dependents();
    const CompressArgs& a = js.job[blockIdx.z];
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
    switch (a.dim) {
        case 64: ring_update_item<64>(a, item, blockIdx.y, lane); break;
        case 128: ring_update_item<128>(a, item, blockIdx.y, lane); break;
        default: ring_update_item<512>(a, item, blockIdx.y, lane); break;
    }
}

static dsa_status_t launch_compress(CompressJobs js, int w, int batch, int max_new, cudaStream_t st) {
    long long warps[kMaxJobs + 1], comp = 0;
    bool split = false;
    for (int k = 0; k < js.n_jobs; ++k) {
        split |= js.job[k].nsub > 1;
        comp += (long long)batch * (js.job[k].entry_items * js.job[k].nsub + js.job[k].token_items);
    }
    // small compressor grids (decode) in CTAs of 2 warps: they fit beside two CTAs of the indexer that follows
    // on an SM, which 8-warp CTAs do not (each SM quarter has its own registers); split entries take whole CTAs
    const int wpc = split ? kSplit : (comp <= 4LL * sm_count() ? 2 : 8);
    for (int k = 0; k < js.n_jobs; ++k) {
        CompressArgs& a = js.job[k];
        a.req_items = (a.entry_items * a.nsub + a.token_items + wpc - 1) / wpc * wpc;
        warps[k] = (long long)batch * a.req_items;
    }
    if (js.has_query) warps[js.n_jobs] = (long long)js.query.nq * js.query.heads;
    long long off = 0;
    for (int k = 0; k < js.n_jobs + js.has_query; ++k) {
        js.cta_off[k] = (int)off;
        off += (warps[k] + wpc - 1) / wpc;
        if (off > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    }
    js.cta_off[js.n_jobs + js.has_query] = (int)off;
    if (off == 0) return DSA_OK;
    dim3 grid((unsigned)off);
    cudaError_t e = w == 8 ? launch_pdl(compress_kernel<8>, grid, dim3(32 * wpc), 0, st, js)
                           : launch_pdl(compress_kernel<128>, grid, dim3(32 * wpc), 0, st, js);
    if (e == cudaSuccess && !js.job[0].fuse_ring && max_new > 0)
        e = launch_pdl(ring_update_kernel, dim3((w + 7) / 8, batch, js.n_jobs), dim3(256), 0, st, js);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    return launch_status();
}

}  // namespace dsa

using namespace dsa;

DSA_TIMELINE_SETTER(dsa_timeline_compress)

// Checks one job's arguments and fills its kernel arguments (the request schedule is set by the caller).
static dsa_status_t make_job(int batch, int max_new, int w, int s, const void* x_new, const float* logit_new,
                             void* state_x, float* state_logit, const float* rms_gamma, float rms_eps,
                             const dsa_rope_t* rope, const dsa_pool_t* out, const dsa_block_table_t* out_bt,
                             const dsa_pool_t* swa, const dsa_block_table_t* swa_bt, int gate_pc, CompressArgs* a) {
    if (!(rms_eps > 0.f)) return DSA_ERR_INVALID_ARG;
    if (!x_new || !logit_new || !state_x || !state_logit || !rope) return DSA_ERR_INVALID_ARG;
    if (!pool_ok(out) || !table_ok(out_bt, batch)) return DSA_ERR_INVALID_ARG;
    if (out->rows_per_block != kBlockPositions / s) return DSA_ERR_INVALID_ARG;
    const int dim = out->dim;
    if (dim != 64 && dim != 128 && dim != 512) return DSA_ERR_UNSUPPORTED;
    if (rope->rope_dim < 0 || rope->rope_dim > dim || (rope->rope_dim & 1) || !(rope->theta > 0.0))
        return DSA_ERR_INVALID_ARG;
    if (rope->rope_dim > 64) return DSA_ERR_UNSUPPORTED;  // the frequency table holds 32 pairs
    if (swa) {
        if (!pool_ok(swa) || !table_ok(swa_bt, batch)) return DSA_ERR_INVALID_ARG;
        if (swa->rows_per_block != kBlockPositions || swa->dim != dim) return DSA_ERR_INVALID_ARG;
        if (swa->dtype == DSA_FP4_E2M1) return DSA_ERR_UNSUPPORTED;
    }
    if (!aligned(x_new, 16) || !aligned(state_x, 16)) return DSA_ERR_INVALID_ARG;
    if (gate_pc != 0 && gate_pc != 1) return DSA_ERR_INVALID_ARG;
    if (gate_pc && (!aligned(logit_new, 16) || !aligned(state_logit, 16))) return DSA_ERR_INVALID_ARG;
    a->w = w;
    a->gate_pc = gate_pc;
    a->s = s;
    a->batch = batch;
    a->dim = dim;
    a->x_new = static_cast<const uint16_t*>(x_new);
    a->logit_new = logit_new;
    a->state_x = static_cast<uint16_t*>(state_x);
    a->state_logit = state_logit;
    a->gamma = rms_gamma;
    a->eps = rms_eps;
    a->rope = make_rope_table(rope->rope_dim, rope->theta);
    a->out = *out;
    a->out_bt = *out_bt;
    a->has_swa = swa != nullptr;
    if (swa) {
        a->swa = *swa;
        a->swa_bt = *swa_bt;
    }
    a->entry_items = max_new / s + 1;
    a->token_items = max_new;
    a->nsub = (w == 128 && !gate_pc) ? kSplit : 1;
    a->fuse_ring = max_new <= 1;
    return DSA_OK;
}

static dsa_status_t make_query(const dsa_query_job_t* q, QueryArgs* a) {
    if (q->nq < 0 || q->heads < 1) return DSA_ERR_INVALID_ARG;
    if (q->dim != 64 && q->dim != 128 && q->dim != 512) return DSA_ERR_UNSUPPORTED;
    if (q->nq > 0 && (!q->q_raw || !q->q_out || !q->q_pos || !q->rope)) return DSA_ERR_INVALID_ARG;
    if (!aligned(q->q_raw, 16) || !aligned(q->q_out, 16) || !(q->rms_eps > 0.f)) return DSA_ERR_INVALID_ARG;
    if (q->rope && (q->rope->rope_dim < 0 || q->rope->rope_dim > q->dim || (q->rope->rope_dim & 1) ||
                    !(q->rope->theta > 0.0)))
        return DSA_ERR_INVALID_ARG;
    if (q->rope && q->rope->rope_dim > 64) return DSA_ERR_UNSUPPORTED;
    a->nq = q->nq;
    a->heads = q->heads;
    a->dim = q->dim;
    a->q_raw = static_cast<const uint16_t*>(q->q_raw);
    a->q_out = static_cast<uint16_t*>(q->q_out);
    a->q_pos = q->q_pos;
    a->gamma = q->rms_gamma;
    a->eps = q->rms_eps;
    if (q->rope) a->rope = make_rope_table(q->rope->rope_dim, q->rope->theta);
    return DSA_OK;
}

static dsa_status_t compress_jobs(int32_t kind, int32_t batch, const int32_t* cu_new, const int32_t* start_pos,
                                  int32_t max_new, const int32_t* state_slot, int32_t num_slots, int32_t n_jobs,
                                  const dsa_compress_job_t* jobs, const dsa_query_job_t* query, int32_t* dev_status,
                                  void* stream) {
    if (kind != DSA_C4A && kind != DSA_C128A) return DSA_ERR_INVALID_ARG;
    if (batch < 0 || max_new < 0 || num_slots <= 0) return DSA_ERR_INVALID_ARG;
    if (n_jobs < 1 || n_jobs > kMaxJobs || !jobs) return DSA_ERR_INVALID_ARG;
    const int w = window_of(kind), s = stride_of(kind);
    CompressJobs js{};
    js.n_jobs = n_jobs;
    if (query) {
        const dsa_status_t e = make_query(query, &js.query);
        if (e != DSA_OK) return e;
        js.query.status = dev_status;
        js.has_query = query->nq > 0;
    }
    if ((batch == 0 || max_new == 0) && !js.has_query) return DSA_OK;
    if (batch > 0 && max_new > 0 && (!cu_new || !start_pos || !state_slot)) return DSA_ERR_INVALID_ARG;
    if (batch == 0 || max_new == 0) {  // only the queries: no compressor work
        js.n_jobs = 0;
        return launch_compress(js, w, 0, 0, static_cast<cudaStream_t>(stream));
    }
    for (int k = 0; k < n_jobs; ++k) {
        const dsa_compress_job_t& j = jobs[k];
        const dsa_status_t e = make_job(batch, max_new, w, s, j.x_new, j.logit_new, j.state_x, j.state_logit,
                                        j.rms_gamma, j.rms_eps, j.rope, j.out, j.out_bt, j.swa, j.swa_bt,
                                        j.gate_per_channel, &js.job[k]);
        if (e != DSA_OK) return e;
        CompressArgs& a = js.job[k];
        a.cu_new = cu_new;
        a.start_pos = start_pos;
        a.state_slot = state_slot;
        a.num_slots = num_slots;
        a.status = dev_status;
    }
    return launch_compress(js, w, batch, max_new, static_cast<cudaStream_t>(stream));
}

extern "C" dsa_status_t dsa_compress(int32_t kind, int32_t batch, const int32_t* cu_new, const int32_t* start_pos,
                                     int32_t max_new, const void* x_new, const float* logit_new, void* state_x,
                                     float* state_logit, const int32_t* state_slot, int32_t num_slots,
                                     const float* rms_gamma, float rms_eps, const dsa_rope_t* rope,
                                     const dsa_pool_t* out, const dsa_block_table_t* out_bt, const dsa_pool_t* swa,
                                     const dsa_block_table_t* swa_bt, int32_t* dev_status, void* stream) {
    if (kind != DSA_C4A && kind != DSA_C128A) return DSA_ERR_INVALID_ARG;
    if (batch < 0 || max_new < 0 || num_slots <= 0 || !(rms_eps > 0.f)) return DSA_ERR_INVALID_ARG;
    if (batch == 0 || max_new == 0) return DSA_OK;
    const dsa_compress_job_t job{x_new, logit_new, state_x, state_logit, rms_gamma, rms_eps, rope, out, out_bt, swa,
                                 swa_bt, 0};
    return compress_jobs(kind, batch, cu_new, start_pos, max_new, state_slot, num_slots, 1, &job, nullptr, dev_status,
                         stream);
}

extern "C" dsa_status_t dsa_compress_jobs(int32_t kind, int32_t batch, const int32_t* cu_new,
                                          const int32_t* start_pos, int32_t max_new, const int32_t* state_slot,
                                          int32_t num_slots, int32_t n_jobs, const dsa_compress_job_t* jobs,
                                          const dsa_query_job_t* query, int32_t* dev_status, void* stream) {
    return compress_jobs(kind, batch, cu_new, start_pos, max_new, state_slot, num_slots, n_jobs, jobs, query,
                         dev_status, stream);
}
