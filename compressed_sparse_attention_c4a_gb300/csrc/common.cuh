// Device and host helpers shared by the libdsa kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <utility>

#include "dsa.h"

namespace dsa {

constexpr int kBlockPositions = 256;  // raw positions per logical block, every cache kind
constexpr double kTwoPi = 6.283185307179586476925286766559;

// -------------------------------------------------------------------------------------
// host side
// -------------------------------------------------------------------------------------
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int window_of(int kind) { return kind == DSA_C4A ? 8 : 128; }
inline int stride_of(int kind) { return kind == DSA_C4A ? 4 : 128; }

inline dsa_status_t launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Every kernel asks for the largest shared-memory carveout: an SM changes its shared-memory / L1 split only
// when it is idle, so a kernel launched with a small carveout (little shared memory) would leave SMs on which
// the next kernel's large CTAs fit once at a time, the second starting only when the first ends.
template <typename... Exp>
inline void prefer_max_shared(void (*kernel)(Exp...)) {
    cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel), cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
}

// As launch_pdl, in clusters of `cluster` CTAs along x (grid.x a multiple of it).
template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl_cluster(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                      int cluster, Act&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    prefer_max_shared(kernel);
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Act&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prefer_max_shared(kernel);
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link dependency).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

inline int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

inline bool pool_ok(const dsa_pool_t* p) {
    if (!p || !p->data || p->num_blocks <= 0 || p->rows_per_block <= 0 || p->dim <= 0) return false;
    if (p->dtype != DSA_BF16 && p->dtype != DSA_FP8_E4M3 && p->dtype != DSA_FP4_E2M1) return false;
    if (p->dtype != DSA_BF16 && (!p->scale || !aligned(p->scale, 16))) return false;
    if (p->dtype == DSA_FP4_E2M1 && (p->dim % 64 || !aligned(p->data, 32))) return false;
    return aligned(p->data, 16);
}

// Bytes of one pool row.
inline long long row_bytes_of(const dsa_pool_t* p) {
    return p->dtype == DSA_BF16 ? 2ll * p->dim : (p->dtype == DSA_FP8_E4M3 ? p->dim : p->dim / 2);
}

inline bool table_ok(const dsa_block_table_t* t, int batch) {
    return t && t->table && t->max_blocks > 0 && t->batch >= batch;
}

// -------------------------------------------------------------------------------------
// device side
// -------------------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with programmatic stream
// serialisation, so it may be scheduled while its predecessor on the stream is still running.  Each
// kernel does only on-chip set-up (barriers, TMEM allocation, shared memory) before pdl_wait(), which
// returns once the predecessor grid has completed and its writes are visible; it then lets its own
// dependent start its set-up (pdl_launch_dependents).  So at most one kernel runs ahead, and only
// through work that touches no global memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Timeline instrumentation, compiled only into builds with -DDSA_TIMELINE (never the library itself):
// DSA_STAMP(k) writes the SM clock to slot k of the CTA's 32-slot record in a buffer that an exported
// setter of the translation unit installs; slots 30 and 31 hold %globaltimer at the CTA's end and start.
#ifdef DSA_TIMELINE
#define DSA_TIMELINE_BUFFER static __device__ unsigned long long* g_timeline;
#define DSA_STAMP(k)                                                                              \
    do {                                                                                          \
        if (g_timeline) {                                                                         \
            unsigned long long c_;                                                                \
            asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_));                                    \
            g_timeline[(unsigned long long)blockIdx.x * 32 + (k)] = c_;                           \
        }                                                                                         \
    } while (0)
#define DSA_STAMP_NS(k)                                                                           \
    do {                                                                                          \
        if (g_timeline) {                                                                         \
            unsigned smid_;                                                                       \
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                    \
            g_timeline[(unsigned long long)blockIdx.x * 32 + 29] = smid_;                         \
            g_timeline[(unsigned long long)blockIdx.x * 32 + (k)] = global_ns();                  \
        }                                                                                         \
    } while (0)
// DSA_TRACE(n, k): the SM clock of event k of work item n of CTAs 0-7 (items below 64), in records 8192 + .
#define DSA_TRACE(n, k)                                                                           \
    do {                                                                                          \
        if (g_timeline && blockIdx.x < 8 && (n) < 64) {                                           \
            unsigned long long c_;                                                                \
            asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_));                                    \
            g_timeline[(8192ull + blockIdx.x * 64 + (n)) * 32 + (k)] = c_;                        \
        }                                                                                         \
    } while (0)
#define DSA_TIMELINE_SETTER(name)                                                                 \
    extern "C" int name(void* p) {                                                                \
        unsigned long long* q = static_cast<unsigned long long*>(p);                              \
        return cudaMemcpyToSymbol(dsa::g_timeline, &q, sizeof(q)) == cudaSuccess ? 0 : 1;         \
    }
#else
#define DSA_TIMELINE_BUFFER
#define DSA_STAMP(k) ((void)0)
#define DSA_STAMP_NS(k) ((void)0)
#define DSA_TRACE(n, k) ((void)0)
#define DSA_TIMELINE_SETTER(name)
#endif
DSA_TIMELINE_BUFFER  // one buffer pointer per translation unit

// Monotone 32-bit key of a score (the top-k's radix digits): a larger float has a larger key; -0 and +0 share
// one key.  Shared by the indexer (which counts each row's top 11 bits while scoring) and the top-k.
__device__ __forceinline__ uint32_t dsa_score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// First error wins; later errors leave the recorded code in place.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// Bounds checks of computed shared-memory and table indexes, compiled into DSA_CHECKED builds only: an index
// outside [0, n) records DSA_ERR_DEVICE_FAULT in the status word and the guarded access is skipped (never a
// trap).  In other builds the check is the constant true and costs nothing.
#ifdef DSA_CHECKED
__device__ __forceinline__ bool dsa_index_ok(long long i, long long n, int32_t* status) {
    if (i >= 0 && i < n) return true;
    report(status, DSA_ERR_DEVICE_FAULT);
    return false;
}
#define DSA_IDX_OK(i, n, status) dsa_index_ok((long long)(i), (long long)(n), (status))
#else
#define DSA_IDX_OK(i, n, status) true
#endif

// Number of entries of a kind (window w, stride s) that T raw tokens form.
__device__ __forceinline__ int entries_formed(long long T, int w, int s) {
    return T < w ? 0 : (int)((T - w) / s + 1);
}

// Physical row of logical row `i` (rows_per_block `epb`) of request `r`, or -1 if the
// block is unmapped, outside the pool or beyond the table.
__device__ __forceinline__ long long physical_row(const dsa_block_table_t& bt, int r, long long i, int epb,
                                                  int num_blocks) {
    long long lb = i / epb;
    if (i < 0 || lb >= bt.max_blocks) return -1;
    int pb = __ldg(bt.table + (long long)r * bt.max_blocks + lb);
    if (pb < 0 || pb >= num_blocks) return -1;
    return (long long)pb * epb + (i - lb * epb);
}

// RoPE frequencies theta^(-2j / rope_dim), j < rope_dim / 2, computed on the host in double precision and
// passed by value in the kernel arguments (no device memory, no device-side pow).
struct RopeTable {
    float f_hi[32], f_lo[32];  // inv_freq of each pair as a float pair: hi + lo carries 48 of its bits
    int rope_dim;
};

inline RopeTable make_rope_table(int rope_dim, double theta) {
    RopeTable t{};
    t.rope_dim = rope_dim;
    for (int j = 0; j < rope_dim / 2 && j < 32; ++j) {
        const double f = pow(theta, -2.0 * j / (double)rope_dim);
        t.f_hi[j] = (float)f;
        t.f_lo[j] = (float)(f - (double)t.f_hi[j]);
    }
    return t;
}

// 2 pi as three floats (Cody-Waite): A + B + C equals 2 pi to within 5e-23; 1 / (2 pi) rounded to float.
constexpr float kTwoPiA = 0x1.921fb6p+2f, kTwoPiB = -0x1.777a5cp-23f, kTwoPiC = -0x1.ee59dap-48f;
constexpr float kInvTwoPiF = 0x1.45f306p-3f;

// cos / sin of pos * inv_freq_j.  A float angle at positions near 2^20 has no fraction bits left, and the
// GPU's fp64 rate is a small fraction of its fp32 rate, so the angle is kept as a float pair instead: the
// product of the position (exact as a float below 2^24) with hi + lo is p + e, e = the product's rounding
// error (one fma, exact) + pos * lo; p is reduced modulo 2 pi with k = rint(p / 2 pi) by one fma per part of
// 2 pi, each rounding a result of magnitude <= 4 once, and e is added last.  The reduced angle is within
// about 3e-7 rad of the exact one below 2^24; larger (or negative) positions take an fp64 reduction.  The
// reduced angle lies in [-pi - 1, pi + 1], where the hardware sine and cosine (__sincosf) are accurate to
// about 5e-7 absolute and take a few instructions (sincosf also carries a long path for huge arguments,
// code that a kernel rotating 8 pairs per lane would repeat 8 times).
__device__ __forceinline__ void rope_cos_sin(long long pos, const RopeTable& t, int j, float* c, float* s) {
    const float hi = t.f_hi[j], lo = t.f_lo[j];
    float r;
    if (pos < 0 || pos >= (1ll << 24)) {
        const double a = (double)pos * ((double)hi + (double)lo);
        r = (float)fma(-kTwoPi, rint(a * (1.0 / kTwoPi)), a);
    } else {
        const float x = (float)pos;
        const float p = x * hi;
        const float e = fmaf(x, hi, -p) + x * lo;
        const float k = rintf(p * kInvTwoPiF);
        r = fmaf(-k, kTwoPiA, p);
        r = fmaf(-k, kTwoPiB, r);
        r = fmaf(-k, kTwoPiC, r) + e;
    }
    __sincosf(r, s, c);
}

__device__ __forceinline__ uint16_t float_to_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// e4m3 encode (round to nearest even, saturate to +-448) and decode via CUDA's conversions.
__device__ __forceinline__ uint8_t float_to_e4m3(float f) {
    return (uint8_t)__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3);
}

// Two values -> one byte of e2m1 codes (x in the low nibble), round to nearest even, saturating (CUDA's conversion).
__device__ __forceinline__ uint8_t float2_to_e2m1x2(float x, float y) {
    return (uint8_t)__nv_cvt_float2_to_fp4x2(make_float2(x, y), __NV_E2M1, cudaRoundNearest);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- shared-memory addresses, mbarriers and bulk copies (PTX) ----------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit_ns` nanoseconds of %globaltimer and returns false.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate copy or MMA

// 16-byte asynchronous copy global -> shared, zero-filled beyond src_bytes (L2 only, not L1).
__device__ __forceinline__ void cp_async16_nc(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on an mbarrier once all of this thread's earlier cp.async copies are complete (the arrival is part
// of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled tensor copy global -> shared with the tensor map's swizzle.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// L2 cache policies for the access hints below: data read once (streamed keys, gathered rows) is marked to
// leave L2 first, so that it does not push out what the step reuses (kernel code, scores, queries, tables).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Raise the barrier's expected transaction bytes without arriving (the arrival comes later).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// 1-D bulk copy from this CTA's shared memory into another CTA's of the cluster (both shared::cluster
// addresses from mapa for the destination and its mbarrier), completing on the destination's mbarrier.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, uint32_t src_smem, uint32_t bytes,
                                               uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_cluster),
                 "r"(src_smem), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}
// 2-D tiled tensor copy shared -> global (a box of the tensor map at {x, y}), tracked by the issuing thread's
// bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x), "r"(y),
                 "r"(smem_u32(src))
                 : "memory");
}
// Wait until at most N of this thread's bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- tcgen05 (5th-generation tensor cores, TMEM accumulators) ---------------------------
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

// N (4, 8 or 16) columns without waiting: the registers are valid only after tmem_wait_ld(), and are
// passed through an empty asm there so that no use can be scheduled before it.
template <int N>
__device__ __forceinline__ void tmem_ld_nowait(uint32_t taddr, float (&v)[N]) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    if constexpr (N == 16)
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
    else if constexpr (N == 8)
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    else
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr)
                     : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// After tmem_wait_ld(): ties the registers of a tmem_ld_nowait to a point after the wait.
template <int N>
__device__ __forceinline__ void tmem_regs_after_wait(float (&v)[N]) {
#pragma unroll
    for (int i = 0; i < N; i += 4) asm volatile("" : "+f"(v[i]), "+f"(v[i + 1]), "+f"(v[i + 2]), "+f"(v[i + 3]));
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// A kind::f16 MMA (A and B from shared-memory descriptors) issued by one elected lane of a converged warp
// (every lane executes the call): issue through elect.sync costs about half the cycles of a single diverged
// thread.
__device__ __forceinline__ void mma_bf16_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_f8_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// Prefetch `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128B swizzle: start address, leading / stride byte offsets.
//   K-major operand: SBO = distance between 8-row groups (LBO unused).
//   MN-major operand: LBO = distance between 64-element (128-byte) atoms along M/N, SBO = distance
//   between 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, M = m (64 or 128), N = n; a_mn = 1
// when A is MN-major (transposed), B K-major.  With M = 64 (one CTA) row r of D sits in TMEM lane
// 32 (r / 16) + r % 16: lanes 0-15 of each warp's quadrant.
__device__ __forceinline__ uint32_t idesc_bf16(int n, int a_mn, int m = 128) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// ---- thread-block clusters (distributed shared memory) -----------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA in the cluster arrives once per phase, then waits for the others.
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float x, float y, float z, float w) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}
// Named barrier over `count` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Arrive at named barrier `id` without waiting (the threads that sync on it see this thread's earlier writes).
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace dsa
