/*
 * dsa.h - C ABI of libdsa.so: one DeepSeek-V4-style compressed sparse attention layer
 * step (c4a / c128a) on a GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" (gentlecold.top)
 *   [P2] "DeepSeek V4 稀疏注意力完全解剖" (zoe.im)
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.  Every pointer argument is DEVICE memory owned by the caller unless the
 *   comment says "host".  The library never allocates or frees memory and keeps no
 *   mutable global state, so calls are reentrant and can be recorded in a CUDA graph.
 *   The one exception is dsa_sparse_attn_decode_static (below): a fixed scratch array in
 *   the library image plus a per-device cache of its address.
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).  Every call only
 *   enqueues work on that stream and returns; none synchronises.
 * Host-side errors.  A call returns DSA_OK or an error code; when the host-side checks
 *   fail no kernel is launched and no memory is touched.
 *     DSA_ERR_INVALID_ARG  null / misaligned pointer, inconsistent sizes
 *     DSA_ERR_UNSUPPORTED  a size outside what the kernels implement (stated per call)
 *     DSA_ERR_CUDA         the CUDA runtime refused a launch
 * Device-side errors.  `dev_status` (optional, one int32 in device memory, may be NULL)
 *   receives the first error that a kernel detects (first writer wins; a zero value is
 *   never overwritten with zero, so the caller clears it):
 *     DSA_ERR_DEVICE_FAULT a needed block is unmapped (-1) or outside the pool, a
 *                          position lies beyond its block table, or an index is out of
 *                          range; the affected row is written as zeros (scores: -inf)
 *     DSA_ERR_TIMEOUT      a bounded wait on an asynchronous copy or MMA expired
 *   Kernels never trap or assert.
 * Paged caches ([P2] 设计 1; [P1] §2.2, §6.1).  A logical block always covers 256 raw
 *   token positions: 64 c4a entries, 2 c128a entries or 256 SWA tokens.  Compressed
 *   entry i (stride s) lives in logical block i / (256/s), row i % (256/s); raw token p
 *   lives in SWA block p / 256, row p % 256.  A request's block table row maps logical
 *   blocks to physical blocks of a pool; -1 marks an unmapped block.
 * RoPE ([P2] 深潜：为什么必须做 Inverse RoPE).  Acts on the last rope_dim dims of a row
 *   in interleaved pairs (dim - rope_dim + 2j, dim - rope_dim + 2j + 1), angle
 *   pos * theta^(-2j / rope_dim); the angle is formed in double precision.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t dsa_status_t;
#define DSA_OK 0
#define DSA_ERR_INVALID_ARG 1
#define DSA_ERR_UNSUPPORTED 2
#define DSA_ERR_CUDA 3
#define DSA_ERR_DEVICE_FAULT 4
#define DSA_ERR_TIMEOUT 5

/* storage formats of a pool row */
#define DSA_BF16 0
#define DSA_FP8_E4M3 1 /* e4m3 bytes + one fp32 scale per row: value = scale * e4m3(code) */
#define DSA_FP4_E2M1 2 /* e2m1 codes packed two per byte (element 2j in the low nibble) + one fp32 scale per
                          row: value = scale * e2m1(code); [P2] 第三层 (the fp4 indexer cache); indexer keys only */

/* compressor kinds ([P1] §5.2, [P2] 机制二) */
#define DSA_C4A 0   /* window 8 raw tokens, stride 4: 64 entries per block */
#define DSA_C128A 1 /* window 128, stride 128: 2 entries per block */

/* A paged pool.  data: [num_blocks][rows_per_block][dim] elements (bf16 or e4m3 bytes; e2m1: dim / 2 bytes
 * per row), row-major and contiguous, 16-byte aligned (e2m1: 32-byte).  scale: [num_blocks][rows_per_block]
 * fp32, required for DSA_FP8_E4M3 and DSA_FP4_E2M1, ignored for DSA_BF16. */
typedef struct dsa_pool {
    void* data;
    float* scale;
    int32_t num_blocks;
    int32_t rows_per_block;
    int32_t dim;
    int32_t dtype;
} dsa_pool_t;

/* Block tables: table[r * max_blocks + b] = physical block of request r's logical block b. */
typedef struct dsa_block_table {
    const int32_t* table;
    int32_t batch;
    int32_t max_blocks;
} dsa_block_table_t;

typedef struct dsa_rope {
    int32_t rope_dim; /* even, <= dim; 64 for the main cache */
    double theta;     /* 10000 */
} dsa_rope_t;

/* Human-readable name of a status code (static string; never NULL). */
const char* dsa_status_string(dsa_status_t status);

/*
 * dsa_compress - compressor + RMSNorm + RoPE + paged insert, and SWA insert.
 * [P1] §5.2 / [P2] 机制二 (c4a: weighted sum of 8 raw tokens at stride 4; c128a: 128 at
 * stride 128), [P2] 融合点 1 (compress -> RMSNorm -> RoPE -> cache insert in one pass),
 * [P2] 设计 2 (the rolling residual of the last w raw tokens), [P2] 融合点 3 (SWA keys:
 * RoPE then insert).
 *
 * Request r appends raw tokens x_new[cu_new[r] .. cu_new[r+1]) at positions
 * start_pos[r], start_pos[r] + 1, ...  Every entry i whose last covered token
 * s*i + w - 1 is among them is formed as
 *     g = softmax_j(z_{s*i+j}),  u = sum_j g_j x_{s*i+j},
 *     v = gamma * u / sqrt(mean(u^2) + eps),  entry = R_{s*i+w-1} v
 * and stored at logical row i of `out` through row r of `out_bt` (bf16, or e4m3 with
 * scale = amax/448 when out->dtype is DSA_FP8_E4M3).  Window tokens older than
 * start_pos[r] are read from the rolling state slot state_slot[r]:
 * state_x[slot][p % w][dim] (bf16) and state_logit[slot][p % w] (fp32).  Afterwards the
 * state holds the request's last w raw tokens (slot position p % w).  With `swa` non-NULL
 * each new token p is also stored as R_p x_p at SWA logical row p through swa_bt.
 *
 * kind       DSA_C4A or DSA_C128A (w, s) = (8, 4) or (128, 128)
 * batch      requests (host int, >= 0; 0 is a no-op)
 * cu_new     [batch + 1] int32, cu_new[0] = 0, non-decreasing
 * start_pos  [batch] int32 >= 0
 * max_new    host int: an upper bound of cu_new[r+1] - cu_new[r] over r (grid sizing)
 * x_new      [cu_new[batch]][dim] bf16;  logit_new [cu_new[batch]] fp32
 * state_*    rolling state; num_slots host int = number of slots; state_slot [batch]
 * rms_gamma  [dim] fp32 or NULL (= all ones);  rms_eps > 0
 * out        bf16, e4m3 or e2m1 pool (e2m1: scale = amax/6), rows_per_block = 256/s;  swa: rows_per_block = 256
 *            (bf16 or e4m3), or NULL
 * Supported: dim in {64, 128, 512}, rope_dim even and <= min(dim, 64).
 * Launched with programmatic dependent launch: cu_new, start_pos, state_slot, the block tables and rms_gamma
 * are read before waiting for the preceding kernel in the stream; the raw tokens, logits and rolling state
 * are read, and the pools and state written, only after it.
 */
dsa_status_t dsa_compress(int32_t kind, int32_t batch, const int32_t* cu_new, const int32_t* start_pos,
                          int32_t max_new, const void* x_new, const float* logit_new, void* state_x,
                          float* state_logit, const int32_t* state_slot, int32_t num_slots,
                          const float* rms_gamma, float rms_eps, const dsa_rope_t* rope,
                          const dsa_pool_t* out, const dsa_block_table_t* out_bt, const dsa_pool_t* swa,
                          const dsa_block_table_t* swa_bt, int32_t* dev_status, void* stream);

/*
 * dsa_compress_jobs - dsa_compress of up to 4 caches of one layer in one launch.  [P2] 融合点 3 (per-token work
 * of one layer that touches different caches runs side by side in one kernel, picked by warp and block index).
 * The jobs share the requests and their new tokens' positions (kind, batch, cu_new, start_pos, max_new,
 * state_slot, num_slots: as dsa_compress); each job has its own raw rows, logits, rolling state, norm weights,
 * RoPE, pool and optional window pool, with the meaning, layout and checks of dsa_compress (a layer's main
 * cache with its window insert, and its indexer cache).  Each job's results equal those of its own
 * dsa_compress call.  The jobs must not share an output row or a rolling state.  n_jobs: 1 .. 4.
 */
typedef struct dsa_compress_job {
    const void* x_new;          /* [cu_new[batch]][dim] bf16 */
    const float* logit_new;     /* [cu_new[batch]] */
    void* state_x;              /* [num_slots][w][dim] bf16 */
    float* state_logit;         /* [num_slots][w] */
    const float* rms_gamma;     /* [dim] or NULL */
    float rms_eps;
    const dsa_rope_t* rope;
    const dsa_pool_t* out;
    const dsa_block_table_t* out_bt;
    const dsa_pool_t* swa;      /* or NULL */
    const dsa_block_table_t* swa_bt;
    int32_t gate_per_channel;   /* 0: one logit per raw token (logit_new [n], state_logit [slots][w]);
                                   1: one per raw token and channel (logit_new [n][dim], state_logit
                                   [slots][w][dim], both 16-byte aligned), a softmax over the window for every
                                   channel c: u_c = sum_j softmax_j(z_{., c}) x_{j, c} (a variant: the pages
                                   say only "weighted sum") */
} dsa_compress_job_t;

/*
 * The query job of dsa_compress_jobs ([P2] 融合点 3: the Q-norm beside the key RoPE and insert): every
 * (query, head) row of q_raw becomes q_out = R_m(gamma * q / sqrt(mean(q^2) + eps)), m = q_pos[query], the
 * rotation on the last rope_dim dims, as bf16 (the queries dsa_sparse_attn_* take, rotated at their
 * position).  q_raw, q_out: [nq][heads][dim] bf16, 16-byte aligned (q_out may be q_raw); q_pos [nq] int32
 * (read before waiting for the preceding kernel; a negative position raises DSA_ERR_DEVICE_FAULT and leaves
 * that row); rms_gamma [dim] fp32 or NULL (ones); rms_eps > 0; dim in {64, 128, 512}; rope_dim even,
 * <= min(dim, 64).  nq = 0 is no work.
 */
typedef struct dsa_query_job {
    int32_t nq;
    int32_t heads;
    int32_t dim;
    const void* q_raw;
    void* q_out;
    const int32_t* q_pos;
    const float* rms_gamma;
    float rms_eps;
    const dsa_rope_t* rope;
} dsa_query_job_t;

/* query: NULL, or the layer's queries, prepared in the same launch by warps of their own (batch or max_new may
 * then be 0: the queries alone). */
dsa_status_t dsa_compress_jobs(int32_t kind, int32_t batch, const int32_t* cu_new, const int32_t* start_pos,
                               int32_t max_new, const int32_t* state_slot, int32_t num_slots, int32_t n_jobs,
                               const dsa_compress_job_t* jobs, const dsa_query_job_t* query, int32_t* dev_status,
                               void* stream);

/*
 * dsa_index_scores - lightning-indexer scores of each query against every visible
 * c4a entry.  [P1] §4.1 (a few heads, FP8), [P2] 机制三.  With e4m3 query codes q8 and
 * per-(query, head) scale sq, e4m3 key codes k8 with per-entry scale sk:
 *     I(m, i) = sum_h w_h * max(0, sq_h * sk_i * <q8_h, k8_i>),  i < n_vis(m),
 * n_vis(m) = number of c4a entries whose last covered token is <= m.
 * Computed on the tensor cores (tcgen05, fp8 x fp8 -> fp32) from key tiles that TMA
 * stages in shared memory.
 *
 * nq         queries (host);  heads in {4, 8, 16};  dim in {64, 128}
 * keys       e4m3 (DSA_FP8_E4M3) or, with dim 128, e2m1 (DSA_FP4_E2M1: the tensor cores take the fp4 codes as
 *            they are, A = e2m1, B = e4m3) pool, rows_per_block 64, dim = dim; bt: its block table
 * q8         [nq][heads][dim] e4m3 bytes;  q_scale, w: [nq][heads] fp32
 * q_pos      [nq] int32 position m of each query;  q_req [nq] int32 request of each query
 * q_group    host int in 1 .. 256/heads: queries g*q_group .. g*q_group + q_group - 1 must
 *            belong to one request (decode: 1; chunked prefill: up to 256/heads, at most 64); a
 *            group that mixes requests raises DSA_ERR_DEVICE_FAULT; at most 4096 groups
 *            (ceil(nq / q_group)), else DSA_ERR_UNSUPPORTED
 * scores     [nq][ld] fp32 out: I(m, i) for i < n_vis(m); -inf for n_vis(m) <= i < the end of
 *            the 128-entry tile holding n_vis(m) - 1; the rest of the row is not written
 * ld         host int, >= n_vis of every query, a multiple of 4
 * n_visible  [nq] int32 out (n_vis per query), or NULL
 * fresh_pos  [batch] int32: for request r, the first raw position whose tokens the preceding kernel in the
 *            stream may still be compressing into the key pool (after dsa_compress of this step: its
 *            start_pos[r]); or NULL.  The entries those tokens can complete, i >= n_vis(fresh_pos[r] - 1)
 *            (c4a: 4i + 7 >= fresh_pos[r]), may still be written; older entries may not.
 * work       NULL (each CTA scores an equal share of the entries), or [2] uint32, 8-byte aligned, zero before the
 *            first call: the CTAs take runs of consecutive (query group, 128-entry tile) items from this counter,
 *            so a CTA that starts late (its SM still busy with another kernel) takes less; the last CTA leaves
 *            it zero again.  Calls that may overlap on the GPU must not share it.
 * Launched with programmatic dependent launch, so the kernel may start before the preceding kernel in
 * the stream has finished.  q_pos, q_req and bt are always read before waiting for it.  Without
 * fresh_pos, keys, queries and every output are touched only after the wait.  With fresh_pos, key pages
 * wholly below entry n_vis(fresh_pos[r] - 1), the queries, and the scores / n_visible outputs may be touched before
 * it: a preceding kernel that releases its dependents early must not write those inputs or read those
 * outputs after releasing them.  The call ends after the preceding kernel in every case.
 */
dsa_status_t dsa_index_scores(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8, const float* q_scale,
                              const float* w, const int32_t* q_pos, const int32_t* q_req, int32_t q_group,
                              const dsa_pool_t* keys, const dsa_block_table_t* bt, float* scores, int32_t ld,
                              int32_t* n_visible, const int32_t* fresh_pos, uint32_t* work, int32_t* dev_status,
                              void* stream);

/*
 * dsa_index_scores_counted / dsa_topk_counted / dsa_index_topk - the indexer and the per-query top-k with the
 * top-k's first pass fused into the indexer.  [P1] §4.1-4.2 (I_t, then S_t = TopK(I_t, k)), [P2] 第四层 (fuse
 * work so that intermediate data is not read back).
 *
 * dsa_index_scores_counted is dsa_index_scores (same arguments, results and launch rules) that, while scoring,
 * also counts each query row's visible scores by the top 11 bits of a monotone 32-bit key of the score:
 * counts [nq][2048] uint32, zero-filled before the call (16-byte aligned).  Rows of at most ld = 16,384 scores.
 * dsa_topk_counted is dsa_topk for such rows (ld <= 16,384, else DSA_ERR_UNSUPPORTED) that starts from those
 * counts: the bucket of the k-th largest score comes from them, so the top-k reads its row once; it selects
 * the same set, in the same order, as dsa_topk and leaves the counts zero-filled again.
 * dsa_index_topk issues the two (for ld > 16,384: dsa_index_scores then dsa_topk), with the counts and the
 * indexer's work counter in `workspace` (>= dsa_index_topk_workspace_size(nq) bytes): zero-filled by the caller
 * before the first call;
 * every call that completes leaves it zero-filled (one that records DSA_ERR_TIMEOUT may not: clear it then).
 * Calls that overlap on the GPU race on it.
 *
 * k          host int, 1 .. 2048;  idx_out [nq][k] int32 out;  n_visible required (the top-k's row lengths)
 * scores     16-byte aligned
 */
size_t dsa_index_topk_workspace_size(int32_t nq);
dsa_status_t dsa_index_scores_counted(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8, const float* q_scale,
                                      const float* w, const int32_t* q_pos, const int32_t* q_req, int32_t q_group,
                                      const dsa_pool_t* keys, const dsa_block_table_t* bt, float* scores, int32_t ld,
                                      int32_t* n_visible, const int32_t* fresh_pos, uint32_t* work, unsigned* counts,
                                      int32_t* dev_status, void* stream);
dsa_status_t dsa_topk_counted(int32_t nq, const float* scores, int32_t ld, const int32_t* n_valid, int32_t k,
                              int32_t* idx_out, unsigned* counts, int32_t* dev_status, void* stream);
dsa_status_t dsa_index_topk(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8, const float* q_scale,
                            const float* w, const int32_t* q_pos, const int32_t* q_req, int32_t q_group,
                            const dsa_pool_t* keys, const dsa_block_table_t* bt, float* scores, int32_t ld,
                            int32_t* n_visible, const int32_t* fresh_pos, int32_t k, int32_t* idx_out,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * dsa_debug_index_scores_stalled - test hook of the bounded waits in dsa_index_scores; the pages have no
 * counterpart.  Launches the indexer as dsa_index_scores would (fresh_pos = NULL), except that the warp that
 * issues the key and query copies issues none and posts no work, so the tensor-core and epilogue warps wait
 * for tiles that never arrive.  Each of their waits gives up after wait_limit_ns nanoseconds (of
 * %globaltimer): the kernel records DSA_ERR_TIMEOUT in dev_status, every warp leaves its loop, the tensor
 * memory is freed and the kernel returns, with nothing in flight.  The scores are not written; n_visible is.
 * wait_limit_ns: 1 .. 2e9 (else DSA_ERR_INVALID_ARG).  Other arguments and checks as dsa_index_scores.
 */
dsa_status_t dsa_debug_index_scores_stalled(int32_t nq, int32_t heads, int32_t dim, const uint8_t* q8,
                                            const float* q_scale, const float* w, const int32_t* q_pos,
                                            const int32_t* q_req, int32_t q_group, const dsa_pool_t* keys,
                                            const dsa_block_table_t* bt, float* scores, int32_t ld, int32_t* n_visible,
                                            uint64_t wait_limit_ns, int32_t* dev_status, void* stream);

/*
 * dsa_topk - per-query top-k of indexer scores.  [P1] §4.2: S_t = TopK(I_{t,:}, k).
 * Row q selects the k largest of scores[q][0 .. n_valid[q]), ties broken toward the
 * lower index, so the selected set is unique; idx_out[q] lists it in increasing index
 * order, padded with -1 when n_valid[q] < k.  Exact (radix select on the fp32 bit
 * patterns); NaN scores are not supported.
 *
 * nq, k      host ints; 1 <= k <= 2048; ld <= 163,840 (else DSA_ERR_UNSUPPORTED)
 * scores     [nq][ld] fp32;  n_valid [nq] int32 in [0, ld]
 * idx_out    [nq][k] int32 out
 */
dsa_status_t dsa_topk(int32_t nq, const float* scores, int32_t ld, const int32_t* n_valid, int32_t k,
                      int32_t* idx_out, int32_t* dev_status, void* stream);

/*
 * dsa_topk_plan - how dsa_topk runs for these sizes on the current device; host only, launches nothing.
 * plan[0] = kernel (0: the row in registers, for ld <= 16,384: one CTA of 1024 threads per row, or, while
 * four CTAs per row fit on the GPU at once, a cluster of four 512-thread CTAs holding a quarter each; 1: a
 * cluster of CTAs per row, each holding one part of the row in shared memory), plan[1] = CTAs per row,
 * plan[2] = threads per CTA.
 * Returns DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED as dsa_topk would for these sizes.
 */
dsa_status_t dsa_topk_plan(int32_t nq, int32_t ld, int32_t k, int32_t* plan);

/*
 * Workspace (bytes) that dsa_sparse_attn_decode / _prefill need for nq query rows of
 * `heads` heads and at most `max_keys` keys per row (compressed + window) on the current
 * device, for either pool format: the fp32 partial outputs and (max, sums) of rows whose keys
 * are split over several groups of CTAs.  0 means the call needs none.
 */
size_t dsa_attn_workspace_size(int32_t nq, int32_t heads, int32_t max_keys);

/*
 * dsa_attn_plan - how dsa_sparse_attn_decode / _prefill split the work for these sizes on
 * the current device and pool format (dtype DSA_BF16 or DSA_FP8_E4M3); host only, launches
 * nothing.  plan[0] = heads per CTA, plan[1] = CTAs per cluster (one query row's keys shared
 * among them), plan[2] = key splits per row, plan[3] = kernels one call launches (1, or 2 with
 * the split merge).  Returns DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED as the attention call
 * would for these sizes.
 */
dsa_status_t dsa_attn_plan(int32_t nq, int32_t heads, int32_t max_keys, int32_t dtype, int32_t* plan);

/*
 * dsa_sparse_attn_decode - main attention of one decode query per request.
 * [P1] §4.2-4.3 (attention over the top-k entries, MQA mode: every entry is shared by
 * all heads), [P2] 机制一 (K = V: one stored row is both key and value), [P2] 机制四 /
 * [P1] §5.3 (a 128-token sliding window of uncompressed tokens is seen together with the
 * compressed entries), [P2] 深潜 (inverse RoPE on the output), [P2] 融合点 2 (fused into
 * the output store).  For query row b at position m = q_pos[b], request b:
 *     keys = {main row i : i in topk[b], i >= 0}  U  {swa row p : max(0, m-window+1) <= p <= m}
 *     p_hj = softmax_j(<q_bh, key_j> * sm_scale),  o_bh = sum_j p_hj key_j
 *     out_bh = o_bh with its last rope_dim dims rotated by R_m^-1.
 * topk == NULL selects every visible entry i < n_vis(m) (the c128a layer).
 *
 * batch      rows (host);  heads in {16, 32, 64, 128}
 * q          [batch][heads][512] bf16, already rotated at m;  q_pos [batch] int32
 * kind       DSA_C4A or DSA_C128A (visibility and rows_per_block of `main`)
 * topk       [batch][k] int32 logical entry ids (-1 = none) or NULL;  k host int <= 2048
 * main, swa  pools with dim 512, bf16 or fp8 (per-row scale);  window: host int, 1..1024
 * sm_scale   host float (1/sqrt(512) in the layer)
 * out        [batch][heads][512] bf16;  lse [batch][heads] fp32 (natural log of the softmax
 *            denominator) or NULL
 * workspace  >= dsa_attn_workspace_size(batch, heads, max_keys) bytes, 256-byte aligned, or
 *            NULL when that size is 0; max_keys = (topk ? k : main_bt->max_blocks *
 *            main->rows_per_block) + window
 * Supported: dim 512, rope_dim <= 64.
 * Launched with programmatic dependent launch: q, q_pos (q_req) and both block tables are read before
 * waiting for the preceding kernel in the stream, so a preceding kernel that releases its dependents
 * early must not write them after releasing; top-k indices, cache rows and every output come after the
 * wait.  A row with a device fault (an unmapped block or an index >= n_vis) is written as zeros, lse -inf.
 */
dsa_status_t dsa_sparse_attn_decode(int32_t batch, int32_t heads, const void* q, const int32_t* q_pos,
                                    int32_t kind, const int32_t* topk, int32_t k, const dsa_pool_t* main,
                                    const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                    const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                    const dsa_rope_t* rope, void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * dsa_sparse_attn_prefill - the same attention for nq query tokens of a chunk, each with
 * its own position, request and top-k row (causal: a token sees only entries and window
 * tokens at or before its position).  Arguments as dsa_sparse_attn_decode, plus
 * q_req [nq] int32 mapping each query row to its request's table rows.
 */
dsa_status_t dsa_sparse_attn_prefill(int32_t nq, int32_t heads, const void* q, const int32_t* q_pos,
                                     const int32_t* q_req, int32_t kind, const int32_t* topk, int32_t k,
                                     const dsa_pool_t* main, const dsa_block_table_t* main_bt,
                                     const dsa_pool_t* swa, const dsa_block_table_t* swa_bt, int32_t window,
                                     float sm_scale, const dsa_rope_t* rope, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                     void* stream);

/*
 * dsa_topk_sparse_attn_decode - dsa_topk followed by dsa_sparse_attn_decode over its output, in one kernel
 * where the work split allows it.  [P1] §4.2 (S_t = TopK(I_t), then attention over S_t), [P2] 第四层 (kernel
 * fusion: adjacent steps of the path share one launch so that the intermediate never leaves the chip): the
 * cluster of CTAs that attends to a query row first selects the row's top-k from its scores, keeps the
 * selected entry ids in shared memory and gathers those rows.
 *     topk_out[b] = dsa_topk's row b of (scores, n_visible, k);  out, lse = dsa_sparse_attn_decode(topk_out)
 * scores     [batch][ld] fp32, 16-byte aligned, ld a multiple of 4;  n_visible [batch] int32
 * topk_out   [batch][k] int32 (required): the selected entry ids, exactly as dsa_topk writes them
 * Other arguments as dsa_sparse_attn_decode with topk = topk_out (workspace sized for max_keys = k + window).
 * One kernel when one cluster of four CTAs per row holds all heads without a key split (64 heads, at most
 * 38 rows on a 152-SM GPU), ld <= 16,384 and k <= 512 (dsa_attn_plan(batch, heads, k + window) gives
 * (64, 4, 1, 1)); else the two calls in sequence.  Programmatic dependent launch as dsa_sparse_attn_decode:
 * scores and n_visible are read after the wait.  Errors: those of both calls.
 */
dsa_status_t dsa_topk_sparse_attn_decode(int32_t batch, int32_t heads, const void* q, const int32_t* q_pos,
                                         int32_t kind, const float* scores, int32_t ld, const int32_t* n_visible,
                                         int32_t k, int32_t* topk_out, const dsa_pool_t* main,
                                         const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                         const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                         const dsa_rope_t* rope, void* out, float* lse, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * dsa_sparse_attn_q8 - the same attention (decode rows when q_req is NULL, else prefill rows as
 * dsa_sparse_attn_prefill) with the output in e4m3 for an fp8 projection that follows: [P2] 融合点 2 (the
 * inverse rotation and the fp8 quantisation fused into one pass over the output, no bf16 round trip).
 * Each 128-dim block of each (row, head) output is scaled by its own amax / 448 (1 for an all-zero block):
 *     out_scale[row][h][b] = max_{d in block b} |o_hd| / 448,   out[row][h][d] = e4m3(o_hd / out_scale[row][h][b])
 * where o is the output dsa_sparse_attn_decode would store in bf16 (R_m^-1 already applied), rounded to nearest
 * even with saturation.
 * out        [nq][heads][512] e4m3 bytes, 16-byte aligned;  out_scale [nq][heads][4] fp32, 16-byte aligned
 * Other arguments, results, workspace and errors as dsa_sparse_attn_decode / _prefill (a faulted row: zero codes,
 * scales 1, lse -inf).
 */
dsa_status_t dsa_sparse_attn_q8(int32_t nq, int32_t heads, const void* q, const int32_t* q_pos, const int32_t* q_req,
                                int32_t kind, const int32_t* topk, int32_t k, const dsa_pool_t* main,
                                const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                const dsa_rope_t* rope, uint8_t* out, float* out_scale, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * dsa_sparse_attn_decode_static - dsa_sparse_attn_decode without a caller workspace, for callers that
 * cannot allocate device memory: a serving loop that forbids cudaMalloc on its hot path (an allocation
 * can synchronise the device and stall every stream), a host whose device memory all belongs to its
 * own arena with no allocator to call, or a plugin that is only handed the input and output pointers.
 * The pages have no counterpart to this call; it exists for those callers only.
 *
 * Arguments and results are those of dsa_sparse_attn_decode minus `workspace` / `workspace_bytes`.
 * The split-K partials live in a fixed array inside the library image, of
 * dsa_attn_static_scratch_bytes() bytes (32 MiB) on every GPU that loads the library, held until the
 * process exits.  A call whose plan needs more than that (dsa_attn_workspace_size() of the same sizes)
 * returns DSA_ERR_UNSUPPORTED without launching anything.  The call allocates and frees nothing.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and caches it; make that first call before any stream capture.  All calls share the
 * one array and its contents persist between calls, so calls that can overlap on the GPU (two streams,
 * or two host threads on one device) race on it and must be serialised by the caller.
 */
dsa_status_t dsa_sparse_attn_decode_static(int32_t batch, int32_t heads, const void* q, const int32_t* q_pos,
                                           int32_t kind, const int32_t* topk, int32_t k, const dsa_pool_t* main,
                                           const dsa_block_table_t* main_bt, const dsa_pool_t* swa,
                                           const dsa_block_table_t* swa_bt, int32_t window, float sm_scale,
                                           const dsa_rope_t* rope, void* out, float* lse, int32_t* dev_status,
                                           void* stream);

/* Size in bytes of the fixed scratch array that dsa_sparse_attn_decode_static uses (32 MiB). */
size_t dsa_attn_static_scratch_bytes(void);

/*
 * dsa_gather_rows - copy the stored bytes of n logical rows, exactly as the attention
 * reads them, into a dense array (a checking hook for the block-table translation of
 * [P1] §2.2 / [P2] 设计 1).  Row j is logical row ids[j] of request req[j].
 * out: [n][dim * element_size] bytes;  out_scale: [n] fp32 (fp8 pools) or NULL.
 * An unmapped or out-of-range row is written as zeros and raises DSA_ERR_DEVICE_FAULT.
 */
dsa_status_t dsa_gather_rows(const dsa_pool_t* pool, const dsa_block_table_t* bt, int32_t n, const int32_t* req,
                             const int32_t* ids, void* out, float* out_scale, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
