// Status strings and the block-table gather hook of libdsa.
//
// dsa_gather_rows copies the stored bytes of logical cache rows through a request's block table
// ([P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" §2.2 PagedAttention; [P2] "DeepSeek V4
// 稀疏注意力完全解剖" 设计 1: 256 raw positions per logical block), with the same translation the
// attention kernels use, so that the translation can be compared bit for bit.
#include "common.cuh"

extern "C" const char* dsa_status_string(dsa_status_t status) {
    switch (status) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported size";
        case DSA_ERR_CUDA: return "CUDA launch failure";
        case DSA_ERR_DEVICE_FAULT: return "device-detected fault (unmapped block, bad position or index)";
        case DSA_ERR_TIMEOUT: return "bounded wait expired";
        default: return "unknown status";
    }
}

namespace dsa {

// One warp per row: 16-byte pieces of the row, then its scale.
__global__ void __launch_bounds__(256) gather_rows_kernel(dsa_pool_t pool, dsa_block_table_t bt, int n,
                                                          const int32_t* req, const int32_t* ids, uint8_t* out,
                                                          float* out_scale, int row_bytes, int32_t* status) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (j >= n) return;
    const int r = req[j];
    long long prow = -1;
    if (r >= 0 && r < bt.batch) prow = physical_row(bt, r, ids[j], pool.rows_per_block, pool.num_blocks);
    uint4* dst = reinterpret_cast<uint4*>(out + (long long)j * row_bytes);
    const int pieces = row_bytes / 16;
    if (prow < 0) {
        for (int c = lane; c < pieces; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        if (lane == 0) {
            if (out_scale) out_scale[j] = 0.f;
            report(status, DSA_ERR_DEVICE_FAULT);
        }
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(pool.data) + prow * row_bytes);
    for (int c = lane; c < pieces; c += 32) dst[c] = src[c];
    if (lane == 0 && out_scale && pool.dtype != DSA_BF16) out_scale[j] = pool.scale[prow];
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_gather_rows(const dsa_pool_t* pool, const dsa_block_table_t* bt, int32_t n,
                                        const int32_t* req, const int32_t* ids, void* out, float* out_scale,
                                        int32_t* dev_status, void* stream) {
    if (n < 0) return DSA_ERR_INVALID_ARG;
    if (n == 0) return DSA_OK;
    if (!pool_ok(pool) || !bt || !bt->table || bt->max_blocks <= 0 || bt->batch <= 0 || !req || !ids || !out)
        return DSA_ERR_INVALID_ARG;
    const int row_bytes = (int)row_bytes_of(pool);
    if (row_bytes % 16 || !aligned(out, 16)) return DSA_ERR_INVALID_ARG;
    if (launch_pdl(gather_rows_kernel, dim3((n + 7) / 8), dim3(256), 0, static_cast<cudaStream_t>(stream), *pool, *bt,
                   n, req, ids, static_cast<uint8_t*>(out), out_scale, row_bytes, dev_status) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_status();
}
