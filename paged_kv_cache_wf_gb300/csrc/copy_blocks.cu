// copy_blocks.cu -- copy-on-write block copy for prefix sharing.
//
// tiny-vllm-py, "Prefix Sharing": requests with a common prefix point their block
// tables at the same physical blocks; before a request appends into a shared,
// partly filled block it needs a private copy.  ember lists the same thing as
// "copy-on-write block tables".  Each (src, dst) pair copies all P slots of block
// src to block dst, in the K pool and in the V pool.
//
// HBM-bound byte copy: grid-stride over (pair, 16-byte chunk), streaming loads of
// the source (read-only for the duration of the call: no block is both a source
// and a destination) and plain stores, with the grid a fixed multiple of the SM
// count.  Ids outside [0, N) are skipped and flagged.
#include "wf_internal.h"

namespace wf {

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                          const int32_t* __restrict__ pairs, int64_t num_pairs,
                                                          int32_t num_blocks, int64_t block_chunks,
                                                          uint32_t* dev_status) {
    const int64_t total = num_pairs * block_chunks;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t pr = i / block_chunks;
        const int64_t c = i - pr * block_chunks;
        const int32_t src = __ldg(pairs + 2 * pr);
        const int32_t dst = __ldg(pairs + 2 * pr + 1);
        if ((unsigned)src >= (unsigned)num_blocks || (unsigned)dst >= (unsigned)num_blocks) {
            if (c == 0) report(dev_status, WF_DEV_BAD_BLOCK);
            continue;
        }
        const uint4 kv = ld_global_stream(k_pool + src * block_chunks + c);
        const uint4 vv = ld_global_stream(v_pool + src * block_chunks + c);
        st_global_v4(k_pool + dst * block_chunks + c, kv);
        st_global_v4(v_pool + dst * block_chunks + c, vv);
    }
}

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int32_t num_pairs,
                               const wf_pool_desc& pool, uint32_t* dev_status, cudaStream_t stream) {
    const int64_t block_bytes =
        (int64_t)pool.block_size * pool.num_kv_heads * pool.head_dim * dtype_bytes(pool.dtype);
    const int64_t block_chunks = block_bytes / 16;
    const int64_t total = (int64_t)num_pairs * block_chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident 256-thread CTAs per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    copy_blocks_kernel<<<(unsigned)blocks, threads, 0, stream>>>((uint4*)k_pool, (uint4*)v_pool, pairs, num_pairs,
                                                                 pool.num_blocks, block_chunks, dev_status);
    return cudaGetLastError();
}

}  // namespace wf
