// reshape_and_cache.cu -- scatter of this step's new K/V rows into the block pool.
//
// weft, "Cache layouts": the paged cache is written by a scatter through
// slot_mapping; token t lands in block slot/P at offset slot%P of the per-layer
// [N, P, H_kv, D] view.  In that row-major view the (block, offset) pair is the
// flat row index block*P + offset == slot, so one [H_kv, D] row is one
// contiguous run of row_bytes at pool + slot*row_bytes.
//
// HBM-bound byte copy: every thread moves 16-byte chunks with a non-allocating
// streaming load and a plain store (fp8 pools: 16 codes per chunk, quantized).  Grid-stride over (token, chunk) pairs so
// the grid is a fixed multiple of the SM count whatever T is.
#include "wf_internal.h"

namespace wf {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
    int64_t num_slots, int row_chunks, uint32_t* dev_status) {
    const int64_t total = num_tokens * row_chunks;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / row_chunks;
        const int c = (int)(i - t * row_chunks);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (c == 0) report(dev_status, WF_DEV_BAD_SLOT);
            continue;
        }
        const uint4 kv = ld_global_stream(k + t * row_chunks + c);
        const uint4 vv = ld_global_stream(v + t * row_chunks + c);
        st_global_v4(k_pool + slot * row_chunks + c, kv);
        st_global_v4(v_pool + slot * row_chunks + c, vv);
    }
}

// fp8 e4m3 pools (ember, "Deliberately out of scope": paged KV quantization): the
// bf16 rows are quantized on the way in, code = e4m3(float(x) * inv_scale_h) with
// round-to-nearest-even and saturation at +-448 (NaN stays NaN), inv_scale_h the
// float32 reciprocal of KV head h's scale.  A thread writes 16 codes (one 16-byte
// chunk of the pool row, inside one head since D % 16 == 0) from 32 bytes of input.
struct InvScales {
    float k[kMaxScaleHeads];
    float v[kMaxScaleHeads];
};

__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
    int64_t num_slots, int row_chunks, int head_chunks, const InvScales inv, uint32_t* dev_status) {
    const int64_t total = num_tokens * row_chunks;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / row_chunks;
        const int c = (int)(i - t * row_chunks);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (c == 0) report(dev_status, WF_DEV_BAD_SLOT);
            continue;
        }
        const int64_t in = (t * row_chunks + c) * 2;   // 16 bf16 = two 16-byte chunks
        uint4 kq, vq;
        // pools with more heads than the table carry one per-tensor scale (the entry
        // point allows per-head scales only up to kMaxScaleHeads heads)
        const int h = min(c / head_chunks, kMaxScaleHeads - 1);
        quantize16_e4m3(ld_global_stream(k + in), ld_global_stream(k + in + 1), inv.k[h], kq);
        quantize16_e4m3(ld_global_stream(v + in), ld_global_stream(v + in + 1), inv.v[h], vq);
        st_global_v4(k_pool + slot * row_chunks + c, kq);
        st_global_v4(v_pool + slot * row_chunks + c, vq);
    }
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                     const int64_t* slot_mapping, int32_t num_tokens,
                                     const wf_pool_desc& pool, uint32_t* dev_status,
                                     cudaStream_t stream) {
    const int64_t row_bytes = (int64_t)pool.num_kv_heads * pool.head_dim * dtype_bytes(pool.dtype);
    const int row_chunks = (int)(row_bytes / 16);
    const int64_t total = (int64_t)num_tokens * row_chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident 256-thread CTAs per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (pool.dtype == WF_DTYPE_FP8_E4M3) {
        const HeadScales sc = head_scales(pool);
        InvScales inv;
        for (int h = 0; h < kMaxScaleHeads; ++h) {
            inv.k[h] = 1.0f / sc.k[h];
            inv.v[h] = 1.0f / sc.v[h];
        }
        reshape_and_cache_fp8_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
            (const uint4*)k, (const uint4*)v, (uint4*)k_pool, (uint4*)v_pool, slot_mapping, num_tokens,
            (int64_t)pool.num_blocks * pool.block_size, row_chunks, pool.head_dim / 16, inv, dev_status);
        return cudaGetLastError();
    }
    reshape_and_cache_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        (const uint4*)k, (const uint4*)v, (uint4*)k_pool, (uint4*)v_pool, slot_mapping, num_tokens,
        (int64_t)pool.num_blocks * pool.block_size, row_chunks, dev_status);
    return cudaGetLastError();
}

}  // namespace wf
