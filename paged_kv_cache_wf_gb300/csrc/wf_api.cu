// wf_api.cu -- the extern "C" boundary of libwf: argument validation (before any
// launch), status mapping, and dispatch to the kernels' launchers.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "wf_internal.h"

namespace wf {

int num_sms() {
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
    cache[dev] = n;
    return n;
}

cudaError_t allow_dynamic_smem(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> done;  // (device, kernel) -> bytes granted
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t key = (reinterpret_cast<uint64_t>(kernel) << 8) ^ (uint64_t)dev;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    if (bytes > 48 * 1024) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (err != cudaSuccess) return err;
    }
    done[key] = bytes;
    return cudaSuccess;
}

cudaError_t encode_tiled_bf16(CUtensorMap* map, void* base, int rank, const uint64_t* dims,
                              const uint64_t* strides, const uint32_t* box) {
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box);
}

cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType type, void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (fn == nullptr) {
            void* f = nullptr;
            cudaDriverEntryPointQueryResult q;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || f == nullptr) return cudaErrorNotSupported;
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        }
    }
    cuuint64_t d[5];
    cuuint64_t s[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) s[i] = strides[i];
    }
    const CUresult r = fn(map, type, (cuuint32_t)rank, base, d, s, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace wf

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

wf_status check_pool(const wf_pool_desc& pool) {
    if (pool.num_blocks < 1 || pool.block_size < 1 || pool.block_size > 1024 ||
        pool.num_kv_heads < 1)
        return WF_ERR_INVALID_ARG;
    if (pool.dtype != WF_DTYPE_F32 && pool.dtype != WF_DTYPE_BF16 && pool.dtype != WF_DTYPE_FP8_E4M3)
        return WF_ERR_UNSUPPORTED;
    if (pool.dtype == WF_DTYPE_FP8_E4M3) {
        auto ok = [](float x) { return x > 0.f && x <= 3.0e38f; };   // finite and positive (NaN fails)
        if (pool.k_head_scales == nullptr && !ok(pool.k_scale)) return WF_ERR_INVALID_ARG;
        if (pool.v_head_scales == nullptr && !ok(pool.v_scale)) return WF_ERR_INVALID_ARG;
        if ((pool.k_head_scales || pool.v_head_scales) && pool.num_kv_heads > wf::kMaxScaleHeads)
            return WF_ERR_UNSUPPORTED;
        for (int h = 0; h < pool.num_kv_heads; ++h) {
            if (pool.k_head_scales && !ok(pool.k_head_scales[h])) return WF_ERR_INVALID_ARG;
            if (pool.v_head_scales && !ok(pool.v_head_scales[h])) return WF_ERR_INVALID_ARG;
        }
    }
    if (pool.head_dim != 64 && pool.head_dim != 128) return WF_ERR_UNSUPPORTED;
    const int64_t slots = (int64_t)pool.num_blocks * pool.block_size;
    if (slots > (int64_t)INT32_MAX * 64) return WF_ERR_INVALID_ARG;
    return WF_OK;
}

wf_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return WF_OK;
    if (e == cudaErrorNotSupported) return WF_ERR_UNSUPPORTED;
    return WF_ERR_CUDA;
}

}  // namespace

extern "C" {

int wf_abi_version(void) { return 104; }

const char* wf_status_string(wf_status s) {
    switch (s) {
        case WF_OK: return "ok";
        case WF_ERR_INVALID_ARG: return "invalid argument";
        case WF_ERR_UNSUPPORTED: return "unsupported configuration";
        case WF_ERR_WORKSPACE: return "workspace missing or too small";
        case WF_ERR_CUDA: return "CUDA error";
        case WF_ERR_NO_BLOCKS: return "not enough free blocks";
    }
    return "unknown status";
}

wf_status wf_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               wf_pool_desc pool, uint32_t* dev_status, cudaStream_t stream) {
    wf_status s = check_pool(pool);
    if (s != WF_OK) return s;
    if (num_tokens < 0) return WF_ERR_INVALID_ARG;
    if (num_tokens == 0) return WF_OK;
    if (!k || !v || !k_pool || !v_pool || !slot_mapping) return WF_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return WF_ERR_INVALID_ARG;
    return from_cuda(wf::launch_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, num_tokens,
                                                  pool, dev_status, stream));
}

wf_status wf_copy_blocks(void* k_pool, void* v_pool, const int32_t* block_pairs, int32_t num_pairs,
                         wf_pool_desc pool, uint32_t* dev_status, cudaStream_t stream) {
    wf_status s = check_pool(pool);
    if (s != WF_OK) return s;
    if (num_pairs < 0) return WF_ERR_INVALID_ARG;
    if (num_pairs == 0) return WF_OK;
    if (!k_pool || !v_pool || !block_pairs) return WF_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || (reinterpret_cast<uintptr_t>(block_pairs) & 3u))
        return WF_ERR_INVALID_ARG;
    return from_cuda(wf::launch_copy_blocks(k_pool, v_pool, block_pairs, num_pairs, pool, dev_status, stream));
}

size_t wf_paged_decode_workspace_size(int32_t B, int32_t num_q_heads, int32_t max_seq_len,
                                      wf_pool_desc pool) {
    if (check_pool(pool) != WF_OK || num_q_heads < 1) return 0;
    return wf::decode_workspace_bytes(B, num_q_heads, max_seq_len, pool);
}

}  // extern "C"

namespace {

// wf_paged_decode's argument rules (WF_OK also for an empty batch, which launches
// nothing).
wf_status decode_args(void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                      int32_t num_q_heads, float scale, const wf_pool_desc& pool, void* workspace,
                      size_t workspace_bytes) {
    wf_status s = check_pool(pool);
    if (s != WF_OK) return s;
    if (B < 0 || num_q_heads < 1 || max_blocks_per_seq < 1 || max_seq_len < 1) return WF_ERR_INVALID_ARG;
    if (num_q_heads % pool.num_kv_heads != 0) return WF_ERR_INVALID_ARG;
    if (num_q_heads / pool.num_kv_heads > 8) return WF_ERR_UNSUPPORTED;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * pool.block_size) return WF_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return WF_ERR_INVALID_ARG;
    if (B == 0) return WF_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens) return WF_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return WF_ERR_INVALID_ARG;
    const size_t need = wf::decode_workspace_bytes(B, num_q_heads, max_seq_len, pool);
    if (need == 0) return WF_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return WF_ERR_WORKSPACE;
    return WF_OK;
}

}  // namespace

extern "C" {

wf_status wf_paged_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                          int32_t num_q_heads, float scale, wf_pool_desc pool,
                          void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                          cudaStream_t stream) {
    const wf_status s = decode_args(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, B,
                                    max_seq_len, num_q_heads, scale, pool, workspace, workspace_bytes);
    if (s != WF_OK || B == 0) return s;
    return from_cuda(wf::launch_paged_decode(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq,
                                             seq_lens, B, max_seq_len, num_q_heads, scale, pool,
                                             workspace, dev_status, stream));
}

}  // extern "C"

namespace {

// wf_paged_prefill's argument rules (WF_OK also for calls that launch nothing).
wf_status prefill_args(void* out, const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* cu_q_lens, int32_t B, int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                       int32_t num_q_heads, float scale, const wf_pool_desc& pool) {
    wf_status s = check_pool(pool);
    if (s != WF_OK) return s;
    if (pool.dtype != WF_DTYPE_BF16) return WF_ERR_UNSUPPORTED;
    if (B < 0 || total_q < 0 || max_q_len < 0 || num_q_heads < 1 || max_blocks_per_seq < 1 ||
        max_seq_len < 0)
        return WF_ERR_INVALID_ARG;
    if (num_q_heads % pool.num_kv_heads != 0) return WF_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * pool.block_size) return WF_ERR_INVALID_ARG;
    if (max_q_len > max_seq_len) return WF_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return WF_ERR_INVALID_ARG;
    if (B == 0 || total_q == 0 || max_q_len == 0) return WF_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !cu_q_lens)
        return WF_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u))
        return WF_ERR_INVALID_ARG;
    return WF_OK;
}

bool prefill_launches(int32_t B, int32_t total_q, int32_t max_q_len) { return B > 0 && total_q > 0 && max_q_len > 0; }

}  // namespace

extern "C" {

wf_status wf_paged_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                           int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                           int32_t num_q_heads, float scale, wf_pool_desc pool,
                           uint32_t* dev_status, cudaStream_t stream) {
    const wf_status s = prefill_args(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens,
                                     B, total_q, max_q_len, max_seq_len, num_q_heads, scale, pool);
    if (s != WF_OK || !prefill_launches(B, total_q, max_q_len)) return s;
    return from_cuda(wf::launch_paged_prefill(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq,
                                              seq_lens, cu_q_lens, B, total_q, max_q_len, max_seq_len,
                                              num_q_heads, scale, pool, dev_status, stream));
}

wf_status wf_paged_prefill_decode(void* pf_out, const void* pf_q, const int32_t* pf_block_tables,
                                  int32_t pf_max_blocks_per_seq, const int32_t* pf_seq_lens,
                                  const int32_t* cu_q_lens, int32_t pf_B, int32_t total_q, int32_t max_q_len,
                                  int32_t pf_max_seq_len, void* dec_out, const void* dec_q,
                                  const int32_t* dec_block_tables, int32_t dec_max_blocks_per_seq,
                                  const int32_t* dec_seq_lens, int32_t dec_B, int32_t dec_max_seq_len,
                                  const void* k_pool, const void* v_pool, int32_t num_q_heads, float scale,
                                  wf_pool_desc pool, void* workspace, size_t workspace_bytes,
                                  uint32_t* dev_status, cudaStream_t stream) {
    wf_status s = prefill_args(pf_out, pf_q, k_pool, v_pool, pf_block_tables, pf_max_blocks_per_seq, pf_seq_lens,
                               cu_q_lens, pf_B, total_q, max_q_len, pf_max_seq_len, num_q_heads, scale, pool);
    if (s != WF_OK) return s;
    s = decode_args(dec_out, dec_q, k_pool, v_pool, dec_block_tables, dec_max_blocks_per_seq, dec_seq_lens, dec_B,
                    dec_max_seq_len, num_q_heads, scale, pool, workspace, workspace_bytes);
    if (s != WF_OK) return s;
    const bool pf = prefill_launches(pf_B, total_q, max_q_len);
    if (!pf && dec_B == 0) return WF_OK;
    return from_cuda(wf::launch_paged_prefill_decode(
        pf_out, pf_q, pf_block_tables, pf_max_blocks_per_seq, pf_seq_lens, cu_q_lens, pf ? pf_B : 0, total_q,
        max_q_len, pf_max_seq_len, dec_out, dec_q, dec_block_tables, dec_max_blocks_per_seq, dec_seq_lens, dec_B,
        dec_max_seq_len, k_pool, v_pool, num_q_heads, scale, pool, workspace, dev_status, stream));
}

wf_status wf_decode_worker(void* out, const void* q, int32_t num_rows, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, int32_t num_table_rows, int32_t max_blocks_per_seq,
                           int32_t num_q_heads, float scale, wf_pool_desc pool, const wf_decode_task* tasks,
                           int32_t task_capacity, wf_worker_mailbox* mailbox, int32_t num_workers,
                           uint64_t idle_timeout_ns, uint32_t* dev_status, cudaStream_t stream) {
    wf_status s = check_pool(pool);
    if (s != WF_OK) return s;
    if (pool.dtype == WF_DTYPE_FP8_E4M3) return WF_ERR_UNSUPPORTED;
    if (num_rows < 0 || num_table_rows < 0 || max_blocks_per_seq < 1 || num_q_heads < 1 || task_capacity < 0)
        return WF_ERR_INVALID_ARG;
    if (num_q_heads % pool.num_kv_heads != 0) return WF_ERR_INVALID_ARG;
    if (num_q_heads / pool.num_kv_heads > 8) return WF_ERR_UNSUPPORTED;
    if (num_workers < 1 || num_workers > 4096 || idle_timeout_ns == 0) return WF_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return WF_ERR_INVALID_ARG;
    if (!mailbox || (reinterpret_cast<uintptr_t>(mailbox) & 15u)) return WF_ERR_INVALID_ARG;
    if (task_capacity > 0 && (!tasks || (reinterpret_cast<uintptr_t>(tasks) & 15u))) return WF_ERR_INVALID_ARG;
    if (num_rows > 0 && (!out || !q || !aligned16(out) || !aligned16(q))) return WF_ERR_INVALID_ARG;
    if (!k_pool || !v_pool || !aligned16(k_pool) || !aligned16(v_pool)) return WF_ERR_INVALID_ARG;
    if (num_table_rows > 0 && (!block_tables || (reinterpret_cast<uintptr_t>(block_tables) & 3u)))
        return WF_ERR_INVALID_ARG;
    return from_cuda(wf::launch_decode_worker(out, q, num_rows, k_pool, v_pool, block_tables, num_table_rows,
                                              max_blocks_per_seq, num_q_heads, scale, pool, tasks, task_capacity,
                                              mailbox, num_workers, idle_timeout_ns, dev_status, stream));
}

int wf_paged_prefill_decode_fused(wf_pool_desc pool, int32_t num_q_heads) {
    if (check_pool(pool) != WF_OK || num_q_heads < 1) return 0;
    return wf::mixed_tc_supported(pool, num_q_heads) ? 1 : 0;
}

int wf_paged_decode_kernel(wf_pool_desc pool, int32_t num_q_heads) {
    if (check_pool(pool) != WF_OK || num_q_heads < 1) return WF_KERNEL_NONE;
    return wf::decode_kernel_kind(pool, num_q_heads);
}

int wf_paged_prefill_kernel(wf_pool_desc pool, int32_t num_q_heads) {
    if (check_pool(pool) != WF_OK || num_q_heads < 1) return WF_KERNEL_NONE;
    return wf::prefill_kernel_kind(pool, num_q_heads);
}

int wf_paged_prefill_persistent(wf_pool_desc pool, int32_t num_q_heads, int32_t B, int32_t max_q_len) {
    if (check_pool(pool) != WF_OK || num_q_heads < 1) return 0;
    if (wf::prefill_kernel_kind(pool, num_q_heads) != WF_KERNEL_TENSOR_CORES) return 0;
    return wf::prefill_tc_persistent(pool, num_q_heads, B, max_q_len) ? 1 : 0;
}

wf_status wf_device_status_fetch(uint32_t* dev_status, uint32_t* host_status, int clear,
                                 cudaStream_t stream) {
    if (!dev_status || !host_status) return WF_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(host_status, dev_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && clear) {
        e = cudaMemsetAsync(dev_status, 0, sizeof(uint32_t), stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return from_cuda(e);
}

}  // extern "C"
