// wf_internal.h -- host-side declarations shared by the libwf translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/wf.h"
#include "wf_device.cuh"

namespace wf {

inline int dtype_bytes(int32_t dtype) { return dtype == WF_DTYPE_F32 ? 4 : (dtype == WF_DTYPE_FP8_E4M3 ? 1 : 2); }

// SM count of the current device (cached per device).
int num_sms();

// Opt a kernel into `bytes` of dynamic shared memory (idempotent, cached).
cudaError_t allow_dynamic_smem(const void* kernel, int bytes);

// Encode a tiled TMA descriptor for a bf16 tensor (128-byte swizzle, no OOB fill).
// dims[0] is the contiguous dimension; strides[] are bytes for dims 1..rank-1.
cudaError_t encode_tiled_bf16(CUtensorMap* map, void* base, int rank, const uint64_t* dims,
                              const uint64_t* strides, const uint32_t* box);
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType type, void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                     const int64_t* slot_mapping, int32_t num_tokens,
                                     const wf_pool_desc& pool, uint32_t* dev_status,
                                     cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int32_t num_pairs,
                               const wf_pool_desc& pool, uint32_t* dev_status, cudaStream_t stream);

// ---- decode -----------------------------------------------------------------
// Positions are cut into fixed spans ("splits") that depend only on the pool
// geometry; each split is one CTA's work and leaves a partial (m, l, o).
struct DecodeGeometry {
    int split_span;   // positions per split (multiple of the tile)
    int tile;         // positions per pipeline stage
    int stages;       // pipeline depth
    int smem_bytes;   // dynamic shared memory per CTA
    int consumer_warps;
    int heads_per_warp;
    int gmax;         // padded GQA group the kernel instance handles
};

bool decode_geometry(const wf_pool_desc& pool, int32_t num_q_heads, DecodeGeometry* g);

// Row of the split partial (o: D floats, (m, l): one float2) of split `split` of
// query head hq of sequence b.  Two layouts, chosen per split kernel by what its
// writes and the combine's reads measured best: split-minor (ps_h = max_splits,
// ps_s = 1), where the splits of one (sequence, query head) are one run of rows,
// and head-minor (ps_h = 1, ps_s = H_q), where one split's query heads are.
__host__ __device__ inline int64_t partial_row(int64_t b, int64_t hq, int64_t split, int64_t H_q,
                                               int64_t max_splits, int64_t ps_h, int64_t ps_s) {
    return b * H_q * max_splits + hq * ps_h + split * ps_s;
}
size_t decode_workspace_bytes(int32_t B, int32_t num_q_heads, int32_t max_seq_len,
                              const wf_pool_desc& pool);

cudaError_t launch_paged_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                void* workspace, uint32_t* dev_status, cudaStream_t stream);
// The wf_kernel value of the decode kernel launch_paged_decode picks for this geometry.
int decode_kernel_kind(const wf_pool_desc& pool, int32_t num_q_heads);

// Tensor-core decode (bf16, D = 128, P % 16 == 0); writes outputs or split
// partials exactly like the CUDA-core kernel, whose combine kernel finishes it.
bool decode_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads);
int decode_tc_span(const wf_pool_desc& pool);   // positions per split
cudaError_t launch_paged_decode_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                   int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                   float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                   cudaStream_t stream);

// Tensor-core decode over fp8 e4m3 pools (H_kv = 8, D = 128, P % 16 == 0,
// G in {2, 4}; bf16 q and outputs); same partials as the bf16 kernel.
bool decode_tc_fp8_supported(const wf_pool_desc& pool, int32_t num_q_heads);
int decode_tc_fp8_span();   // positions per work item of the fp8 kernel
cudaError_t launch_paged_decode_tc_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                       int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                       float2* ws_ml, int32_t max_splits, uint32_t* queue, void* prep,
                                       uint32_t* dev_status, cudaStream_t stream);
// fp8 pools: the scale of each KV head (the per-head arrays when given, else the
// per-tensor scale for every head), read on the host and passed by value.
constexpr int kMaxScaleHeads = 64;
struct HeadScales {
    float k[kMaxScaleHeads];
    float v[kMaxScaleHeads];
};
inline HeadScales head_scales(const wf_pool_desc& pool) {
    HeadScales s;
    for (int h = 0; h < kMaxScaleHeads; ++h) {
        const bool in = h < pool.num_kv_heads;
        s.k[h] = in && pool.k_head_scales ? pool.k_head_scales[h] : pool.k_scale;
        s.v[h] = in && pool.v_head_scales ? pool.v_head_scales[h] : pool.v_scale;
    }
    return s;
}
// Workspace the fp8 decode needs beyond the partials: the prepared q parts and scales.
size_t decode_fp8_prep_bytes(int32_t B, int32_t num_q_heads);

// Persistent decode worker fed while it runs (decode_worker.cu).
cudaError_t launch_decode_worker(void* out, const void* q, int32_t num_rows, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, int32_t num_table_rows, int32_t max_blocks_per_seq,
                                 int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                 const wf_decode_task* tasks, int32_t task_capacity, wf_worker_mailbox* mailbox,
                                 int32_t num_workers, uint64_t idle_timeout_ns, uint32_t* dev_status,
                                 cudaStream_t stream);

// ---- mixed step (paged_mixed_tc.cu) -------------------------------------------
// One launch for a step's prefill and decode over one pool: bf16, both tensor-core
// kernels, H_kv a multiple of 8, groups of 1, 2 or 4.
bool mixed_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads);
cudaError_t launch_paged_mixed_tc(void* pf_out, const void* pf_q, const int32_t* pf_block_tables,
                                  int32_t pf_max_blocks_per_seq, const int32_t* pf_seq_lens, const int32_t* cu_q_lens,
                                  int32_t pf_B, int32_t total_q, int32_t max_q_len, int32_t pf_max_seq_len,
                                  void* dec_out, const void* dec_q, const int32_t* dec_block_tables,
                                  int32_t dec_max_blocks_per_seq, const int32_t* dec_seq_lens, int32_t dec_B,
                                  int32_t dec_max_seq_len, const void* k_pool, const void* v_pool,
                                  int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                  float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                  cudaStream_t stream);
// The step's prefill and decode: one launch when mixed_tc_supported, else the two
// calls one after the other (paged_decode.cu).
cudaError_t launch_paged_prefill_decode(void* pf_out, const void* pf_q, const int32_t* pf_block_tables,
                                       int32_t pf_max_blocks_per_seq, const int32_t* pf_seq_lens,
                                       const int32_t* cu_q_lens, int32_t pf_B, int32_t total_q, int32_t max_q_len,
                                       int32_t pf_max_seq_len, void* dec_out, const void* dec_q,
                                       const int32_t* dec_block_tables, int32_t dec_max_blocks_per_seq,
                                       const int32_t* dec_seq_lens, int32_t dec_B, int32_t dec_max_seq_len,
                                       const void* k_pool, const void* v_pool, int32_t num_q_heads, float scale,
                                       const wf_pool_desc& pool, void* workspace, uint32_t* dev_status,
                                       cudaStream_t stream);

// ---- prefill ------------------------------------------------------------------
// Pipelined tcgen05 prefill (bf16, P % 16 == 0, G in {1, 2, 4, 8}, D in {64, 128}).
bool prefill_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads);
cudaError_t launch_paged_prefill_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                                    int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                                    int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                    uint32_t* dev_status, cudaStream_t stream);

// The wf_kernel value of the prefill kernel launch_paged_prefill picks.
int prefill_kernel_kind(const wf_pool_desc& pool, int32_t num_q_heads);
// Whether the pipelined tensor-core prefill runs this batch shape as its persistent grid.
bool prefill_tc_persistent(const wf_pool_desc& pool, int32_t num_q_heads, int32_t B, int32_t max_q_len);
cudaError_t launch_paged_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                                 int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                                 int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                 uint32_t* dev_status, cudaStream_t stream);

}  // namespace wf
