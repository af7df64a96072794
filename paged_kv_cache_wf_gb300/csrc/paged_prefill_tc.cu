// paged_prefill_tc.cu -- launchers of the pipelined tensor-core prefill: the
// persistent grid (paged_prefill_persist.cuh) when the batch is within its list
// build's limits, else one CTA per query block (paged_prefill_tc.cuh).
#include "paged_prefill_persist.cuh"

namespace wf {

namespace {

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const PfParams p) {
    extern __shared__ unsigned char smem_raw[];
    prefill_tc_body<D, G>(tm_q, tm_k, tm_v, p, smem_raw, (int)blockIdx.x, (int)blockIdx.y);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v, const PfParams p) {
    extern __shared__ unsigned char smem_raw[];
    prefill_tc_persist<D, G>(tm_q, tm_k, tm_v, p, smem_raw, (int)blockIdx.x, (int)gridDim.x);
}

template <int D, int G>
cudaError_t launch_pf(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, PfParams p,
                      cudaStream_t stream) {
    const int pgrid = prefill_persist_grid<D, G>(p.B, p.max_q_len, p.H_kv, num_sms());
    if (pgrid > 0) {
        const int smem = PpLayout<D, G>::total + 1024;
        auto kern = paged_prefill_persist_kernel<D, G>;
        cudaError_t err = allow_dynamic_smem((const void*)kern, smem);
        if (err != cudaSuccess) return err;
        kern<<<pgrid, kThreads, smem, stream>>>(tq, tk, tv, p);
        return cudaGetLastError();
    }
    using L = PfLayout<D, G>;
    p.nqblk = (p.max_q_len + L::BMQ - 1) / L::BMQ;
    const int smem = L::total + 1024;
    auto kern = paged_prefill_tc_kernel<D, G>;
    cudaError_t err = allow_dynamic_smem((const void*)kern, smem);
    if (err != cudaSuccess) return err;
    dim3 grid(p.B * p.H_kv, p.nqblk);
    kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads) {
    if (pool.dtype != WF_DTYPE_BF16 || pool.block_size % 16 != 0) return false;
    if (pool.head_dim != 64 && pool.head_dim != 128) return false;
    if (num_q_heads % pool.num_kv_heads != 0) return false;
    const int G = num_q_heads / pool.num_kv_heads;
    return G == 1 || G == 2 || G == 4 || G == 8;
}

cudaError_t launch_paged_prefill_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                                    int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                                    int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                    uint32_t* dev_status, cudaStream_t stream) {
    const int D = pool.head_dim;
    const int G = num_q_heads / pool.num_kv_heads;
    CUtensorMap tq, tk, tv;
    PfParams p;
    cudaError_t e = prefill_tc_prepare(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens,
                                       B, total_q, max_q_len, max_seq_len, num_q_heads, scale, pool, dev_status, tq,
                                       tk, tv, p);
    if (e != cudaSuccess) return e;
    if (D == 128) {
        switch (G) {
            case 1: return launch_pf<128, 1>(tq, tk, tv, p, stream);
            case 2: return launch_pf<128, 2>(tq, tk, tv, p, stream);
            case 4: return launch_pf<128, 4>(tq, tk, tv, p, stream);
            default: return launch_pf<128, 8>(tq, tk, tv, p, stream);
        }
    }
    switch (G) {
        case 1: return launch_pf<64, 1>(tq, tk, tv, p, stream);
        case 2: return launch_pf<64, 2>(tq, tk, tv, p, stream);
        case 4: return launch_pf<64, 4>(tq, tk, tv, p, stream);
        default: return launch_pf<64, 8>(tq, tk, tv, p, stream);
    }
}

}  // namespace wf
