// paged_decode_tc.cu -- launchers of the tensor-core decode (the kernel body and
// its design notes are in paged_decode_tc.cuh).
#include "paged_decode_tc.cuh"

namespace wf {

namespace {

template <int G, int D, int HT>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    decode_tc_body<G, D, HT>(tm_k, tm_v, tm_q, p, smem_raw, (int)blockIdx.x, (int)gridDim.x);
}



template <int G, int D, int HT>
cudaError_t launch_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q, const TcParams& p,
                      int64_t items, cudaStream_t stream) {
    using L = TcCfg<G, D>;
    const int smem = L::total + 1024;
    auto kern = paged_decode_tc_kernel<G, D, HT>;
    cudaError_t err = allow_dynamic_smem((const void*)kern, smem);
    if (err != cudaSuccess) return err;
    const int64_t ctas = num_sms();
    const int grid = (int)(items < ctas ? items : ctas);
    // a programmatic dependent of the reset: its set-up overlaps, its producer waits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, tm_q, p);
}

template <int D, int G>
cudaError_t launch_g(int HT, const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                     const TcParams& p, int64_t items, cudaStream_t stream) {
    switch (HT) {
        case 8: return launch_tc<G, D, 8>(tm_k, tm_v, tm_q, p, items, stream);
        case 4: return launch_tc<G, D, 4>(tm_k, tm_v, tm_q, p, items, stream);
        case 2: return launch_tc<G, D, 2>(tm_k, tm_v, tm_q, p, items, stream);
        default: return launch_tc<G, D, 1>(tm_k, tm_v, tm_q, p, items, stream);
    }
}

template <int D>
cudaError_t launch_d(int G, int HT, const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                     const TcParams& p, int64_t items, cudaStream_t stream) {
    if (G == 1) return launch_g<D, 1>(HT, tm_k, tm_v, tm_q, p, items, stream);
    if (G == 2) return launch_g<D, 2>(HT, tm_k, tm_v, tm_q, p, items, stream);
    return launch_g<D, 4>(HT, tm_k, tm_v, tm_q, p, items, stream);
}

}  // namespace

bool decode_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads) {
    if (pool.dtype != WF_DTYPE_BF16 || (pool.head_dim != 64 && pool.head_dim != 128)) return false;
    if (pool.block_size % kBoxPos != 0 || pool.num_kv_heads < 1 || num_q_heads % pool.num_kv_heads != 0) return false;
    const int G = num_q_heads / pool.num_kv_heads;
    return G == 1 || G == 2 || G == 4;
}

int decode_tc_span(const wf_pool_desc& pool) { return tc_span(pool.head_dim, 8 / heads_per_box(pool.num_kv_heads)); }

cudaError_t launch_paged_decode_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                   int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                   float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                   cudaStream_t stream) {
    const int G = num_q_heads / pool.num_kv_heads;
    const int D = pool.head_dim;
    const int HT = heads_per_box(pool.num_kv_heads);
    CUtensorMap tm_k, tm_v, tm_q;
    TcParams p;
    int64_t items = 0;
    cudaError_t e = decode_tc_prepare(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, B,
                                      max_seq_len, num_q_heads, scale, pool, ws_o, ws_ml, max_splits, queue,
                                      dev_status, tm_k, tm_v, tm_q, p, items);
    if (e != cudaSuccess) return e;
    decode_queue_reset_kernel<<<1, 32, 0, stream>>>(queue);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return D == 64 ? launch_d<64>(G, HT, tm_k, tm_v, tm_q, p, items, stream)
                   : launch_d<128>(G, HT, tm_k, tm_v, tm_q, p, items, stream);
}

}  // namespace wf
