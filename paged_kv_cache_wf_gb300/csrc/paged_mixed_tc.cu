// paged_mixed_tc.cu -- one launch for the attention of a mixed continuous-batching
// step: the causal prefill of the step's new requests and the decode of its running
// sequences, both over the same paged pool.
//
// The step mixes prefill and decode work (tiny-vllm-py, "Inference Server Flow";
// ember, "Deliberately out of scope": a proper prefill/decode mix per step).  Issued
// as two launches, each ends in a ragged tail: the prefill's last CTAs (its longest
// query blocks, one per request and KV head) leave most SMs idle while they finish,
// and the decode only starts after them.  Here one grid carries both programs:
//
//   * CTAs 0 .. n_pf - 1 run the pipelined tensor-core prefill (paged_prefill_tc.cuh),
//     one per (request, KV head, query block), longest query blocks first;
//   * the n_dec CTAs after them run the persistent tensor-core decode
//     (paged_decode_tc.cuh), claiming work items from its queue.
//
// CTAs are dispatched in index order as SMs free up, so the decode CTAs start on
// the SMs the prefill's tail leaves idle and take decode items from one queue until
// it is empty: no SM is set aside for either kind of work.  (The standalone prefill
// runs as a persistent grid whose CTAs finish together; here the one-CTA-per-block
// grid's ragged end is what the decode fills, and it measured 1.1% faster a step.)  The block has the
// prefill's 12 warps; a decode CTA runs on its first 6 (the others leave at once,
// and the decode's block-wide barriers are named barriers over those 6 warps).
// Both programs only read the pool, and they write disjoint outputs, so the result
// is the same as the two separate calls.
#include "paged_decode_tc.cuh"
#include "paged_prefill_tc.cuh"

namespace wf {

namespace {

static_assert(kThreads >= kDecodeThreads, "a decode CTA runs on the first warps of the block");

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    paged_mixed_tc_kernel(const __grid_constant__ CUtensorMap pf_q, const __grid_constant__ CUtensorMap pf_k,
                          const __grid_constant__ CUtensorMap pf_v, const PfParams pp,
                          const __grid_constant__ CUtensorMap dec_k, const __grid_constant__ CUtensorMap dec_v,
                          const __grid_constant__ CUtensorMap dec_q, const TcParams dp, int n_pf, int pf_gx) {
    extern __shared__ unsigned char smem_raw[];
    const int cta = (int)blockIdx.x;
    if (cta < n_pf) {
        prefill_tc_body<D, G>(pf_q, pf_k, pf_v, pp, smem_raw, cta % pf_gx, cta / pf_gx);
        return;
    }
    if (threadIdx.x >= kDecodeThreads) return;
    decode_tc_body<G, D, 8>(dec_k, dec_v, dec_q, dp, smem_raw, cta - n_pf, (int)gridDim.x - n_pf);
}

template <int D, int G>
cudaError_t launch_mixed(const CUtensorMap& pq, const CUtensorMap& pk, const CUtensorMap& pv, PfParams pp,
                         const CUtensorMap& dk, const CUtensorMap& dv, const CUtensorMap& dq, const TcParams& dp,
                         int64_t items, cudaStream_t stream) {
    using PL = PfLayout<D, G>;
    using DL = TcCfg<G, D>;
    pp.nqblk = (pp.max_q_len + PL::BMQ - 1) / PL::BMQ;
    const int pf_gx = pp.B * pp.H_kv;
    const int64_t n_pf = (int64_t)pf_gx * pp.nqblk;
    const int64_t sms = num_sms();
    const int64_t n_dec = items < sms ? items : sms;
    if (n_pf + n_dec > INT32_MAX) return cudaErrorInvalidValue;
    const int smem = (PL::total > DL::total ? PL::total : DL::total) + 1024;
    auto kern = paged_mixed_tc_kernel<D, G>;
    cudaError_t err = allow_dynamic_smem((const void*)kern, smem);
    if (err != cudaSuccess) return err;
    // a programmatic dependent of the decode queue's reset: the prefill CTAs never
    // wait for it, the decode CTAs do before their first claim
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_pf + n_dec));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, pq, pk, pv, pp, dk, dv, dq, dp, (int)n_pf, pf_gx);
}

}  // namespace

bool mixed_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads) {
    const int G = pool.num_kv_heads > 0 ? num_q_heads / pool.num_kv_heads : 0;
    return decode_tc_supported(pool, num_q_heads) && prefill_tc_supported(pool, num_q_heads) &&
           pool.num_kv_heads % 8 == 0 && (G == 1 || G == 2 || G == 4) &&
           (int64_t)pool.num_blocks * pool.block_size <= INT32_MAX;
}

cudaError_t launch_paged_mixed_tc(void* pf_out, const void* pf_q, const int32_t* pf_block_tables,
                                  int32_t pf_max_blocks_per_seq, const int32_t* pf_seq_lens, const int32_t* cu_q_lens,
                                  int32_t pf_B, int32_t total_q, int32_t max_q_len, int32_t pf_max_seq_len,
                                  void* dec_out, const void* dec_q, const int32_t* dec_block_tables,
                                  int32_t dec_max_blocks_per_seq, const int32_t* dec_seq_lens, int32_t dec_B,
                                  int32_t dec_max_seq_len, const void* k_pool, const void* v_pool,
                                  int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                  float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                  cudaStream_t stream) {
    CUtensorMap pq, pk, pv, dk, dv, dq;
    PfParams pp;
    TcParams dp;
    int64_t items = 0;
    cudaError_t e = prefill_tc_prepare(pf_out, pf_q, k_pool, v_pool, pf_block_tables, pf_max_blocks_per_seq,
                                       pf_seq_lens, cu_q_lens, pf_B, total_q, max_q_len, pf_max_seq_len, num_q_heads,
                                       scale, pool, dev_status, pq, pk, pv, pp);
    if (e != cudaSuccess) return e;
    e = decode_tc_prepare(dec_out, dec_q, k_pool, v_pool, dec_block_tables, dec_max_blocks_per_seq, dec_seq_lens,
                          dec_B, dec_max_seq_len, num_q_heads, scale, pool, ws_o, ws_ml, max_splits, queue,
                          dev_status, dk, dv, dq, dp, items);
    if (e != cudaSuccess) return e;
    decode_queue_reset_kernel<<<1, 32, 0, stream>>>(queue);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int G = num_q_heads / pool.num_kv_heads;
    if (pool.head_dim == 64) {
        if (G == 1) return launch_mixed<64, 1>(pq, pk, pv, pp, dk, dv, dq, dp, items, stream);
        if (G == 2) return launch_mixed<64, 2>(pq, pk, pv, pp, dk, dv, dq, dp, items, stream);
        return launch_mixed<64, 4>(pq, pk, pv, pp, dk, dv, dq, dp, items, stream);
    }
    if (G == 1) return launch_mixed<128, 1>(pq, pk, pv, pp, dk, dv, dq, dp, items, stream);
    if (G == 2) return launch_mixed<128, 2>(pq, pk, pv, pp, dk, dv, dq, dp, items, stream);
    return launch_mixed<128, 4>(pq, pk, pv, pp, dk, dv, dq, dp, items, stream);
}

}  // namespace wf
