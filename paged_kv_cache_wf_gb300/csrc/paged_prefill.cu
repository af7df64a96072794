// paged_prefill.cu -- causal varlen attention of new tokens over the paged pool,
// with QK^T and PV on the 5th-generation tensor cores (tcgen05, TMEM).
//
// What is computed (tiny-vllm-py, "KV Cache": prefill attention is causal;
// "Dense vs. Ragged batching": requests packed back to back by offsets):
//   request b owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1; with n_b rows and
//   a cached prefix of c_b = seq_lens[b] - n_b tokens, row i (position c_b + i)
//   attends to positions 0 .. c_b + i, read from the [N, P, H_kv, D] pool through
//   block_table[b][p / P], offset p % P (ember, "The core idea"); query head g uses
//   KV head g / (H_q / H_kv) (weft, "Shapes and symbols").
//
// GB300 design (one CTA = 128 query rows of one request and one query head):
//   * Q, K and V tiles are staged in shared memory in the 128-byte-swizzled
//     K-major layout the tensor cores read directly (K and V rows are gathered per
//     position through the block table; rows past the causal end are zero-filled).
//   * One thread issues S = Q K^T (M=128, N=128 keys, K=D) as tcgen05.mma
//     kind::f16 with bf16 operands from shared memory and the fp32 accumulator in
//     tensor memory; completion is signalled by tcgen05.commit on an mbarrier.
//   * 4 warps (thread i <-> TMEM lane i <-> query row i) read S with tcgen05.ld,
//     apply the causal mask, run the online softmax in fp32 (exp2 domain), rescale
//     the O accumulator in TMEM when the row max moves, and write P as bf16 into a
//     swizzled shared tile.
//   * One thread issues O += P V (M=128, N=D, K=128 keys) with V read as an
//     MN-major operand -- no transpose pass.  The epilogue reads O from TMEM,
//     divides by the row sum and stores bf16.
#include "wf_internal.h"
#include "paged_prefill_persist.cuh"

namespace wf {

namespace {

constexpr int BM = 128;  // query rows per CTA (= TMEM lanes = threads)
constexpr int BN = 128;  // keys per tile

struct PrefillParams {
    __nv_bfloat16* out;
    const __nv_bfloat16* q;
    const char* k_pool;
    const char* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    uint32_t* dev_status;
    int32_t M, B, total_q, max_q_len, max_seq_len, H_q, H_kv, G, N, P;
    float scale_log2;
};

// Byte offset of 16-byte chunk `c` of row `r` in a [128 rows x (8*chunks)] bf16
// tile stored as 64-element column blocks of 128 rows x 128 B (16 KB each), each
// made of 8-row x 128-byte swizzle atoms (chunk index XOR row-in-atom).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)((c >> 3) * (128 * 128) + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(128, 1) paged_prefill_kernel(const PrefillParams p) {
    constexpr int CH = D / 8;             // 16-byte chunks per row
    constexpr int TILE_BYTES = BM * D * 2;
    const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;

    const int q_begin = __ldg(p.cu_q_lens + b);
    const int q_end = __ldg(p.cu_q_lens + b + 1);
    const int n = q_end - q_begin;
    const int len = __ldg(p.seq_lens + b);
    const bool bad = q_begin < 0 || n < 0 || q_end > p.total_q || n > p.max_q_len || len < n ||
                     len > p.max_seq_len || (int64_t)len > (int64_t)p.M * p.P;
    if (bad) {
        if (qt == 0 && hq == 0 && tid == 0) report(p.dev_status, WF_DEV_BAD_SEQLEN);
        return;
    }
    const int i0 = qt * BM;
    if (i0 >= n) return;
    const int c = len - n;                 // cached prefix
    const int rows = min(BM, n - i0);
    const int kend = c + i0 + rows;        // keys this tile needs: [0, kend)
    const int ntiles = (kend + BN - 1) / BN;
    const int h = hq / p.G;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sQ = smem;
    unsigned char* sK = sQ + TILE_BYTES;
    unsigned char* sV = sK + TILE_BYTES;
    unsigned char* sP = sV + TILE_BYTES;  // 128 x 128 bf16
    uint64_t* bar = reinterpret_cast<uint64_t*>(sP + BM * BN * 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

    if (warp == 0) {
        tc::alloc(tmem_slot, 256);
        tc::relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // ---- Q tile ---------------------------------------------------------------
    for (int idx = tid; idx < BM * CH; idx += BM) {
        const int r = idx / CH, cc = idx % CH;
        const int i = i0 + r;
        const bool valid = i < n;
        const __nv_bfloat16* src = valid ? p.q + ((int64_t)(q_begin + i) * p.H_q + hq) * D + cc * 8 : p.q;
        cp_async16(sQ + sw128_off(r, cc), src, valid ? 16u : 0u);
    }
    cp_async_commit();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;         // columns [0, 128): S (fp32)
    const uint32_t tO = tmem + 128;   // columns [128, 128 + D): O (fp32)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    const int row = tid;
    const int qi = i0 + row;
    const bool row_valid = qi < n;
    const int last_key = c + qi;      // row sees keys 0 .. last_key
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t phase = 0;
    bool ok_run = true;
    constexpr uint32_t kIdS = tc::idesc_bf16_f32(BM, BN, 0, 0);
    constexpr uint32_t kIdO = tc::idesc_bf16_f32(BM, D, 0, 1);
    const int64_t pool_row = (int64_t)p.H_kv * D * 2;

    for (int j = 0; j < ntiles && ok_run; ++j) {
        const int k0 = j * BN;
        // ---- K, V tile j, gathered through the block table ------------------
        for (int idx = tid; idx < BN * CH; idx += BM) {
            const int r = idx / CH, cc = idx % CH;
            const int kp = k0 + r;
            const bool valid = kp < kend;
            int blk = 0;
            if (valid) blk = __ldg(p.block_tables + (int64_t)b * p.M + kp / p.P);
            const bool okb = valid && (unsigned)blk < (unsigned)p.N;
            if (valid && !okb && cc == 0) report(p.dev_status, WF_DEV_BAD_BLOCK);
            const int64_t off = okb ? ((int64_t)blk * p.P + kp % p.P) * pool_row + (int64_t)h * D * 2 + cc * 16 : 0;
            cp_async16(sK + sw128_off(r, cc), p.k_pool + off, okb ? 16u : 0u);
            cp_async16(sV + sw128_off(r, cc), p.v_pool + off, okb ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // ---- S = Q K^T --------------------------------------------------------
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                tc::mma_f16(tS, tc::sdesc_sw128(smem_u32(sQ) + off, 16, 1024),
                            tc::sdesc_sw128(smem_u32(sK) + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
            }
            tc::commit(bar);
        }
        if (!mbar_wait(bar, phase)) {
            if (tid == 0) report(p.dev_status, WF_DEV_TIMEOUT);
            ok_run = false;
        }
        phase ^= 1;
        tc::fence_after_sync();

        // ---- online softmax of row `row` over this tile ----------------------
        float s[4][32];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) tc::ld_32cols(tS + lane_base + c4 * 32, s[c4]);
        tc::wait_ld();
        float mt = -INFINITY;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int kp = k0 + c4 * 32 + e;
                const bool vis = row_valid && kp <= last_key;
                s[c4][e] = vis ? s[c4][e] * p.scale_log2 : -INFINITY;
                mt = fmaxf(mt, s[c4][e]);
            }
        const float m_new = fmaxf(m_run, mt);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m_run - m_use);
        float psum = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int e8 = 0; e8 < 4; ++e8) {
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float a = exp2f(s[c4][e8 * 8 + 2 * u] - m_use);
                    const float bb = exp2f(s[c4][e8 * 8 + 2 * u + 1] - m_use);
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, bb);
                    const float2 back = __bfloat1622float2(h2);
                    psum += back.x + back.y;  // sum the weights PV actually uses
                    w[u] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                const int chunk = c4 * 4 + e8;
                *reinterpret_cast<uint4*>(sP + sw128_off(row, chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        // rescale O (in TMEM) where the row max moved; PV of tile j-1 is complete
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                float o[32];
                tc::ld_32cols(tO + lane_base + c4 * 32, o);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= alpha;
                tc::st_32cols(tO + lane_base + c4 * 32, o);
            }
            tc::wait_st();
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // ---- O += P V ---------------------------------------------------------
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                const uint64_t ad = tc::sdesc_sw128(smem_u32(sP) + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t bd = tc::sdesc_sw128(smem_u32(sV) + kk * 2048, 16384, 1024);
                tc::mma_f16(tO, ad, bd, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit(bar);
        }
        if (!mbar_wait(bar, phase)) {
            if (tid == 0) report(p.dev_status, WF_DEV_TIMEOUT);
            ok_run = false;
        }
        phase ^= 1;
        tc::fence_after_sync();
    }

    // ---- epilogue: O / l -> bf16 --------------------------------------------------
    if (ok_run) {
        const float inv = row_valid ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
            float o[32];
            tc::ld_32cols(tO + lane_base + c4 * 32, o);
            tc::wait_ld();
            if (row_valid) {
                __nv_bfloat16* dst = p.out + ((int64_t)(q_begin + qi) * p.H_q + hq) * D + c4 * 32;
#pragma unroll
                for (int e8 = 0; e8 < 4; ++e8) {
                    uint4 v;
                    v.x = pack_bf16x2(o[e8 * 8 + 0] * inv, o[e8 * 8 + 1] * inv);
                    v.y = pack_bf16x2(o[e8 * 8 + 2] * inv, o[e8 * 8 + 3] * inv);
                    v.z = pack_bf16x2(o[e8 * 8 + 4] * inv, o[e8 * 8 + 5] * inv);
                    v.w = pack_bf16x2(o[e8 * 8 + 6] * inv, o[e8 * 8 + 7] * inv);
                    *reinterpret_cast<uint4*>(dst + e8 * 8) = v;
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::dealloc(tmem, 256);
    }
}

template <int D>
cudaError_t launch_d(const PrefillParams& p, cudaStream_t stream) {
    const int smem = 1024 + 3 * BM * D * 2 + BM * BN * 2 + 64;
    auto k = paged_prefill_kernel<D>;
    cudaError_t err = allow_dynamic_smem((const void*)k, smem);
    if (err != cudaSuccess) return err;
    dim3 grid((p.max_q_len + BM - 1) / BM, p.H_q, p.B);
    k<<<grid, BM, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_persistent(const wf_pool_desc& pool, int32_t num_q_heads, int32_t B, int32_t max_q_len) {
    if (!prefill_tc_supported(pool, num_q_heads) || B < 1 || max_q_len < 1) return false;
    const int G = num_q_heads / pool.num_kv_heads;
    const int H_kv = pool.num_kv_heads;
    // the grid's yes / no does not depend on the SM count (1 here)
    if (pool.head_dim == 128) {
        switch (G) {
            case 1: return prefill_persist_grid<128, 1>(B, max_q_len, H_kv, 1) > 0;
            case 2: return prefill_persist_grid<128, 2>(B, max_q_len, H_kv, 1) > 0;
            case 4: return prefill_persist_grid<128, 4>(B, max_q_len, H_kv, 1) > 0;
            default: return prefill_persist_grid<128, 8>(B, max_q_len, H_kv, 1) > 0;
        }
    }
    switch (G) {
        case 1: return prefill_persist_grid<64, 1>(B, max_q_len, H_kv, 1) > 0;
        case 2: return prefill_persist_grid<64, 2>(B, max_q_len, H_kv, 1) > 0;
        case 4: return prefill_persist_grid<64, 4>(B, max_q_len, H_kv, 1) > 0;
        default: return prefill_persist_grid<64, 8>(B, max_q_len, H_kv, 1) > 0;
    }
}

int prefill_kernel_kind(const wf_pool_desc& pool, int32_t num_q_heads) {
    if (pool.dtype != WF_DTYPE_BF16 || (pool.head_dim != 64 && pool.head_dim != 128)) return WF_KERNEL_NONE;
    if (pool.num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % pool.num_kv_heads != 0) return WF_KERNEL_NONE;
    if (prefill_tc_supported(pool, num_q_heads) && (int64_t)pool.num_blocks * pool.block_size <= INT32_MAX)
        return WF_KERNEL_TENSOR_CORES;
    return WF_KERNEL_TENSOR_CORES_SIMPLE;
}

cudaError_t launch_paged_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                                 int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                                 int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                 uint32_t* dev_status, cudaStream_t stream) {
    if (prefill_tc_supported(pool, num_q_heads) &&
        (int64_t)pool.num_blocks * pool.block_size <= INT32_MAX && total_q > 0) {
        return launch_paged_prefill_tc(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens,
                                       B, total_q, max_q_len, max_seq_len, num_q_heads, scale, pool, dev_status,
                                       stream);
    }
    PrefillParams p;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k_pool = static_cast<const char*>(k_pool);
    p.v_pool = static_cast<const char*>(v_pool);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.dev_status = dev_status;
    p.M = max_blocks_per_seq;
    p.B = B;
    p.total_q = total_q;
    p.max_q_len = max_q_len;
    p.max_seq_len = max_seq_len;
    p.H_q = num_q_heads;
    p.H_kv = pool.num_kv_heads;
    p.G = num_q_heads / pool.num_kv_heads;
    p.N = pool.num_blocks;
    p.P = pool.block_size;
    p.scale_log2 = scale * 1.4426950408889634f;
    return pool.head_dim == 64 ? launch_d<64>(p, stream) : launch_d<128>(p, stream);
}

}  // namespace wf
