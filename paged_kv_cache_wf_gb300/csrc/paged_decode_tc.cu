// paged_decode_tc.cu -- paged decode on the 5th-generation tensor cores, for bf16
// pools with H_kv = 8 KV heads, D = 64 or 128, a block size that is a multiple of
// 16 and GQA groups of 2 or 4 (H_q = 16 or 32).
//
// Same contract and split-K structure as the CUDA-core decode in
// paged_decode.cu (ember, "The core idea"; tiny-vllm-py, "KV Cache"; weft,
// "Shapes and symbols"): a work item is (sequence b, split of tc_span(D) positions), the
// split boundaries depend only on the pool geometry, and the items of a
// multi-split sequence leave (m, l, o) partials for the combine kernel.
//
// Why tensor cores: per KV byte the GQA group needs 2 FMAs plus a widening; on
// CUDA cores that instruction stream, not HBM, limits decode.  Here a tile is one
// 16-position run of a block for all 8 KV heads -- 128 rows r = (head, position)
// -- and the group's work is two dense products issued by one thread:
//     S^T[128 rows x H_q]  = K[128 rows x D] . Q^T[D x H_q]
//     O^T[128 d x H_q]     = V^T[128 d x 128 rows] . P^T[128 rows x H_q]
// (at D = 64 the upper 64 rows of V^T read a zero tile: same MMA shape, zero rows
// of O^T that nobody stores)
// with bf16 operands and fp32 accumulators in tensor memory.  Row r only belongs
// to the G query heads of its KV head: S entries outside that diagonal block are
// ignored and P^T is block-diagonal (its off-diagonal entries stay zero).
//
// Loads: the K and V pools are described to the TMA unit as (d, slot, head) so
// that one 16-slot box of all 8 heads lands as 8 contiguous 16-row, 128-byte-
// swizzled head tiles, i.e. the UMMA K-major layout with rows (head, position).
// A tile is 4 boxes of 16 KB (K and V, two 64-wide halves of D), each issued by
// its own producer lane: the copy engine keeps one request per issuing thread in
// flight, so spreading large copies over lanes is what reaches HBM bandwidth.
//
// CTA (persistent, one per SM), 6 warps:
//   warp 0   producer (TMA): tiles into a 3-stage ring; q of an item into one of two
//            q buffers; mbarrier transaction counts mark arrival.
//   warp 1   MMA issuer: S(t) into one of two TMEM S buffers, then O(t-1) = V^T P^T
//            into one of two TMEM O buffers; commits free stages and buffers.
//   warps 2-5  (thread i):  (a) as the owner of row i = (head i/16, position i%16),
//            runs the online softmax of the current tile for the head's G query heads
//            (reductions over the 16 positions stay inside a half-warp) and writes
//            P^T as bf16; the four warps then meet and release P.V of the tile;
//            (b) as the owner of head dim d = i, folds the previous tile's O^T row
//            into fp32 registers with the per-head rescale factors, and at the end
//            of an item stores the output or the partial.  Doing (b) after (a) keeps
//            the wait for P.V(t-1) off the path from one softmax to the next.
#include <cuda.h>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kRows = 128;       // MMA M: 8 heads x 16 positions (and D = 128 for P.V)
constexpr int kHeads = 8;        // KV heads per tile
constexpr int kPosT = 16;        // positions per tile
// Positions per item (split): 256 at D = 128 (1 MB of K and V over the 8 KV heads;
// half the partials of 128, measured 287 -> 275 us a call at the Llama-3-8B batch),
// 128 at D = 64 (64 measured slower there).
__host__ __device__ constexpr int tc_span(int D) { return D == 128 ? 256 : 128; }
constexpr int kNq = 32;          // max H_q handled (MMA N, padded to a multiple of 16)
constexpr int kEndTile = -1;
constexpr int kHalf = kRows * 128;             // one 64-wide half of a K or V tile: 16 KB
constexpr int kQHalf = kNq * 128;              // one 64-wide half of q: 32 rows x 128 B
constexpr int kPHalf = kNq * 128;              // one 64-row half of P^T (32 q rows x 128 B)
constexpr int kPBytes = 2 * kPHalf;

struct TcParams {
    void* out;
    float* ws_o;
    float2* ws_ml;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    uint32_t* dev_status;
    uint32_t* queue;     // next unclaimed work item; zero at launch
    int32_t M, B, max_seq_len, H_q, H_kv, G, N, P, max_splits;
    float scale_log2;
};

struct TcMeta {
    int32_t b, split, nsplit, p0, nvalid, first, last, item;
};

// Per head dimension D (64 or 128): a K or V tile is D/64 halves of 64 columns
// (16 KB each).  At D = 64 the P.V product still runs as M = 128 rows of V^T, the
// upper 64 of which read a zero half, so one MMA shape and TMEM layout serve both.
template <int D>
struct TcSmemT {  // byte offsets from the 1024-aligned base
    static constexpr int NH = D / 64;
    static constexpr int kStages = D == 128 ? 3 : 5;
    static constexpr int kStageBytes = 2 * NH * kHalf;     // K halves, then V halves
    static constexpr int kQBytes = NH * kQHalf;
    static constexpr int stage = 0;
    static constexpr int zero = kStages * kStageBytes;      // D = 64: V^T rows 64..127
    static constexpr int qbuf = zero + (D == 64 ? kHalf : 0);
    static constexpr int pbuf = qbuf + 2 * kQBytes;
    static constexpr int bars = pbuf + 2 * kPBytes;
    // full[S] empty[S] s_full[2] s_free[2] p_full[2] o_full[2] o_free[2] q_free[2] grp
    static constexpr int nbars = 2 * kStages + 13;
    static constexpr int meta = (bars + nbars * 8 + 15) / 16 * 16;   // alpha/l/m below are read as float4
    static constexpr int alpha = meta + kStages * (int)sizeof(TcMeta);  // [3][kNq]: tile t in t % 3
    static constexpr int lbuf = alpha + 3 * kNq * 4;                    // [3][kNq]: item k in k % 3
    static constexpr int mbuf = lbuf + 3 * kNq * 4;                     // [3][kNq]
    static constexpr int tmem_slot = mbuf + 3 * kNq * 4;
    static constexpr int total = tmem_slot + 16;
};
static_assert(TcSmemT<128>::total + 1024 <= 232448 && TcSmemT<64>::total + 1024 <= 232448,
              "tensor-core decode exceeds shared memory");
static_assert(TcSmemT<128>::alpha % 16 == 0 && TcSmemT<128>::lbuf % 16 == 0 && TcSmemT<128>::mbuf % 16 == 0 &&
                  TcSmemT<64>::alpha % 16 == 0 && TcSmemT<64>::lbuf % 16 == 0 && TcSmemT<64>::mbuf % 16 == 0,
              "alpha, l and m buffers are read with 16-byte loads");
static_assert(TcSmemT<64>::zero % 1024 == 0 && TcSmemT<64>::qbuf % 1024 == 0, "swizzle atoms stay 1024-aligned");

template <int D>
__device__ __forceinline__ unsigned char* stage_k(unsigned char* base, int st, int c) {
    return base + TcSmemT<D>::stage + st * TcSmemT<D>::kStageBytes + c * kHalf;
}
template <int D>
__device__ __forceinline__ unsigned char* stage_v(unsigned char* base, int st, int c) {
    return base + TcSmemT<D>::stage + st * TcSmemT<D>::kStageBytes + TcSmemT<D>::NH * kHalf + c * kHalf;
}

// Byte offset of bf16 element (row, k) of a K-major 128-byte-swizzled tile whose
// 64-element column blocks are `block_bytes` apart.
__device__ __forceinline__ uint32_t sw_elem(int row, int k, int block_bytes) {
    const int chunk = (k & 63) >> 3;
    return (uint32_t)((k >> 6) * block_bytes + (row >> 3) * 1024 + (row & 7) * 128 +
                      ((chunk ^ (row & 7)) << 4) + (k & 7) * 2);
}

// 32 consecutive fp32 TMEM columns / 16 of them, this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) { tc::ld_32cols(taddr, v); }

template <int G, int D>
__global__ void __launch_bounds__(192, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, const TcParams p) {
    constexpr int HQ = kHeads * G;                 // query heads (MMA N)
    constexpr int kSpan = tc_span(D);
    using L = TcSmemT<D>;
    constexpr int kStages = L::kStages;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* s_full = bars + 2 * kStages;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* o_full = p_full + 2;
    uint64_t* o_free = o_full + 2;
    uint64_t* q_free = o_free + 2;
    // the four softmax warps meet here each tile (bounded waits, so a warp that stops
    // on a timed-out wait cannot leave the others blocked)
    uint64_t* grp = q_free + 2;
    TcMeta* meta = reinterpret_cast<TcMeta*>(smem + L::meta);
    float* alpha_buf = reinterpret_cast<float*>(smem + L::alpha);
    float* l_buf = reinterpret_cast<float*>(smem + L::lbuf);
    float* m_buf = reinterpret_cast<float*>(smem + L::mbuf);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the combine grid that follows may be scheduled now; it waits for this grid to
    // finish before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 1) {
        tc::alloc(tmem_slot, 128);
        tc::relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 4);
            mbar_init(&q_free[i], 1);
        }
        mbar_init(grp, 4);
        fence_mbar_init();
    }
    // P^T is block-diagonal: zero both buffers once; only diagonal entries are rewritten.
    for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem + L::pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (D == 64) {   // the zero half standing for V^T rows 64..127
        for (int i = threadIdx.x; i < kHalf / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(smem + L::zero)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S buffers [0,32) [32,64); O buffers [64,96) [96,128)

    if (warp == 0) {
        // ============================ producer ==================================
        // the queue is zeroed by the grid this one depends on
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const uint64_t pol = l2_policy_evict_first();
        int t = 0, k = 0;          // tiles and items issued
        int b = 0, len = 0, nsp = 0;
        int64_t cum = 0;
        bool ok = true;
        const int64_t cap = min((int64_t)p.max_seq_len, (int64_t)p.M * p.P);   // longest valid sequence
        ItemWalk walk;
        item_walk_load(walk, p.seq_lens, p.B, kSpan, cap, p.dev_status, lane);
        // Items come from a queue shared by all CTAs (one atomic increment per item,
        // claimed one item ahead so the round trip overlaps the current item's
        // copies).  Each CTA's claims increase, so its walk over the sequences only
        // moves forward.
        uint32_t claim = lane == 0 ? atomicAdd(p.queue, 1u) : 0u;
        for (int64_t item = __shfl_sync(0xffffffffu, claim, 0); ok; item = __shfl_sync(0xffffffffu, claim, 0)) {
            if (!item_walk_find(walk, item, p.seq_lens, p.B, kSpan, cap, p.dev_status, lane, b, len, nsp, cum))
                break;
            claim = lane == 0 ? atomicAdd(p.queue, 1u) : 0u;
            const int split = (int)(item - cum);
            const int s0 = split * kSpan;
            const int s1 = min(len, s0 + kSpan);
            const int ntiles = (s1 - s0 + kPosT - 1) / kPosT;
            const int qb = k & 1;
            if (k >= 2 && !mbar_wait(&q_free[qb], ((k >> 1) - 1) & 1)) {
                if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                ok = false;
                break;
            }
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int st = t % kStages;
                if (t >= kStages && !mbar_wait(&empty[st], ((t / kStages) - 1) & 1)) {
                    if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                    ok = false;
                    break;
                }
                const int p0 = s0 + j * kPosT;
                const int nvalid = min(kPosT, s1 - p0);
                const int blk = __ldg(p.block_tables + (int64_t)b * p.M + p0 / p.P);
                const bool okb = (unsigned)blk < (unsigned)p.N;
                const uint32_t bytes = (okb ? (uint32_t)L::kStageBytes : 0u) + (j == 0 ? 2u * HQ * (uint32_t)D : 0u);
                if (lane == 0) {
                    if (!okb) report(p.dev_status, WF_DEV_BAD_BLOCK);
                    TcMeta m;
                    m.b = b; m.split = split; m.nsplit = nsp; m.p0 = p0; m.nvalid = nvalid;
                    m.first = (j == 0); m.last = (j == ntiles - 1); m.item = k;
                    meta[st] = m;
                    mbar_arrive_expect_tx(&full[st], bytes);
                }
                __syncwarp();
                const int slot = blk * p.P + p0 % p.P;
                if (okb && lane < 2 * L::NH) {   // one 16 KB box per lane: K halves, then V halves
                    const bool isv = lane >= L::NH;
                    const int c = lane % L::NH;
                    unsigned char* dst = isv ? stage_v<D>(smem, st, c) : stage_k<D>(smem, st, c);
                    tma_load_3d(dst, isv ? &tm_v : &tm_k, c * 64, slot, 0, &full[st], pol);
                }
                if (j == 0 && lane >= 4 && lane < 4 + L::NH) {
                    tma_load_2d(smem + L::qbuf + qb * L::kQBytes + (lane - 4) * kQHalf, &tm_q, (lane - 4) * 64,
                                b * p.H_q, &full[st]);
                }
            }
            ++k;
        }
        if (ok) {
            const int st = t % kStages;
            if (t < kStages || mbar_wait(&empty[st], ((t / kStages) - 1) & 1)) {
                if (lane == 0) {
                    meta[st].nvalid = kEndTile;
                    mbar_arrive_expect_tx(&full[st], 0);
                }
            } else if (lane == 0) {
                report(p.dev_status, WF_DEV_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ================================
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16_f32(kRows, HQ < 16 ? 16 : HQ, 0, 0);
            constexpr uint32_t idO = tc::idesc_bf16_f32(kRows, HQ < 16 ? 16 : HQ, 1, 0);
            auto issue_pv = [&](int u) {
                const int su = u % kStages, ub = u & 1;
                tc::fence_after_sync();
                const uint32_t vbase = smem_u32(stage_v<D>(smem, su, 0));
                const uint32_t pb = smem_u32(smem + L::pbuf + ub * kPBytes);
                // V^T rows 64..127: the tile's second half (D = 128) or the zero half (D = 64)
                const uint32_t lbo = D == 128 ? (uint32_t)kHalf : smem_u32(smem + L::zero) - vbase;
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk) {
                    const uint64_t ad = tc::sdesc_sw128(vbase + kk * 2048, lbo, 1024);
                    const uint64_t bd = tc::sdesc_sw128(pb + (kk >> 2) * kPHalf + (kk & 3) * 32, 16, 1024);
                    tc::mma_f16(tmem + 64 + ub * 32, ad, bd, idO, kk > 0 ? 1u : 0u);
                }
                tc::commit(&o_full[ub]);
                tc::commit(&empty[su]);
            };
            // Event loop: issue P.V(tp) as soon as its weights are ready (it frees the
            // stage), otherwise S(tq) as soon as its tile has landed.
            int tq = 0, tp = 0;
            bool end_seen = false;
            uint32_t idle = 0;
            while (!(end_seen && tp == tq)) {
                bool did = false;
                if (tp < tq) {
                    const int ub = tp & 1;
                    if (mbar_test(&p_full[ub], (tp >> 1) & 1) &&
                        (tp < 2 || mbar_test(&o_free[ub], ((tp >> 1) - 1) & 1))) {
                        issue_pv(tp);
                        ++tp;
                        did = true;
                    }
                }
                if (!end_seen) {
                    const int st = tq % kStages;
                    if (mbar_test(&full[st], (tq / kStages) & 1)) {
                        const TcMeta m = meta[st];
                        if (m.nvalid == kEndTile) {
                            end_seen = true;
                        } else if (tq < 2 || mbar_test(&s_free[tq & 1], ((tq >> 1) - 1) & 1)) {
                            const int sb = tq & 1;
                            tc::fence_after_sync();
                            const uint32_t kbase = smem_u32(stage_k<D>(smem, st, 0));
                            const uint32_t qbase = smem_u32(smem + L::qbuf + (m.item & 1) * L::kQBytes);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t ad = tc::sdesc_sw128(kbase + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                                const uint64_t bd = tc::sdesc_sw128(qbase + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024);
                                tc::mma_f16(tmem + sb * 32, ad, bd, idS, kk > 0 ? 1u : 0u);
                            }
                            tc::commit(&s_full[sb]);
                            if (m.last) tc::commit(&q_free[m.item & 1]);
                            ++tq;
                            did = true;
                        }
                    }
                }
                if (did) {
                    idle = 0;
                } else {
                    if (++idle > (1u << 24)) {
                        report(p.dev_status, WF_DEV_TIMEOUT);
                        break;
                    }
                    if (idle > 8) __nanosleep(64);  // leave issue slots to the softmax warp on this SMSP
                }
            }
        }
    } else {
        // ==================== accumulate / softmax warps ===========================
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int i = quad * 32 + lane;            // row (softmax) / head dim (accumulate)
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const int hk = i >> 4;                     // KV head of row i
        const int pos = i & 15;                    // position of row i within the tile
        const int upper = lane >> 4;               // which of the warp's two heads
        float acc[kNq];                            // O^T row d = i, all query heads
#pragma unroll
        for (int c = 0; c < kNq; ++c) acc[c] = 0.f;
        float m_run[G], l_part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_part[g] = 0.f;
        }
        TcMeta prev;
        bool have_prev = false;

        auto accumulate = [&](int u, const TcMeta& m) {
            const int ub = u & 1;
            if (!mbar_wait(&o_full[ub], (u >> 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            tc::fence_after_sync();
            float o[32];
            tmem_ld32(tmem + lane_addr + 64 + ub * 32, o);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[ub]);
            const float* al = alpha_buf + (u % 3) * kNq;
#pragma unroll
            for (int c = 0; c < HQ; c += 4) {
                const float4 a4 = ld_shared_f4(al + c);
                acc[c] = acc[c] * a4.x + o[c];
                acc[c + 1] = acc[c + 1] * a4.y + o[c + 1];
                acc[c + 2] = acc[c + 2] * a4.z + o[c + 2];
                acc[c + 3] = acc[c + 3] * a4.w + o[c + 3];
            }
            if (m.last) {
                const float* Lsum = l_buf + (m.item % 3) * kNq;
                const float* Mx = m_buf + (m.item % 3) * kNq;
                if (m.nsplit == 1) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (int64_t)m.b * p.H_q * D + i;
                    if (i < D) {
#pragma unroll
                        for (int c = 0; c < HQ; ++c) dst[c * D] = __float2bfloat16_rn(acc[c] / Lsum[c]);
                    }
                } else {
                    const int64_t base = ((int64_t)m.b * p.max_splits + m.split) * p.H_q;
                    if (i < D) {
#pragma unroll
                        for (int c = 0; c < HQ; ++c) p.ws_o[(base + c) * D + i] = acc[c];
                    }
                    if (i < HQ) p.ws_ml[base + i] = make_float2(Mx[i], Lsum[i]);
                }
            }
        };

        int t = 0;
        for (;; ++t) {
            const int st = t % kStages;
            if (!mbar_wait(&full[st], (t / kStages) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            const TcMeta m = meta[st];
            if (m.nvalid == kEndTile) break;
            // (a) softmax of this tile
            const int sb = t & 1;
            if (!mbar_wait(&s_full[sb], (t >> 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            tc::fence_after_sync();
            // this warp's two KV heads' query-head columns [2G*quad, 2G*quad + 2G), width-aligned
            float sv[2 * G];
            if constexpr (G == 4) {
                tc::ld_8cols(tmem + lane_addr + sb * 32 + quad * 8, sv);
            } else {
                tc::ld_4cols(tmem + lane_addr + sb * 32 + quad * 4, sv);
            }
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);
            if (m.first) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_part[g] = 0.f;
                }
            }
            const bool live = pos < m.nvalid;
            float al[G];
            unsigned char* pb = smem + L::pbuf + sb * kPBytes;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float raw = upper ? sv[G + g] : sv[g];
                const float s = live ? raw * p.scale_log2 : -INFINITY;
                float mx = s;
#pragma unroll
                for (int mask = 8; mask >= 1; mask >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
                const float m_new = fmaxf(m_run[g], mx);
                al[g] = exp2f(m_run[g] - m_new);       // 0 on an item's first tile
                const __nv_bfloat16 eb = __float2bfloat16_rn(exp2f(s - m_new));
                l_part[g] = l_part[g] * al[g] + __bfloat162float(eb);
                m_run[g] = m_new;
                *reinterpret_cast<__nv_bfloat16*>(pb + sw_elem(hk * G + g, i, kPHalf)) = eb;
            }
            if (pos == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) alpha_buf[(t % 3) * kNq + hk * G + g] = al[g];
            }
            if (m.last) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float x = l_part[g];
#pragma unroll
                    for (int mask = 8; mask >= 1; mask >>= 1) x += __shfl_xor_sync(0xffffffffu, x, mask);
                    if (pos == 0) {
                        l_buf[(m.item % 3) * kNq + hk * G + g] = x;
                        m_buf[(m.item % 3) * kNq + hk * G + g] = m_run[g];
                    }
                }
            }
            if (!live) {
                // rows past the sequence end: zero V so their 0-weights cannot meet NaN/Inf
#pragma unroll
                for (int c = 0; c < L::NH; ++c) {
                    uint4* row = reinterpret_cast<uint4*>(stage_v<D>(smem, st, c) + (i >> 3) * 1024 + (i & 7) * 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q) row[q] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(grp);
            if (!mbar_wait(grp, t & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            if (lane == 0) mbar_arrive(&p_full[sb]);
            // (b) fold in the previous tile's P.V while this tile's runs: it completed
            // during this softmax (alpha of tile t-1 sits in ring slot (t-1) % 3, which
            // softmax(t+2) rewrites only after every warp has met at tile t+1)
            if (have_prev) accumulate(t - 1, prev);
            prev = m;
            have_prev = true;
        }
        if (have_prev) accumulate(t - 1, prev);
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, 128);
    }
}

// Zeroes the decode's work-item queue; the decode grid is launched as its
// programmatic dependent.
__global__ void decode_queue_reset_kernel(uint32_t* queue) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) *queue = 0u;
}

}  // namespace

bool decode_tc_supported(const wf_pool_desc& pool, int32_t num_q_heads) {
    const int G = pool.num_kv_heads > 0 ? num_q_heads / pool.num_kv_heads : 0;
    return pool.dtype == WF_DTYPE_BF16 && (pool.head_dim == 64 || pool.head_dim == 128) &&
           pool.block_size % kPosT == 0 &&
           pool.num_kv_heads == kHeads && num_q_heads % pool.num_kv_heads == 0 && (G == 2 || G == 4);
}

int decode_tc_span(int head_dim) { return tc_span(head_dim); }

cudaError_t launch_paged_decode_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                   int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                   float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                   cudaStream_t stream) {
    const int G = num_q_heads / pool.num_kv_heads;
    const int D = pool.head_dim;
    CUtensorMap tm_k, tm_v, tm_q;
    const uint64_t slots = (uint64_t)pool.num_blocks * pool.block_size;
    {
        // (d, slot, head): one box = 16 slots x 8 heads x 64 d, head-major in shared memory
        const uint64_t dims[3] = {(uint64_t)D, slots, (uint64_t)kHeads};
        const uint64_t strides[2] = {(uint64_t)kHeads * D * 2, (uint64_t)D * 2};
        const uint32_t box[3] = {64, (uint32_t)kPosT, (uint32_t)kHeads};
        cudaError_t e = encode_tiled_bf16(&tm_k, const_cast<void*>(k_pool), 3, dims, strides, box);
        if (e != cudaSuccess) return e;
        e = encode_tiled_bf16(&tm_v, const_cast<void*>(v_pool), 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)B * num_q_heads};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64, (uint32_t)num_q_heads};
        cudaError_t e = encode_tiled_bf16(&tm_q, const_cast<void*>(q), 2, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    TcParams p;
    p.out = out;
    p.ws_o = ws_o;
    p.ws_ml = ws_ml;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.dev_status = dev_status;
    p.queue = queue;
    p.M = max_blocks_per_seq;
    p.B = B;
    p.max_seq_len = max_seq_len;
    p.H_q = num_q_heads;
    p.H_kv = pool.num_kv_heads;
    p.G = G;
    p.N = pool.num_blocks;
    p.P = pool.block_size;
    p.max_splits = max_splits;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int smem = (D == 64 ? TcSmemT<64>::total : TcSmemT<128>::total) + 1024;
    const int64_t items = (int64_t)B * max_splits;
    const int grid = (int)(items < num_sms() ? items : num_sms());
    decode_queue_reset_kernel<<<1, 32, 0, stream>>>(queue);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const void* kern = D == 64 ? (G == 4 ? (const void*)paged_decode_tc_kernel<4, 64> : (const void*)paged_decode_tc_kernel<2, 64>)
                               : (G == 4 ? (const void*)paged_decode_tc_kernel<4, 128>
                                         : (const void*)paged_decode_tc_kernel<2, 128>);
    err = allow_dynamic_smem(kern, smem);
    if (err != cudaSuccess) return err;
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
    if (D == 64) {
        if (G == 4) return cudaLaunchKernelEx(&cfg, paged_decode_tc_kernel<4, 64>, tm_k, tm_v, tm_q, p);
        return cudaLaunchKernelEx(&cfg, paged_decode_tc_kernel<2, 64>, tm_k, tm_v, tm_q, p);
    }
    if (G == 4) return cudaLaunchKernelEx(&cfg, paged_decode_tc_kernel<4, 128>, tm_k, tm_v, tm_q, p);
    return cudaLaunchKernelEx(&cfg, paged_decode_tc_kernel<2, 128>, tm_k, tm_v, tm_q, p);
}

}  // namespace wf
