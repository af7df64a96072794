// paged_decode_tc.cuh -- paged decode on the 5th-generation tensor cores, for bf16
// pools with any number of KV heads H_kv, GQA groups G = H_q / H_kv of 1, 2 or 4
// (MHA included), D = 64 or 128, and a block size that is a multiple of 16.
//
// Same contract and split-K structure as the CUDA-core decode in
// paged_decode.cu (ember, "The core idea"; tiny-vllm-py, "KV Cache"; weft,
// "Shapes and symbols"): a split is tc_span(D) positions of one sequence, the
// split boundaries depend only on the pool geometry, and the splits of a
// multi-split sequence leave (m, l, o) partials for the combine kernel.
//
// Why tensor cores: per KV byte the GQA group needs 2 FMAs plus a widening; on
// CUDA cores that instruction stream, not HBM, limits decode.  A sub-tile is 128
// rows r = (box, KV head, position): NB = 8 / HT TMA boxes of 16 consecutive
// positions of HT KV heads (HT = the largest power of two <= 8 that divides H_kv; a
// work item covers one group of HT heads).  A stage holds SUB sub-tiles, 64 KB of
// K and V: one at D = 128, two at D = 64 (so that each step of the per-tile chain
// below moves the same bytes at both head dims).  The group's work is two dense
// products per sub-tile, issued by one thread:
//     S^T[128 rows x HT*G]  = K[128 rows x D] . Q^T[D x HT*G]
//     O^T[128 d x 8*G]     += V^T[128 d x 128 rows] . P^T[128 rows x 8*G]
// with bf16 operands and fp32 accumulators in tensor memory (the P.V products of
// both sub-tiles add into one accumulator).  Row r only belongs to the G query
// heads of its KV head: other S entries are ignored, and P^T has one column per
// (box, KV head, query head) -- the column of row r's box and head, zero elsewhere.
// Each box position of a sub-tile is therefore its own online-softmax stream with
// its own running max and sum (shared by the sub-tiles of a stage), and the streams
// of one query head are merged when the item ends.  (At D = 64 the upper 64 rows of
// V^T read the next 16 KB of the stage: rows of O^T that nobody reads.)
//
// Loads: the pools are described to the TMA unit as (d, slot, head); one box is 16
// slots x HT heads x 64 d and lands as HT contiguous 16-row, 128-byte-swizzled head
// tiles, i.e. the UMMA K-major layout with rows (head, position).  Every box is
// issued by its own producer lane: the copy engine keeps one request per issuing
// thread in flight, so spreading copies over lanes is what reaches HBM bandwidth.
//
// CTA (persistent, one per SM), 6 warps:
//   warp 0   producer (TMA): tiles into a 3-stage ring; q of an item into one of
//            two q buffers; mbarrier transaction counts mark arrival.
//   warp 1   MMA issuer: S(t) into one of two TMEM S buffers, then O(t-1) = V^T P^T
//            into one of two TMEM O buffers; commits free stages and buffers.
//   warps 2-5  (thread i):  (a) as the owner of row i of every sub-tile, runs the
//            online softmax of the current tile for its KV head's G query heads
//            (the 16 rows of a box and head are one half-warp) and writes P^T as
//            bf16; the four warps then meet and release P.V of the tile; (b) as the
//            owner of head dim d = i, folds the previous tile's O^T row into fp32
//            registers with the per-column rescale factors, and at the end of an
//            item merges the box streams and stores the output or the partial.
//            Doing (b) after (a) keeps the wait for P.V(t-1) off the path from one
//            softmax to the next.
#pragma once

#include <cuda.h>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kRows = 128;          // MMA M: rows (box, head, position) of a tile; d rows of O^T
constexpr int kBoxPos = 16;         // positions per TMA box (P % 16 == 0: a box stays in one block)
constexpr int kHalf = kRows * 128;  // one 64-wide half of a K or V tile: 16 KB
constexpr int kEndTile = -1;
constexpr int kDecodeThreads = 192;   // 6 warps
// Positions per item (split): 256 at D = 128 (1 MB of K and V over 8 KV heads;
// half the partials of 128, measured 287 -> 275 us a call at the Llama-3-8B batch),
// 128 at D = 64, and never less than one tile (SUB * 16 * NB positions).
__host__ __device__ constexpr int tc_span(int D, int NB) {
    return (D == 128 ? 256 : 128) > (D == 64 ? 32 : 16) * NB ? (D == 128 ? 256 : 128) : (D == 64 ? 32 : 16) * NB;
}

struct TcParams {
    void* out;
    float* ws_o;
    float2* ws_ml;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    uint32_t* dev_status;
    uint32_t* queue;     // next unclaimed work item; zero at launch
    int32_t M, B, max_seq_len, H_q, H_kv, N, P, max_splits;
    int32_t HT;          // KV heads per box
    int32_t NB;          // boxes per sub-tile (8 / HT)
    int32_t HGRP;        // head groups per split (H_kv / HT)
    int32_t span;        // positions per split
    float scale_log2;
};

struct TcMeta {
    int32_t b, split, nsplit, hg, nvalid, item;
    int32_t flags;      // bit 0: first tile of its item, bit 1: last; bits 8..: boxes loaded
    int32_t pad;
    __device__ bool first() const { return flags & 1; }
    __device__ bool last() const { return (flags >> 1) & 1; }
    __device__ uint32_t okmask() const { return (uint32_t)flags >> 8; }
};

// Shared-memory layout per (G, D): byte offsets from the 1024-aligned base.
template <int G, int D>
struct TcCfg {
    static constexpr int NH = D / 64;                   // 64-wide halves of D
    static constexpr int SUB = D == 64 ? 2 : 1;         // sub-tiles per stage
    static constexpr int NOC = 8 * G;                   // P^T / O^T columns: (box, head, query head)
    static constexpr int NCOL = NOC < 16 ? 16 : NOC;    // MMA N (padded); S uses at most NOC columns
    static constexpr int kStages = 3;
    static constexpr int kStageBytes = 4 * kHalf;       // 64 KB: two K and two V slots of 16 KB
    // D = 64 puts V first: rows 64..127 of a P.V operand read the 16 KB after its V
    // slot, which must stay inside the stage
    static constexpr bool kVFirst = D == 64;
    static constexpr int kQHalf = NCOL * 128;           // q rows of one 64-wide half
    static constexpr int kQBytes = NH * kQHalf;
    static constexpr int kPHalf = NCOL * 128;           // one 64-row half of a sub-tile's P^T
    static constexpr int kPBytes = 2 * kPHalf;          // a sub-tile's P^T
    // P^T buffers: two at D = 128 (softmax(t) writes one while P.V(t-1) reads the
    // other).  At D = 64 sub-tile s's P^T goes into K slot s of the tile's own stage,
    // free once S(t) is done and released with the stage after P.V(t).
    static constexpr int kPBufs = SUB == 1 ? 2 : 0;
    static_assert(kPBytes <= kHalf, "P^T of a sub-tile fits in a K slot");
    static constexpr int stage = 0;
    static constexpr int qbuf = kStages * kStageBytes;
    static constexpr int pbuf = qbuf + 2 * kQBytes;
    static constexpr int bars = pbuf + kPBufs * SUB * kPBytes;
    // full[S] empty[S] s_full[2] s_free[2] p_full[2] o_full[2] o_free[2] q_free[2] grp
    static constexpr int nbars = 2 * kStages + 13;
    static constexpr int meta = (bars + nbars * 8 + 15) / 16 * 16;
    static constexpr int alpha = (meta + kStages * (int)sizeof(TcMeta) + 15) / 16 * 16;  // [3][NCOL]: tile t in t % 3
    static constexpr int lbuf = alpha + 3 * NCOL * 4;                                     // [3][NCOL]: item k in k % 3
    static constexpr int mbuf = lbuf + 3 * NCOL * 4;                                      // [3][NCOL]
    static constexpr int tmem_slot = mbuf + 3 * NCOL * 4;
    static constexpr int total = tmem_slot + 16;
    // TMEM: S buffers (SUB * NCOL columns each) at [0, 2 SUB NCOL); O buffers after them
    static constexpr int kSCols = SUB * NCOL;
    static constexpr int kOBase = 2 * kSCols;
    static constexpr int TMEM = kOBase + 2 * NCOL <= 32 ? 32 : kOBase + 2 * NCOL <= 64 ? 64
                                : kOBase + 2 * NCOL <= 128 ? 128 : 256;
    static_assert(total + 1024 <= 232448, "tensor-core decode exceeds shared memory");
    static_assert(alpha % 16 == 0 && lbuf % 16 == 0 && mbuf % 16 == 0, "alpha, l and m are read with 16-byte loads");
    static_assert(qbuf % 1024 == 0 && pbuf % 1024 == 0 && kQHalf % 1024 == 0 && kPHalf % 1024 == 0,
                  "swizzle atoms stay 1024-aligned");
    static_assert(NOC % 4 == 0, "alpha is read four columns at a time");
    static_assert(SUB * NH == 2, "a stage holds two 16 KB slots of V and two of K");
};

// Slot `sl` (0 or 1) of V / K in stage `st`: the two 64-wide halves of D at D = 128,
// the two sub-tiles at D = 64.
template <int G, int D>
__device__ __forceinline__ unsigned char* stage_v(unsigned char* base, int st, int sl) {
    return base + TcCfg<G, D>::stage + st * TcCfg<G, D>::kStageBytes + ((TcCfg<G, D>::kVFirst ? 0 : 2) + sl) * kHalf;
}
template <int G, int D>
__device__ __forceinline__ unsigned char* stage_k(unsigned char* base, int st, int sl) {
    return base + TcCfg<G, D>::stage + st * TcCfg<G, D>::kStageBytes + ((TcCfg<G, D>::kVFirst ? 2 : 0) + sl) * kHalf;
}

// Byte offset of bf16 element (row, k) of a K-major 128-byte-swizzled tile whose
// 64-element column blocks are `block_bytes` apart.
__device__ __forceinline__ uint32_t sw_elem(int row, int k, int block_bytes) {
    const int chunk = (k & 63) >> 3;
    return (uint32_t)((k >> 6) * block_bytes + (row >> 3) * 1024 + (row & 7) * 128 +
                      ((chunk ^ (row & 7)) << 4) + (k & 7) * 2);
}

// N consecutive fp32 TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[N]);
template <>
__device__ __forceinline__ void ld_cols<1>(uint32_t taddr, float (&v)[1]) { tc::ld_1col(taddr, v); }
template <>
__device__ __forceinline__ void ld_cols<2>(uint32_t taddr, float (&v)[2]) { tc::ld_2cols(taddr, v); }
template <>
__device__ __forceinline__ void ld_cols<4>(uint32_t taddr, float (&v)[4]) { tc::ld_4cols(taddr, v); }
template <>
__device__ __forceinline__ void ld_cols<8>(uint32_t taddr, float (&v)[8]) { tc::ld_8cols(taddr, v); }
template <>
__device__ __forceinline__ void ld_cols<16>(uint32_t taddr, float (&v)[16]) { tc::ld_16cols(taddr, v); }
template <>
__device__ __forceinline__ void ld_cols<32>(uint32_t taddr, float (&v)[32]) { tc::ld_32cols(taddr, v); }

// The kernel's body for CTA `cta` of `ncta` persistent CTAs, run by threads
// 0 .. kDecodeThreads - 1 of its block (other threads of a larger block must not
// enter); its block-wide barriers are named barrier 1 over those threads.
template <int G, int D, int HT>
__device__ __forceinline__ void decode_tc_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                               const CUtensorMap& tm_q, const TcParams& p,
                                               unsigned char* smem_raw, int cta, int ncta) {
    using L = TcCfg<G, D>;
    constexpr int NOC = L::NOC;
    constexpr int NCOL = L::NCOL;
    constexpr int SUB = L::SUB;
    constexpr int kStages = L::kStages;
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
    constexpr int NB = 8 / HT;             // boxes per sub-tile
    constexpr int NS = HT * G;             // S columns in use: the query heads of the item's HT KV heads
    constexpr int kSpan = tc_span(D, NB);
    if (warp == 1) {
        tc::alloc(tmem_slot, L::TMEM);
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
    // P^T has one nonzero block per row group: zero the buffers once; only those
    // entries are ever rewritten (D = 128; at D = 64 the softmax writes whole rows).
    for (int i = threadIdx.x; i < L::kPBufs * SUB * L::kPBytes / 16; i += kDecodeThreads)
        reinterpret_cast<uint4*>(smem + L::pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    named_bar_sync(1, kDecodeThreads);
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ============================ producer ==================================
        const uint64_t pol = l2_policy_evict_first();
        const int PT = SUB * kBoxPos * NB;           // positions per tile
        const int per_box = 2 * L::NH;               // copies per box: K halves (needed first), then V
        const int gb = lane / per_box;               // this lane's box in the tile (sub-tile major)
        const int rem = lane - gb * per_box;
        const bool isv = rem >= L::NH;
        const int c = isv ? rem - L::NH : rem;       // half of D
        const int sub = gb / NB;
        const int sl = sub * L::NH + c;              // V / K slot of the stage
        const int boff = (gb - sub * NB) * HT * kBoxPos * 128;   // the box's offset in its slot
        const uint32_t box_bytes = (uint32_t)(HT * kBoxPos * 128);
        int t = 0, k = 0;          // tiles and items issued
        int b = 0, len = 0, nitems = 0;
        int64_t cum = 0;
        bool ok = true;
        const int64_t cap = min((int64_t)p.max_seq_len, (int64_t)p.M * p.P);   // longest valid sequence
        ItemWalk walk;
        item_walk_load(walk, p.seq_lens, p.B, kSpan, cap, p.dev_status, lane, p.HGRP);
        // CTA c starts with item c, so its first copies go out without waiting for
        // anything; later items come from a queue shared by all CTAs (item ncta
        // + the queue's count; one atomic increment per item, claimed one item ahead,
        // after the current item's first tile, so the round trip overlaps its copies).
        // Each CTA's items increase, so its walk over the sequences only moves
        // forward.  The queue is zeroed by the grid this one depends on: the first
        // claim waits for it (griddepcontrol.wait).  Everything else this kernel
        // reads was written before that grid started.
        uint32_t claim = lane == 0 ? (uint32_t)cta : 0u;
        bool waited = false;
        for (int64_t item = __shfl_sync(0xffffffffu, claim, 0); ok; item = __shfl_sync(0xffffffffu, claim, 0)) {
            if (!item_walk_find(walk, item, p.seq_lens, p.B, kSpan, cap, p.dev_status, lane, b, len, nitems, cum,
                                p.HGRP))
                break;
            const int kin = (int)(item - cum);           // split-major within the sequence
            const int split = kin / p.HGRP;
            const int hg = kin - split * p.HGRP;
            const int s0 = split * kSpan;
            const int s1 = min(len, s0 + kSpan);
            const int ntiles = (s1 - s0 + PT - 1) / PT;
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
                const int p0 = s0 + j * PT;
                const int nvalid = min(PT, s1 - p0);
                const int pb0 = p0 + gb * kBoxPos;           // first position of this lane's box
                const bool need = gb < SUB * NB && gb * kBoxPos < nvalid;
                const int blk = need ? __ldg(p.block_tables + (int64_t)b * p.M + pb0 / p.P) : -1;
                const bool okb = need && (unsigned)blk < (unsigned)p.N;
                if (need && !okb && rem == 0) report(p.dev_status, WF_DEV_BAD_BLOCK);
                const unsigned okl = __ballot_sync(0xffffffffu, okb);
                if (lane == 0) {
                    uint32_t okmask = 0;
                    for (int x = 0; x < SUB * NB; ++x) okmask |= ((okl >> (x * per_box)) & 1u) << x;
                    TcMeta m;
                    m.b = b; m.split = split; m.nsplit = (len + kSpan - 1) / kSpan; m.hg = hg; m.nvalid = nvalid; m.item = k;
                    m.flags = (j == 0 ? 1 : 0) | (j == ntiles - 1 ? 2 : 0) | (int)(okmask << 8);
                    m.pad = 0;
                    meta[st] = m;
                    const uint32_t bytes = (uint32_t)__popc(okl) * box_bytes + (j == 0 ? 2u * NS * D : 0u);
                    mbar_arrive_expect_tx(&full[st], bytes);
                }
                __syncwarp();
                if (okb) {   // one box per lane: 16 slots x HT heads x 64 d
                    unsigned char* dst = (isv ? stage_v<G, D>(smem, st, sl) : stage_k<G, D>(smem, st, sl)) + boff;
                    tma_load_3d(dst, isv ? &tm_v : &tm_k, c * 64, blk * p.P + pb0 % p.P, hg * HT, &full[st], pol);
                }
                if (j == 0 && lane < L::NH) {
                    tma_load_2d(smem + L::qbuf + qb * L::kQBytes + lane * L::kQHalf, &tm_q, lane * 64,
                                b * p.H_q + hg * NS, &full[st]);
                }
                if (j == 0) {   // claim the next item
                    if (!waited) {
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        waited = true;
                    }
                    claim = lane == 0 ? (uint32_t)ncta + atomicAdd(p.queue, 1u) : 0u;
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
            constexpr uint32_t idS = tc::idesc_bf16_f32(kRows, NS < 16 ? 16 : NS, 0, 0);
            constexpr uint32_t idO = tc::idesc_bf16_f32(kRows, NCOL, 1, 0);
            auto issue_pv = [&](int u) {
                const int su = u % kStages, ub = u & 1;
                tc::fence_after_sync();
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    // A = V^T of sub-tile s; its rows 64..127 are the next 16 KB slot: the
                    // second half of D (D = 128), or rows of O^T nobody reads (D = 64)
                    const uint32_t vbase = smem_u32(stage_v<G, D>(smem, su, s));
                    const uint32_t pb = L::kPBufs == 2 ? smem_u32(smem + L::pbuf + ub * L::kPBytes)
                                                       : smem_u32(stage_k<G, D>(smem, su, s));
#pragma unroll
                    for (int kk = 0; kk < kRows / 16; ++kk) {
                        const uint64_t ad = tc::sdesc_sw128(vbase + kk * 2048, kHalf, 1024);
                        const uint64_t bd = tc::sdesc_sw128(pb + (kk >> 2) * L::kPHalf + (kk & 3) * 32, 16, 1024);
                        tc::mma_f16(tmem + L::kOBase + ub * NCOL, ad, bd, idO, (s > 0 || kk > 0) ? 1u : 0u);
                    }
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
                        const int mnvalid = meta[st].nvalid;
                        if (mnvalid == kEndTile) {
                            end_seen = true;
                        } else if (tq < 2 || mbar_test(&s_free[tq & 1], ((tq >> 1) - 1) & 1)) {
                            const int sb = tq & 1;
                            tc::fence_after_sync();
                            const int mitem = meta[st].item;
                            const bool mlast = meta[st].last();
                            const uint32_t qbase = smem_u32(smem + L::qbuf + (mitem & 1) * L::kQBytes);
#pragma unroll
                            for (int s = 0; s < SUB; ++s) {
                                const uint32_t kbase = smem_u32(stage_k<G, D>(smem, st, s * L::NH));
#pragma unroll
                                for (int kk = 0; kk < D / 16; ++kk) {
                                    const uint64_t ad =
                                        tc::sdesc_sw128(kbase + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                                    const uint64_t bd =
                                        tc::sdesc_sw128(qbase + (kk >> 2) * L::kQHalf + (kk & 3) * 32, 16, 1024);
                                    tc::mma_f16(tmem + sb * L::kSCols + s * NCOL, ad, bd, idS, kk > 0 ? 1u : 0u);
                                }
                            }
                            tc::commit(&s_full[sb]);
                            if (mlast) tc::commit(&q_free[mitem & 1]);
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
        const int rg = i >> 4;                     // row group: box * HT + head in the box
        const int bx = rg / HT;                    // box of row i in its sub-tile
        const int pos = i & 15;                    // position of row i within its box
        const int upper = lane >> 4;               // which of the warp's two row groups
        // S columns of this warp: the query heads of its two row groups' KV heads
        // (HT >= 2: two different heads, 2G columns; HT = 1: one head, G columns)
        const int colw = HT >= 2 ? ((2 * quad) % HT) * G : 0;   // (HT is a power of two)
        float acc[NOC];                            // O^T row d = i, every (box, head, query head) column
#pragma unroll
        for (int cc = 0; cc < NOC; ++cc) acc[cc] = 0.f;
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
            float o[NOC];
            ld_cols<NOC>(tmem + lane_addr + L::kOBase + ub * NCOL, o);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[ub]);
            const float* al = alpha_buf + (u % 3) * NCOL;
            // (alpha is 0 on an item's first tile; with several streams a stream's
            // accumulator is also restarted explicitly, since it may hold nothing yet)
            const bool restart = NB * SUB > 1 && m.first();
#pragma unroll
            for (int cc = 0; cc < NOC; cc += 4) {
                const float4 a4 = ld_shared_f4(al + cc);
                acc[cc] = restart ? o[cc] : acc[cc] * a4.x + o[cc];
                acc[cc + 1] = restart ? o[cc + 1] : acc[cc + 1] * a4.y + o[cc + 1];
                acc[cc + 2] = restart ? o[cc + 2] : acc[cc + 2] * a4.z + o[cc + 2];
                acc[cc + 3] = restart ? o[cc + 3] : acc[cc + 3] * a4.w + o[cc + 3];
            }
            if (m.last()) {
                const float* Lsum = l_buf + (m.item % 3) * NCOL;
                const float* Mx = m_buf + (m.item % 3) * NCOL;
                const int64_t qbase = (int64_t)m.b * p.H_q + (int64_t)m.hg * NS;   // first query head of the item
                // split-minor partial rows: the item's first query head; query head qh is max_splits rows on
                const int64_t wrow = partial_row(m.b, (int64_t)m.hg * NS, m.split, p.H_q, p.max_splits, p.max_splits, 1);
                if constexpr (NB == 1) {
                    // one stream per query head (column qh)
#pragma unroll
                    for (int cc = 0; cc < NOC; ++cc) {
                        if (cc >= NS) continue;
                        if (m.nsplit == 1) {
                            if (i < D)
                                static_cast<__nv_bfloat16*>(p.out)[(qbase + cc) * D + i] =
                                    __float2bfloat16_rn(acc[cc] / Lsum[cc]);
                        } else if (i < D) {
                            p.ws_o[(wrow + (int64_t)cc * p.max_splits) * D + i] = acc[cc];
                        }
                    }
                    if (m.nsplit != 1 && quad == 0 && lane < NS)
                        p.ws_ml[wrow + (int64_t)lane * p.max_splits] = make_float2(Mx[lane], Lsum[lane]);
                } else {
                    // Merge the box streams: query head qh of the item owns columns
                    // qh + x * NS (x < NB).  Lane c works out the weight 2^(m_c - M_qh)
                    // of column c, and lane qh the merged max M_qh and sum L_qh; the
                    // warp shares them by shuffles.  Each column is weighed, then the
                    // columns of each query head are added with a halving fold.
                    float w_c = 0.f, m_q = -INFINITY, l_q = 0.f;
                    if (lane < NOC) {
                        const int qh = lane % NS;
                        float mq = -INFINITY;
                        for (int x = 0; x < NB; ++x) mq = fmaxf(mq, Mx[qh + x * NS]);
                        const float mc = Mx[lane];
                        w_c = mc == -INFINITY ? 0.f : exp2f(mc - mq);
                    }
                    if (lane < NS) {
                        for (int x = 0; x < NB; ++x) m_q = fmaxf(m_q, Mx[lane + x * NS]);
                        for (int x = 0; x < NB; ++x) {
                            const float mc = Mx[lane + x * NS];
                            if (mc != -INFINITY) l_q += Lsum[lane + x * NS] * exp2f(mc - m_q);
                        }
                    }
#pragma unroll
                    for (int cc = 0; cc < NOC; ++cc) acc[cc] *= __shfl_sync(0xffffffffu, w_c, cc);
#pragma unroll
                    for (int s = NOC / 2; s >= 1; s >>= 1) {
                        if (s >= NS) {
#pragma unroll
                            for (int cc = 0; cc < s; ++cc) acc[cc] += acc[cc + s];
                        }
                    }
#pragma unroll
                    for (int cc = 0; cc < NOC; ++cc) {
                        const float lq = __shfl_sync(0xffffffffu, l_q, cc);
                        if (cc >= NS) continue;
                        if (m.nsplit == 1) {
                            if (i < D)
                                static_cast<__nv_bfloat16*>(p.out)[(qbase + cc) * D + i] =
                                    __float2bfloat16_rn(acc[cc] / lq);
                        } else if (i < D) {
                            p.ws_o[(wrow + (int64_t)cc * p.max_splits) * D + i] = acc[cc];
                        }
                    }
                    if (m.nsplit != 1 && quad == 0 && lane < NS) p.ws_ml[wrow + (int64_t)lane * p.max_splits] = make_float2(m_q, l_q);
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
            float sv[SUB][2 * G];
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                const uint32_t sa = tmem + lane_addr + sb * L::kSCols + s * NCOL;
                if constexpr (HT >= 2) {
                    ld_cols<2 * G>(sa + colw, sv[s]);
                } else {
                    float s1[G];
                    ld_cols<G>(sa, s1);
#pragma unroll
                    for (int g = 0; g < G; ++g) sv[s][g] = sv[s][G + g] = s1[g];
                }
            }
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);
            if (m.first()) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_part[g] = 0.f;
                }
            }
            bool live[SUB];
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                const int gbox = s * NB + bx;
                live[s] = gbox * kBoxPos + pos < m.nvalid && ((m.okmask() >> gbox) & 1);
            }
            float al[G];
            __nv_bfloat16 eb[SUB][G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float sc[SUB];
                float mx = -INFINITY;
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    const float raw = upper ? sv[s][G + g] : sv[s][g];
                    sc[s] = live[s] ? raw * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sc[s]);
                }
#pragma unroll
                for (int mask = 8; mask >= 1; mask >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
                const float m_new = fmaxf(m_run[g], mx);
                float lsum = 0.f;
                if constexpr (NB * SUB == 1) {
                    // one box: every tile of an item has a live row, so m_new is finite
                    al[g] = exp2f(m_run[g] - m_new);   // 0 on an item's first tile
                    eb[0][g] = __float2bfloat16_rn(exp2f(sc[0] - m_new));
                    lsum = __bfloat162float(eb[0][g]);
                } else {
                    // a stream with no live row yet keeps m = -inf: its factor and weights are 0
                    al[g] = m_new == -INFINITY ? 0.f : exp2f(m_run[g] - m_new);
#pragma unroll
                    for (int s = 0; s < SUB; ++s) {
                        eb[s][g] = __float2bfloat16_rn(live[s] ? exp2f(sc[s] - m_new) : 0.f);
                        lsum += __bfloat162float(eb[s][g]);
                    }
                }
                l_part[g] = l_part[g] * al[g] + lsum;
                m_run[g] = m_new;
            }
            if constexpr (L::kPBufs == 2) {
                unsigned char* pb = smem + L::pbuf + sb * L::kPBytes;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    *reinterpret_cast<__nv_bfloat16*>(pb + sw_elem(rg * G + g, i, L::kPHalf)) = eb[0][g];
            } else {
                // P^T of sub-tile s over K slot s of this stage (S(t) is done with it):
                // the 8 threads of a group of 8 rows zero the 16-byte chunks of those
                // rows in every column, then each writes its nonzero entries
                const int kg = i >> 3, r = i & 7;
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    unsigned char* pb = stage_k<G, D>(smem, st, s);
#pragma unroll
                    for (int cm = 0; cm < NCOL / 8; ++cm) {
                        const int c = r + 8 * cm;
                        *reinterpret_cast<uint4*>(pb + (kg >> 3) * L::kPHalf + (c >> 3) * 1024 + (c & 7) * 128 +
                                                  (((kg & 7) ^ (c & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                __syncwarp();
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    unsigned char* pb = stage_k<G, D>(smem, st, s);
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        *reinterpret_cast<__nv_bfloat16*>(pb + sw_elem(rg * G + g, i, L::kPHalf)) = eb[s][g];
                }
            }
            if (pos == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) alpha_buf[(t % 3) * NCOL + rg * G + g] = al[g];
            }
            if (m.last()) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float x = l_part[g];
#pragma unroll
                    for (int mask = 8; mask >= 1; mask >>= 1) x += __shfl_xor_sync(0xffffffffu, x, mask);
                    if (pos == 0) {
                        l_buf[(m.item % 3) * NCOL + rg * G + g] = x;
                        m_buf[(m.item % 3) * NCOL + rg * G + g] = m_run[g];
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                if (!live[s]) {
                    // rows past the sequence end or of a skipped box: zero V so their
                    // 0-weights cannot meet NaN/Inf
#pragma unroll
                    for (int c = 0; c < L::NH; ++c) {
                        uint4* row = reinterpret_cast<uint4*>(stage_v<G, D>(smem, st, s * L::NH + c) + (i >> 3) * 1024 +
                                                              (i & 7) * 128);
#pragma unroll
                        for (int q = 0; q < 8; ++q) row[q] = make_uint4(0u, 0u, 0u, 0u);
                    }
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
    named_bar_sync(1, kDecodeThreads);
    // the combine grid that follows may be scheduled now (it waits for this grid to
    // finish before it reads anything); signalled late, so that its CTAs do not
    // take room on the SMs while this grid streams (measured 0.7 us a call faster
    // than at the start at the Llama-3.2-1B batch)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, L::TMEM);
    }
}

// Zeroes the decode's work-item queue; the decode grid is launched as its
// programmatic dependent.
__global__ void decode_queue_reset_kernel(uint32_t* queue) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) *queue = 0u;
}

// KV heads per box: the largest power of two <= 8 that divides H_kv.
inline int heads_per_box(int H_kv) {
    int ht = 8;
    while (ht > 1 && H_kv % ht != 0) ht >>= 1;
    return ht;
}

// Host side: the tensor maps and parameters of a tensor-core decode launch, and
// the number of work items it can have (an upper bound: B * splits * head groups).
inline cudaError_t decode_tc_prepare(void* out, const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                     int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                     float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                     CUtensorMap& tm_k, CUtensorMap& tm_v, CUtensorMap& tm_q, TcParams& p,
                                     int64_t& items) {
    const int H_kv = pool.num_kv_heads;
    const int G = num_q_heads / H_kv;
    const int D = pool.head_dim;
    const int HT = heads_per_box(H_kv);
    const uint64_t slots = (uint64_t)pool.num_blocks * pool.block_size;
    {
        // (d, slot, head): one box = 16 slots x HT heads x 64 d, head-major in shared memory
        const uint64_t dims[3] = {(uint64_t)D, slots, (uint64_t)H_kv};
        const uint64_t strides[2] = {(uint64_t)H_kv * D * 2, (uint64_t)D * 2};
        const uint32_t box[3] = {64, (uint32_t)kBoxPos, (uint32_t)HT};
        cudaError_t e = encode_tiled_bf16(&tm_k, const_cast<void*>(k_pool), 3, dims, strides, box);
        if (e != cudaSuccess) return e;
        e = encode_tiled_bf16(&tm_v, const_cast<void*>(v_pool), 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        // q rows of one item: the HT * G query heads of its KV heads
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)B * num_q_heads};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64, (uint32_t)(HT * G)};
        cudaError_t e = encode_tiled_bf16(&tm_q, const_cast<void*>(q), 2, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
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
    p.H_kv = H_kv;
    p.N = pool.num_blocks;
    p.P = pool.block_size;
    p.max_splits = max_splits;
    p.HT = HT;
    p.NB = 8 / HT;
    p.HGRP = H_kv / HT;
    p.span = tc_span(D, p.NB);
    p.scale_log2 = scale * 1.4426950408889634f;
    items = (int64_t)B * max_splits * p.HGRP;
    return cudaSuccess;
}

}  // namespace
}  // namespace wf
