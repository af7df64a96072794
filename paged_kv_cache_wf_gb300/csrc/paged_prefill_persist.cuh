// paged_prefill_persist.cuh -- the tensor-core prefill as a persistent grid: each CTA
// runs a list of query blocks, longest first, with one K/V pipeline across them.
//
// What is computed is the causal prefill of paged_prefill_tc.cuh (tiny-vllm-py, "KV
// Cache"; ember, "The core idea"; weft, "Shapes and symbols"), with the same per-query-
// block arithmetic, so the outputs are the same bytes.  What changes is the schedule.
// One CTA per query block pays a start (TMEM allocation, the query tile's and the
// first K tile's loads: ~2.4 us before the first softmax) and an end (the last P.V,
// the epilogue, the launch of the next CTA: ~3-4 us) per block, and the grid's order
// (query block index, longest first) leaves SMs idle at the end when requests differ
// in length.  Here:
//   * every CTA computes the same longest-first order of the (request, query block)
//     pairs -- a counting sort on the number of 128-key tiles a block reads, ties in
//     (request, block) order -- expands each pair to its H_kv KV heads and deals the
//     items to the CTAs in a snake (round r: CTA c takes item r * ncta + c, or
//     r * ncta + ncta - 1 - c when r is odd), which balances the per-CTA work;
//   * a K warp and a V warp stream the items' K and V tiles through their rings
//     without a break, and a third warp reloads each query tile as soon as its last
//     S product of the previous item is done, so the next block's first tiles are in
//     flight while the current block finishes, and the MMA warp issues the next
//     block's first S = Q K^T while the softmax warps run the current block's
//     epilogue;
//   * the V tile an item ends in gets the rows of its last, partial 16-key block
//     copied by hand (the rest zeroed) before it is handed over, so no warp waits
//     for its own copy to land.
// The ring's slots, the query tile and every barrier keep counting across items; each
// role walks the same item list and derives every barrier phase from it.
#pragma once

#include "paged_prefill_tc.cuh"

namespace wf {

namespace {

template <int D, int G>
struct PpLayout {
    using B0 = PfLayout<D, G>;
    static constexpr int QT = B0::QT, TOKT = B0::TOKT, BMQ = B0::BMQ, NC = B0::NC;
    static constexpr int QTILE = B0::QTILE, SLOT = B0::SLOT, ATOM = B0::ATOM, HALF_OFF = B0::HALF_OFF,
                         BOX = B0::BOX;
    // K ring and V ring: K tile number g (counted over the CTA's items) in K slot g % KS,
    // V tile g in V slot KS + g % VS
    static constexpr int KS = D == 128 ? 2 : 4;
    static constexpr int VS = D == 128 ? 2 : 4;
    static constexpr int NSLOT = KS + VS;
    static constexpr int LMAX = 256;     // items one CTA can hold (the host sizes the grid)
    static constexpr int RMAX = 1024;    // requests the list build takes
    static constexpr int PMAX = 4096;    // (request, query block) pairs it sorts
    static constexpr int NB = 1024;      // sort buckets: tiles read, capped
    static constexpr int q = 0;
    static constexpr int kv = QT * QTILE;
    static constexpr int list = kv + NSLOT * SLOT;
    static constexpr int bars = list + LMAX * 8;
    // per query tile q_full, q_empty; slot_full[NSLOT], slot_empty[NSLOT]; per query
    // tile s_full, p_full, pv_done
    static constexpr int nbars = 2 * QT + 2 * NSLOT + 3 * QT;
    static constexpr int tmem_slot = bars + nbars * 8;
    static constexpr int misc = tmem_slot + 16;   // [0] items of this CTA, [1] abort, [2] pairs
    static constexpr int total = misc + 16;
    // list-build scratch, on the K/V ring before its first load
    static constexpr int s_req = kv;
    static constexpr int s_key = s_req + RMAX * 4;
    static constexpr int s_pair = s_key + PMAX * 4;
    static constexpr int s_cnt = s_pair + PMAX * 4;
    static_assert(s_cnt + NB * 4 <= list, "list-build scratch exceeds the K/V ring");
    static constexpr int SCOL = 128, OCOL = 256, TMEM_COLS = 512;
    static_assert(total + 1024 <= 232448, "persistent prefill CTA exceeds shared memory");
};

// One query block of one KV head: what every role derives from a list entry.
struct PfItem {
    int b, h, q_begin, n, c, i0, rows_tok, kend, ntiles, nt0, nt1;
};

template <class L>
__device__ __forceinline__ PfItem pf_item(const PfParams& p, int2 e) {
    PfItem it;
    it.b = e.x & 0xffff;
    const int qb = e.x >> 16;
    it.h = e.y;
    it.q_begin = __ldg(p.cu_q_lens + it.b);
    it.n = __ldg(p.cu_q_lens + it.b + 1) - it.q_begin;
    it.c = __ldg(p.seq_lens + it.b) - it.n;
    it.i0 = qb * L::BMQ;
    it.rows_tok = min(L::BMQ, it.n - it.i0);
    it.kend = it.c + it.i0 + it.rows_tok;
    it.ntiles = (it.kend + PN - 1) / PN;
    const int toks1 = it.rows_tok - L::TOKT;
    it.nt0 = (it.c + it.i0 + min(L::TOKT, it.rows_tok) + PN - 1) / PN;
    it.nt1 = toks1 > 0 ? (it.c + it.i0 + L::TOKT + toks1 + PN - 1) / PN : 0;
    return it;
}

// This CTA's work list (all threads; ends with a barrier).  Requests that fail the
// argument checks are reported and contribute no pairs.
template <class L>
__device__ void pf_build_list(const PfParams& p, unsigned char* smem, int cta, int ncta) {
    int* s_req = reinterpret_cast<int*>(smem + L::s_req);
    int* s_key = reinterpret_cast<int*>(smem + L::s_key);
    int* s_pair = reinterpret_cast<int*>(smem + L::s_pair);
    int* s_cnt = reinterpret_cast<int*>(smem + L::s_cnt);
    int* misc = reinterpret_cast<int*>(smem + L::misc);
    int2* list = reinterpret_cast<int2*>(smem + L::list);
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
    // keys run up to ceil(max_seq_len / PN), capped: only those buckets are used
    const int nbk = min((p.max_seq_len + PN - 1) / PN + 1, L::NB);
    for (int x = tid; x < nbk; x += nthr) s_cnt[x] = 0;
    for (int b = tid; b < p.B; b += nthr) {
        const int q_begin = __ldg(p.cu_q_lens + b);
        const int q_end = __ldg(p.cu_q_lens + b + 1);
        const int n = q_end - q_begin;
        const int len = __ldg(p.seq_lens + b);
        const bool bad = q_begin < 0 || n < 0 || q_end > p.total_q || n > p.max_q_len || len < n ||
                         len > p.max_seq_len || (int64_t)len > (int64_t)p.M * p.P;
        if (bad && cta == 0) report(p.dev_status, WF_DEV_BAD_SEQLEN);
        s_req[b] = bad ? 0 : (n + L::BMQ - 1) / L::BMQ;
    }
    __syncthreads();
    if (tid < 32) {   // first pair of each request (exclusive prefix sum)
        int run = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            const int v = b < p.B ? s_req[b] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (b < p.B) s_req[b] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) misc[2] = run;
    }
    __syncthreads();
    const int npairs = misc[2];
    for (int b = tid; b < p.B; b += nthr) {   // sort key: 128-key tiles the block reads
        const int first = s_req[b];
        const int last = b + 1 < p.B ? s_req[b + 1] : npairs;
        if (first == last) continue;
        const int q_begin = __ldg(p.cu_q_lens + b);
        const int n = __ldg(p.cu_q_lens + b + 1) - q_begin;
        const int c = __ldg(p.seq_lens + b) - n;
        for (int qb = 0; qb < last - first; ++qb) {
            const int kend = c + min((qb + 1) * L::BMQ, n);
            const int key = min((kend + PN - 1) / PN, L::NB - 1);
            s_key[first + qb] = key;
            s_pair[first + qb] = b | (qb << 16);
            atomicAdd(&s_cnt[key], 1);
        }
    }
    __syncthreads();
    if (tid < 32) {
        // bucket starts, longest first: start(x) = pairs whose key is above x
        int run = 0;
        for (int top = nbk; top > 0; top -= 32) {
            const int x = top - 1 - lane;
            const int v = x >= 0 ? s_cnt[x] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (x >= 0) s_cnt[x] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        // stable ranks within a bucket (32 pairs a round, in pair order) and the deal
        for (int base = 0; base < npairs; base += 32) {
            const int pi = base + lane;
            const bool in = pi < npairs;
            const int key = in ? s_key[pi] : -1 - lane;
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int before = __popc(peers & ((1u << lane) - 1u));
            const int rank = in ? s_cnt[key] + before : 0;
            __syncwarp();
            if (in && before == 0) s_cnt[key] += __popc(peers);
            __syncwarp();
            if (in) {
                // items rank * H_kv + hh, hh < H_kv: round k / ncta, position k % ncta
                const int k0 = rank * p.H_kv;
                int round = k0 / ncta, pos = k0 - round * ncta;
                for (int hh = 0; hh < p.H_kv; ++hh) {
                    const int owner = (round & 1) ? ncta - 1 - pos : pos;
                    if (owner == cta && round < L::LMAX) list[round] = make_int2(s_pair[pi], hh);
                    if (++pos == ncta) {
                        pos = 0;
                        ++round;
                    }
                }
            }
        }
        if (lane == 0) {
            const int total = npairs * p.H_kv;
            const int R = total / ncta, rem = total - R * ncta;
            const int pos = (R & 1) ? ncta - 1 - cta : cta;
            const int mine = R + (pos < rem ? 1 : 0);
            misc[0] = mine < L::LMAX ? mine : L::LMAX;
            misc[1] = 0;
        }
    }
    // the scratch was written through the generic proxy; the ring is next written by TMA
    tc::fence_proxy_async_smem();
    __syncthreads();
}

// The persistent kernel's body for CTA `cta` of `ncta`, run by all kThreads threads.
template <int D, int G>
__device__ __forceinline__ void prefill_tc_persist(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                                   const CUtensorMap& tm_v, const PfParams& p,
                                                   unsigned char* smem_raw, int cta, int ncta) {
    using L = PpLayout<D, G>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
    uint64_t* q_full = bars;              // [t]
    uint64_t* q_empty = bars + L::QT;     // [t]
    uint64_t* slot_full = bars + 2 * L::QT;
    uint64_t* slot_empty = slot_full + L::NSLOT;
    uint64_t* tb = slot_empty + L::NSLOT;
    auto s_full = [&](int t) { return tb + t * 3; };
    auto p_full = [&](int t) { return tb + t * 3 + 1; };
    auto pv_done = [&](int t) { return tb + t * 3 + 2; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + L::misc);
    const int2* list = reinterpret_cast<const int2*>(smem + L::list);
    auto kslot = [&](int g) { return g % L::KS; };
    auto vslot = [&](int g) { return L::KS + g % L::VS; };
    auto slot_ptr = [&](int s) { return smem + L::kv + s * L::SLOT; };
    auto fail = [&]() {
        report(p.dev_status, WF_DEV_TIMEOUT);
        misc[1] = 1;
    };

    if (warp == kMma) {
        tc::alloc(tmem_slot, L::TMEM_COLS);
        tc::relinquish();
    }
    if (threadIdx.x == 0) {
        for (int t = 0; t < L::QT; ++t) {
            mbar_init(&q_full[t], 1);
            mbar_init(&q_empty[t], 1);
        }
        for (int i = 0; i < L::NSLOT; ++i) {
            mbar_init(&slot_full[i], 1);
            mbar_init(&slot_empty[i], 1);
        }
        for (int t = 0; t < L::QT; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 4);
            mbar_init(pv_done(t), 1);
        }
        fence_mbar_init();
    }
    pf_build_list<L>(p, smem, cta, ncta);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int n_my = misc[0];

    if (warp >= kSoft && warp < kMma) {
        // ============================= producers ====================================
        // producer 0: K tiles, producer 1: V tiles, producer 2: query tiles, each in
        // item order; a 16-key box per lane, its block id read from the table in global
        // memory (L2-resident) one tile ahead of its use.
        const int pw = warp - kSoft;
        if (pw == 2) {
            // query tile t of item i once tile t's S products of the previous item are
            // done; tile 1 only for items whose second query tile has rows
            int nb = 0;   // earlier items with a second query tile
            for (int i = 0; i < n_my && !misc[1]; ++i) {
                const PfItem it = pf_item<L>(p, list[i]);
#pragma unroll
                for (int t = 0; t < L::QT; ++t) {
                    if (t == 1 && it.nt1 == 0) continue;
                    const int prev = t == 0 ? i : nb;
                    if (prev > 0 && !mbar_wait(&q_empty[t], (prev - 1) & 1)) {
                        if (lane == 0) fail();
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&q_full[t], (uint32_t)L::QTILE);
#pragma unroll
                        for (int cb = 0; cb < L::NC; ++cb)
                            tma_load_3d_nohint(smem + L::q + t * L::QTILE + cb * (PM * 128), &tm_q, cb * 64, it.h * G,
                                               it.q_begin + it.i0 + t * L::TOKT, &q_full[t]);
                    }
                    __syncwarp();
                }
                if (it.nt1 > 0) ++nb;
            }
        } else {
            const bool isv = pw == 1;
            const CUtensorMap* tm = isv ? &tm_v : &tm_k;
            int g = 0;   // tiles of this ring issued so far
            for (int i = 0; i < n_my && !misc[1]; ++i) {
                const PfItem it = pf_item<L>(p, list[i]);
                const int32_t* trow = p.block_tables + (int64_t)it.b * p.M;
                int blk_next = 0;
                if (lane * 16 < min(PN, it.kend)) blk_next = __ldg(trow + (lane * 16) / p.P);
                for (int j = 0; j < it.ntiles; ++j, ++g) {
                    const int s = isv ? vslot(g) : kslot(g);
                    const int round = isv ? g / L::VS : g / L::KS;
                    const int k0 = j * PN;
                    const int kt = min(PN, it.kend - k0);
                    const int nbox = (kt + 15) >> 4;
                    const int blk = blk_next;
                    if (j + 1 < it.ntiles && lane * 16 < min(PN, it.kend - k0 - PN))
                        blk_next = __ldg(trow + (k0 + PN + lane * 16) / p.P);
                    if (round > 0 && !mbar_wait(&slot_empty[s], (round - 1) & 1)) {
                        if (lane == 0) fail();
                        break;
                    }
                    if (lane < nbox && (unsigned)blk >= (unsigned)p.N && !isv) report(p.dev_status, WF_DEV_BAD_BLOCK);
                    unsigned char* base = slot_ptr(s);
                    // V of the item's last tile: keys past its end must not be NaN (their
                    // weights are 0, but 0 * NaN is NaN in P.V).  16-key blocks past the end
                    // are zeroed; a block the end falls inside is copied row by row, its
                    // rows past the end zeroed, before the tile is handed over
                    const bool tail = isv && j == it.ntiles - 1 && kt < PN;
                    const bool part = tail && (kt & 15) != 0;
                    const int ntma = part ? kt >> 4 : nbox;   // blocks the TMA loads
                    if (tail) {
                        for (int rr = nbox * 16 + lane; rr < PN; rr += 32) {
#pragma unroll
                            for (int cb = 0; cb < L::NC; ++cb) {
                                uint4* row = reinterpret_cast<uint4*>(base + (rr >> 3) * L::ATOM +
                                                                      cb * L::HALF_OFF + (rr & 7) * 128);
#pragma unroll
                                for (int qq = 0; qq < 8; ++qq) row[qq] = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                    if (part) {
                        const int pb = kt >> 4;                 // the block within the tile
                        const int vr = kt & 15;                 // its rows before the end
                        const int pblk = __shfl_sync(0xffffffffu, blk, pb);
                        const bool pok = (unsigned)pblk < (unsigned)p.N;
                        const int pos0 = k0 + pb * 16;
                        unsigned char* pbase = base + pb * L::BOX;
                        // 16-byte chunk c of row r, half hf, at its 128-byte-swizzled place
                        for (int qd = lane; qd < 16 * L::NC * 8; qd += 32) {
                            const int r = qd / (L::NC * 8), hf = (qd >> 3) % L::NC, c = qd & 7;
                            uint4 v = make_uint4(0u, 0u, 0u, 0u);
                            if (r < vr && pok) {
                                const int64_t slot = (int64_t)pblk * p.P + (pos0 + r) % p.P;
                                v = __ldg(reinterpret_cast<const uint4*>(p.v_pool + (slot * p.H_kv + it.h) * D +
                                                                         hf * 64 + c * 8));
                            }
                            *reinterpret_cast<uint4*>(pbase + (r >> 3) * L::ATOM + hf * L::HALF_OFF + (r & 7) * 128 +
                                                      ((c ^ (r & 7)) << 4)) = v;
                        }
                    }
                    if (tail) tc::fence_proxy_async_smem();   // generic writes before the tensor core reads
                    const bool okb = lane < ntma && (unsigned)blk < (unsigned)p.N;
                    const unsigned okm = __ballot_sync(0xffffffffu, okb);
                    if (lane == 0) mbar_arrive_expect_tx(&slot_full[s], (uint32_t)__popc(okm) * (uint32_t)L::BOX);
                    __syncwarp();
                    if (okb) {
                        const int slot = blk * p.P + (k0 + lane * 16) % p.P;   // multiple of 16
                        unsigned char* dst = base + lane * L::BOX;
                        if constexpr (L::NC == 2) {
                            tma_load_5d(dst, tm, 0, 0, 0, slot >> 3, it.h, &slot_full[s]);
                        } else {
                            tma_load_3d_nohint(dst, tm, 0, slot, it.h, &slot_full[s]);
                        }
                    }
                }
            }
        }
    } else if (warp == kMma) {
        // ============================= MMA issuer ===================================
        // The event loop of paged_prefill_tc.cuh over each item in turn; tile and step
        // counters run on across items.  A query tile's last S product of an item releases
        // it (q_empty[t]); its first S product of the next item waits for the new one.
        constexpr uint32_t idS = tc::idesc_bf16_f32(PM, PN, 0, 0);
        constexpr uint32_t idO = tc::idesc_bf16_f32(PM, D, 0, 1);
        const uint64_t qdesc = tc::sdesc_sw128(smem_u32(smem + L::q), 16, 1024);
        const uint64_t kvdesc_k = tc::sdesc_sw128(smem_u32(smem + L::kv), 16, L::ATOM);
        const uint64_t kvdesc_v = tc::sdesc_sw128(smem_u32(smem + L::kv), L::HALF_OFF, L::ATOM);
        int g = 0;                    // K/V tiles of earlier items (both rings advance alike)
        int gs0 = 0, gs1 = 0;         // S/P steps of earlier items, per query tile
        int nb = 0;                   // earlier items with a second query tile
        bool ok = true;
        for (int i = 0; i < n_my && ok; ++i) {
            const PfItem it = pf_item<L>(p, list[i]);
            const int nt_t[2] = {it.nt0, it.nt1};
            const int gs_t[2] = {gs0, gs1};
            const uint32_t qpar[2] = {(uint32_t)i & 1u, (uint32_t)nb & 1u};
            int sq[2] = {0, 0}, sp[2] = {0, 0};
            uint32_t idle = 0;
            while (ok && (sp[0] < nt_t[0] || sp[1] < nt_t[1])) {
                bool did = false;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int o = t ^ 1;
                    const int u = sp[t];
                    if (u < sq[t]) {
                        const int gv = g + u;
                        const int vs = vslot(gv);
                        const bool rdy = mbar_test(p_full(t), (gs_t[t] + u) & 1) &&
                                         mbar_test(&slot_full[vs], (gv / L::VS) & 1);
                        if (__shfl_sync(0xffffffffu, (int)rdy, 0)) {
                            tc::fence_after_sync();
                            const uint32_t dO = tmem + L::OCOL + t * D;
                            const uint32_t pcol = tmem + t * L::SCOL;
                            const uint64_t vd = kvdesc_v + (uint64_t)((vs * L::SLOT) >> 4);
                            if (lane == 0) {
#pragma unroll
                                for (int kk = 0; kk < PN / 16; ++kk)
                                    tc::mma_f16_tmem_a(dO, pcol + kk * 8 + (kk >= 4 ? 32 : 0),
                                                       vd + (uint64_t)((kk * 2 * L::ATOM) >> 4), idO,
                                                       (u > 0 || kk > 0) ? 1u : 0u);
                                tc::commit(pv_done(t));
                                if (sp[o] > u || u >= nt_t[o]) tc::commit(&slot_empty[vs]);
                            }
                            __syncwarp();
                            sp[t] = u + 1;
                            did = true;
                        }
                    }
                    const int j = sq[t];
                    if (j < nt_t[t] && j == sp[t]) {
                        const int gk = g + j;
                        const int ks = kslot(gk);
                        const bool rdy = mbar_test(&slot_full[ks], (gk / L::KS) & 1) &&
                                         (j > 0 || mbar_test(&q_full[t], qpar[t]));
                        if (__shfl_sync(0xffffffffu, (int)rdy, 0)) {
                            tc::fence_after_sync();
                            const uint32_t dS = tmem + t * L::SCOL;
                            const uint64_t qd = qdesc + (uint64_t)((t * L::QTILE) >> 4);
                            const uint64_t kd = kvdesc_k + (uint64_t)((ks * L::SLOT) >> 4);
                            if (lane == 0) {
#pragma unroll
                                for (int kk = 0; kk < D / 16; ++kk) {
                                    const uint32_t qoff = (kk >> 2) * (PM * 128) + (kk & 3) * 32;
                                    const uint32_t koff = (kk >> 2) * L::HALF_OFF + (kk & 3) * 32;
                                    tc::mma_f16(dS, qd + (uint64_t)(qoff >> 4), kd + (uint64_t)(koff >> 4), idS,
                                                kk > 0 ? 1u : 0u);
                                }
                                tc::commit(s_full(t));
                                if (sq[o] > j || j >= nt_t[o]) tc::commit(&slot_empty[ks]);
                                if (j + 1 == nt_t[t]) tc::commit(&q_empty[t]);
                            }
                            __syncwarp();
                            sq[t] = j + 1;
                            did = true;
                        }
                    }
                }
                if (did) {
                    idle = 0;
                } else {
                    if (misc[1] || ++idle > (1u << 24)) {
                        if (lane == 0) fail();
                        ok = false;
                        break;
                    }
                    if (idle > 8) __nanosleep(32);
                }
            }
            g += it.ntiles;
            gs0 += it.nt0;
            gs1 += it.nt1;
            if (it.nt1 > 0) ++nb;
        }
    } else {
        // ============================= softmax ======================================
        // paged_prefill_tc.cuh's softmax and epilogue, item after item.
        const int t = warp >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const uint32_t sbase = tmem + lane_addr + t * L::SCOL;
        const uint32_t obase = tmem + lane_addr + L::OCOL + t * D;
        const int R = t * PM + r;
        const int tok = R / G, g = R % G;
        int gs = 0;   // S/P steps of this query tile in earlier items
        bool ok = true;
        for (int i = 0; i < n_my && ok && !misc[1]; ++i) {
            const PfItem it = pf_item<L>(p, list[i]);
            const int nt = t == 0 ? it.nt0 : it.nt1;
            if (nt == 0) continue;
            const int qi = it.i0 + tok;
            const bool row_valid = qi < it.n;
            const int last_key = it.c + qi;
            const int first_key_t = it.c + it.i0 + t * L::TOKT;
            float m_ref = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nt; ++j) {
                const int k0 = j * PN;
                if (!mbar_wait(s_full(t), (gs + j) & 1)) {
                    fail();
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const bool masked = (k0 + PN - 1 > first_key_t) || !row_valid;
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
                auto load_half = [&](int hh, float (&s)[2][32]) {
                    tc::ld_32cols(sbase + hh * 64, s[0]);
                    tc::ld_32cols(sbase + hh * 64 + 32, s[1]);
                    tc::wait_ld();
                    if (masked) {
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const bool vis = row_valid && k0 + hh * 64 + c2 * 32 + e <= last_key;
                                s[c2][e] = vis ? s[c2][e] : -INFINITY;
                            }
                    }
                };
                float s[2][32];
                load_half(0, s);
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                    for (int e = 0; e < 16; ++e) m8[e & 7] = fmax3(m8[e & 7], s[c2][e], s[c2][e + 16]);
                load_half(1, s);
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                    for (int e = 0; e < 16; ++e) m8[e & 7] = fmax3(m8[e & 7], s[c2][e], s[c2][e + 16]);
                const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float mt = mraw * p.scale_log2;
                float alpha = 1.f;
                if (m_ref == -INFINITY) {
                    m_ref = mt;
                } else if (mt > m_ref + kLazy) {
                    alpha = ex2(m_ref - mt);
                    m_ref = mt;
                }
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    if (!mbar_wait(pv_done(t), (gs + j - 1) & 1)) fail();
                    tc::fence_after_sync();
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        float o[32];
                        tc::ld_32cols(obase + c4 * 32, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tc::st_32cols(obase + c4 * 32, o);
                    }
                    tc::wait_st();
                }
                l_run *= alpha;
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(-m_use, -m_use);
                float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                auto weights = [&](int hh) {
                    uint32_t pw[32];
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float2 x = __ffma2_rn(make_float2(s[c2][2 * u], s[c2][2 * u + 1]), sc2, nm2);
                            const float2 e2 = make_float2(ex2(x.x), ex2(x.y));
                            ps[u & 3] = __fadd2_rn(ps[u & 3], e2);
                            pw[c2 * 16 + u] = pack_bf16x2(e2.x, e2.y);
                        }
                    }
                    tc::st_32words(sbase + hh * 64, pw);
                };
                weights(1);
                load_half(0, s);
                weights(0);
                tc::wait_st();
                const float2 ps01 = __fadd2_rn(ps[0], ps[1]), ps23 = __fadd2_rn(ps[2], ps[3]);
                const float2 pst = __fadd2_rn(ps01, ps23);
                l_run += pst.x + pst.y;
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(t));
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 ----------------------------------------------
            if (!mbar_wait(pv_done(t), (gs + nt - 1) & 1)) {
                fail();
                break;
            }
            tc::fence_after_sync();
            const float inv = row_valid ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                float o[32];
                tc::ld_32cols(obase + c4 * 32, o);
                tc::wait_ld();
                if (row_valid) {
                    __nv_bfloat16* dst =
                        p.out + ((int64_t)(it.q_begin + qi) * p.H_q + it.h * G + g) * D + c4 * 32;
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
            // O is read: the next item's first P.V (issued after this warpgroup's next P)
            // may overwrite it
            tc::fence_before_sync();
            gs += nt;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMma) {
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, L::TMEM_COLS);
    }
}

// Grid of the persistent prefill: one CTA per SM, more when the items' upper bound
// (every request at max_q_len) exceeds what the CTAs' lists hold.  0 when the batch is
// beyond the list build's limits (the one-CTA-per-block grid runs it instead).
template <int D, int G>
inline int prefill_persist_grid(int32_t B, int32_t max_q_len, int32_t H_kv, int sms) {
    using L = PpLayout<D, G>;
    if (B > L::RMAX) return 0;
    const int64_t pairs = (int64_t)B * ((max_q_len + L::BMQ - 1) / L::BMQ);
    if (pairs > L::PMAX) return 0;
    const int64_t items = pairs * H_kv;
    if (items > (int64_t)1 << 30) return 0;
    int64_t grid = items < sms ? items : sms;
    if (grid * L::LMAX < items) grid = (items + L::LMAX - 1) / L::LMAX;
    return grid < 1 ? 1 : (int)grid;
}

}  // namespace
}  // namespace wf
