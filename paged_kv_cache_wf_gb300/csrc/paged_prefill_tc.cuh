// paged_prefill_tc.cuh -- pipelined, warp-specialised causal prefill on tcgen05 for
// bf16 pools whose block size is a multiple of 16.
//
// What is computed (tiny-vllm-py, "KV Cache": prefill attention is causal;
// "Dense vs. Ragged batching"): query row i of request b (position c_b + i, c_b =
// seq_lens[b] - n_b) attends to positions 0 .. c_b + i of its KV head, read from the
// [N, P, H_kv, D] pool through block_table[b][p / P], offset p % P (ember, "The core
// idea"); query head g uses KV head g / G (weft, "Shapes and symbols").
//
// GB300 design.  One CTA = one request, one KV head and two query tiles of 128
// rows r = (token, g): 128/G consecutive query tokens times the G query heads that
// share the KV head.  Every 128-key K/V tile loaded serves both query tiles (256
// rows), and every MMA has N >= 128.  12 warps:
//   warps 0-7   softmax, one warpgroup per query tile; thread r <-> row r <-> TMEM
//               lane r: causal mask (only on tiles that cross the diagonal), online
//               softmax in the exp2 domain with a lazy rescale (O in TMEM is rescaled
//               only when a row max grows by more than 2^8), P written as bf16 pairs
//               over S columns already read (keys 0-63 into columns 0-31, keys 64-127
//               into columns 64-95); the epilogue divides O by the row sum.
//   warps 8-10  producers: TMA loads of the two Q tiles (3D box d x head x token) and,
//               tile by tile, of 128 keys of K and V gathered 16-key block by block
//               through the block table (one box per lane, 128-byte swizzle) into a
//               ring of K and V slots.  The producer of a CTA's last V tile, when
//               that tile runs past the CTA's last key, zeroes the rows past it (their
//               weights are 0, but 0 * NaN is NaN in P.V) and releases the tile to
//               P.V through its own barrier, off the softmax's path.
//   warp 11     MMA issuer, event loop over both query tiles: S_t(j) = Q_t K_j^T
//               (M=128, N=128 keys, K=D) into TMEM, O_t += P_t(j) V_j (M=128, N=D,
//               K=128 keys, P from TMEM, V MN-major from shared memory); commits hand
//               S to the softmax and release ring slots.
#pragma once

#include <cuda.h>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int PM = 128;          // rows per query tile (TMEM lanes, MMA M)
constexpr int PN = 128;          // keys per K/V tile (MMA N of S = Q K^T)
constexpr float kLazy = 8.f;     // rescale O only when the row max grows by more than 2^8
// warps 0-7 softmax (two warpgroups, one per query tile), then kProd producer warps,
// then the MMA warp.  12 warps leave 168 registers per thread.
constexpr int kSoft = 8;
constexpr int kProd = 3;         // producer warps: ring slot s is refilled by producer s % kProd
constexpr int kMma = kSoft + kProd;
constexpr int kThreads = (kMma + 1) * 32;

struct PfParams {
    __nv_bfloat16* out;
    const __nv_bfloat16* v_pool;   // rows of a V tile's last partial block are copied by hand
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    uint32_t* dev_status;
    int32_t M, B, total_q, max_q_len, max_seq_len, H_q, H_kv, G, N, P, nqblk;
    float scale_log2;
};

// One CTA per SM.  Two 128-row query tiles (A, B) share every K/V tile, which
// doubles the work per loaded byte.  Each query tile has its own softmax
// warpgroup, S accumulator and O accumulator in TMEM; while one group computes
// its softmax the tensor core runs the other tile's products.  Every MMA has
// N >= 128 (S: 128 keys, P.V: N = D), which a single issuing thread keeps fed.
template <int D, int G>
struct PfLayout {
    static constexpr int QT = 2;                    // query tiles per CTA
    static constexpr int TOKT = PM / G;             // query tokens per tile
    static constexpr int BMQ = QT * TOKT;           // query tokens per CTA
    static constexpr int NC = D / 64;               // 64-wide column blocks of D
    static constexpr int QTILE = PM * D * 2;        // one query tile
    static constexpr int SLOT = PN * D * 2;         // one K or V tile
    // K/V ring: K(j) is load unit 2j, V(j) unit 2j + 1, unit u in slot u % NSLOT, so a
    // K tile is released after its S products and a V tile after its P.V products.
    static constexpr int NSLOT = D == 128 ? 4 : 8;
    static constexpr int TBL = 2048;                // block-table entries staged in shared memory
    // D = 128: one 4 KB box per 16-key block holds both 64-wide halves, laid out
    // [8-key group][half][8 keys][64 d] -- atoms 2048 B apart, halves 1024 B apart.
    // D = 64: one 2 KB box per block, [16 keys][64 d] -- atoms 1024 B apart.
    static constexpr int ATOM = NC == 2 ? 2048 : 1024;   // stride between 8-key atoms
    static constexpr int HALF_OFF = 1024;                 // offset of the second 64-wide half
    static constexpr int BOX = NC * 2048;                 // bytes of one block's box
    static constexpr int q = 0;
    static constexpr int kv = QT * QTILE;
    static constexpr int tbl = kv + NSLOT * SLOT;
    static constexpr int bars = tbl + TBL * 4;
    // q_full, slot_full[NSLOT], slot_empty[NSLOT], then per query tile: s_full,
    // p_full, pv_done, then v_fixed
    static constexpr int nbars = 1 + 2 * NSLOT + QT * 3 + 1;
    static constexpr int tmem_slot = bars + nbars * 8;
    static constexpr int total = tmem_slot + 16;
    // TMEM: S of query tile t in columns [128 t, 128 t + 128) -- its softmax weights
    // P (bf16 pairs) replace columns 0-31 (keys 0-63) and 64-95 (keys 64-127) of
    // them -- and O of tile t at 256 + D t.
    static constexpr int SCOL = 128;
    static constexpr int OCOL = 256;
    static constexpr int TMEM_COLS = 512;
    static_assert(total + 1024 <= 232448, "prefill CTA exceeds shared memory");
};

// The kernel's body for the CTA of (request, KV head) bx and query-block index by
// (query block p.nqblk - 1 - by), run by all kThreads threads of the block.
template <int D, int G>
__device__ __forceinline__ void prefill_tc_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                                const CUtensorMap& tm_v, const PfParams& p,
                                                unsigned char* smem_raw, int bx, int by) {
    using L = PfLayout<D, G>;
    const int qb = p.nqblk - 1 - by;   // the longest query blocks start first
    const int hb = bx;                      // (request, KV head)
    const int h = hb % p.H_kv, b = hb / p.H_kv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int q_begin = __ldg(p.cu_q_lens + b);
    const int q_end = __ldg(p.cu_q_lens + b + 1);
    const int n = q_end - q_begin;
    const int len = __ldg(p.seq_lens + b);
    const bool bad = q_begin < 0 || n < 0 || q_end > p.total_q || n > p.max_q_len || len < n ||
                     len > p.max_seq_len || (int64_t)len > (int64_t)p.M * p.P;
    if (bad) {
        if (by == 0 && h == 0 && threadIdx.x == 0) report(p.dev_status, WF_DEV_BAD_SEQLEN);
        return;
    }
    const int i0 = qb * L::BMQ;
    if (i0 >= n) return;
    const int c = len - n;                            // cached prefix
    const int rows_tok = min(L::BMQ, n - i0);
    const int kend = c + i0 + rows_tok;               // keys this CTA needs: [0, kend)
    const int ntiles = (kend + PN - 1) / PN;
    // K/V tiles query tile t takes part in: those holding keys its rows see (0 when
    // the tile has no query rows; tile 0 always has some)
    int nt_t[L::QT];
#pragma unroll
    for (int t = 0; t < L::QT; ++t) {
        const int toks = min(L::TOKT, rows_tok - t * L::TOKT);
        nt_t[t] = toks > 0 ? (c + i0 + t * L::TOKT + toks + PN - 1) / PN : 0;
    }

    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
    uint64_t* q_full = bars;
    uint64_t* slot_full = bars + 1;
    uint64_t* slot_empty = slot_full + L::NSLOT;
    uint64_t* tb = slot_empty + L::NSLOT;             // per query tile: s_full, p_full, pv_done
    auto s_full = [&](int t) { return tb + t * 3; };
    auto p_full = [&](int t) { return tb + t * 3 + 1; };
    auto pv_done = [&](int t) { return tb + t * 3 + 2; };
    // the last V tile of a CTA whose last key tile is partial, once its rows past kend
    // are zero
    uint64_t* v_fixed = tb + 3 * L::QT;
    const bool partial = kend % PN != 0;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);
    int32_t* tbl = reinterpret_cast<int32_t*>(smem + L::tbl);
    // load unit u (K(j): u = 2j, V(j): u = 2j + 1)
    auto unit_slot = [&](int u) { return smem + L::kv + (u % L::NSLOT) * L::SLOT; };

    if (warp == kMma) {
        tc::alloc(tmem_slot, L::TMEM_COLS);
        tc::relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < L::NSLOT; ++i) {
            mbar_init(&slot_full[i], 1);
            mbar_init(&slot_empty[i], 1);
        }
        for (int t = 0; t < L::QT; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 4);
            mbar_init(pv_done(t), 1);
        }
        mbar_init(v_fixed, 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kSoft && warp < kMma) {
        // ============================= producers ====================================
        // A thread's TMA copies complete one after another, so the load units are spread
        // over several warps, one 16-key box per lane, to keep many copies in flight.
        const int pw = warp - kSoft;                     // producer index
        if (pw == 0 && lane == 0) {
            mbar_arrive_expect_tx(q_full, (uint32_t)(L::QT * L::QTILE));
#pragma unroll
            for (int t = 0; t < L::QT; ++t)
#pragma unroll
                for (int cb = 0; cb < L::NC; ++cb)
                    tma_load_3d_nohint(smem + L::q + t * L::QTILE + cb * (PM * 128), &tm_q, cb * 64, h * G,
                                       q_begin + i0 + t * L::TOKT, q_full);
        }
        // the CTA's block-table slice, staged once when it fits
        const int nblk = (kend + p.P - 1) / p.P;
        const int32_t* trow = p.block_tables + (int64_t)b * p.M;
        const bool staged = nblk <= L::TBL;
        if (staged) {
            for (int i = threadIdx.x - kSoft * 32; i < nblk; i += kProd * 32) tbl[i] = __ldg(trow + i);
            named_bar_sync(2, kProd * 32);
        }
        // Each ring slot is refilled by one producer warp (slot s by producer s % kProd),
        // in order: a parity wait tells phase r from phase r - 2 only if the waiter is at
        // most one phase ahead, so no warp may move on to a slot's next round before the
        // previous one was issued.  A warp takes its units in increasing order.
        for (int u = 0; u < 2 * ntiles; ++u) {
            const int j = u >> 1, isv = u & 1;
            const int sl = u % L::NSLOT;
            if (sl % kProd != pw) continue;
            const int k0 = j * PN;
            const int kt = min(PN, kend - k0);
            const int nbox = (kt + 15) >> 4;            // 16-key blocks in this tile (<= 8)
            if (u >= L::NSLOT && !mbar_wait(&slot_empty[sl], ((u / L::NSLOT) - 1) & 1)) {
                if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            bool okb = false;
            int blk = 0;
            if (lane < nbox) {
                const int bi = (k0 + lane * 16) / p.P;
                blk = staged ? tbl[bi] : __ldg(trow + bi);
                okb = (unsigned)blk < (unsigned)p.N;
                if (!okb && isv == 0) report(p.dev_status, WF_DEV_BAD_BLOCK);
            }
            if (isv && partial && j == ntiles - 1) {
                // rows of 16-key blocks past the CTA's end are not loaded: zero them now
                for (int rr = nbox * 16 + lane; rr < PN; rr += 32) {
#pragma unroll
                    for (int cb = 0; cb < L::NC; ++cb) {
                        uint4* row = reinterpret_cast<uint4*>(unit_slot(u) + (rr >> 3) * L::ATOM + cb * L::HALF_OFF +
                                                              (rr & 7) * 128);
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq) row[qq] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            const unsigned okm = __ballot_sync(0xffffffffu, okb);
            if (lane == 0) mbar_arrive_expect_tx(&slot_full[sl], (uint32_t)__popc(okm) * (uint32_t)L::BOX);
            __syncwarp();
            if (okb) {
                const int slot = blk * p.P + (k0 + lane * 16) % p.P;   // multiple of 16
                unsigned char* dst = unit_slot(u) + lane * L::BOX;
                if constexpr (L::NC == 2) {
                    tma_load_5d(dst, isv ? &tm_v : &tm_k, 0, 0, 0, slot >> 3, h, &slot_full[sl]);
                } else {
                    tma_load_3d_nohint(dst, isv ? &tm_v : &tm_k, 0, slot, h, &slot_full[sl]);
                }
            }
            if (isv && partial && j == ntiles - 1) {
                // keys past the CTA's end were not loaded (or hold whatever the pool has
                // there): their P is 0, but 0 * NaN is NaN in P.V, so their V rows are
                // zeroed once the tile has landed, before P.V may read it
                if (!mbar_wait(&slot_full[sl], (uint32_t)(u / L::NSLOT) & 1u)) {
                    if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
                for (int rr = kend - k0 + lane; rr < nbox * 16; rr += 32) {   // the last block's tail
#pragma unroll
                    for (int cb = 0; cb < L::NC; ++cb) {
                        uint4* row = reinterpret_cast<uint4*>(unit_slot(u) + (rr >> 3) * L::ATOM + cb * L::HALF_OFF +
                                                              (rr & 7) * 128);
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq) row[qq] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(v_fixed);
            }
        }
    } else if (warp == kMma) {
        // ============================= MMA issuer ===================================
        // Per query tile t the products run in order S_t(0), P_t(0).V_0, S_t(1), ...:
        // S_t(j+1) overwrites the columns P_t(j) lives in, and the tensor core executes
        // one thread's MMAs in issue order.  O_t += P_t(j) V_j is issued as soon as the
        // softmax has written P_t(j) and V_j has landed; S_t(j+1) = Q_t K_{j+1}^T right
        // after it once K_{j+1} has landed.  A K or V slot is released by the product
        // of the last query tile that reads it.
        // The whole warp runs the loop (lane 0's barrier observations decide, broadcast
        // by shuffle) so that control flow and descriptors stay warp-uniform; lane 0
        // alone issues.  Descriptors are built once and advanced by adding the byte
        // offset >> 4 to their start-address field.
        constexpr uint32_t idS = tc::idesc_bf16_f32(PM, PN, 0, 0);
        constexpr uint32_t idO = tc::idesc_bf16_f32(PM, D, 0, 1);
        const bool ok = mbar_wait(q_full, 0);
        if (!ok && lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
        const uint64_t qdesc = tc::sdesc_sw128(smem_u32(smem + L::q), 16, 1024);
        const uint64_t kvdesc_k = tc::sdesc_sw128(smem_u32(smem + L::kv), 16, L::ATOM);
        // V as MN-major B: 64-wide halves HALF_OFF apart, 8-key atoms ATOM apart
        const uint64_t kvdesc_v = tc::sdesc_sw128(smem_u32(smem + L::kv), L::HALF_OFF, L::ATOM);
        int sq[L::QT], sp[L::QT];   // next S and next P.V of each query tile
#pragma unroll
        for (int t = 0; t < L::QT; ++t) sq[t] = sp[t] = 0;
        uint32_t idle = 0;
        while (ok && (sp[0] < nt_t[0] || sp[1] < nt_t[1])) {
            bool did = false;
#pragma unroll
            for (int t = 0; t < L::QT; ++t) {
                const int o = t ^ 1;
                const int u = sp[t];
                if (u < sq[t]) {
                    const int vu = 2 * u + 1;
                    const bool vlast = partial && u == ntiles - 1;
                    const bool rdy = mbar_test(p_full(t), u & 1) &&
                                     (vlast ? mbar_test(v_fixed, 0)
                                            : mbar_test(&slot_full[vu % L::NSLOT], (vu / L::NSLOT) & 1));
                    if (__shfl_sync(0xffffffffu, (int)rdy, 0)) {
                        tc::fence_after_sync();
                        const uint32_t dO = tmem + L::OCOL + t * D;
                        const uint32_t pcol = tmem + t * L::SCOL;
                        const uint64_t vd = kvdesc_v + (uint64_t)(((vu % L::NSLOT) * L::SLOT) >> 4);
                        if (lane == 0) {
#pragma unroll
                            for (int kk = 0; kk < PN / 16; ++kk)
                                tc::mma_f16_tmem_a(dO, pcol + kk * 8 + (kk >= 4 ? 32 : 0),
                                                   vd + (uint64_t)((kk * 2 * L::ATOM) >> 4), idO,
                                                   (u > 0 || kk > 0) ? 1u : 0u);
                            tc::commit(pv_done(t));
                            if (sp[o] > u || u >= nt_t[o]) tc::commit(&slot_empty[vu % L::NSLOT]);
                        }
                        __syncwarp();
                        sp[t] = u + 1;
                        did = true;
                    }
                }
                const int j = sq[t];
                if (j < nt_t[t] && j == sp[t]) {
                    const int ku = 2 * j;
                    const bool rdy = mbar_test(&slot_full[ku % L::NSLOT], (ku / L::NSLOT) & 1);
                    if (__shfl_sync(0xffffffffu, (int)rdy, 0)) {
                        tc::fence_after_sync();
                        const uint32_t dS = tmem + t * L::SCOL;
                        const uint64_t qd = qdesc + (uint64_t)((t * L::QTILE) >> 4);
                        const uint64_t kd = kvdesc_k + (uint64_t)(((ku % L::NSLOT) * L::SLOT) >> 4);
                        if (lane == 0) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t qoff = (kk >> 2) * (PM * 128) + (kk & 3) * 32;
                                const uint32_t koff = (kk >> 2) * L::HALF_OFF + (kk & 3) * 32;
                                tc::mma_f16(dS, qd + (uint64_t)(qoff >> 4), kd + (uint64_t)(koff >> 4), idS,
                                            kk > 0 ? 1u : 0u);
                            }
                            tc::commit(s_full(t));
                            if (sq[o] > j || j >= nt_t[o]) tc::commit(&slot_empty[ku % L::NSLOT]);
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
                if (++idle > (1u << 24)) {
                    if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
                if (idle > 8) __nanosleep(32);
            }
        }
    } else {
        // ============================= softmax ======================================
        const int t = warp >> 2;                         // query tile of this warpgroup
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                  // row / TMEM lane
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const uint32_t sbase = tmem + lane_addr + t * L::SCOL;
        const uint32_t obase = tmem + lane_addr + L::OCOL + t * D;
        const int R = t * PM + r;                        // row within the CTA
        const int tok = R / G, g = R % G;
        const int qi = i0 + tok;
        const bool row_valid = qi < n;
        const int last_key = c + qi;                     // row sees keys 0 .. last_key
        const int first_key_t = c + i0 + t * L::TOKT;    // smallest last_key in this tile
        const int nt = nt_t[t];
        float m_ref = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nt && ok; ++j) {
            const int k0 = j * PN;
            if (!mbar_wait(s_full(t), j & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                ok = false;
                break;
            }
            tc::fence_after_sync();
            // keys some row of the tile may not see are masked.  Three round trips to
            // TMEM: keys 0-63 (their maximum), keys 64-127 (kept in registers for their
            // weights), keys 0-63 again.  The row max is taken on raw scores (scale > 0)
            // and scaled once.
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
            // lazy online softmax: move the reference max only when it grows by > 2^8
            float alpha = 1.f;
            if (m_ref == -INFINITY) {
                m_ref = mt;
            } else if (mt > m_ref + kLazy) {
                alpha = ex2(m_ref - mt);
                m_ref = mt;
            }
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                // O must hold P.V of tile j-1 before it is rescaled
                if (!mbar_wait(pv_done(t), (j - 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
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
            // weights of the half in registers -> bf16 pairs -> TMEM (keys 64-127 into
            // columns 64-95, keys 0-63 into columns 0-31: S there is consumed)
            auto weights = [&](int hh) {
                uint32_t pw[32];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        // exponent = s * scale*log2(e) - m_ref, two keys per fp32x2 FMA
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
        // ---- epilogue: O / l -> bf16 --------------------------------------------------
        if (ok && nt > 0) {
            if (!mbar_wait(pv_done(t), (nt - 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            tc::fence_after_sync();
            const float inv = row_valid ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                float o[32];
                tc::ld_32cols(obase + c4 * 32, o);
                tc::wait_ld();
                if (row_valid) {
                    __nv_bfloat16* dst = p.out + ((int64_t)(q_begin + qi) * p.H_q + h * G + g) * D + c4 * 32;
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
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMma) {
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, L::TMEM_COLS);
    }
}

// Host side: the tensor maps and parameters of a prefill launch (p.nqblk is set
// by the launcher, which knows the instance's query block).
inline cudaError_t prefill_tc_prepare(void* out, const void* q, const void* k_pool, const void* v_pool,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                                      int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                                      int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                      uint32_t* dev_status, CUtensorMap& tq, CUtensorMap& tk, CUtensorMap& tv,
                                      PfParams& p) {
    const int D = pool.head_dim;
    const int G = num_q_heads / pool.num_kv_heads;
    {
        const uint64_t dims[3] = {(uint64_t)D, (uint64_t)num_q_heads, (uint64_t)total_q};
        const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)num_q_heads * D * 2};
        const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)(PM / G)};
        cudaError_t e = encode_tiled_bf16(&tq, const_cast<void*>(q), 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t slots = (uint64_t)pool.num_blocks * pool.block_size;
        const uint64_t row = (uint64_t)pool.num_kv_heads * D * 2;   // bytes of one pool slot
        cudaError_t e;
        if (D == 128) {
            // (d 0-63, slot % 8, d half, slot / 8, head): a 16-slot box of one head holds both
            // halves of D as [slot/8 % 2][half][slot % 8][64]
            const uint64_t dims[5] = {64, 8, 2, slots / 8, (uint64_t)pool.num_kv_heads};
            const uint64_t strides[4] = {row, 128, 8 * row, (uint64_t)D * 2};
            const uint32_t box[5] = {64, 8, 2, 2, 1};
            e = encode_tiled_bf16(&tk, const_cast<void*>(k_pool), 5, dims, strides, box);
            if (e != cudaSuccess) return e;
            e = encode_tiled_bf16(&tv, const_cast<void*>(v_pool), 5, dims, strides, box);
        } else {
            const uint64_t dims[3] = {(uint64_t)D, slots, (uint64_t)pool.num_kv_heads};
            const uint64_t strides[2] = {row, (uint64_t)D * 2};
            const uint32_t box[3] = {64, 16, 1};
            e = encode_tiled_bf16(&tk, const_cast<void*>(k_pool), 3, dims, strides, box);
            if (e != cudaSuccess) return e;
            e = encode_tiled_bf16(&tv, const_cast<void*>(v_pool), 3, dims, strides, box);
        }
        if (e != cudaSuccess) return e;
    }
    p.out = static_cast<__nv_bfloat16*>(out);
    p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
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
    p.G = G;
    p.N = pool.num_blocks;
    p.P = pool.block_size;
    p.nqblk = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    return cudaSuccess;
}

}  // namespace
}  // namespace wf
