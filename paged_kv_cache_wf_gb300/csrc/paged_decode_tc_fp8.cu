// paged_decode_tc_fp8.cu -- paged decode on the 5th-generation tensor cores for
// fp8 e4m3 pools with H_kv = 8 KV heads, D = 64 or 128, a block size that is a
// multiple of 16 and GQA groups of 2 or 4; q and outputs are bf16.
//
// What is computed (ember, "Deliberately out of scope": paged KV quantization; the
// attention itself as in paged_decode_tc.cu): K_p = k_scale_h * value(code),
// V_p = v_scale_h * value(code) with the scales of KV head h (per head, or one per
// tensor), out = softmax_p(scale * q.K_p) V_p.
//
// The stored codes feed the tensor cores as they are (kind::f8f6f4, e4m3 x e4m3 ->
// fp32): nothing widens K or V.  The other operand of each product is split into
// two e4m3 parts whose sum carries its precision:
//   - q row n is scaled by a power of two 2^e_n (its largest magnitude lands in
//     [128, 256)) and written as hi + lo with hi = e4m3(q 2^e_n) and
//     lo = e4m3(q 2^e_n - hi).  A bf16 value has 8 significant bits, hi keeps 4 and
//     the remainder fits lo's 4, so hi + lo is q 2^e_n exactly unless lo falls
//     below the e4m3 normal range (error <= 2^-10 on a scale where the row's
//     largest entry is >= 128).  S = K (hi + lo)^T takes two MMAs per k-step and
//     2^-e_n, the row's K scale and the softmax scale fold into the exponent.
//   - the softmax weights p in [0, 1] are written as hi + lo of 256 p the same way
//     (about 8 significant bits, what the bf16 kernel keeps), and l sums exactly
//     the hi + lo that the P.V product uses; the factor 256 cancels in o / l, and
//     the V scale of each query head's KV head multiplies its output column.
//
// Work split, tiles and the (m, l, o) partials are those of the bf16 kernel: a work
// item is (sequence b, split of 256 positions), a tile is one 16-position run of a
// block for all 8 KV heads -- 128 rows r = (head, position):
//     S^T[128 rows x H_q] = K[128 rows x 128 d] . Q^T           (K-major A and B)
//     O^T[128 d x H_q]    = V^T[128 d x 128 rows] . P^T          (V^T: MN-major A)
// At D = 128 a tile is two 16 KB boxes (K and V, one 128-byte swizzled row per
// (head, position)), so a stage is half the bf16 kernel's and the ring holds five.
// At D = 64 a row is 64 bytes (64-byte swizzle) and a stage holds two such 16-
// position sub-tiles, so each step of the per-tile chain still moves 32 KB; their
// S products go to two TMEM column blocks, their P.V products add into one
// accumulator (the upper 64 rows of each V^T operand read the next 8 KB of shared
// memory: rows of O^T that nobody reads), and the softmax treats a row of both
// sub-tiles as one stream.
//
// A small grid runs first (fp8_q_prepare_kernel): it splits every q row into its
// e4m3 parts once per call, into the workspace, and zeroes the work-item queue.  The
// decode grid is its programmatic dependent: set-up overlaps, the producer waits.
//
// CTA (persistent, one per SM), 11 warps:
//   warp 0   producer: claims items from the launch's queue; per item, a TMA copy
//            of the sequence's q parts into one of two q buffers; per tile, TMA
//            copies of K and V (alternating lane pairs) and the tile's meta.
//   warp 1   S issuer: S(t) into one of two TMEM S buffers.
//   warps 2-5  softmax of tile t (thread i = row i): P^T parts, and a record of the
//            tile's rescale factors (and, at an item's end, l and m) in a ring.
//   warps 7-10 fold P.V(t) into fp32 registers (thread i = head dim i) with the
//            tile's record, beside the next softmax; store outputs or partials.
//   warp 6   P.V issuer: P.V(t) into one of two TMEM O buffers; its commits free
//            the stage and signal the softmax warps.
#include <cuda.h>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kRows = 128;       // MMA M: 8 heads x 16 positions (and D = 128 for P.V)
constexpr int kHeads = 8;        // KV heads per tile
constexpr int kPosT = 16;        // positions per tile
// positions per item (split): 256 one-byte positions make an item the size of the
// bf16 kernel's (512 KB over 8 KV heads); half as many partials to combine as with
// 128 (measured 184 -> 176 us a call at the Llama-3-8B batch)
constexpr int kSpanTc = 256;
constexpr int kNq = 32;          // max H_q handled (MMA N)
constexpr int kStages = 5;
constexpr int kEndTile = -1;
constexpr int kStageBytes = 32 * 1024;          // K sub-tiles, then V sub-tiles
constexpr int kPart = kNq * 128;                // one e4m3 part of q or P^T: 32 rows x (up to) 128 B
constexpr int kPartsBytes = 2 * kPart;          // hi then lo

// Per head dim D (64 or 128): SUB sub-tiles of 16 positions per stage, whose K (or
// V) codes are kSub bytes each; K, V and q rows of D bytes use the 128-byte swizzle
// at D = 128 and the 64-byte swizzle at D = 64 (8-row atoms of 8 * D bytes).
template <int D>
struct Fp8Cfg {
    static constexpr int SUB = D == 128 ? 1 : 2;
    static constexpr int kSub = kRows * D;
    static constexpr int kSbo = 8 * D;
    static constexpr int kPBytes = SUB * kPartsBytes;   // P^T parts of one tile
    static constexpr int kSCols = SUB * 32;             // TMEM columns of one S buffer
    static constexpr int kOBase = 2 * kSCols;           // the two O buffers (32 columns each) follow
    static constexpr int TMEM = kOBase + 64 <= 128 ? 128 : 256;
    static_assert(2 * SUB * kSub == kStageBytes, "a stage holds 32 KB of codes");
};

template <int D>
__device__ __forceinline__ uint64_t sdesc_kv(uint32_t addr, uint32_t lbo) {
    return D == 128 ? tc::sdesc_sw128(addr, lbo, 1024) : tc::sdesc_sw64(addr, lbo, 512);
}
constexpr int kRing = 8;         // per-tile records from the softmax warps to the accumulate warps
constexpr int kThreadsFp8 = 352;

struct Fp8Params {
    void* out;
    const float* qinv;   // [B * H_q]: 2^-e of each prepared q row
    float* ws_o;
    float2* ws_ml;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    uint32_t* dev_status;
    uint32_t* queue;     // next unclaimed work item; zero at launch
    int32_t M, B, max_seq_len, H_q, H_kv, G, N, P, max_splits;
    float scale_log2;   // softmax scale * log2(e)
    float k_head[kHeads];   // K scale of each KV head
    float v_head[kHeads];   // V scale of each KV head
};

struct Fp8Meta {
    int32_t b, split, nsplit, okmask, nvalid, first, last, item;   // okmask: sub-tiles loaded
    float qinv[kNq];    // 2^-e_n of q row n
};

struct AccRec {     // what the accumulate warps need of tile t, in ring slot t % kRing
    int32_t b, split, nsplit, last, end, pad[3];
    float alpha[kNq];   // rescale of the running output, per query head
    float l[kNq];       // at an item's last tile: the softmax denominators (x 256)
    float m[kNq];       //   and the running maxima (log2 units)
};

template <int D>
struct Fp8Smem {  // byte offsets from the 1024-aligned base
    static constexpr int stage = 0;
    static constexpr int qbuf = kStages * kStageBytes;       // [2 items][hi, lo]
    static constexpr int pbuf = qbuf + 2 * kPartsBytes;      // [2 tiles][sub-tile][hi, lo]
    static constexpr int bars = pbuf + 2 * Fp8Cfg<D>::kPBytes;
    // full[S] empty[S] s_full[2] s_free[2] p_full[2] o_full[2] o_free[2] q_free[2]
    // a_full[R] a_free[R]
    static constexpr int nbars = 2 * kStages + 12 + 2 * kRing;
    static constexpr int meta = (bars + nbars * 8 + 15) / 16 * 16;
    static constexpr int ring = meta + kStages * (int)sizeof(Fp8Meta);
    static constexpr int tmem_slot = ring + kRing * (int)sizeof(AccRec);
    static constexpr int total = tmem_slot + 16;
};
static_assert(Fp8Smem<64>::total + 1024 <= 232448 && Fp8Smem<128>::total + 1024 <= 232448,
              "fp8 tensor-core decode exceeds shared memory");
static_assert(Fp8Smem<64>::ring % 16 == 0 && Fp8Smem<128>::ring % 16 == 0 && sizeof(AccRec) % 16 == 0,
              "alpha is read with 16-byte loads");
static_assert(sizeof(Fp8Meta) % 16 == 0, "meta entries stay 16-byte aligned");

// Byte offset of 16-byte chunk j of row r in a tile of 128-byte rows with the
// 128-byte swizzle (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t sw_chunk(int r, int j) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

// Byte offset of 8-bit element (row, k), k < 128, in such a tile.
__device__ __forceinline__ uint32_t sw_byte(int row, int k) { return sw_chunk(row, k >> 4) + (k & 15); }

// (x0, x1) -> e4m3 hi codes and lo codes of the remainders, packed in the low 16 bits;
// used receives float(hi) + float(lo) of both.
__device__ __forceinline__ void split2_e4m3(float x0, float x1, uint32_t& hi, uint32_t& lo, float2& used) {
    hi = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)hi, __NV_E4M3);
    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    lo = __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
    const __half2_raw lr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)lo, __NV_E4M3);
    const float2 lf = __half22float2(*reinterpret_cast<const __half2*>(&lr));
    used = make_float2(hf.x + lf.x, hf.y + lf.y);
}

template <int G, int D>
__global__ void __launch_bounds__(kThreadsFp8, 1)
    paged_decode_tc_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                               const __grid_constant__ CUtensorMap tm_q, const Fp8Params p) {
    constexpr int HQ = kHeads * G;                 // query heads (MMA N)
    using C = Fp8Cfg<D>;
    using Fp8Smem = wf::Fp8Smem<D>;
    constexpr int SUB = C::SUB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Fp8Smem::bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* s_full = bars + 2 * kStages;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* o_full = p_full + 2;
    uint64_t* o_free = o_full + 2;
    uint64_t* q_free = o_free + 2;
    uint64_t* a_full = q_free + 2;   // record of tile t written (4 softmax warps)
    uint64_t* a_free = a_full + kRing;  // record of tile t read (4 accumulate warps)
    Fp8Meta* meta = reinterpret_cast<Fp8Meta*>(smem + Fp8Smem::meta);
    AccRec* ring = reinterpret_cast<AccRec*>(smem + Fp8Smem::ring);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Fp8Smem::tmem_slot);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == 1) {
        tc::alloc(tmem_slot, C::TMEM);
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
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&a_free[i], 4);
        }
        fence_mbar_init();
    }
    // P^T is block-diagonal: zero both buffers once; only diagonal entries are rewritten.
    for (int i = threadIdx.x; i < 2 * C::kPBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem + Fp8Smem::pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S buffers [0, kSCols) [kSCols, 2 kSCols) (32 per sub-tile); O
    // buffers [kOBase, kOBase + 32) [kOBase + 32, kOBase + 64)

    if (warp == 0) {
        // ============================ producer ==================================
        // the q parts, the row scales and the zeroed queue come from the preparing grid
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const uint64_t pol = l2_policy_evict_first();
        int t = 0, k = 0;          // tiles and items issued
        int b = 0, len = 0, nsp = 0;
        int64_t cum = 0;
        bool ok = true;
        const int64_t cap = min((int64_t)p.max_seq_len, (int64_t)p.M * p.P);   // longest valid sequence
        ItemWalk walk;
        item_walk_load(walk, p.seq_lens, p.B, kSpanTc, cap, p.dev_status, lane);
        constexpr int PT = SUB * kPosT;            // positions per tile
        // Items come from a queue shared by all CTAs (one atomic increment per item,
        // claimed one item ahead so the round trip overlaps the current item's
        // copies).  Each CTA's claims increase, so its walk over the sequences only
        // moves forward.
        uint32_t claim = lane == 0 ? atomicAdd(p.queue, 1u) : 0u;
        for (int64_t item = __shfl_sync(0xffffffffu, claim, 0); ok; item = __shfl_sync(0xffffffffu, claim, 0)) {
            if (!item_walk_find(walk, item, p.seq_lens, p.B, kSpanTc, cap, p.dev_status, lane, b, len, nsp, cum))
                break;
            claim = lane == 0 ? atomicAdd(p.queue, 1u) : 0u;
            const int split = (int)(item - cum);
            const int s0 = split * kSpanTc;
            const int s1 = min(len, s0 + kSpanTc);
            const int ntiles = (s1 - s0 + PT - 1) / PT;
            const int qb = k & 1;
            if (k >= 2 && !mbar_wait(&q_free[qb], ((k >> 1) - 1) & 1)) {
                if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                ok = false;
                break;
            }
            // the sequence's q parts arrive by TMA with the item's first tile; its row
            // scales travel in the tiles' meta
            const float qinv = lane < p.H_q ? __ldg(p.qinv + (int64_t)b * p.H_q + lane) : 1.f;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int st = t % kStages;
                if (t >= kStages && !mbar_wait(&empty[st], ((t / kStages) - 1) & 1)) {
                    if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                    ok = false;
                    break;
                }
                if constexpr (SUB == 1) {
                // D = 128: one block per tile (this path is the one the kernel was tuned with)
                const int p0 = s0 + j * kPosT;
                const int nvalid = min(kPosT, s1 - p0);
                const int blk = __ldg(p.block_tables + (int64_t)b * p.M + p0 / p.P);
                const bool okb = (unsigned)blk < (unsigned)p.N;
                meta[st].qinv[lane] = qinv;
                __syncwarp();
                if (lane == 0) {
                    if (!okb) report(p.dev_status, WF_DEV_BAD_BLOCK);
                    Fp8Meta& m = meta[st];
                    m.b = b; m.split = split; m.nsplit = nsp; m.okmask = okb ? 1 : 0; m.nvalid = nvalid;
                    m.first = (j == 0); m.last = (j == ntiles - 1); m.item = k;
                    mbar_arrive_expect_tx(&full[st], (okb ? (uint32_t)kStageBytes : 0u) +
                                                         (j == 0 ? 2u * (uint32_t)HQ * 128u : 0u));
                }
                __syncwarp();
                if (j == 0 && (lane == 8 || lane == 9)) {   // hi rows, then lo rows
                    tma_load_2d(smem + Fp8Smem::qbuf + qb * kPartsBytes + (lane - 8) * kPart, &tm_q, 0,
                                (lane - 8) * p.B * p.H_q + b * p.H_q, &full[st]);
                }
                const int slot = blk * p.P + p0 % p.P;
                const int base_lane = (t & 3) * 2;   // a thread's copies complete in order: rotate lanes
                if (okb && (lane == base_lane || lane == base_lane + 1)) {
                    const bool isv = lane == base_lane + 1;
                    tma_load_3d(smem + Fp8Smem::stage + st * kStageBytes + (isv ? C::kSub : 0), isv ? &tm_v : &tm_k,
                                0, slot, 0, &full[st], pol);
                }
                } else {
                const int p0 = s0 + j * PT;
                const int nvalid = min(PT, s1 - p0);
                // sub-tile s covers positions p0 + 16 s .. + 15 (one block: P % 16 == 0)
                const int sl = lane & (SUB - 1);
                const bool need = sl * kPosT < nvalid;
                const int blk = need ? __ldg(p.block_tables + (int64_t)b * p.M + (p0 + sl * kPosT) / p.P) : -1;
                const bool okb = need && (unsigned)blk < (unsigned)p.N;
                const uint32_t needl = nvalid > kPosT ? (1u << SUB) - 1u : 1u;
                // a tile with a block id out of range is skipped whole (none of its copies
                // is issued and no row of it is live)
                const uint32_t okl = (__ballot_sync(0xffffffffu, okb) & needl) == needl ? needl : 0u;
                meta[st].qinv[lane] = qinv;
                __syncwarp();
                if (lane == 0) {
                    if (okl != needl) report(p.dev_status, WF_DEV_BAD_BLOCK);
                    Fp8Meta& m = meta[st];
                    m.b = b; m.split = split; m.nsplit = nsp; m.okmask = (int)okl; m.nvalid = okl ? nvalid : 0;
                    m.first = (j == 0); m.last = (j == ntiles - 1); m.item = k;
                    mbar_arrive_expect_tx(&full[st], (uint32_t)__popc(okl) * 2u * (uint32_t)C::kSub +
                                                         (j == 0 ? 2u * (uint32_t)HQ * (uint32_t)D : 0u));
                }
                __syncwarp();
                if (j == 0 && (lane == 8 || lane == 9)) {   // hi rows, then lo rows
                    tma_load_2d(smem + Fp8Smem::qbuf + qb * kPartsBytes + (lane - 8) * kPart, &tm_q, 0,
                                (lane - 8) * p.B * p.H_q + b * p.H_q, &full[st]);
                }
                // copies: K of each sub-tile, then V; a thread's copies complete in order,
                // so they rotate over lanes (lane base + c, c = kind * SUB + sub-tile)
                const int base_lane = (t & 3) * 2 * SUB;
                const int c = lane - base_lane;
                const int cs = c & (SUB - 1);
                const int cblk = __shfl_sync(0xffffffffu, blk, cs);
                if (c >= 0 && c < 2 * SUB && ((okl >> cs) & 1u)) {
                    const bool isv = c >= SUB;
                    const int slot = cblk * p.P + (p0 + cs * kPosT) % p.P;
                    tma_load_3d(smem + Fp8Smem::stage + st * kStageBytes + (isv ? SUB : 0) * C::kSub + cs * C::kSub,
                                isv ? &tm_v : &tm_k, 0, slot, 0, &full[st], pol);
                }
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
        // ============================ S issuer ==================================
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_e4m3_f32(kRows, HQ < 16 ? 16 : HQ, 0, 0);
            // (each sub-tile's S goes to its own 32 columns of the buffer)
            for (int tq = 0;; ++tq) {
                const int st = tq % kStages, sb = tq & 1;
                if (!mbar_wait(&full[st], (tq / kStages) & 1)) {
                    report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
                const int nvalid = meta[st].nvalid, item = meta[st].item, last = meta[st].last;
                if (nvalid == kEndTile) break;
                if (tq >= 2 && !mbar_wait(&s_free[sb], ((tq >> 1) - 1) & 1)) {
                    report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t qbase = smem_u32(smem + Fp8Smem::qbuf + (item & 1) * kPartsBytes);
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    const uint32_t kbase = smem_u32(smem + Fp8Smem::stage + st * kStageBytes + s * C::kSub);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const uint64_t ad = sdesc_kv<D>(kbase + kk * 32, 16);
                            const uint64_t bd = sdesc_kv<D>(qbase + part * kPart + kk * 32, 16);
                            tc::mma_f8f6f4(tmem + sb * C::kSCols + s * 32, ad, bd, idS, (part | kk) ? 1u : 0u);
                        }
                }
                tc::commit(&s_full[sb]);
                if (last) tc::commit(&q_free[item & 1]);
            }
        }
    } else if (warp == 6) {
        // ============================ P.V issuer ================================
        // A second issuing thread: one thread's MMAs issue one after another, and S
        // and P.V of a tile would otherwise queue behind each other.
        if (lane == 0) {
            constexpr uint32_t idO = tc::idesc_e4m3_f32(kRows, HQ < 16 ? 16 : HQ, 1, 0);
            for (int tp = 0;; ++tp) {
                const int su = tp % kStages, ub = tp & 1;
                // the stage is released by this thread's own commit below, so this wait
                // cannot fall two phases behind
                if (!mbar_wait(&full[su], (tp / kStages) & 1)) {
                    report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
                if (meta[su].nvalid == kEndTile) break;
                if (!mbar_wait(&p_full[ub], (tp >> 1) & 1) ||
                    (tp >= 2 && !mbar_wait(&o_free[ub], ((tp >> 1) - 1) & 1))) {
                    report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    const uint32_t vbase = smem_u32(smem + Fp8Smem::stage + su * kStageBytes + (SUB + s) * C::kSub);
                    const uint32_t pb = smem_u32(smem + Fp8Smem::pbuf + ub * C::kPBytes + s * kPartsBytes);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int kk = 0; kk < kRows / 32; ++kk) {
                            // V^T: 32 rows (k) per MMA = four 8-row swizzle atoms; its M rows
                            // beyond D read the next kSub bytes (rows of O^T nobody reads)
                            const uint64_t ad = sdesc_kv<D>(vbase + kk * 32 * D, C::kSub);
                            const uint64_t bd = tc::sdesc_sw128(pb + part * kPart + kk * 32, 16, 1024);
                            tc::mma_f8f6f4(tmem + C::kOBase + ub * 32, ad, bd, idO, (s | part | kk) ? 1u : 0u);
                        }
                }
                tc::commit(&o_full[ub]);
                tc::commit(&empty[su]);
            }
        }
    } else if (warp < 6) {
        // ============================ softmax warps =============================
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int i = quad * 32 + lane;            // tile row
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const int hk = i >> 4;                     // KV head of row i
        const int pos = i & 15;                    // position of row i within the tile
        const int upper = lane >> 4;               // which of the warp's two heads
        float m_run[G], l_part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_part[g] = 0.f;
        }
        for (int t = 0;; ++t) {
            const int st = t % kStages, sb = t & 1, rs = t % kRing;
            if (!mbar_wait(&full[st], (t / kStages) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            const Fp8Meta& ms = meta[st];
            const int nvalid = ms.nvalid;
            // the record slot of tile t must have been read for tile t - kRing
            if (t >= kRing && !mbar_wait(&a_free[rs], ((t / kRing) - 1) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            AccRec& rec = ring[rs];
            if (nvalid == kEndTile) {
                if (warp == 2 && lane == 0) rec.end = 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[rs]);
                break;
            }
            const int mfirst = ms.first, mlast = ms.last;
            if (warp == 2 && lane == 0) {
                rec.b = ms.b; rec.split = ms.split; rec.nsplit = ms.nsplit; rec.last = mlast; rec.end = 0;
            }
            float colscale[G];                     // softmax scale * log2(e) * k_scale * 2^-e_n
#pragma unroll
            for (int g = 0; g < G; ++g) colscale[g] = p.scale_log2 * p.k_head[hk] * ms.qinv[hk * G + g];

            if (!mbar_wait(&s_full[sb], (t >> 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            tc::fence_after_sync();
            if constexpr (SUB == 1) {
            // D = 128: one sub-tile (this path is the one the kernel was tuned with)
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
            if (mfirst) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_part[g] = 0.f;
                }
            }
            const bool live = pos < nvalid;
            float al[G], x256[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float raw = upper ? sv[G + g] : sv[g];
                const float sc = live ? raw * colscale[g] : -INFINITY;
                float mx = sc;
#pragma unroll
                for (int mask = 8; mask >= 1; mask >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
                const float m_new = fmaxf(m_run[g], mx);
                al[g] = exp2f(m_run[g] - m_new);       // 0 on an item's first tile
                x256[g] = 256.f * exp2f(sc - m_new);
                m_run[g] = m_new;
            }
            // P^T buffer sb was last read by P.V(t-2); o_full of that product cannot have
            // moved on to P.V(t), which needs this tile's weights
            if (t >= 2 && !mbar_wait(&o_full[sb], ((t >> 1) - 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            unsigned char* pb = smem + Fp8Smem::pbuf + sb * C::kPBytes;
#pragma unroll
            for (int g = 0; g < G; g += 2) {
                uint32_t hi, lo;
                float2 used;
                split2_e4m3(x256[g], x256[g + 1], hi, lo, used);
                l_part[g] = l_part[g] * al[g] + used.x;
                l_part[g + 1] = l_part[g + 1] * al[g + 1] + used.y;
                pb[sw_byte(hk * G + g, i)] = (unsigned char)(hi & 0xffu);
                pb[sw_byte(hk * G + g + 1, i)] = (unsigned char)((hi >> 8) & 0xffu);
                pb[kPart + sw_byte(hk * G + g, i)] = (unsigned char)(lo & 0xffu);
                pb[kPart + sw_byte(hk * G + g + 1, i)] = (unsigned char)((lo >> 8) & 0xffu);
            }
            if (pos == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) rec.alpha[hk * G + g] = al[g];
            }
            if (mlast) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float x = l_part[g];
#pragma unroll
                    for (int mask = 8; mask >= 1; mask >>= 1) x += __shfl_xor_sync(0xffffffffu, x, mask);
                    if (pos == 0) {
                        rec.l[hk * G + g] = x;
                        rec.m[hk * G + g] = m_run[g];
                    }
                }
            }
            if (!live) {
                // rows past the sequence end: zero V so their 0-weights cannot meet NaN codes
                uint4* row = reinterpret_cast<uint4*>(smem + Fp8Smem::stage + st * kStageBytes + C::kSub +
                                                      (i >> 3) * 1024 + (i & 7) * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            } else {
            // this warp's two KV heads' query-head columns [2G*quad, 2G*quad + 2G) of each
            // sub-tile's S block, width-aligned
            float sv[SUB][2 * G];
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                if constexpr (G == 4) {
                    tc::ld_8cols(tmem + lane_addr + sb * C::kSCols + s * 32 + quad * 8, sv[s]);
                } else {
                    tc::ld_4cols(tmem + lane_addr + sb * C::kSCols + s * 32 + quad * 4, sv[s]);
                }
            }
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);
            if (mfirst) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_part[g] = 0.f;
                }
            }
            bool live[SUB];
#pragma unroll
            for (int s = 0; s < SUB; ++s) live[s] = s * kPosT + pos < nvalid;
            float al[G], x256[SUB][G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float sc[SUB];
                float mx = -INFINITY;
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    const float raw = upper ? sv[s][G + g] : sv[s][g];
                    sc[s] = live[s] ? raw * colscale[g] : -INFINITY;
                    mx = fmaxf(mx, sc[s]);
                }
#pragma unroll
                for (int mask = 8; mask >= 1; mask >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
                const float m_new = fmaxf(m_run[g], mx);
                // 0 on an item's first tile; a tile with no live row (a skipped block)
                // keeps the stream as it was
                al[g] = m_new == -INFINITY ? 1.f : exp2f(m_run[g] - m_new);
#pragma unroll
                for (int s = 0; s < SUB; ++s) x256[s][g] = live[s] ? 256.f * exp2f(sc[s] - m_new) : 0.f;
                m_run[g] = m_new;
            }
            // P^T buffer sb was last read by P.V(t-2); o_full of that product cannot have
            // moved on to P.V(t), which needs this tile's weights
            if (t >= 2 && !mbar_wait(&o_full[sb], ((t >> 1) - 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
#pragma unroll
            for (int g = 0; g < G; ++g) l_part[g] *= al[g];
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                unsigned char* pb = smem + Fp8Smem::pbuf + sb * C::kPBytes + s * kPartsBytes;
#pragma unroll
                for (int g = 0; g < G; g += 2) {
                    uint32_t hi, lo;
                    float2 used;
                    split2_e4m3(x256[s][g], x256[s][g + 1], hi, lo, used);
                    l_part[g] += used.x;
                    l_part[g + 1] += used.y;
                    pb[sw_byte(hk * G + g, i)] = (unsigned char)(hi & 0xffu);
                    pb[sw_byte(hk * G + g + 1, i)] = (unsigned char)((hi >> 8) & 0xffu);
                    pb[kPart + sw_byte(hk * G + g, i)] = (unsigned char)(lo & 0xffu);
                    pb[kPart + sw_byte(hk * G + g + 1, i)] = (unsigned char)((lo >> 8) & 0xffu);
                }
            }
            if (pos == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) rec.alpha[hk * G + g] = al[g];
            }
            if (mlast) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float x = l_part[g];
#pragma unroll
                    for (int mask = 8; mask >= 1; mask >>= 1) x += __shfl_xor_sync(0xffffffffu, x, mask);
                    if (pos == 0) {
                        rec.l[hk * G + g] = x;
                        rec.m[hk * G + g] = m_run[g];
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                if (!live[s]) {
                    // rows past the sequence end or of a skipped block: zero V so their
                    // 0-weights cannot meet NaN codes (row i is D contiguous bytes of its
                    // swizzle atom)
                    uint4* row = reinterpret_cast<uint4*>(smem + Fp8Smem::stage + st * kStageBytes + (SUB + s) * C::kSub +
                                                          (i >> 3) * (8 * D) + (i & 7) * D);
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&p_full[sb]);
                mbar_arrive(&a_full[rs]);
            }
        }
    } else {
        // ======================= accumulate warps (7-10) ==========================
        // Thread i owns row d = i of O^T for every query head and folds in each tile's
        // P.V with that tile's rescale factors; this runs beside the next softmax.
        const int quad = warp & 3;
        const int i = quad * 32 + lane;            // head dim
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        float acc[kNq];                            // O^T row d = i (code units x 256), all query heads
#pragma unroll
        for (int c = 0; c < kNq; ++c) acc[c] = 0.f;
        for (int t = 0;; ++t) {
            const int ub = t & 1, rs = t % kRing;
            if (!mbar_wait(&a_full[rs], (t / kRing) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            const AccRec& rec = ring[rs];
            if (rec.end) break;
            if (!mbar_wait(&o_full[ub], (t >> 1) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            tc::fence_after_sync();
            float o[32];
            tc::ld_32cols(tmem + lane_addr + C::kOBase + ub * 32, o);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[ub]);
#pragma unroll
            for (int c = 0; c < HQ; c += 4) {
                const float4 a4 = ld_shared_f4(rec.alpha + c);
                acc[c] = acc[c] * a4.x + o[c];
                acc[c + 1] = acc[c + 1] * a4.y + o[c + 1];
                acc[c + 2] = acc[c + 2] * a4.z + o[c + 2];
                acc[c + 3] = acc[c + 3] * a4.w + o[c + 3];
            }
            // At an item's end, everything the stores need comes out of the record
            // first: the record is released before the global stores are issued, so
            // the release (which orders this thread's earlier writes) does not wait
            // for them (measured 14 us a call at the Llama-3-8B batch otherwise).
            const bool last = rec.last;
            const bool direct = rec.nsplit == 1;
            const int ob = rec.b, osplit = rec.split;
            float mi = 0.f, li = 0.f;
            if (last) {
#pragma unroll
                for (int c = 0; c < HQ; ++c)   // acc restarts at the next item's first tile (alpha 0)
                    acc[c] = direct ? acc[c] * p.v_head[c / G] / rec.l[c] : acc[c] * p.v_head[c / G];
                if (i < HQ) {
                    mi = rec.m[i];
                    li = rec.l[i];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_free[rs]);
            if (last) {
                if (direct) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (int64_t)ob * p.H_q * D + i;
                    if (i < D) {
#pragma unroll
                        for (int c = 0; c < HQ; ++c) dst[c * D] = __float2bfloat16_rn(acc[c]);
                    }
                } else {
                    if (i < D) {
#pragma unroll
                        for (int c = 0; c < HQ; ++c)   // head-minor partial rows: one split's heads are contiguous
                            p.ws_o[partial_row(ob, c, osplit, p.H_q, p.max_splits, 1, p.H_q) * D + i] = acc[c];
                    }
                    if (i < HQ) p.ws_ml[partial_row(ob, i, osplit, p.H_q, p.max_splits, 1, p.H_q)] = make_float2(mi, li);
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    // the combine grid that follows may be scheduled now (it waits for this grid to
    // finish before it reads anything); signalled at the end so that its CTAs take
    // no room on the SMs while this grid streams
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, C::TMEM);
    }
}

// q [rows = B * H_q, D] bf16 -> the e4m3 parts of q 2^e_r: hi in rows [0, rows),
// lo in rows [rows, 2 rows) of `parts` (D bytes a row), and qinv[r] = 2^-e_r, with
// e_r chosen so that the row's largest magnitude lands in [128, 256).  One warp per
// row, lane l holding d = VL l .. VL l + VL - 1 (VL = D / 32).  Block 0 also zeroes
// the decode's work-item queue.  Run once per call, so every split of a sequence
// reads the same parts.
template <int D>
__global__ void __launch_bounds__(256) fp8_q_prepare_kernel(const __nv_bfloat16* __restrict__ q,
                                                            unsigned char* __restrict__ parts,
                                                            float* __restrict__ qinv, int64_t rows,
                                                            uint32_t* queue) {
    constexpr int VL = D / 32;
    // the decode grid may start its set-up now; it waits for this grid before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *queue = 0u;
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= rows) return;
    float x[4];
    if constexpr (VL == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(q + r * D + 4 * lane);
        const float2 a = bf16x2_to_float2(v.x), c = bf16x2_to_float2(v.y);
        x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
    } else {
        const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(q + r * D + 2 * lane));
        x[0] = a.x; x[1] = a.y; x[2] = 0.f; x[3] = 0.f;
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, mask));
    int e = 0;
    if (amax > 0.f && amax <= 3.0e38f) {
        // floor(log2 amax) from the exponent bits (subnormals count as 2^-126)
        const int E = max(-126, (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127);
        e = min(126, max(-126, 7 - E));
    }
    const float qs = __uint_as_float((uint32_t)(e + 127) << 23);
    uint32_t h0, l0, h1, l1;
    float2 u0, u1;
    split2_e4m3(x[0] * qs, x[1] * qs, h0, l0, u0);
    if constexpr (VL == 4) {
        split2_e4m3(x[2] * qs, x[3] * qs, h1, l1, u1);
        *reinterpret_cast<uint32_t*>(parts + r * D + 4 * lane) = (h0 & 0xffffu) | (h1 << 16);
        *reinterpret_cast<uint32_t*>(parts + (rows + r) * D + 4 * lane) = (l0 & 0xffffu) | (l1 << 16);
    } else {
        *reinterpret_cast<uint16_t*>(parts + r * D + 2 * lane) = (uint16_t)(h0 & 0xffffu);
        *reinterpret_cast<uint16_t*>(parts + (rows + r) * D + 2 * lane) = (uint16_t)(l0 & 0xffffu);
    }
    if (lane == 0) qinv[r] = __uint_as_float((uint32_t)(127 - e) << 23);
}

template <int D>
cudaError_t launch_fp8(int G, const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                       const Fp8Params& p, int grid, cudaStream_t stream) {
    const int smem = Fp8Smem<D>::total + 1024;
    const void* kern = G == 4 ? (const void*)paged_decode_tc_fp8_kernel<4, D> : (const void*)paged_decode_tc_fp8_kernel<2, D>;
    cudaError_t err = allow_dynamic_smem(kern, smem);
    if (err != cudaSuccess) return err;
    // launched as a programmatic dependent of the preparing grid: its set-up overlaps
    // that grid, and its producer waits (griddepcontrol.wait) before reading anything
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsFp8);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (G == 4) return cudaLaunchKernelEx(&cfg, paged_decode_tc_fp8_kernel<4, D>, tm_k, tm_v, tm_q, p);
    return cudaLaunchKernelEx(&cfg, paged_decode_tc_fp8_kernel<2, D>, tm_k, tm_v, tm_q, p);
}

}  // namespace

size_t decode_fp8_prep_bytes(int32_t B, int32_t num_q_heads) {
    const int64_t rows = (int64_t)B * num_q_heads;
    return (size_t)(2 * rows * 128 + rows * 4 + 256);
}

int decode_tc_fp8_span() { return kSpanTc; }

bool decode_tc_fp8_supported(const wf_pool_desc& pool, int32_t num_q_heads) {
    const int G = pool.num_kv_heads > 0 ? num_q_heads / pool.num_kv_heads : 0;
    return pool.dtype == WF_DTYPE_FP8_E4M3 && (pool.head_dim == 64 || pool.head_dim == 128) &&
           pool.block_size % kPosT == 0 &&
           pool.num_kv_heads == kHeads && num_q_heads % pool.num_kv_heads == 0 && (G == 2 || G == 4);
}

cudaError_t launch_paged_decode_tc_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                       int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                       float2* ws_ml, int32_t max_splits, uint32_t* queue, void* prep,
                                       uint32_t* dev_status, cudaStream_t stream) {
    const int G = num_q_heads / pool.num_kv_heads;
    const int D = pool.head_dim;
    const int64_t rows = (int64_t)B * num_q_heads;
    // prep: the q parts (2 rows x D bytes per q row), then the row scales
    unsigned char* parts = static_cast<unsigned char*>(prep);
    float* qinv = reinterpret_cast<float*>(parts + 2 * rows * 128);
    const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tm_k, tm_v, tm_q;
    const uint64_t slots = (uint64_t)pool.num_blocks * pool.block_size;
    {
        // (d, slot, head) over the code pools: one box = 16 slots x 8 heads x D codes
        const uint64_t dims[3] = {(uint64_t)D, slots, (uint64_t)kHeads};
        const uint64_t strides[2] = {(uint64_t)kHeads * D, (uint64_t)D};
        const uint32_t box[3] = {(uint32_t)D, (uint32_t)kPosT, (uint32_t)kHeads};
        cudaError_t e = encode_tiled(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(k_pool), 3, dims,
                                     strides, box, swz);
        if (e != cudaSuccess) return e;
        e = encode_tiled(&tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(v_pool), 3, dims, strides, box,
                         swz);
        if (e != cudaSuccess) return e;
    }
    {
        // (d, part row): one box = one sequence's H_q rows of one part
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)(2 * rows)};
        const uint64_t strides[1] = {(uint64_t)D};
        const uint32_t box[2] = {(uint32_t)D, (uint32_t)num_q_heads};
        cudaError_t e = encode_tiled(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, parts, 2, dims, strides, box, swz);
        if (e != cudaSuccess) return e;
    }
    if (D == 128)
        fp8_q_prepare_kernel<128><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(q), parts, qinv, rows, queue);
    else
        fp8_q_prepare_kernel<64><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(q), parts, qinv, rows, queue);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    Fp8Params p;
    p.out = out;
    p.qinv = qinv;
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
    const HeadScales sc = head_scales(pool);
    for (int h = 0; h < kHeads; ++h) {
        p.k_head[h] = sc.k[h];
        p.v_head[h] = sc.v[h];
    }
    const int64_t items = (int64_t)B * max_splits;
    const int grid = (int)(items < num_sms() ? items : num_sms());
    return D == 128 ? launch_fp8<128>(G, tm_k, tm_v, tm_q, p, grid, stream)
                    : launch_fp8<64>(G, tm_k, tm_v, tm_q, p, grid, stream);
}

}  // namespace wf
