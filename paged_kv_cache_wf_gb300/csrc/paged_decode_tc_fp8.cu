// paged_decode_tc_fp8.cu -- paged decode on the 5th-generation tensor cores for
// fp8 e4m3 pools with H_kv = 8 KV heads, D = 128, a block size that is a multiple of
// 16 and GQA groups of 2 or 4; q and outputs are bf16.
//
// What is computed (ember, "Deliberately out of scope": paged KV quantization; the
// attention itself as in paged_decode_tc.cu): K_p = k_scale * value(code),
// V_p = v_scale * value(code).  Every e4m3 value is exactly an fp16 value, so the
// two products run as fp16 MMAs (kind::f16) on the codes' exact values; k_scale is
// folded into the softmax exponent and v_scale into the final normalisation.
//
// Work split, tiles and the (m, l, o) partials are those of the bf16 kernel: a work
// item is (sequence b, split of 128 positions), a tile is one 16-position run of a
// block for all 8 KV heads, 128 rows r = (head, position).  Per tile:
//   - TMA brings the fp8 K and V tiles (16 KB each, one box per operand: (d, slot,
//     head) with d the contiguous 128 bytes) into a 3-stage ring;
//   - converter warps (thread r <-> row r <-> TMEM lane r) widen K row r to fp16
//     and store it into TMEM, where it is the A operand of S^T = K . Q^T, and widen
//     V row r into a 128-byte-swizzled fp16 tile in shared memory, the MN-major A
//     operand of O^T = V^T . P^T (rows past the sequence's end are written as 0).
//     On an item's first tile they also convert its q (bf16 -> fp16) in place.  The
//     fp8 stage is free as soon as it is converted;
//   - the MMA warp and the softmax / accumulate warps work as in the bf16 kernel,
//     with fp16 q, K, V and P.
//
// CTA (persistent, one per SM), 10 warps:
//   warp 0     producer (TMA): fp8 tiles into the ring (lanes of alternate parity take
//              alternate tiles, since a thread's copies complete one after another),
//              q of an item into one of two q buffers.
//   warp 1     MMA issuer: S(t) into one of two TMEM S buffers, O(t-1) into one of two
//              TMEM O buffers; commits free converted buffers and S / O buffers.
//   warps 2-5  accumulate / softmax, as in the bf16 kernel.
//   warps 6-9  converters.
#include <cuda.h>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kRows = 128;       // MMA M: 8 heads x 16 positions (and D = 128 for P.V)
constexpr int kHeads = 8;        // KV heads per tile
constexpr int kPosT = 16;        // positions per tile
constexpr int kSpanTc = 128;     // positions per item (split)
constexpr int kD = 128;
constexpr int kNq = 32;          // max H_q handled (MMA N)
constexpr int kStages = 3;       // fp8 landing stages
constexpr int kEndTile = -1;
constexpr int kTile8 = kRows * kD;              // one fp8 K or V tile: 16 KB
constexpr int kStageBytes = 2 * kTile8;         // K then V
constexpr int kHalf = kRows * 128;              // one 64-wide fp16 half of a V tile: 16 KB
constexpr int kVBytes = 2 * kHalf;
constexpr int kQHalf = kNq * 128;               // one half of q: 32 rows x 128 B
constexpr int kQBytes = 2 * kQHalf;
constexpr int kPHalf = kNq * 128;               // one 64-row half of P^T (32 q rows x 128 B)
constexpr int kPBytes = 2 * kPHalf;
constexpr int kThreadsFp8 = 320;

struct Fp8Params {
    void* out;
    float* ws_o;
    float2* ws_ml;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    uint32_t* dev_status;
    uint32_t* queue;     // next unclaimed work item; zero at launch
    int32_t M, B, max_seq_len, H_q, H_kv, G, N, P, max_splits;
    float scale_log2;   // softmax scale * log2(e) * k_scale
    float v_scale;
};

struct Fp8Meta {
    int32_t b, split, nsplit, p0, nvalid, first, last, item;
};

struct Fp8Smem {  // byte offsets from the 1024-aligned base
    static constexpr int stage = 0;
    static constexpr int vbuf = kStages * kStageBytes;
    static constexpr int qbuf = vbuf + 2 * kVBytes;
    static constexpr int pbuf = qbuf + 2 * kQBytes;
    static constexpr int bars = pbuf + 2 * kPBytes;
    // full[3] empty[3] conv_full[2] conv_free[2] s_full[2] s_free[2] p_full[2] o_full[2]
    // o_free[2] q_free[2] grp
    static constexpr int nbars = 2 * kStages + 17;
    static constexpr int meta = (bars + nbars * 8 + 15) / 16 * 16;
    static constexpr int cmeta = meta + kStages * (int)sizeof(Fp8Meta);   // [2] per converted buffer
    static constexpr int alpha = cmeta + 2 * (int)sizeof(Fp8Meta);      // [3][kNq]: tile t in t % 3
    static constexpr int lbuf = alpha + 3 * kNq * 4;                    // [3][kNq]: item k in k % 3
    static constexpr int mbuf = lbuf + 3 * kNq * 4;                     // [3][kNq]
    static constexpr int tmem_slot = mbuf + 3 * kNq * 4;
    static constexpr int total = tmem_slot + 16;
};
static_assert(Fp8Smem::total + 1024 <= 232448, "fp8 tensor-core decode exceeds shared memory");
static_assert(Fp8Smem::alpha % 16 == 0 && Fp8Smem::lbuf % 16 == 0 && Fp8Smem::mbuf % 16 == 0,
              "alpha, l and m buffers are read with 16-byte loads");

// Byte offset of 16-byte chunk j of row r in a tile of 128-byte rows with the
// 128-byte swizzle (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t sw_chunk(int r, int j) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

// Byte offset of bf16/fp16 element (row, k) of a K-major 128-byte-swizzled tile
// whose 64-element column blocks are `block_bytes` apart.
__device__ __forceinline__ uint32_t sw_elem(int row, int k, int block_bytes) {
    const int chunk = (k & 63) >> 3;
    return (uint32_t)((k >> 6) * block_bytes + (row >> 3) * 1024 + (row & 7) * 128 +
                      ((chunk ^ (row & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ bool fp8_len_ok(int len, const Fp8Params& p) {
    return len >= 1 && len <= p.max_seq_len && (int64_t)len <= (int64_t)p.M * p.P;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
    const float2 f = bf16x2_to_float2(u);
    const __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <int G>
__global__ void __launch_bounds__(kThreadsFp8, 1)
    paged_decode_tc_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                               const __grid_constant__ CUtensorMap tm_q, const Fp8Params p) {
    constexpr int HQ = kHeads * G;                 // query heads (MMA N)
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Fp8Smem::bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* conv_full = bars + 2 * kStages;
    uint64_t* conv_free = conv_full + 2;
    uint64_t* s_full = conv_free + 2;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* o_full = p_full + 2;
    uint64_t* o_free = o_full + 2;
    uint64_t* q_free = o_free + 2;
    uint64_t* grp = q_free + 2;      // the four softmax warps meet here each tile
    Fp8Meta* meta = reinterpret_cast<Fp8Meta*>(smem + Fp8Smem::meta);
    Fp8Meta* cmeta = reinterpret_cast<Fp8Meta*>(smem + Fp8Smem::cmeta);
    float* alpha_buf = reinterpret_cast<float*>(smem + Fp8Smem::alpha);
    float* l_buf = reinterpret_cast<float*>(smem + Fp8Smem::lbuf);
    float* m_buf = reinterpret_cast<float*>(smem + Fp8Smem::mbuf);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Fp8Smem::tmem_slot);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the combine grid that follows may be scheduled now; it waits for this grid to
    // finish before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 1) {
        tc::alloc(tmem_slot, 256);
        tc::relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&conv_full[i], 4);
            mbar_init(&conv_free[i], 1);
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
        reinterpret_cast<uint4*>(smem + Fp8Smem::pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S buffers [0,32) [32,64); O buffers [64,96) [96,128);
    // fp16 K tiles [128,192) [192,256) (a column holds the fp16 pair d = 2c, 2c + 1)

    if (warp == 0) {
        // ============================ producer ==================================
        const uint64_t pol = l2_policy_evict_first();
        int t = 0, k = 0;          // tiles and items issued
        int b = 0, len = 0, nsp = -1;
        int64_t cum = 0;
        bool ok = true;
        // Items come from a queue shared by all CTAs (one atomic increment per item,
        // claimed one item ahead so the round trip overlaps the current item's
        // copies).  Each CTA's claims increase, so the walk over sequences below
        // only moves forward.
        uint32_t claim = lane == 0 ? atomicAdd(p.queue, 1u) : 0u;
        for (int64_t item = __shfl_sync(0xffffffffu, claim, 0); ok; item = __shfl_sync(0xffffffffu, claim, 0)) {
            while (b < p.B) {
                if (nsp < 0) {
                    len = __ldg(p.seq_lens + b);
                    if (fp8_len_ok(len, p)) {
                        nsp = (len + kSpanTc - 1) / kSpanTc;
                    } else {
                        nsp = 0;
                        if (lane == 0) report(p.dev_status, WF_DEV_BAD_SEQLEN);
                    }
                }
                if (item < cum + nsp) break;
                cum += nsp;
                ++b;
                nsp = -1;
            }
            if (b >= p.B) break;
            claim = lane == 0 ? atomicAdd(p.queue, 1u) : 0u;
            const int split = (int)(item - cum);
            const int s0 = split * kSpanTc;
            const int s1 = min(len, s0 + kSpanTc);
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
                const uint32_t bytes = (okb ? (uint32_t)kStageBytes : 0u) + (j == 0 ? 2u * HQ * 128u : 0u);
                if (lane == 0) {
                    if (!okb) report(p.dev_status, WF_DEV_BAD_BLOCK);
                    Fp8Meta m;
                    m.b = b; m.split = split; m.nsplit = nsp; m.p0 = p0; m.nvalid = nvalid;
                    m.first = (j == 0); m.last = (j == ntiles - 1); m.item = k;
                    meta[st] = m;
                    mbar_arrive_expect_tx(&full[st], bytes);
                }
                __syncwarp();
                const int slot = blk * p.P + p0 % p.P;
                const int base_lane = (t & 1) * 2;   // lanes 0-1 on even tiles, 2-3 on odd ones
                if (okb && (lane == base_lane || lane == base_lane + 1)) {
                    const bool isv = lane == base_lane + 1;
                    tma_load_3d(smem + Fp8Smem::stage + st * kStageBytes + (isv ? kTile8 : 0), isv ? &tm_v : &tm_k,
                                0, slot, 0, &full[st], pol);
                }
                if (j == 0 && (lane == 4 || lane == 5)) {
                    tma_load_2d(smem + Fp8Smem::qbuf + qb * kQBytes + (lane - 4) * kQHalf, &tm_q, (lane - 4) * 64,
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
            constexpr uint32_t idS = tc::idesc_f16_f32(kRows, HQ < 16 ? 16 : HQ, 0, 0);
            constexpr uint32_t idO = tc::idesc_f16_f32(kD, HQ < 16 ? 16 : HQ, 1, 0);
            auto issue_pv = [&](int u) {
                const int ub = u & 1;
                tc::fence_after_sync();
                const uint32_t vbase = smem_u32(smem + Fp8Smem::vbuf + ub * kVBytes);
                const uint32_t pb = smem_u32(smem + Fp8Smem::pbuf + ub * kPBytes);
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk) {
                    const uint64_t ad = tc::sdesc_sw128(vbase + kk * 2048, kHalf, 1024);
                    const uint64_t bd = tc::sdesc_sw128(pb + (kk >> 2) * kPHalf + (kk & 3) * 32, 16, 1024);
                    tc::mma_f16(tmem + 64 + ub * 32, ad, bd, idO, kk > 0 ? 1u : 0u);
                }
                tc::commit(&o_full[ub]);
                tc::commit(&conv_free[ub]);   // K in TMEM (read by S(u)) and V in shared memory
            };
            // Event loop: issue P.V(tp) as soon as its weights are ready (it frees the
            // converted buffers), otherwise S(tq) as soon as its tile is converted.
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
                    const int cb = tq & 1;
                    if (mbar_test(&conv_full[cb], (tq >> 1) & 1)) {
                        const Fp8Meta m = cmeta[cb];
                        if (m.nvalid == kEndTile) {
                            end_seen = true;
                        } else if (tq < 2 || mbar_test(&s_free[cb], ((tq >> 1) - 1) & 1)) {
                            tc::fence_after_sync();
                            const uint32_t qbase = smem_u32(smem + Fp8Smem::qbuf + (m.item & 1) * kQBytes);
#pragma unroll
                            for (int kk = 0; kk < kD / 16; ++kk) {
                                const uint64_t bd = tc::sdesc_sw128(qbase + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024);
                                tc::mma_f16_tmem_a(tmem + cb * 32, tmem + 128 + cb * 64 + kk * 8, bd, idS,
                                                   kk > 0 ? 1u : 0u);
                            }
                            tc::commit(&s_full[cb]);
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
    } else if (warp < 6) {
        // ==================== accumulate / softmax warps ===========================
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int i = quad * 32 + lane;            // row (softmax) / head dim (accumulate)
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const int hk = i >> 4;                     // KV head of row i
        const int pos = i & 15;                    // position of row i within the tile
        const int upper = lane >> 4;               // which of the warp's two heads
        float acc[kNq];                            // O^T row d = i (code units), all query heads
#pragma unroll
        for (int c = 0; c < kNq; ++c) acc[c] = 0.f;
        float m_run[G], l_part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_part[g] = 0.f;
        }
        Fp8Meta prev;
        bool have_prev = false;

        auto accumulate = [&](int u, const Fp8Meta& m) {
            const int ub = u & 1;
            if (!mbar_wait(&o_full[ub], (u >> 1) & 1)) report(p.dev_status, WF_DEV_TIMEOUT);
            tc::fence_after_sync();
            float o[32];
            tc::ld_32cols(tmem + lane_addr + 64 + ub * 32, o);
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
                const float* L = l_buf + (m.item % 3) * kNq;
                const float* Mx = m_buf + (m.item % 3) * kNq;
                if (m.nsplit == 1) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (int64_t)m.b * p.H_q * kD + i;
#pragma unroll
                    for (int c = 0; c < HQ; ++c) dst[c * kD] = __float2bfloat16_rn(acc[c] * p.v_scale / L[c]);
                } else {
                    const int64_t base = ((int64_t)m.b * p.max_splits + m.split) * p.H_q;
#pragma unroll
                    for (int c = 0; c < HQ; ++c) p.ws_o[(base + c) * kD + i] = acc[c] * p.v_scale;
                    if (i < HQ) p.ws_ml[base + i] = make_float2(Mx[i], L[i]);
                }
            }
        };

        int t = 0;
        for (;; ++t) {
            const int cb = t & 1;
            if (!mbar_wait(&conv_full[cb], (t >> 1) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            const Fp8Meta m = cmeta[cb];
            if (m.nvalid == kEndTile) break;
            // (a) softmax of this tile
            const int sb = cb;
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
            unsigned char* pb = smem + Fp8Smem::pbuf + sb * kPBytes;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float raw = upper ? sv[G + g] : sv[g];
                const float s = live ? raw * p.scale_log2 : -INFINITY;
                float mx = s;
#pragma unroll
                for (int mask = 8; mask >= 1; mask >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
                const float m_new = fmaxf(m_run[g], mx);
                al[g] = exp2f(m_run[g] - m_new);       // 0 on an item's first tile
                const __half eh = __float2half_rn(exp2f(s - m_new));
                l_part[g] = l_part[g] * al[g] + __half2float(eh);
                m_run[g] = m_new;
                *reinterpret_cast<__half*>(pb + sw_elem(hk * G + g, i, kPHalf)) = eh;
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
    } else {
        // ============================ converters ================================
        const int quad = warp & 3;
        const int r = quad * 32 + lane;            // tile row (head r / 16, position r % 16) = TMEM lane
        const int pos = r & 15;
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        for (int t = 0;; ++t) {
            const int st = t % kStages, cb = t & 1;
            if (!mbar_wait(&full[st], (t / kStages) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            const Fp8Meta m = meta[st];
            // the buffers of tile t - 2 must have been read by its products
            if (t >= 2 && !mbar_wait(&conv_free[cb], ((t >> 1) - 1) & 1)) {
                report(p.dev_status, WF_DEV_TIMEOUT);
                break;
            }
            if (m.nvalid != kEndTile) {
                if (m.first && r < HQ) {
                    // q row r (bf16 -> fp16, in place): two 128-byte halves of 8 chunks
                    unsigned char* qrow = smem + Fp8Smem::qbuf + (m.item & 1) * kQBytes;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint4* ch = reinterpret_cast<uint4*>(qrow + c * kQHalf + sw_chunk(r, j));
                            const uint4 v = *ch;
                            *ch = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                                             bf16x2_to_f16x2(v.w));
                        }
                }
                const unsigned char* k8 = smem + Fp8Smem::stage + st * kStageBytes;
                const unsigned char* v8 = k8 + kTile8;
                // K row r -> 64 fp16 pairs -> TMEM lane r, columns [128 + 64 cb, + 64)
#pragma unroll
                for (int hcol = 0; hcol < 2; ++hcol) {
                    uint32_t w[32];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        uint32_t x[8];
                        e4m3x16_to_f16(*reinterpret_cast<const uint4*>(k8 + sw_chunk(r, hcol * 4 + jj)), x);
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[jj * 8 + e] = x[e];
                    }
                    tc::st_32words(tmem + lane_addr + 128 + cb * 64 + hcol * 32, w);
                }
                // V row r -> fp16 into the swizzled tile (zeros past the sequence's end)
                unsigned char* vb = smem + Fp8Smem::vbuf + cb * kVBytes;
                const bool live = pos < m.nvalid;
#pragma unroll
                for (int J = 0; J < 8; ++J) {
                    uint32_t x[8];
                    if (live) {
                        e4m3x16_to_f16(*reinterpret_cast<const uint4*>(v8 + sw_chunk(r, J)), x);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = 0u;
                    }
                    const int c = J >> 2, j0 = 2 * (J & 3);   // d 16J .. 16J+15: half c, chunks j0, j0 + 1
                    *reinterpret_cast<uint4*>(vb + c * kHalf + sw_chunk(r, j0)) = make_uint4(x[0], x[1], x[2], x[3]);
                    *reinterpret_cast<uint4*>(vb + c * kHalf + sw_chunk(r, j0 + 1)) =
                        make_uint4(x[4], x[5], x[6], x[7]);
                }
                tc::wait_st();
            }
            if (threadIdx.x == 6 * 32) cmeta[cb] = m;
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[st]);
                mbar_arrive(&conv_full[cb]);
            }
            if (m.nvalid == kEndTile) break;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, 256);
    }
}

}  // namespace

bool decode_tc_fp8_supported(const wf_pool_desc& pool, int32_t num_q_heads) {
    const int G = pool.num_kv_heads > 0 ? num_q_heads / pool.num_kv_heads : 0;
    return pool.dtype == WF_DTYPE_FP8_E4M3 && pool.head_dim == kD && pool.block_size % kPosT == 0 &&
           pool.num_kv_heads == kHeads && num_q_heads % pool.num_kv_heads == 0 && (G == 2 || G == 4);
}

cudaError_t launch_paged_decode_tc_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                       int32_t num_q_heads, float scale, const wf_pool_desc& pool, float* ws_o,
                                       float2* ws_ml, int32_t max_splits, uint32_t* queue, uint32_t* dev_status,
                                       cudaStream_t stream) {
    const int G = num_q_heads / pool.num_kv_heads;
    CUtensorMap tm_k, tm_v, tm_q;
    const uint64_t slots = (uint64_t)pool.num_blocks * pool.block_size;
    {
        // (d, slot, head) over the fp8 pools: one box = 16 slots x 8 heads x 128 codes
        const uint64_t dims[3] = {(uint64_t)kD, slots, (uint64_t)kHeads};
        const uint64_t strides[2] = {(uint64_t)kHeads * kD, (uint64_t)kD};
        const uint32_t box[3] = {(uint32_t)kD, (uint32_t)kPosT, (uint32_t)kHeads};
        cudaError_t e = encode_tiled(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(k_pool), 3, dims,
                                     strides, box);
        if (e != cudaSuccess) return e;
        e = encode_tiled(&tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(v_pool), 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)B * num_q_heads};
        const uint64_t strides[1] = {(uint64_t)kD * 2};
        const uint32_t box[2] = {64, (uint32_t)num_q_heads};
        cudaError_t e = encode_tiled_bf16(&tm_q, const_cast<void*>(q), 2, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    Fp8Params p;
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
    p.scale_log2 = scale * 1.4426950408889634f * pool.k_scale;
    p.v_scale = pool.v_scale;
    const int smem = Fp8Smem::total + 1024;
    const int64_t items = (int64_t)B * max_splits;
    const int grid = (int)(items < num_sms() ? items : num_sms());
    cudaError_t err;
    if (G == 4) {
        err = allow_dynamic_smem((const void*)paged_decode_tc_fp8_kernel<4>, smem);
        if (err != cudaSuccess) return err;
        paged_decode_tc_fp8_kernel<4><<<grid, kThreadsFp8, smem, stream>>>(tm_k, tm_v, tm_q, p);
    } else {
        err = allow_dynamic_smem((const void*)paged_decode_tc_fp8_kernel<2>, smem);
        if (err != cudaSuccess) return err;
        paged_decode_tc_fp8_kernel<2><<<grid, kThreadsFp8, smem, stream>>>(tm_k, tm_v, tm_q, p);
    }
    return cudaGetLastError();
}

}  // namespace wf
