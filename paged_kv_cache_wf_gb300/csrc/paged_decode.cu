// paged_decode.cu -- split-K ("flash-decoding") attention of one query per
// sequence over its paged KV cache, plus the combine kernel across splits.
//
// What is computed (ember, "The core idea"; tiny-vllm-py, "KV Cache"):
//   out[b, g] = sum_p softmax_p(scale * q[b,g] . K[b,p]) V[b,p],  p = 0 .. seq_len-1,
// where K[b,p] is row (block_table[b][p / P], p % P, g / G) of the [N, P, H_kv, D]
// pool and G = H_q / H_kv (weft, "Shapes and symbols").
//
// GB300 design:
//   * Work item = (sequence b, split j, group of HC <= 8 KV heads).  A split is a
//     fixed span of positions that depends only on the pool geometry, so a
//     sequence's result is the same whatever else is in the batch.
//   * Persistent CTAs, one per SM (two per SM, with half the ring stages each, for
//     group sizes up to 2, whose per-tile chain is short and latency-bound: two
//     items in flight per SM).  CTA c takes items c, c + grid, ... (its
//     producer maps an item to its sequence by a warp-parallel walk over 32
//     sequence lengths per load round) and streams their K and V rows, tile by
//     tile (T positions), from
//     HBM into a ring of shared-memory stages with the bulk-copy (TMA) engine,
//     without a pipeline restart between items.  Completion is an mbarrier
//     transaction count; each stage also carries the tile's item description.
//     Rows of one block that are contiguous in the pool go in one copy.  L2
//     policy evict-first: KV is read once.
//   * Two consumer warps per KV head, each owning half of the head dimension and
//     the head's whole GQA group (up to 8 query heads): each K/V byte is read
//     from HBM once and used G times.
//       q.K: a lane owns 8 dims of a few tile positions; fp32x2 FMAs; partial dot
//            products are finished by a transposing butterfly over the lanes that
//            share the positions, then the two halves are added through shared
//            memory (one named barrier per tile).
//       softmax: running max and sum per query head in fp32 registers (exp2
//            domain, q prescaled by scale*log2 e); both warps of a pair compute
//            the same weights.
//       P.V: a lane owns D/64 output dims of every query head of the group;
//            positions are paired so one fp32x2 FMA adds two positions.
//   * A sequence that fits in one split writes its output directly; otherwise each
//     split leaves (m, l, o) in the workspace and the combine kernel merges them
//     with a warp-shuffle log-sum-exp reduction.
#include <type_traits>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kMaxHC = 8;     // KV heads per CTA
constexpr int kEnd = -1;      // tile meta sentinel: no more work
// positions per split of this file's CUDA-core kernel: small batches of MHA models
// (GPT-2 shapes) have too few 128-position items to spread over the SMs; 64 was
// measured 22% faster there, and 32 slower than 64
constexpr int kSpan = 64;

struct DecodeParams {
    void* out;
    const void* q;
    const char* k_pool;
    const char* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    float* ws_o;     // [B, max_splits, H_q, D]
    float2* ws_ml;   // [B, max_splits, H_q]  (running max in log2 units, sum)
    uint32_t* dev_status;
    int32_t M, B, max_seq_len, H_q, H_kv, G, N, P;
    int32_t HC;          // KV heads per CTA
    int32_t HG;          // head groups: H_kv / HC
    int32_t split_span;  // positions per split
    int32_t max_splits;
    int32_t ps_h, ps_s;  // partial-row strides of a query head and a split (partial_row)
    int32_t stages;
    float scale_log2;    // scale * log2(e)
    // fp8 e4m3 pools: the scale of each KV head's K and V codes (a code c of head h
    // stands for k_head[h] * value(c)); unused for fp32 and bf16 pools
    float k_head[kMaxScaleHeads];
    float v_head[kMaxScaleHeads];
};

// q and the outputs: the pool's type, except that fp8 pools take bf16 ones.
template <typename E>
struct QType {
    using type = E;
};
template <>
struct QType<FP8> {
    using type = BF16;
};

// What the producer tells the consumers about the tile in a stage.
struct TileMeta {
    int32_t b, split, hg, p0;
    int32_t nvalid;   // positions in the tile; kEnd = stop
    int32_t nsplit;   // splits of sequence b
    int32_t first, last;
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ bool len_ok(int len, const DecodeParams& p) {
    return len >= 1 && len <= p.max_seq_len && (int64_t)len <= (int64_t)p.M * p.P;
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <typename E, int D, int GMAX>
struct Shape {
    static constexpr int EB = E::kBytes;
    static constexpr int T = GMAX >= 8 ? 8 : 16;                  // positions per tile
    static constexpr int DH = D / 2;                              // dims per warp of a pair
    static constexpr int DPL = (GMAX >= 8 && D == 64) ? 4 : 8;    // dims per lane in q.K
    static constexpr int LB = DPL * EB < 16 ? DPL * EB : 16;      // bytes per shared load
    static constexpr int NCH = DPL * EB / LB;                     // loads per lane per position
    static constexpr int EPL = LB / EB;                           // elements per load
    static constexpr int DG = DH / DPL;                           // lanes sharing a position
    static constexpr int PS = 32 / DG;                            // positions per pass
    static constexpr int NPL = T / PS;                            // positions per lane per tile
    static constexpr int NV = NPL * GMAX;                         // partial dots per lane
    static constexpr int NF = NV / DG > 0 ? NV / DG : 1;          // finished dots per lane
    static constexpr int VPL = DH / 32;                           // P.V output dims per lane
    static_assert(DG >= GMAX, "a lane's finished dots must belong to one query head");
    static_assert(NPL >= 1 && T % 4 == 0 && EPL % 2 == 0 && DH % 32 == 0, "bad decode shape");
};

// Butterfly that finishes NV partial sums held by each of DG lanes (lane bits
// [0, log2 DG)), halving the set each round while it can.  A lane ends with
// NF = max(1, NV/DG) totals; total j has original index
// j + sum_r bit_r(lane) * (NV >> (r+1)) over the halving rounds r (mask DG/2 first).
template <int NV, int DG>
__device__ __forceinline__ void transpose_reduce(float (&v)[NV], int lane) {
    int n = NV;
#pragma unroll
    for (int mask = DG / 2; mask >= 1; mask >>= 1) {
        if (n >= 2) {
            const int half = n / 2;
            const bool upper = (lane & mask) != 0;
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
        }
    }
}

template <int NV, int DG>
__device__ __forceinline__ int reduced_offset(int lane) {
    int off = 0, n = NV;
#pragma unroll
    for (int mask = DG / 2; mask >= 1; mask >>= 1) {
        if (n >= 2) {
            if (lane & mask) off += n / 2;
            n /= 2;
        }
    }
    return off;
}

// Does lane bit `mask` select the query head of a lane's finished dots?
template <int NV, int NPL, int DG>
__host__ __device__ constexpr bool head_bit(int mask) {
    return mask < DG && (ilog2(DG / mask) - 1) < ilog2(NV) &&
           (ilog2(NV) - 1 - (ilog2(DG / mask) - 1)) >= ilog2(NPL);
}
// Does lane bit `mask` only duplicate values (a plain butterfly round)?
template <int NV, int DG>
__host__ __device__ constexpr bool dup_bit(int mask) {
    return mask < DG && (ilog2(DG / mask) - 1) >= ilog2(NV);
}
// A lane whose finished dots belong to query head g.
template <int NV, int NPL, int DG>
__device__ __forceinline__ int head_lane(int g) {
    int lane = 0;
#pragma unroll
    for (int mask = DG / 2; mask >= 1; mask >>= 1) {
        if (head_bit<NV, NPL, DG>(mask)) {
            const int k = ilog2(NV) - 1 - (ilog2(DG / mask) - 1);  // index bit of this round
            if ((g >> (k - ilog2(NPL))) & 1) lane |= mask;
        }
    }
    return lane;
}

template <typename E, int LB>
__device__ __forceinline__ void load_widen(const unsigned char* src, float* f) {
    if constexpr (E::kBytes == 1) {  // LB e4m3 codes
        if constexpr (LB == 8) {
            const uint2 u = ld_shared_v2(src);
            const float2 a = e4m3x2_to_float2(u.x), b = e4m3x2_to_float2(u.x >> 16);
            const float2 c = e4m3x2_to_float2(u.y), d = e4m3x2_to_float2(u.y >> 16);
            f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
            f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
        } else {
            static_assert(LB == 4, "fp8 K loads of 4 or 8 codes");
            const uint32_t u = *reinterpret_cast<const uint32_t*>(src);
            const float2 a = e4m3x2_to_float2(u), b = e4m3x2_to_float2(u >> 16);
            f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        }
    } else if constexpr (LB == 16) {
        widen_chunk<E>(ld_shared_v4(src), f);
    } else {  // 8 bytes of bf16
        const uint2 u = ld_shared_v2(src);
        const float2 a = bf16x2_to_float2(u.x), b = bf16x2_to_float2(u.y);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
}

// One lane's VPL dims of V at one position, as fp32 (0 when `live` is false).
template <typename E, int VPL>
__device__ __forceinline__ void load_v(const unsigned char* src, bool live, float* f) {
    if constexpr (E::kBytes == 1) {  // e4m3 codes
        if constexpr (VPL == 2) {
            const float2 x = e4m3x2_to_float2(live ? (uint32_t)(*reinterpret_cast<const uint16_t*>(src)) : 0u);
            f[0] = x.x;
            f[1] = x.y;
        } else {
            f[0] = e4m3x2_to_float2(live ? (uint32_t)(*src) : 0u).x;
        }
    } else if constexpr (E::kBytes == 2) {
        if constexpr (VPL == 2) {
            const uint32_t u = live ? *reinterpret_cast<const uint32_t*>(src) : 0u;
            f[0] = __uint_as_float(u << 16);
            f[1] = __uint_as_float(u & 0xffff0000u);
        } else {
            const uint32_t u = live ? (uint32_t)(*reinterpret_cast<const uint16_t*>(src)) : 0u;
            f[0] = __uint_as_float(u << 16);
        }
    } else {
        if constexpr (VPL == 2) {
            const float2 x = live ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
            f[0] = x.x;
            f[1] = x.y;
        } else {
            f[0] = live ? *reinterpret_cast<const float*>(src) : 0.f;
        }
    }
}

template <typename E, int D, int GMAX, int MINB>
__global__ void __launch_bounds__((2 * kMaxHC + 1) * 32, MINB) paged_decode_kernel(const DecodeParams p) {
    using S = Shape<E, D, GMAX>;
    constexpr int T = S::T;
    constexpr int EB = S::EB;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NCW = 2 * p.HC;  // consumer warps
    const int row_bytes = p.HC * D * EB;
    const int tile_bytes = T * row_bytes;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sK = smem;
    unsigned char* sV = sK + (size_t)p.stages * tile_bytes;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(sV + (size_t)p.stages * tile_bytes);
    uint64_t* empty_bar = full_bar + p.stages;
    TileMeta* sMeta = reinterpret_cast<TileMeta*>(empty_bar + p.stages);
    float* sX = reinterpret_cast<float*>(sMeta + p.stages);   // [HC][parity][half][32][NF]
    float* sP = sX + p.HC * 2 * 2 * 32 * S::NF;                // [NCW][GMAX][T]
    // [HC]: the two warps of a KV head meet here each tile (bounded waits, so a warp
    // that stops on a timed-out wait cannot leave its partner blocked)
    uint64_t* pair_bar = reinterpret_cast<uint64_t*>(sP + NCW * GMAX * T);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
        for (int i = 0; i < p.HC; ++i) mbar_init(&pair_bar[i], 2);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ======================= producer warp ==============================
        const uint64_t pol = l2_policy_evict_first();
        const int64_t pool_row = (int64_t)p.H_kv * D * EB;  // bytes of one pool slot
        const bool whole_rows = (p.HC == p.H_kv);           // slots contiguous across positions
        int t = 0;
        int b = 0, len_b = 0, nsp_b = 0;
        int64_t cum = 0;  // splits of sequences before b
        bool ok = true;
        // the item -> sequence map walks 32 sequence lengths per load round (a CTA's
        // items only move forward)
        const int64_t cap = min((int64_t)p.max_seq_len, (int64_t)p.M * p.P);
        ItemWalk walk;
        item_walk_load(walk, p.seq_lens, p.B, p.split_span, cap, p.dev_status, lane);
        for (int64_t item = blockIdx.x; ok; item += gridDim.x) {
            const int64_t u = item / p.HG;
            const int hg = (int)(item % p.HG);
            if (!item_walk_find(walk, u, p.seq_lens, p.B, p.split_span, cap, p.dev_status, lane, b, len_b, nsp_b, cum))
                break;
            const int split = (int)(u - cum);
            const int s0 = split * p.split_span;
            const int s1 = min(len_b, s0 + p.split_span);
            const int ntiles = (s1 - s0 + T - 1) / T;
            const int32_t* table = p.block_tables + (int64_t)b * p.M;
            const int64_t head_off = (int64_t)hg * p.HC * D * EB;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int st = t % p.stages;
                if (t >= p.stages && !mbar_wait(&empty_bar[st], ((t / p.stages) - 1) & 1)) {
                    if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                    ok = false;
                    break;
                }
                const int p0 = s0 + j * T;
                const int nvalid = min(T, s1 - p0);
                const int pos = p0 + lane;
                const bool valid = lane < nvalid;
                int blk = 0, off = 0;
                if (valid) {
                    blk = __ldg(table + pos / p.P);
                    off = pos % p.P;
                }
                const bool okb = valid && (unsigned)blk < (unsigned)p.N;
                if (valid && !okb && (lane == 0 || off == 0)) report(p.dev_status, WF_DEV_BAD_BLOCK);
                const unsigned okmask = __ballot_sync(0xffffffffu, okb);
                const uint32_t bytes = (uint32_t)__popc(okmask) * (uint32_t)row_bytes * 2u;
                if (lane == 0) {
                    TileMeta m;
                    m.b = b; m.split = split; m.hg = hg; m.p0 = p0; m.nvalid = nvalid; m.nsplit = nsp_b;
                    m.first = (j == 0); m.last = (j == ntiles - 1);
                    sMeta[st] = m;
                    mbar_arrive_expect_tx(&full_bar[st], bytes);
                }
                __syncwarp();
                const bool start = okb && (!whole_rows || lane == 0 || off == 0);
                if (start) {
                    const int run = whole_rows ? min(p.P - off, nvalid - lane) : 1;
                    const int64_t src = ((int64_t)blk * p.P + off) * pool_row + head_off;
                    bulk_g2s(sK + (size_t)st * tile_bytes + lane * row_bytes, p.k_pool + src,
                             (uint32_t)(run * row_bytes), &full_bar[st], pol);
                    bulk_g2s(sV + (size_t)st * tile_bytes + lane * row_bytes, p.v_pool + src,
                             (uint32_t)(run * row_bytes), &full_bar[st], pol);
                }
            }
        }
        if (ok) {  // tell the consumers to stop
            const int st = t % p.stages;
            if (t < p.stages || mbar_wait(&empty_bar[st], ((t / p.stages) - 1) & 1)) {
                if (lane == 0) {
                    sMeta[st].nvalid = kEnd;
                    mbar_arrive_expect_tx(&full_bar[st], 0);
                }
                ++t;
            } else if (lane == 0) {
                report(p.dev_status, WF_DEV_TIMEOUT);
            }
        }
        // Never leave with copies in flight: the last stages' fills must have landed.
        if (lane == 0) {
            const int first = t > p.stages ? t - p.stages : 0;
            for (int tt = first; tt < t; ++tt) mbar_wait(&full_bar[tt % p.stages], (tt / p.stages) & 1, 1u << 20);
        }
        return;
    }

    // ========================= consumer warps ===============================
    const int pair = warp >> 1;   // KV head within the CTA
    const int half = warp & 1;    // which half of the head dimension
    const int dg = lane % S::DG;
    const int ps = lane / S::DG;
    const int G = p.G;
    float* sPw = sP + warp * GMAX * T;
    float* sXp = sX + pair * (2 * 2 * 32 * S::NF);
    const int off_r = reduced_offset<S::NV, S::DG>(lane);
    const int g_lane = off_r / S::NPL;  // query head of this lane's finished dots

    using QE = typename QType<E>::type;                // q and output element type
    constexpr int QB = S::EPL * QE::kBytes;            // bytes of q per K load chunk
    constexpr bool kCodes = E::kBytes == 1;            // fp8 e4m3 pool
    float2 q2[GMAX][S::DPL / 2];
    float2 acc[GMAX][S::VPL];
    float m_run = -INFINITY, l_run = 0.f;
    int hq0 = 0;
    int meets = 0;

    for (int t = 0;; ++t) {
        const int st = t % p.stages;
        if (!mbar_wait(&full_bar[st], (t / p.stages) & 1)) {
            if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
            return;
        }
        const TileMeta mt = sMeta[st];
        if (mt.nvalid == kEnd) break;
        const int nvalid = mt.nvalid;
        if (mt.first) {
            hq0 = (mt.hg * p.HC + pair) * G;
#pragma unroll
            for (int g = 0; g < GMAX; ++g) {
#pragma unroll
                for (int k = 0; k < S::NCH; ++k) {
                    const int c = dg + S::DG * ((k + ps) % S::NCH);
                    float f[S::EPL];
                    if (g < G) {
                        const char* src = static_cast<const char*>(p.q) +
                                          (((int64_t)mt.b * p.H_q + hq0 + g) * D + half * S::DH) * QE::kBytes + c * QB;
                        if constexpr (QB == 16) {
                            widen_chunk<QE>(*reinterpret_cast<const uint4*>(src), f);
                        } else {
                            const uint2 u = *reinterpret_cast<const uint2*>(src);
                            const float2 a = bf16x2_to_float2(u.x), bb = bf16x2_to_float2(u.y);
                            f[0] = a.x; f[1] = a.y; f[2] = bb.x; f[3] = bb.y;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < S::EPL; ++e) f[e] = 0.f;
                    }
                    // fp8: scores are formed from the code values, so the K scale of this
                    // warp's KV head goes into q
                    float qs = p.scale_log2;
                    if constexpr (kCodes) qs = p.scale_log2 * p.k_head[mt.hg * p.HC + pair];
#pragma unroll
                    for (int e = 0; e < S::EPL / 2; ++e)
                        q2[g][k * S::EPL / 2 + e] = make_float2(f[2 * e] * qs, f[2 * e + 1] * qs);
                }
            }
#pragma unroll
            for (int g = 0; g < GMAX; ++g)
#pragma unroll
                for (int v = 0; v < S::VPL; ++v) acc[g][v] = make_float2(0.f, 0.f);
            m_run = -INFINITY;
            l_run = 0.f;
        }
        const unsigned char* tK = sK + (size_t)st * tile_bytes + pair * D * EB + half * S::DH * EB;
        const unsigned char* tV = sV + (size_t)st * tile_bytes + pair * D * EB + half * S::DH * EB;

        // ---- q . K over this warp's half of D --------------------------------
        float2 part[GMAX][S::NPL];
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int i = 0; i < S::NPL; ++i) part[g][i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < S::NPL; ++i) {
            const int pl = ps + S::PS * i;
#pragma unroll
            for (int k = 0; k < S::NCH; ++k) {
                const int c = dg + S::DG * ((k + ps) % S::NCH);
                float f[S::EPL];
                load_widen<E, S::LB>(tK + pl * row_bytes + c * S::LB, f);
#pragma unroll
                for (int e = 0; e < S::EPL / 2; ++e) {
                    const float2 kk = make_float2(f[2 * e], f[2 * e + 1]);
#pragma unroll
                    for (int g = 0; g < GMAX; ++g)
                        part[g][i] = ffma2(q2[g][k * S::EPL / 2 + e], kk, part[g][i]);
                }
            }
        }
        float v[S::NV];
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int i = 0; i < S::NPL; ++i) v[g * S::NPL + i] = part[g][i].x + part[g][i].y;
        transpose_reduce<S::NV, S::DG>(v, lane);

        // ---- add the other half of D (the partner warp) ------------------------
        {
            const int par = t & 1;
            float* mine = sXp + ((par * 2 + half) * 32 + lane) * S::NF;
            const float* theirs = sXp + ((par * 2 + (1 - half)) * 32 + lane) * S::NF;
#pragma unroll
            for (int j = 0; j < S::NF; ++j) mine[j] = v[j];
            __syncwarp();
            if (lane == 0) mbar_arrive(&pair_bar[pair]);
            if (!mbar_wait(&pair_bar[pair], meets & 1) && lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
            ++meets;
#pragma unroll
            for (int j = 0; j < S::NF; ++j) v[j] += theirs[j];
        }

        // ---- online softmax for query head g_lane -------------------------------
        float s[S::NF];
        int plj[S::NF];
        float mtile = -INFINITY;
#pragma unroll
        for (int j = 0; j < S::NF; ++j) {
            plj[j] = ps + S::PS * ((off_r + j) % S::NPL);
            s[j] = plj[j] < nvalid ? v[j] : -INFINITY;
            mtile = fmaxf(mtile, s[j]);
        }
#pragma unroll
        for (int mask = 1; mask < 32; mask <<= 1)
            if (!head_bit<S::NV, S::NPL, S::DG>(mask)) mtile = fmaxf(mtile, __shfl_xor_sync(0xffffffffu, mtile, mask));
        const float m_new = fmaxf(m_run, mtile);
        const float alpha = exp2f(m_run - m_new);  // 0 on an item's first tile
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < S::NF; ++j) {
            const float pj = exp2f(s[j] - m_new);   // 0 for positions past the tile end
            psum += pj;
            sPw[g_lane * T + plj[j]] = pj;
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        float a[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) a[g] = __shfl_sync(0xffffffffu, alpha, head_lane<S::NV, S::NPL, S::DG>(g));
        __syncwarp();
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int vv = 0; vv < S::VPL; ++vv) acc[g][vv] = make_float2(acc[g][vv].x * a[g], acc[g][vv].y * a[g]);

        // ---- P . V, two positions per fp32x2 FMA ------------------------------
        const unsigned char* vcol = tV + lane * S::VPL * EB;
#pragma unroll
        for (int pl = 0; pl < T; pl += 4) {
            float vf[4][S::VPL];
#pragma unroll
            for (int k = 0; k < 4; ++k) load_v<E, S::VPL>(vcol + (pl + k) * row_bytes, pl + k < nvalid, vf[k]);
#pragma unroll
            for (int g = 0; g < GMAX; ++g) {
                const float4 w = ld_shared_f4(sPw + g * T + pl);
#pragma unroll
                for (int vv = 0; vv < S::VPL; ++vv) {
                    acc[g][vv] = ffma2(make_float2(w.x, w.y), make_float2(vf[0][vv], vf[1][vv]), acc[g][vv]);
                    acc[g][vv] = ffma2(make_float2(w.z, w.w), make_float2(vf[2][vv], vf[3][vv]), acc[g][vv]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);

        if (mt.last) {
            // ---- finish the item: per-head sums, then output or partial ----------
            float lt = l_run;
#pragma unroll
            for (int mask = 1; mask < 32; mask <<= 1)
                if (!head_bit<S::NV, S::NPL, S::DG>(mask) && !dup_bit<S::NV, S::DG>(mask))
                    lt += __shfl_xor_sync(0xffffffffu, lt, mask);
            float Lh[GMAX], Mh[GMAX];
#pragma unroll
            for (int g = 0; g < GMAX; ++g) {
                const int src = head_lane<S::NV, S::NPL, S::DG>(g);
                Lh[g] = __shfl_sync(0xffffffffu, lt, src);
                Mh[g] = __shfl_sync(0xffffffffu, m_run, src);
            }
            const int dcol = half * S::DH + lane * S::VPL;
            if (mt.nsplit == 1) {
#pragma unroll
                for (int g = 0; g < GMAX; ++g) {
                    if (g < G) {
                        float inv = 1.f / Lh[g];
                        if constexpr (kCodes) inv *= p.v_head[mt.hg * p.HC + pair];   // the V scale
                        float o[S::VPL];
#pragma unroll
                        for (int vv = 0; vv < S::VPL; ++vv) o[vv] = (acc[g][vv].x + acc[g][vv].y) * inv;
                        char* dst =
                            static_cast<char*>(p.out) + (((int64_t)mt.b * p.H_q + hq0 + g) * D + dcol) * QE::kBytes;
                        store_out<QE, S::VPL>(dst, o);
                    }
                }
            } else {
#pragma unroll
                for (int g = 0; g < GMAX; ++g) {
                    if (g < G) {
                        const int64_t row = partial_row(mt.b, hq0 + g, mt.split, p.H_q, p.max_splits, p.ps_h, p.ps_s);
                        float* dst = p.ws_o + row * D + dcol;
                        float vsc = 1.f;
                        if constexpr (kCodes) vsc = p.v_head[mt.hg * p.HC + pair];   // partials carry the V scale
#pragma unroll
                        for (int vv = 0; vv < S::VPL; ++vv) dst[vv] = (acc[g][vv].x + acc[g][vv].y) * vsc;
                        if (half == 0 && lane == 0) p.ws_ml[row] = make_float2(Mh[g], Lh[g]);
                    }
                }
            }
        }
    }
}

// Merge the splits of every (sequence, query head) with more than one split:
//   out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j.
// One warp per (b, query head); lanes own D/32 output dims.  The merge is bound by
// the latency of reading the partials: each round of up to kChunk splits issues
// its (m, l) loads and every o row load at once, before using any of them, and
// folds the round in with an online rescale, so a merge of up to kChunk splits is
// one round trip.  Launched as a programmatic dependent of the split kernel: the
// grid may start while the split kernel drains, and waits for it
// (griddepcontrol.wait) before reading the workspace.
template <typename E, int D>
__global__ void __launch_bounds__(128, D == 128 ? 6 : 4) paged_decode_combine_kernel(const DecodeParams p) {
    constexpr int VPL = D / 32;
    // o rows in flight per lane: 12 at D = 128 (80 registers, six 4-warp CTAs an SM:
    // the Llama-3-8B batch's 7392 rows merge in two waves instead of three, which
    // measured 1.3 us a call faster than 24 rows at four CTAs an SM), 32 at D = 64
    constexpr int kChunk = D == 128 ? 12 : 32;
    using Vec = typename std::conditional<VPL == 4, float4, float2>::type;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.x * 4 + warp;
    const int b = blockIdx.y;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (hq >= p.H_q) return;
    const int len = __ldg(p.seq_lens + b);
    if (!len_ok(len, p)) return;
    const int n = (len + p.split_span - 1) / p.split_span;
    if (n <= 1) return;
    const int64_t row0 = partial_row(b, hq, 0, p.H_q, p.max_splits, p.ps_h, p.ps_s);
    const Vec* orow = reinterpret_cast<const Vec*>(p.ws_o + row0 * D) + lane;   // + j * ps_s * (D / VPL)
    const float2* mrow = p.ws_ml + row0;                                        // + j * ps_s
    float M = -INFINITY, den = 0.f;
    float o[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) o[k] = 0.f;
    for (int j0 = 0; j0 < n; j0 += kChunk) {
        const int cnt = min(kChunk, n - j0);
        Vec x[kChunk];
#pragma unroll
        for (int u = 0; u < kChunk; ++u)
            if (u < cnt) x[u] = __ldcg(orow + (int64_t)(j0 + u) * p.ps_s * (D / VPL));
        const float2 ml = lane < cnt ? __ldcg(mrow + (int64_t)(j0 + lane) * p.ps_s) : make_float2(-INFINITY, 0.f);
        float cm = ml.x;
#pragma unroll
        for (int mask = 16; mask >= 1; mask >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, mask));
        const float Mn = fmaxf(M, cm);                     // finite: every split has a live position
        const float a = M == -INFINITY ? 0.f : exp2f(M - Mn);
        den *= a;
#pragma unroll
        for (int k = 0; k < VPL; ++k) o[k] *= a;
        const float wl = lane < cnt ? exp2f(ml.x - Mn) : 0.f;
        den += wl * ml.y;                                  // per lane; summed over the warp at the end
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            const float w = __shfl_sync(0xffffffffu, wl, u);
            if (u < cnt) {
                if constexpr (VPL == 4) {
                    o[0] += w * x[u].x; o[1] += w * x[u].y; o[2] += w * x[u].z; o[3] += w * x[u].w;
                } else {
                    o[0] += w * x[u].x; o[1] += w * x[u].y;
                }
            }
        }
        M = Mn;
    }
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(0xffffffffu, den, mask);
    const float inv = 1.f / den;
#pragma unroll
    for (int k = 0; k < VPL; ++k) o[k] *= inv;
    char* dst = static_cast<char*>(p.out) + (((int64_t)b * p.H_q + hq) * D + lane * VPL) * E::kBytes;
    store_out<E, VPL>(dst, o);
}

// The combine kernel as a programmatic dependent launch of the split kernel before it.
template <typename E, int D>
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.H_q + 3) / 4, p.B);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, paged_decode_combine_kernel<E, D>, p);
}

int pow2_at_least(int x) {
    int r = 1;
    while (r < x) r <<= 1;
    return r;
}

template <typename E, int D, int GMAX>
int smem_bytes_for(int hc, int stages) {
    using S = Shape<E, D, GMAX>;
    const int tile_bytes = S::T * hc * D * S::EB;
    return stages * (2 * tile_bytes + 16 + (int)sizeof(TileMeta)) + hc * 2 * 2 * 32 * S::NF * 4 +
           2 * hc * GMAX * S::T * 4 + hc * 8;
}

template <typename E, int D, int GMAX, int MINB = 1>
int pick_stages(int hc) {
    constexpr int kBudget = MINB == 1 ? 216 * 1024 : 108 * 1024;
    int st = 8;
    while (st > 2 && smem_bytes_for<E, D, GMAX>(hc, st) > kBudget) --st;
    return st;
}

template <typename E, int D, int GMAX>
cudaError_t launch_typed(DecodeParams& p, cudaStream_t stream) {
    // small group sizes run two CTAs per SM (half the stages each)
    constexpr int MINB = GMAX <= 2 ? 2 : 1;
    auto kern = paged_decode_kernel<E, D, GMAX, MINB>;
    p.stages = pick_stages<E, D, GMAX, MINB>(p.HC);
    const int smem = smem_bytes_for<E, D, GMAX>(p.HC, p.stages);
    cudaError_t err = allow_dynamic_smem((const void*)kern, smem);
    if (err != cudaSuccess) return err;
    const int64_t items = (int64_t)p.B * p.max_splits * p.HG;
    const int grid = (int)(items < MINB * num_sms() ? items : MINB * num_sms());
    kern<<<grid, (2 * p.HC + 1) * 32, smem, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return p.max_splits > 1 ? launch_combine<typename QType<E>::type, D>(p, stream) : cudaSuccess;
}

template <typename E, int D>
cudaError_t launch_group(DecodeParams& p, int gmax, cudaStream_t stream) {
    switch (gmax) {
        case 1: return launch_typed<E, D, 1>(p, stream);
        case 2: return launch_typed<E, D, 2>(p, stream);
        case 4: return launch_typed<E, D, 4>(p, stream);
        default: return launch_typed<E, D, 8>(p, stream);
    }
}

}  // namespace

// fp8 pools run the tensor-core kernel where it takes their shape, else this file's
// CUDA-core kernel on the codes.
static bool fp8_on_tensor_cores(const wf_pool_desc& pool, int32_t num_q_heads) {
    return decode_tc_fp8_supported(pool, num_q_heads) && (int64_t)pool.num_blocks * pool.block_size <= INT32_MAX;
}

bool decode_geometry(const wf_pool_desc& pool, int32_t num_q_heads, DecodeGeometry* g) {
    if (pool.num_kv_heads < 1 || num_q_heads % pool.num_kv_heads != 0) return false;
    const int G = num_q_heads / pool.num_kv_heads;
    if (G < 1 || G > 8) return false;
    if (pool.head_dim != 64 && pool.head_dim != 128) return false;
    int hc = 1;
    for (int c = kMaxHC; c >= 1; --c)
        if (pool.num_kv_heads % c == 0) {
            hc = c;
            break;
        }
    // the tensor-core kernels (bf16, and every fp8 pool) have their own item spans
    g->split_span = pool.dtype == WF_DTYPE_FP8_E4M3
                        ? (fp8_on_tensor_cores(pool, num_q_heads) ? decode_tc_fp8_span() : kSpan)
                    : decode_tc_supported(pool, num_q_heads) ? decode_tc_span(pool)
                                                             : kSpan;
    g->tile = G > 4 ? 8 : 16;
    g->stages = 0;  // chosen per kernel instance at launch
    g->consumer_warps = 2 * hc;
    g->heads_per_warp = 1;
    g->gmax = pow2_at_least(G);
    g->smem_bytes = 0;
    return true;
}

int decode_kernel_kind(const wf_pool_desc& pool, int32_t num_q_heads) {
    DecodeGeometry g;
    if (!decode_geometry(pool, num_q_heads, &g)) return WF_KERNEL_NONE;
    const int64_t slots = (int64_t)pool.num_blocks * pool.block_size;
    if (decode_tc_supported(pool, num_q_heads) && slots <= INT32_MAX) return WF_KERNEL_TENSOR_CORES;
    if (pool.dtype == WF_DTYPE_FP8_E4M3 && fp8_on_tensor_cores(pool, num_q_heads)) return WF_KERNEL_TENSOR_CORES;
    return WF_KERNEL_CUDA_CORES;
}

size_t decode_workspace_bytes(int32_t B, int32_t num_q_heads, int32_t max_seq_len,
                              const wf_pool_desc& pool) {
    DecodeGeometry g;
    if (B < 0 || max_seq_len < 1 || !decode_geometry(pool, num_q_heads, &g)) return 0;
    const int64_t max_splits = (max_seq_len + g.split_span - 1) / g.split_span;
    const int64_t rows = (int64_t)B * max_splits * num_q_heads;
    const int64_t o_bytes = rows * pool.head_dim * 4;
    const int64_t ml_bytes = rows * 8;
    const int64_t base = ((o_bytes + 255) / 256) * 256 + ml_bytes + 256;
    // fp8 pools: the prepared q parts and row scales follow, 256-byte aligned
    if (pool.dtype == WF_DTYPE_FP8_E4M3) return (size_t)((base + 255) / 256 * 256) + decode_fp8_prep_bytes(B, num_q_heads);
    return (size_t)base;
}

// The decode's parameters, with the workspace carved into split partials and the
// tensor-core kernels' work-item queue.
static bool decode_setup(void* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t B,
                         int32_t max_seq_len, int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                         void* workspace, uint32_t* dev_status, DecodeGeometry& g, DecodeParams& p,
                         uint32_t*& queue) {
    if (!decode_geometry(pool, num_q_heads, &g)) return false;
    p.out = out;
    p.q = q;
    p.k_pool = static_cast<const char*>(k_pool);
    p.v_pool = static_cast<const char*>(v_pool);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.dev_status = dev_status;
    p.M = max_blocks_per_seq;
    p.B = B;
    p.max_seq_len = max_seq_len;
    p.H_q = num_q_heads;
    p.H_kv = pool.num_kv_heads;
    p.G = num_q_heads / pool.num_kv_heads;
    p.N = pool.num_blocks;
    p.P = pool.block_size;
    p.HC = g.consumer_warps / 2;
    p.HG = pool.num_kv_heads / p.HC;
    p.split_span = g.split_span;
    p.max_splits = (max_seq_len + g.split_span - 1) / g.split_span;
    // split-minor partial rows; the fp8 tensor-core kernel writes head-minor ones
    const bool fp8_tc = pool.dtype == WF_DTYPE_FP8_E4M3 && fp8_on_tensor_cores(pool, num_q_heads);
    p.ps_h = fp8_tc ? 1 : p.max_splits;
    p.ps_s = fp8_tc ? num_q_heads : 1;
    p.stages = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int64_t rows = (int64_t)B * p.max_splits * num_q_heads;
    const int64_t o_bytes = ((rows * pool.head_dim * 4 + 255) / 256) * 256;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + o_bytes);
    // the tensor-core kernels' work-item queue: one word after the (m, l) partials,
    // inside the workspace's slack, zeroed by a small grid that runs before each
    // decode grid (for fp8 pools, the grid that prepares q)
    queue = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + o_bytes + (rows * 8 + 15) / 16 * 16);
    return true;
}

cudaError_t launch_paged_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                void* workspace, uint32_t* dev_status, cudaStream_t stream) {
    DecodeGeometry g;
    DecodeParams p;
    uint32_t* queue = nullptr;
    if (!decode_setup(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, B, max_seq_len, num_q_heads,
                      scale, pool, workspace, dev_status, g, p, queue))
        return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)B * p.max_splits * num_q_heads;
    const int64_t o_bytes = ((rows * pool.head_dim * 4 + 255) / 256) * 256;
    const int64_t slots = (int64_t)pool.num_blocks * pool.block_size;
    if (decode_tc_supported(pool, num_q_heads) && slots <= INT32_MAX) {
        cudaError_t err = launch_paged_decode_tc(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, B,
                                     max_seq_len, num_q_heads, scale, pool, p.ws_o, p.ws_ml, p.max_splits, queue,
                                     dev_status, stream);
        if (err != cudaSuccess) return err;
        if (p.max_splits <= 1) return cudaSuccess;
        return pool.head_dim == 64 ? launch_combine<BF16, 64>(p, stream) : launch_combine<BF16, 128>(p, stream);
    }
    if (pool.dtype == WF_DTYPE_FP8_E4M3 && !fp8_on_tensor_cores(pool, num_q_heads)) {
        // other shapes: the CUDA-core kernel widens the codes; per-head scales by value
        const HeadScales hs = head_scales(pool);
        for (int h = 0; h < kMaxScaleHeads; ++h) {
            p.k_head[h] = hs.k[h];
            p.v_head[h] = hs.v[h];
        }
        return pool.head_dim == 64 ? launch_group<FP8, 64>(p, g.gmax, stream)
                                   : launch_group<FP8, 128>(p, g.gmax, stream);
    }
    if (pool.dtype == WF_DTYPE_FP8_E4M3) {
        // the preparing grid zeroes the queue; its q parts follow the partials
        void* prep = static_cast<char*>(workspace) + (o_bytes + rows * 8 + 256 + 255) / 256 * 256;
        cudaError_t err = launch_paged_decode_tc_fp8(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq,
                                                     seq_lens, B, max_seq_len, num_q_heads, scale, pool, p.ws_o,
                                                     p.ws_ml, p.max_splits, queue, prep, dev_status, stream);
        if (err != cudaSuccess) return err;
        if (p.max_splits <= 1) return cudaSuccess;
        return pool.head_dim == 64 ? launch_combine<BF16, 64>(p, stream) : launch_combine<BF16, 128>(p, stream);
    }
    if (pool.dtype == WF_DTYPE_F32) {
        return pool.head_dim == 64 ? launch_group<F32, 64>(p, g.gmax, stream)
                                   : launch_group<F32, 128>(p, g.gmax, stream);
    }
    return pool.head_dim == 64 ? launch_group<BF16, 64>(p, g.gmax, stream)
                               : launch_group<BF16, 128>(p, g.gmax, stream);
}

cudaError_t launch_paged_prefill_decode(void* pf_out, const void* pf_q, const int32_t* pf_block_tables,
                                       int32_t pf_max_blocks_per_seq, const int32_t* pf_seq_lens,
                                       const int32_t* cu_q_lens, int32_t pf_B, int32_t total_q, int32_t max_q_len,
                                       int32_t pf_max_seq_len, void* dec_out, const void* dec_q,
                                       const int32_t* dec_block_tables, int32_t dec_max_blocks_per_seq,
                                       const int32_t* dec_seq_lens, int32_t dec_B, int32_t dec_max_seq_len,
                                       const void* k_pool, const void* v_pool, int32_t num_q_heads, float scale,
                                       const wf_pool_desc& pool, void* workspace, uint32_t* dev_status,
                                       cudaStream_t stream) {
    const bool has_pf = pf_B > 0 && total_q > 0 && max_q_len > 0;
    if (!has_pf || dec_B == 0 || !mixed_tc_supported(pool, num_q_heads)) {
        // nothing to share a launch, or shapes the one-launch kernel does not take:
        // the two calls one after the other
        if (has_pf) {
            cudaError_t err = launch_paged_prefill(pf_out, pf_q, k_pool, v_pool, pf_block_tables,
                                                   pf_max_blocks_per_seq, pf_seq_lens, cu_q_lens, pf_B, total_q,
                                                   max_q_len, pf_max_seq_len, num_q_heads, scale, pool, dev_status,
                                                   stream);
            if (err != cudaSuccess) return err;
        }
        if (dec_B == 0) return cudaSuccess;
        return launch_paged_decode(dec_out, dec_q, k_pool, v_pool, dec_block_tables, dec_max_blocks_per_seq,
                                   dec_seq_lens, dec_B, dec_max_seq_len, num_q_heads, scale, pool, workspace,
                                   dev_status, stream);
    }
    DecodeGeometry g;
    DecodeParams p;
    uint32_t* queue = nullptr;
    if (!decode_setup(dec_out, dec_q, k_pool, v_pool, dec_block_tables, dec_max_blocks_per_seq, dec_seq_lens, dec_B,
                      dec_max_seq_len, num_q_heads, scale, pool, workspace, dev_status, g, p, queue))
        return cudaErrorInvalidValue;
    cudaError_t err = launch_paged_mixed_tc(pf_out, pf_q, pf_block_tables, pf_max_blocks_per_seq, pf_seq_lens,
                                            cu_q_lens, pf_B, total_q, max_q_len, pf_max_seq_len, dec_out, dec_q,
                                            dec_block_tables, dec_max_blocks_per_seq, dec_seq_lens, dec_B,
                                            dec_max_seq_len, k_pool, v_pool, num_q_heads, scale, pool, p.ws_o,
                                            p.ws_ml, p.max_splits, queue, dev_status, stream);
    if (err != cudaSuccess) return err;
    if (p.max_splits <= 1) return cudaSuccess;
    return pool.head_dim == 64 ? launch_combine<BF16, 64>(p, stream) : launch_combine<BF16, 128>(p, stream);
}

}  // namespace wf
