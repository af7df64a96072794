// paged_decode.cu -- split-K ("flash-decoding") attention of one query per
// sequence over its paged KV cache, plus the combine kernel across splits.
//
// What is computed (ember, "The core idea"; tiny-vllm-py, "KV Cache"):
//   out[b, g] = sum_p softmax_p(scale * q[b,g] . K[b,p]) V[b,p],  p = 0 .. seq_len-1,
// where K[b,p] is row (block_table[b][p / P], p % P, g / G) of the [N, P, H_kv, D]
// pool and G = H_q / H_kv (weft, "Shapes and symbols").
//
// GB300 design:
//   * The work unit is (sequence b, split j, group of HC KV heads).  A split is a
//     fixed span of positions that depends only on the pool geometry, so a
//     sequence's result is the same whatever else is in the batch.
//   * One producer warp streams K and V rows of the split, tile by tile
//     (kTile positions), from HBM into a ring of shared-memory stages with the
//     bulk-copy (TMA) engine; completion is tracked by mbarrier transaction
//     counts, release by a second mbarrier per stage.  Rows of one block that are
//     contiguous in the pool go in one copy.  L2 policy evict-first: KV is read once.
//   * One consumer warp per KV head holds the head's whole GQA group (up to 8
//     query heads): each K/V byte is read from HBM once and used G times.
//   * q.K: a lane owns 16 (or 8) head dims of a few tile positions; partial dot
//     products are finished with a transposing butterfly over the lanes that share
//     the positions.  Online softmax keeps the running max and sum in fp32
//     registers (exp2 domain, q prescaled by scale*log2 e).  P.V: a lane owns D/32
//     output dims of every query head of the group, with packed fp32x2 FMAs.
//   * A sequence that fits in one split writes its output directly; otherwise each
//     split leaves (m, l, o) in the workspace and the combine kernel merges them
//     with a warp-shuffle log-sum-exp reduction.
#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kTile = 16;  // positions per pipeline stage (one producer lane each)

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
    int32_t HC;          // KV heads per CTA (= consumer warps)
    int32_t split_span;  // positions per split
    int32_t max_splits;
    int32_t stages;
    float scale_log2;    // scale * log2(e)
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Sequence-length check shared by the split and combine kernels.
__device__ __forceinline__ bool len_ok(int len, const DecodeParams& p) {
    return len >= 1 && len <= p.max_seq_len && (int64_t)len <= (int64_t)p.M * p.P;
}

template <typename E, int D, int GMAX>
struct Shape {
    static constexpr int EPC = E::kPerChunk;                   // elements per 16-byte chunk
    static constexpr int DPL = GMAX >= 8 ? 8 : 16;             // head dims per lane in q.K
    static constexpr int DG = D / DPL;                         // lanes sharing one position
    static constexpr int PS = 32 / DG;                         // positions in flight per warp
    static constexpr int NPL = kTile / PS;                     // positions per lane per tile
    static constexpr int CPL = DPL / EPC;                      // chunks per lane per position
    static constexpr int NV = NPL * GMAX;                      // partial dot products per lane
    static constexpr int VPL = D / 32;                         // output dims per lane in P.V
    static constexpr int NSE = (kTile * GMAX + 31) / 32;       // softmax entries per lane
    static_assert(D % DPL == 0 && 32 % DG == 0 && kTile % PS == 0, "bad decode shape");
    static_assert(DPL % EPC == 0 && VPL % 2 == 0, "bad decode shape");
};

// Butterfly that finishes NV partial sums held by each of DG lanes (lane bits
// [0, log2 DG)), halving the set each round while it can.  Lane ends with
// NF = max(1, NV/DG) totals; total j of a lane has original index
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
__device__ __forceinline__ int reduced_index(int j, int lane) {
    int idx = j, n = NV;
#pragma unroll
    for (int mask = DG / 2; mask >= 1; mask >>= 1) {
        if (n >= 2) {
            if (lane & mask) idx += n / 2;
            n /= 2;
        }
    }
    return idx;
}

template <typename E, int D, int GMAX>
__global__ void __launch_bounds__(9 * 32) paged_decode_split_kernel(const DecodeParams p) {
    using S = Shape<E, D, GMAX>;
    constexpr int EB = E::kBytes;
    const int split = blockIdx.x;
    const int b = blockIdx.y;
    const int hg = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NW = p.HC;

    const int len = __ldg(p.seq_lens + b);
    if (!len_ok(len, p)) {
        if (split == 0 && hg == 0 && threadIdx.x == 0) report(p.dev_status, WF_DEV_BAD_SEQLEN);
        return;
    }
    const int nsplit = (len + p.split_span - 1) / p.split_span;
    if (split >= nsplit) return;
    const int s0 = split * p.split_span;
    const int s1 = min(len, s0 + p.split_span);
    const int ntiles = (s1 - s0 + kTile - 1) / kTile;
    const int blk0 = s0 / p.P;
    const int nblk = (s1 - 1) / p.P - blk0 + 1;

    // ---- shared memory carve-up -------------------------------------------
    extern __shared__ __align__(128) unsigned char smem[];
    const int row_bytes = p.HC * D * EB;             // one position, this CTA's heads
    const int tile_bytes = kTile * row_bytes;
    unsigned char* sK = smem;
    unsigned char* sV = smem + (size_t)p.stages * tile_bytes;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(sV + (size_t)p.stages * tile_bytes);
    uint64_t* empty_bar = full_bar + p.stages;
    float* sS = reinterpret_cast<float*>(empty_bar + p.stages);       // [NW][kTile*GMAX]
    int32_t* sTable = reinterpret_cast<int32_t*>(sS + NW * kTile * GMAX);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NW);
        }
        fence_mbar_init();
    }
    const int32_t* table = p.block_tables + (int64_t)b * p.M + blk0;
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) sTable[i] = __ldg(table + i);
    __syncthreads();

    if (warp == NW) {
        // ===================== producer warp ================================
        const uint64_t pol = l2_policy_evict_first();
        const int64_t pool_row = (int64_t)p.H_kv * D * EB;     // bytes of one pool slot
        const int64_t head_off = (int64_t)hg * p.HC * D * EB;  // this CTA's heads in a slot
        const bool whole_rows = (p.HC == p.H_kv);              // slots contiguous across positions
        int issued = 0;
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % p.stages;
            if (t >= p.stages) {
                if (!mbar_wait(&empty_bar[st], ((t / p.stages) - 1) & 1)) {
                    if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
                    break;
                }
            }
            const int p0 = s0 + t * kTile;
            const int nvalid = min(kTile, s1 - p0);
            const int pos = p0 + lane;
            const bool valid = lane < nvalid;
            int blk = 0, off = 0;
            if (valid) {
                blk = sTable[pos / p.P - blk0];
                off = pos % p.P;
            }
            const bool ok = valid && (unsigned)blk < (unsigned)p.N;
            if (valid && !ok && (lane == 0 || off == 0)) report(p.dev_status, WF_DEV_BAD_BLOCK);
            const unsigned okmask = __ballot_sync(0xffffffffu, ok);
            const uint32_t bytes = (uint32_t)__popc(okmask) * (uint32_t)row_bytes * 2u;
            if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], bytes);
            __syncwarp();
            const bool start = ok && (!whole_rows || lane == 0 || off == 0);
            if (start) {
                const int run = whole_rows ? min(p.P - off, nvalid - lane) : 1;
                const int64_t src = ((int64_t)blk * p.P + off) * pool_row + head_off;
                bulk_g2s(sK + (size_t)st * tile_bytes + lane * row_bytes, p.k_pool + src,
                         (uint32_t)(run * row_bytes), &full_bar[st], pol);
                bulk_g2s(sV + (size_t)st * tile_bytes + lane * row_bytes, p.v_pool + src,
                         (uint32_t)(run * row_bytes), &full_bar[st], pol);
            }
            ++issued;
        }
        // Never leave with copies in flight: the last stages' fills must have landed.
        if (lane == 0) {
            const int first = issued > p.stages ? issued - p.stages : 0;
            for (int t = first; t < issued; ++t)
                mbar_wait(&full_bar[t % p.stages], (t / p.stages) & 1, 1u << 20);
        }
        return;
    }

    // ======================= consumer warps =================================
    const int dg = lane % S::DG;
    const int ps = lane / S::DG;
    const int h_local = warp;                      // KV head within the CTA
    const int hq0 = (hg * p.HC + h_local) * p.G;   // first query head of the group
    const int G = p.G;

    // q of the group, the lane's chunks, prescaled into the exp2 domain
    float2 q2[GMAX][S::CPL][S::EPC / 2];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
#pragma unroll
        for (int k = 0; k < S::CPL; ++k) {
            const int c = dg + S::DG * ((k + ps) % S::CPL);
            float f[S::EPC];
            if (g < G) {
                const char* src = static_cast<const char*>(p.q) +
                                  (((int64_t)b * p.H_q + hq0 + g) * D + c * S::EPC) * EB;
                widen_chunk<E>(*reinterpret_cast<const uint4*>(src), f);
            } else {
#pragma unroll
                for (int e = 0; e < S::EPC; ++e) f[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < S::EPC / 2; ++e)
                q2[g][k][e] = make_float2(f[2 * e] * p.scale_log2, f[2 * e + 1] * p.scale_log2);
        }
    }

    float2 acc[GMAX][S::VPL / 2];
#pragma unroll
    for (int g = 0; g < GMAX; ++g)
#pragma unroll
        for (int v = 0; v < S::VPL / 2; ++v) acc[g][v] = make_float2(0.f, 0.f);
    float m_run = -INFINITY;  // running max of head (lane % GMAX), log2 units
    float l_run = 0.f;        // this lane's share of that head's running sum
    float* sSw = sS + warp * kTile * GMAX;
    bool timed_out = false;

    for (int t = 0; t < ntiles; ++t) {
        const int st = t % p.stages;
        if (!mbar_wait(&full_bar[st], (t / p.stages) & 1)) {
            if (lane == 0) report(p.dev_status, WF_DEV_TIMEOUT);
            timed_out = true;
            break;
        }
        const int p0 = s0 + t * kTile;
        const int nvalid = min(kTile, s1 - p0);
        const unsigned char* tK = sK + (size_t)st * tile_bytes + h_local * D * EB;
        const unsigned char* tV = sV + (size_t)st * tile_bytes + h_local * D * EB;

        // ---- scores: q . K for the lane's positions, all heads of the group --
        float2 part[GMAX][S::NPL];
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int i = 0; i < S::NPL; ++i) part[g][i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < S::NPL; ++i) {
            const int pl = ps + S::PS * i;
            if (pl < nvalid) {
#pragma unroll
                for (int k = 0; k < S::CPL; ++k) {
                    const int c = dg + S::DG * ((k + ps) % S::CPL);
                    float f[S::EPC];
                    widen_chunk<E>(ld_shared_v4(tK + pl * row_bytes + c * 16), f);
#pragma unroll
                    for (int e = 0; e < S::EPC / 2; ++e) {
                        const float2 kk = make_float2(f[2 * e], f[2 * e + 1]);
#pragma unroll
                        for (int g = 0; g < GMAX; ++g) part[g][i] = ffma2(q2[g][k][e], kk, part[g][i]);
                    }
                }
            }
        }
        float v[S::NV];
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int i = 0; i < S::NPL; ++i) v[g * S::NPL + i] = part[g][i].x + part[g][i].y;
        transpose_reduce<S::NV, S::DG>(v, lane);
        constexpr int NF = S::NV / S::DG > 0 ? S::NV / S::DG : 1;
#pragma unroll
        for (int j = 0; j < NF; ++j) {
            const int idx = reduced_index<S::NV, S::DG>(j, lane);
            const int g = idx / S::NPL;
            const int pl = ps + S::PS * (idx % S::NPL);
            sSw[pl * GMAX + g] = v[j];
        }
        __syncwarp();

        // ---- online softmax (per query head, exp2 domain) --------------------
        float sv[S::NSE];
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < S::NSE; ++k) {
            const int e = lane + 32 * k;
            const bool live = e < kTile * GMAX && (e / GMAX) < nvalid;
            sv[k] = live ? sSw[e] : -INFINITY;
            mt = fmaxf(mt, sv[k]);
        }
#pragma unroll
        for (int mask = GMAX; mask < 32; mask <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, mask));
        const float m_new = fmaxf(m_run, mt);
        const float alpha = exp2f(m_run - m_new);   // 0 on the first tile
        float psum = 0.f;
#pragma unroll
        for (int k = 0; k < S::NSE; ++k) {
            const int e = lane + 32 * k;
            const float pe = exp2f(sv[k] - m_new);  // exp2(-inf) = 0 for dead entries
            psum += pe;
            if (e < kTile * GMAX) sSw[e] = pe;
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        float a[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) a[g] = __shfl_sync(0xffffffffu, alpha, g);
        __syncwarp();
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int vv = 0; vv < S::VPL / 2; ++vv) {
                acc[g][vv].x *= a[g];
                acc[g][vv].y *= a[g];
            }

        // ---- P . V ----------------------------------------------------------
        for (int pl = 0; pl < nvalid; ++pl) {
            float pw[GMAX];
            if constexpr (GMAX >= 4) {
#pragma unroll
                for (int g4 = 0; g4 < GMAX; g4 += 4) {
                    const float4 w4 = ld_shared_f4(sSw + pl * GMAX + g4);
                    pw[g4] = w4.x; pw[g4 + 1] = w4.y; pw[g4 + 2] = w4.z; pw[g4 + 3] = w4.w;
                }
            } else {
#pragma unroll
                for (int g = 0; g < GMAX; ++g) pw[g] = sSw[pl * GMAX + g];
            }
            float vf[S::VPL];
            const unsigned char* src = tV + pl * row_bytes + lane * S::VPL * EB;
            if constexpr (EB == 2) {
                if constexpr (S::VPL == 4) {
                    const uint2 u = *reinterpret_cast<const uint2*>(src);
                    const float2 x = bf16x2_to_float2(u.x), y = bf16x2_to_float2(u.y);
                    vf[0] = x.x; vf[1] = x.y; vf[2] = y.x; vf[3] = y.y;
                } else {
                    const float2 x = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(src));
                    vf[0] = x.x; vf[1] = x.y;
                }
            } else {
                if constexpr (S::VPL == 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src);
                    vf[0] = x.x; vf[1] = x.y; vf[2] = x.z; vf[3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2*>(src);
                    vf[0] = x.x; vf[1] = x.y;
                }
            }
#pragma unroll
            for (int g = 0; g < GMAX; ++g)
#pragma unroll
                for (int vv = 0; vv < S::VPL / 2; ++vv)
                    acc[g][vv] = ffma2(make_float2(pw[g], pw[g]),
                                       make_float2(vf[2 * vv], vf[2 * vv + 1]), acc[g][vv]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
    }
    if (timed_out) return;

    // ---- finish: per-head sums, then output or partial ------------------------
#pragma unroll
    for (int mask = GMAX; mask < 32; mask <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, mask);
    float l_h[GMAX], m_h[GMAX];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        l_h[g] = __shfl_sync(0xffffffffu, l_run, g);
        m_h[g] = __shfl_sync(0xffffffffu, m_run, g);
    }
    if (nsplit == 1) {
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            if (g < G) {
                const float inv = 1.f / l_h[g];
                float o[S::VPL];
#pragma unroll
                for (int vv = 0; vv < S::VPL / 2; ++vv) {
                    o[2 * vv] = acc[g][vv].x * inv;
                    o[2 * vv + 1] = acc[g][vv].y * inv;
                }
                char* dst = static_cast<char*>(p.out) +
                            (((int64_t)b * p.H_q + hq0 + g) * D + lane * S::VPL) * EB;
                store_out<E, S::VPL>(dst, o);
            }
        }
    } else {
        const int64_t base = ((int64_t)b * p.max_splits + split) * p.H_q + hq0;
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            if (g < G) {
                float* dst = p.ws_o + (base + g) * D + lane * S::VPL;
#pragma unroll
                for (int vv = 0; vv < S::VPL / 2; ++vv)
                    reinterpret_cast<float2*>(dst)[vv] = acc[g][vv];
                if (lane == 0) p.ws_ml[base + g] = make_float2(m_h[g], l_h[g]);
            }
        }
    }
}

// Merge the splits of every (sequence, query head) with more than one split:
//   out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j.
// One warp per (b, query head); lanes own D/32 output dims.
template <typename E, int D>
__global__ void __launch_bounds__(128) paged_decode_combine_kernel(const DecodeParams p) {
    constexpr int VPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.x * 4 + warp;
    const int b = blockIdx.y;
    if (hq >= p.H_q) return;
    const int len = __ldg(p.seq_lens + b);
    if (!len_ok(len, p)) return;
    const int n = (len + p.split_span - 1) / p.split_span;
    if (n <= 1) return;
    const int64_t base = (int64_t)b * p.max_splits * p.H_q + hq;  // + j * H_q
    float mx = -INFINITY;
    for (int j = lane; j < n; j += 32) mx = fmaxf(mx, p.ws_ml[base + (int64_t)j * p.H_q].x);
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
    float den = 0.f;
    for (int j = lane; j < n; j += 32) {
        const float2 ml = p.ws_ml[base + (int64_t)j * p.H_q];
        den += exp2f(ml.x - mx) * ml.y;
    }
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(0xffffffffu, den, mask);
    float o[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) o[k] = 0.f;
    for (int j = 0; j < n; ++j) {
        const int64_t row = base + (int64_t)j * p.H_q;
        const float w = exp2f(p.ws_ml[row].x - mx);
        const float* src = p.ws_o + row * D + lane * VPL;
        if constexpr (VPL == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            o[0] += w * x.x; o[1] += w * x.y; o[2] += w * x.z; o[3] += w * x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(src);
            o[0] += w * x.x; o[1] += w * x.y;
        }
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int k = 0; k < VPL; ++k) o[k] *= inv;
    char* dst = static_cast<char*>(p.out) + (((int64_t)b * p.H_q + hq) * D + lane * VPL) * E::kBytes;
    store_out<E, VPL>(dst, o);
}

int pow2_at_least(int x) {
    int r = 1;
    while (r < x) r <<= 1;
    return r;
}

template <typename E, int D, int GMAX>
cudaError_t launch_typed(const DecodeParams& p, const DecodeGeometry& g, cudaStream_t stream) {
    auto split = paged_decode_split_kernel<E, D, GMAX>;
    cudaError_t err = allow_dynamic_smem((const void*)split, g.smem_bytes);
    if (err != cudaSuccess) return err;
    dim3 grid(p.max_splits, p.B, p.H_kv / p.HC);
    split<<<grid, (p.HC + 1) * 32, g.smem_bytes, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (p.max_splits > 1) {
        dim3 cgrid((p.H_q + 3) / 4, p.B);
        paged_decode_combine_kernel<E, D><<<cgrid, 128, 0, stream>>>(p);
        err = cudaGetLastError();
    }
    return err;
}

template <typename E, int D>
cudaError_t launch_group(const DecodeParams& p, const DecodeGeometry& g, cudaStream_t stream) {
    switch (g.gmax) {
        case 1: return launch_typed<E, D, 1>(p, g, stream);
        case 2: return launch_typed<E, D, 2>(p, g, stream);
        case 4: return launch_typed<E, D, 4>(p, g, stream);
        default: return launch_typed<E, D, 8>(p, g, stream);
    }
}

}  // namespace

bool decode_geometry(const wf_pool_desc& pool, int32_t num_q_heads, DecodeGeometry* g) {
    if (pool.num_kv_heads < 1 || num_q_heads % pool.num_kv_heads != 0) return false;
    const int G = num_q_heads / pool.num_kv_heads;
    if (G < 1 || G > 8) return false;
    if (pool.head_dim != 64 && pool.head_dim != 128) return false;
    int hc = 1;
    for (int c = 8; c >= 1; --c)
        if (pool.num_kv_heads % c == 0) { hc = c; break; }
    const int eb = dtype_bytes(pool.dtype);
    const int row_bytes = hc * pool.head_dim * eb;
    const int stage_bytes = 2 * kTile * row_bytes;  // K + V
    int stages = (192 * 1024) / stage_bytes;
    if (stages < 2) stages = 2;
    if (stages > 6) stages = 6;
    const int gmax = pow2_at_least(G);
    const int span = 128;
    const int table_ints = span / 1 + 2;  // P = 1 worst case: one entry per position
    g->split_span = span;
    g->tile = kTile;
    g->stages = stages;
    g->consumer_warps = hc;
    g->heads_per_warp = 1;
    g->gmax = gmax;
    g->smem_bytes = stages * stage_bytes + 2 * stages * 8 + hc * kTile * gmax * 4 + table_ints * 4;
    return true;
}

size_t decode_workspace_bytes(int32_t B, int32_t num_q_heads, int32_t max_seq_len,
                              const wf_pool_desc& pool) {
    DecodeGeometry g;
    if (B < 0 || max_seq_len < 1 || !decode_geometry(pool, num_q_heads, &g)) return 0;
    const int64_t max_splits = (max_seq_len + g.split_span - 1) / g.split_span;
    const int64_t rows = (int64_t)B * max_splits * num_q_heads;
    const int64_t o_bytes = rows * pool.head_dim * 4;
    const int64_t ml_bytes = rows * 8;
    return (size_t)(((o_bytes + 255) / 256) * 256 + ml_bytes + 256);
}

cudaError_t launch_paged_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                void* workspace, uint32_t* dev_status, cudaStream_t stream) {
    DecodeGeometry g;
    if (!decode_geometry(pool, num_q_heads, &g)) return cudaErrorInvalidValue;
    DecodeParams p;
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
    p.HC = g.consumer_warps;
    p.split_span = g.split_span;
    p.max_splits = (max_seq_len + g.split_span - 1) / g.split_span;
    p.stages = g.stages;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int64_t rows = (int64_t)B * p.max_splits * num_q_heads;
    const int64_t o_bytes = ((rows * pool.head_dim * 4 + 255) / 256) * 256;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + o_bytes);
    if (pool.dtype == WF_DTYPE_F32) {
        return pool.head_dim == 64 ? launch_group<F32, 64>(p, g, stream)
                                   : launch_group<F32, 128>(p, g, stream);
    }
    return pool.head_dim == 64 ? launch_group<BF16, 64>(p, g, stream)
                               : launch_group<BF16, 128>(p, g, stream);
}

}  // namespace wf
