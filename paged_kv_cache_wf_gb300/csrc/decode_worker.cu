// decode_worker.cu -- a persistent decode worker that takes its tasks while it
// runs: GPU-driven control flow on one GPU.
//
// The Weaver summary (Awesome System Papers wiki, WEAVER, "核心方法") describes a
// receiving GPU whose kernel spins on a task counter, runs the attention work it
// finds there and bumps a completion counter, so no host launch sits between a
// request and its attention.  This file is the single-GPU form of that loop:
//
//   * the worker grid is launched once; a feeder outside it (a host thread
//     copying through the copy engine on another stream, or anything else that
//     writes device memory) appends task records to an array and then raises
//     `posted` in a mailbox in device memory;
//   * each CTA claims the next task index with one atomic increment, waits until
//     the task is posted (polling with acquire loads and a nanosleep back-off),
//     reads the record, decodes that one sequence against the paged pool, writes
//     its output and bumps `done`;
//   * `stop` ends the loop once every posted task has been claimed;
//   * every wait is bounded by a per-launch idle limit (globaltimer nanoseconds,
//     with a poll-count backstop): a CTA that waits longer reports WF_DEV_TIMEOUT
//     and returns.  Nothing is in flight while a CTA waits (no bulk copy, no MMA:
//     the task body uses plain loads), so a timed-out CTA leaves cleanly.
//
// What a task computes is the decode of the attention pages (ember, "The core
// idea": position p of the sequence is row block_table[p / P], offset p % P of
// the pool; tiny-vllm-py, "KV Cache": the query attends to every cached position
// including its own; weft, "Shapes and symbols": query head g reads KV head
// g / (H_q / H_kv)).  One CTA decodes the whole sequence: warp w takes KV heads
// w, w + 8, ...; inside a warp, groups of lanes own one position at a time (one
// 16-byte load of K and of V per lane), keep an online softmax per query head of
// the group in fp32, and are merged by shuffles at the end.  The loads of four
// positions are issued before any of them is used.
#include <type_traits>

#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kWorkerThreads = 256;
constexpr int kWorkerWarps = kWorkerThreads / 32;

struct WorkerParams {
    void* out;
    const void* q;
    const char* k_pool;
    const char* v_pool;
    const int32_t* block_tables;
    const wf_decode_task* tasks;
    wf_worker_mailbox* mb;
    uint32_t* dev_status;
    int32_t rows, table_rows, M, H_q, H_kv, G, N, P, capacity;
    float scale_log2;
    uint64_t idle_timeout_ns;
};

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A task record as it is now in memory (not from a cache line read earlier).
__device__ __forceinline__ wf_decode_task ld_task(const wf_decode_task* p) {
    int4 r;
    asm volatile("ld.relaxed.gpu.global.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    wf_decode_task t;
    t.seq_len = r.x;
    t.table_row = r.y;
    t.q_row = r.z;
    t.out_row = r.w;
    return t;
}

// Claim the next task and wait for it.  Returns the task index, -1 when the
// feeder has stopped with nothing left for this claim, -2 on timeout.
__device__ int64_t claim_task(const WorkerParams& p) {
    const uint32_t t = atomicAdd(&p.mb->claimed, 1u);
    if ((int64_t)t >= (int64_t)p.capacity) return -1;   // past the task array: nothing can come
    const uint64_t t0 = global_ns();
    // backstop in case the timer stalls: each poll sleeps >= ~32 ns
    const uint64_t max_polls = (p.idle_timeout_ns >> 5) + 4096;
    for (uint64_t polls = 0;; ++polls) {
        if (ld_acquire_u32(&p.mb->posted) > t) return (int64_t)t;
        if (ld_acquire_u32(&p.mb->stop) != 0u) {
            // the feeder raises `stop` after its last `posted`: read that again
            return ld_acquire_u32(&p.mb->posted) > t ? (int64_t)t : -1;
        }
        if (global_ns() - t0 > p.idle_timeout_ns || polls > max_polls) return -2;
        __nanosleep(256);
    }
}

template <typename E, int D, int GMAX>
__global__ void __launch_bounds__(kWorkerThreads, 1) decode_worker_kernel(const WorkerParams p) {
    constexpr int EB = E::kBytes;
    constexpr int EPL = 16 / EB;     // elements of a row per lane (one 16-byte load)
    constexpr int LPR = D / EPL;     // lanes per row
    constexpr int RPW = 32 / LPR;    // rows (positions) a warp holds at once
    constexpr int U = 4;             // positions per lane group whose loads go out together
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "worker row layout");
    __shared__ long long s_task;
    __shared__ wf_decode_task s_rec;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane / LPR;       // which row of the warp this lane works on
    const int d0 = (lane % LPR) * EPL;
    const int64_t slot_bytes = (int64_t)p.H_kv * D * EB;
    using QE = typename std::conditional<std::is_same<E, F32>::value, F32, BF16>::type;

    for (;;) {
        if (threadIdx.x == 0) {
            const int64_t t = claim_task(p);
            if (t == -2) report(p.dev_status, WF_DEV_TIMEOUT);
            if (t >= 0) s_rec = ld_task(p.tasks + t);
            s_task = t;
        }
        __syncthreads();
        const int64_t t = s_task;
        if (t < 0) break;
        const wf_decode_task rec = s_rec;
        const bool ok = rec.seq_len >= 1 && (int64_t)rec.seq_len <= (int64_t)p.M * p.P && rec.table_row >= 0 &&
                        rec.table_row < p.table_rows && rec.q_row >= 0 && rec.q_row < p.rows && rec.out_row >= 0 &&
                        rec.out_row < p.rows;
        if (!ok) {
            if (threadIdx.x == 0) report(p.dev_status, WF_DEV_BAD_TASK);
        } else {
            const int L = rec.seq_len;
            const int32_t* bt = p.block_tables + (int64_t)rec.table_row * p.M;
            for (int h = warp; h < p.H_kv; h += kWorkerWarps) {
                float qv[GMAX][EPL];
                float m[GMAX], l[GMAX], acc[GMAX][EPL];
#pragma unroll
                for (int g = 0; g < GMAX; ++g) {
                    m[g] = -INFINITY;
                    l[g] = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        acc[g][e] = 0.f;
                        qv[g][e] = 0.f;
                    }
                    if (g < p.G) {
                        const int64_t qi = ((int64_t)rec.q_row * p.H_q + h * p.G + g) * D + d0;
                        const char* src = static_cast<const char*>(p.q) + qi * QE::kBytes;
                        if constexpr (std::is_same<QE, F32>::value) {
                            const uint4 c = *reinterpret_cast<const uint4*>(src);
                            float f[4];
                            widen_chunk<F32>(c, f);
#pragma unroll
                            for (int e = 0; e < EPL; ++e) qv[g][e] = f[e] * p.scale_log2;
                        } else {
                            const uint4 c = *reinterpret_cast<const uint4*>(src);
                            float f[8];
                            widen_chunk<BF16>(c, f);
#pragma unroll
                            for (int e = 0; e < EPL; ++e) qv[g][e] = f[e] * p.scale_log2;
                        }
                    }
                }
                // the loop bound is the same for every lane of the warp (the shuffles
                // below take the whole warp); each lane group masks its own positions
                for (int base = 0; base < L; base += RPW * U) {
                    uint4 kc[U], vc[U];
                    bool live[U];
#pragma unroll
                    for (int j = 0; j < U; ++j) {
                        const int pos = base + j * RPW + rg;
                        live[j] = pos < L;
                        kc[j] = make_uint4(0u, 0u, 0u, 0u);
                        vc[j] = kc[j];
                        if (live[j]) {
                            const int blk = __ldg(bt + pos / p.P);
                            if ((unsigned)blk < (unsigned)p.N) {
                                const int64_t off = ((int64_t)blk * p.P + pos % p.P) * slot_bytes +
                                                    (int64_t)(h * D + d0) * EB;
                                kc[j] = ld_global_stream(p.k_pool + off);
                                vc[j] = ld_global_stream(p.v_pool + off);
                            } else {
                                live[j] = false;
                                report(p.dev_status, WF_DEV_BAD_BLOCK);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < U; ++j) {
                        float kf[EPL], vf[EPL];
                        widen_chunk<E>(kc[j], kf);
                        widen_chunk<E>(vc[j], vf);
#pragma unroll
                        for (int g = 0; g < GMAX; ++g) {
                            float s = 0.f;
#pragma unroll
                            for (int e = 0; e < EPL; ++e) s = fmaf(qv[g][e], kf[e], s);
#pragma unroll
                            for (int mask = 1; mask < LPR; mask <<= 1) s += __shfl_xor_sync(0xffffffffu, s, mask);
                            if (live[j] && g < p.G) {
                                const float mn = fmaxf(m[g], s);
                                const float a = exp2f(m[g] - mn);   // 0 while m is -inf
                                const float w = exp2f(s - mn);
                                l[g] = l[g] * a + w;
#pragma unroll
                                for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(w, vf[e], acc[g][e] * a);
                                m[g] = mn;
                            }
                        }
                    }
                }
                // merge the warp's rows (lanes that hold the same dims)
#pragma unroll
                for (int mask = LPR; mask < 32; mask <<= 1) {
#pragma unroll
                    for (int g = 0; g < GMAX; ++g) {
                        const float mo = __shfl_xor_sync(0xffffffffu, m[g], mask);
                        const float lo = __shfl_xor_sync(0xffffffffu, l[g], mask);
                        const float mn = fmaxf(m[g], mo);
                        const float a = mn == -INFINITY ? 0.f : exp2f(m[g] - mn);
                        const float b = mn == -INFINITY ? 0.f : exp2f(mo - mn);
                        l[g] = l[g] * a + lo * b;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            const float ao = __shfl_xor_sync(0xffffffffu, acc[g][e], mask);
                            acc[g][e] = acc[g][e] * a + ao * b;
                        }
                        m[g] = mn;
                    }
                }
                if (rg == 0) {
#pragma unroll
                    for (int g = 0; g < GMAX; ++g) {
                        if (g >= p.G) continue;
                        const float inv = 1.f / l[g];
                        float o[EPL];
#pragma unroll
                        for (int e = 0; e < EPL; ++e) o[e] = acc[g][e] * inv;
                        const int64_t oi = ((int64_t)rec.out_row * p.H_q + h * p.G + g) * D + d0;
                        char* dst = static_cast<char*>(p.out) + oi * QE::kBytes;
#pragma unroll
                        for (int e = 0; e < EPL; e += 4) store_out<QE, 4>(dst + e * QE::kBytes, o + e);
                    }
                }
            }
        }
        // every output of the task is written before it counts as done
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&p.mb->done, 1u);
        }
    }
}

template <typename E, int D>
cudaError_t launch_worker_g(const WorkerParams& p, int gmax, int workers, cudaStream_t stream) {
    switch (gmax) {
        case 1: decode_worker_kernel<E, D, 1><<<workers, kWorkerThreads, 0, stream>>>(p); break;
        case 2: decode_worker_kernel<E, D, 2><<<workers, kWorkerThreads, 0, stream>>>(p); break;
        case 4: decode_worker_kernel<E, D, 4><<<workers, kWorkerThreads, 0, stream>>>(p); break;
        default: decode_worker_kernel<E, D, 8><<<workers, kWorkerThreads, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_worker(void* out, const void* q, int32_t num_rows, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, int32_t num_table_rows, int32_t max_blocks_per_seq,
                                 int32_t num_q_heads, float scale, const wf_pool_desc& pool,
                                 const wf_decode_task* tasks, int32_t task_capacity, wf_worker_mailbox* mailbox,
                                 int32_t num_workers, uint64_t idle_timeout_ns, uint32_t* dev_status,
                                 cudaStream_t stream) {
    WorkerParams p;
    p.out = out;
    p.q = q;
    p.k_pool = static_cast<const char*>(k_pool);
    p.v_pool = static_cast<const char*>(v_pool);
    p.block_tables = block_tables;
    p.tasks = tasks;
    p.mb = mailbox;
    p.dev_status = dev_status;
    p.rows = num_rows;
    p.table_rows = num_table_rows;
    p.M = max_blocks_per_seq;
    p.H_q = num_q_heads;
    p.H_kv = pool.num_kv_heads;
    p.G = num_q_heads / pool.num_kv_heads;
    p.N = pool.num_blocks;
    p.P = pool.block_size;
    p.capacity = task_capacity;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.idle_timeout_ns = idle_timeout_ns;
    // the worker's own counters start at zero; `posted` and `stop` belong to the feeder
    cudaError_t err = cudaMemsetAsync(&mailbox->claimed, 0, 2 * sizeof(uint32_t), stream);
    if (err != cudaSuccess) return err;
    int gmax = 1;
    while (gmax < p.G) gmax *= 2;
    if (pool.dtype == WF_DTYPE_F32)
        return pool.head_dim == 64 ? launch_worker_g<F32, 64>(p, gmax, num_workers, stream)
                                   : launch_worker_g<F32, 128>(p, gmax, num_workers, stream);
    return pool.head_dim == 64 ? launch_worker_g<BF16, 64>(p, gmax, num_workers, stream)
                               : launch_worker_g<BF16, 128>(p, gmax, num_workers, stream);
}

}  // namespace wf
