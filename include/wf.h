/*
 * wf.h -- C ABI of libwf: attention over a paged KV cache on GB300 (sm_103a).
 *
 * Three calls make up one attention step of an LLM serving engine that keeps
 * its KV cache in fixed-size blocks:
 *
 *   wf_reshape_and_cache  write this step's new K/V rows into the block pool
 *   wf_paged_decode       one query per sequence over its whole cached context
 *   wf_paged_prefill      causal attention of new tokens over prefix + themselves
 *
 * Sources (page title, section):
 *   weft, "Shapes and symbols": B, H_q, H_kv (H_q / H_kv = GQA group), D, N, P, T_total.
 *   weft, "Cache layouts": per-layer paged view [N, P, H_kv, D]; write = scatter
 *     via slot_mapping; read = gather by block_table; blocks handed out per request.
 *   ember, "The core idea, in one picture": position p of a sequence lives in
 *     block block_table[p // P] at offset p % P.
 *   tiny-vllm-py, "KV Cache": the cache holds RoPE-rotated K and plain V; at
 *     decode the new token attends to every earlier position and to itself; prefill
 *     attention is causal ("Mistakes I made in Initial Implementation").
 *
 * Conventions for every call
 *   - Every pointer argument is DEVICE memory owned by the caller, dense and
 *     row-major as documented, 16-byte aligned (the optional per-head fp8 scale
 *     arrays inside wf_pool_desc are the one exception: small host arrays).  The library allocates nothing,
 *     keeps no per-call state, and never synchronises the stream (except
 *     wf_device_status_fetch).  Calls are asynchronous and stream-ordered.
 *   - q, k, v, pools and outputs all use the pool's dtype (float32 or bfloat16);
 *     arithmetic is float32.  Outputs are rounded to nearest-even.
 *   - Argument errors are returned synchronously, before anything is launched.
 *   - Values that only the device can see (slots, block ids, sequence lengths)
 *     are bounds-checked by the kernels: a bad one is skipped (never read or
 *     written out of bounds) and a bit is OR-ed into *dev_status (a device
 *     uint32_t; may be NULL to not record).  Read it with wf_device_status_fetch.
 *   - Outputs never alias inputs.  K and V pools are separate buffers.
 */
#ifndef WF_H
#define WF_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum wf_status {
    WF_OK = 0,
    WF_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, H_q % H_kv != 0 */
    WF_ERR_UNSUPPORTED = 2,  /* dtype / head_dim / group size this build does not handle     */
    WF_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the *_workspace_size value */
    WF_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed                  */
    WF_ERR_NO_BLOCKS = 5     /* block manager: not enough free blocks (nothing was changed)  */
} wf_status;

typedef enum wf_dtype {
    WF_DTYPE_F32 = 0,
    WF_DTYPE_BF16 = 1,
    /* fp8 e4m3 pools (OCP E4M3: 4 exponent bits, bias 7, 3 mantissa bits, largest
     * 448, no infinities).  q, new k/v rows and outputs stay bfloat16; the pools
     * hold codes that stand for k_scale * value (V: v_scale * value).
     * (ember, "Deliberately out of scope": paged KV quantization (fp8/int8)) */
    WF_DTYPE_FP8_E4M3 = 2
} wf_dtype;

/* Bits the kernels OR into *dev_status. */
#define WF_DEV_BAD_SLOT    0x1u  /* slot_mapping[t] >= N*P: token t not written              */
#define WF_DEV_BAD_BLOCK   0x2u  /* block id outside [0, N): that block's rows were skipped
                                    (fp8 pools at D = 64: the 32 positions of its tile)       */
#define WF_DEV_BAD_SEQLEN  0x4u  /* seq_lens[b] < 1, > max_seq_len, > M*P, or < q_len:
                                    sequence b was skipped and its output left unwritten    */
#define WF_DEV_TIMEOUT     0x8u  /* a wait gave up: an internal pipeline wait (should never
                                    happen), or a decode worker idle past its limit          */
#define WF_DEV_BAD_TASK    0x10u /* decode worker: a task record out of range (skipped)     */

/* One layer's pool geometry.  k_pool and v_pool are each [N, P, H_kv, D]. */
typedef struct wf_pool_desc {
    int32_t num_blocks;    /* N: blocks in the pool                       */
    int32_t block_size;    /* P: tokens per block, 1 .. 1024              */
    int32_t num_kv_heads;  /* H_kv                                        */
    int32_t head_dim;      /* D: 64 or 128                                */
    int32_t dtype;         /* wf_dtype of the pools; q, k, v and outputs
                              have it too, except that fp8 pools take
                              bfloat16 q, k, v and give bfloat16 outputs  */
    float k_scale;         /* fp8 pools: a K code c stands for k_scale *
                              value(c); the scatter stores
                              e4m3(float(k) * (1.0f / k_scale)), rounded
                              to nearest even and saturated at +-448.
                              Must be finite and > 0 for fp8; ignored
                              otherwise.                                  */
    float v_scale;         /* the same for V                              */
    const float* k_head_scales; /* fp8 pools, optional: NULL, or host memory
                              holding num_kv_heads scales (num_kv_heads <= 64),
                              one per KV head, read during the call and not
                              kept.  When set, codes of head h stand for
                              k_head_scales[h] * value(c) and k_scale is not
                              used.  Each must be finite and > 0.          */
    const float* v_head_scales; /* the same for V                         */
} wf_pool_desc;

/*
 * wf_reshape_and_cache -- scatter new K/V rows into the block pool.
 * (weft, "Cache layouts": "write: scatter via slot_mapping")
 *
 *   k, v          [T, H_kv, D]   rows of this step's T new tokens
 *   k_pool,v_pool [N, P, H_kv, D] updated in place
 *   slot_mapping  [T] int64: token t goes to block slot/P, offset slot%P.
 *                 A negative slot means "padding token": nothing is written.
 *                 Two tokens with the same slot: one of them wins (unspecified).
 *   num_tokens    T >= 0 (0 is a no-op)
 * Pure byte copy: pool bytes equal the input bytes exactly.  fp8 pools: k, v are
 * bfloat16 and each element of KV head h is stored as the e4m3 code of
 * float(x) * (1.0f / scale_h) (scale_h = k_head_scales[h] if given, else
 * k_scale; likewise for V), rounded to nearest even, saturated at +-448, NaN kept.
 * Slots >= N*P are skipped and flagged WF_DEV_BAD_SLOT.
 */
wf_status wf_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               wf_pool_desc pool, uint32_t* dev_status, cudaStream_t stream);

/*
 * wf_copy_blocks -- copy-on-write block copy for prefix sharing.
 * (tiny-vllm-py, "Prefix Sharing": requests with a common prefix share its blocks,
 *  and a shared, partly filled block is copied before a request appends to it;
 *  ember, "Deliberately out of scope": copy-on-write block tables)
 *
 *   k_pool, v_pool  [N, P, H_kv, D], 16-byte aligned, modified in place
 *   block_pairs     [num_pairs, 2] int32 device array of (src, dst) block ids:
 *                   block dst of both pools becomes a byte copy of block src.
 *   Destinations must be distinct and no block may be both a source and a
 *   destination (the copies run in parallel); otherwise the result is undefined.
 *   Ids outside [0, N) are skipped and flagged WF_DEV_BAD_BLOCK in *dev_status.
 * num_pairs == 0 is a no-op.  Any pool dtype.
 */
wf_status wf_copy_blocks(void* k_pool, void* v_pool, const int32_t* block_pairs, int32_t num_pairs,
                         wf_pool_desc pool, uint32_t* dev_status, cudaStream_t stream);

/*
 * Bytes of caller-allocated device workspace wf_paged_decode needs for a batch
 * of at most B sequences of at most max_seq_len tokens.  Depends only on its
 * arguments; 0 if they are invalid.
 */
size_t wf_paged_decode_workspace_size(int32_t B, int32_t num_q_heads, int32_t max_seq_len,
                                      wf_pool_desc pool);

/*
 * wf_paged_decode -- one query token per sequence against its paged context.
 * (ember, "The core idea"; tiny-vllm-py, "KV Cache": decode is not causal over
 *  the cache and includes the just-written token)
 *
 *   out          [B, H_q, D]  out[b,g] = softmax_p(scale * q[b,g].K_p) V_p
 *   q            [B, H_q, D]
 *   k_pool, v_pool [N, P, H_kv, D] (already holding this step's new token)
 *   block_tables [B, max_blocks_per_seq] int32, row-major.  Only the first
 *                ceil(seq_lens[b] / P) entries of row b are read.
 *   seq_lens     [B] int32: positions 0 .. seq_lens[b]-1 of sequence b are attended.
 *                Must satisfy 1 <= seq_lens[b] <= max_seq_len <= max_blocks_per_seq*P.
 *   num_q_heads  H_q; query head g reads KV head g / (H_q / H_kv).  H_q/H_kv <= 8.
 *   scale        softmax scale (normally 1/sqrt(D))
 *   workspace    device scratch of >= wf_paged_decode_workspace_size(B, H_q,
 *                max_seq_len, pool) bytes, 16-byte aligned; contents need no
 *                initialisation and are clobbered.  Calls that overlap in time
 *                must not share a workspace.
 * Launches a split-K kernel and, when any sequence spans more than one split, a
 * combine kernel.  The split boundaries depend only on the pool geometry, so a
 * sequence's output does not depend on the rest of the batch.
 * fp8 e4m3 pools: q and out are bfloat16; K_p and V_p are k_scale_h * value and
 * v_scale_h * value of the stored codes (h the KV head; per-pool or per-head
 * scales).  Every geometry of the bf16 path is supported.  For H_kv = 8, D = 128,
 * P a multiple of 16, H_q / H_kv in {2, 4} and N*P <= 2^31 - 1 both products run
 * on the tensor cores on the codes (e4m3 x e4m3 -> fp32): q is split into two e4m3
 * parts whose sum is q exactly, and the softmax weights into two parts (about 8
 * significant bits).  Other shapes run on the CUDA cores, which widen the codes to
 * fp32 exactly and keep fp32 weights.
 */
wf_status wf_paged_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                          int32_t num_q_heads, float scale, wf_pool_desc pool,
                          void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                          cudaStream_t stream);

/*
 * wf_paged_prefill -- causal varlen attention of new tokens over the pool.
 * (tiny-vllm-py, "KV Cache": prefill is causal; "Dense vs. Ragged batching":
 *  requests are packed back to back with per-request offsets, no padding)
 *
 *   out        [T_total, H_q, D]
 *   q          [T_total, H_q, D]: request b owns rows cu_q_lens[b] .. cu_q_lens[b+1]-1
 *   cu_q_lens  [B+1] int32, cu_q_lens[0] = 0, non-decreasing, cu_q_lens[B] = T_total
 *   seq_lens   [B] int32: tokens of request b in the pool INCLUDING its n_b new ones
 *              (already written by wf_reshape_and_cache).  With c_b = seq_lens[b] - n_b,
 *              query row i of request b attends to positions 0 .. c_b + i.
 *   max_q_len  >= every n_b (sizes the launch)
 * bfloat16 only; QK^T and PV run on the tensor cores (bf16 operands, fp32
 * accumulation in tensor memory); the softmax weights are rounded to bf16 for PV.
 * Schedule (no effect on the result: the same bytes either way): a batch of at
 * most 1024 requests and 4096 (request, query block) pairs -- a query block is
 * 256 (token, query head) rows of one KV head -- runs as one persistent grid, one
 * CTA per SM, each taking its share of the blocks longest first; a larger batch
 * runs one CTA per query block.
 */
wf_status wf_paged_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t B,
                           int32_t total_q, int32_t max_q_len, int32_t max_seq_len,
                           int32_t num_q_heads, float scale, wf_pool_desc pool,
                           uint32_t* dev_status, cudaStream_t stream);

/*
 * wf_paged_prefill_decode -- the attention of a mixed continuous-batching step:
 * wf_paged_prefill of the step's new requests and wf_paged_decode of its running
 * sequences, over one pool, in one call.
 * (tiny-vllm-py, "Inference Server Flow": a step mixes prefill and decode work;
 *  ember, "Deliberately out of scope": a proper prefill/decode mix per step)
 *
 * The pf_* arguments are those of wf_paged_prefill, the dec_* ones those of
 * wf_paged_decode (its workspace too), and both share the pools, num_q_heads,
 * scale and pool descriptor; every rule of the two calls applies.  The outputs
 * are those of the two calls (the prefill and the decode outputs must not
 * overlap).  For bf16 pools whose prefill and decode both run on the tensor cores,
 * H_kv a multiple of 8 and GQA groups of 1, 2 or 4, both run in one grid: its first
 * CTAs are the prefill's, the rest are persistent decode CTAs that take decode
 * work from a queue as the prefill's CTAs finish, so the decode fills the SMs the
 * prefill's tail leaves idle.  Other shapes run the two calls one after the other.
 */
wf_status wf_paged_prefill_decode(void* pf_out, const void* pf_q, const int32_t* pf_block_tables,
                                  int32_t pf_max_blocks_per_seq, const int32_t* pf_seq_lens,
                                  const int32_t* cu_q_lens, int32_t pf_B, int32_t total_q, int32_t max_q_len,
                                  int32_t pf_max_seq_len, void* dec_out, const void* dec_q,
                                  const int32_t* dec_block_tables, int32_t dec_max_blocks_per_seq,
                                  const int32_t* dec_seq_lens, int32_t dec_B, int32_t dec_max_seq_len,
                                  const void* k_pool, const void* v_pool, int32_t num_q_heads, float scale,
                                  wf_pool_desc pool, void* workspace, size_t workspace_bytes,
                                  uint32_t* dev_status, cudaStream_t stream);
/* 1 when wf_paged_prefill_decode runs both in one grid for this geometry, else 0
 * (host-only, no CUDA call). */
int wf_paged_prefill_decode_fused(wf_pool_desc pool, int32_t num_q_heads);

/*
 * Size of the fixed device array wf_paged_decode_static_scratch uses as its
 * workspace (32 MiB).  A device holds it from the first
 * wf_paged_decode_static_scratch call on that device until the process exits.
 */
#define WF_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * wf_paged_decode_static_scratch -- wf_paged_decode for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a library
 * convenience, not part of the method.
 *
 * Some callers cannot call cudaMalloc when they run attention: an allocator or
 * memory manager that must not re-enter itself, a plugin whose host framework
 * owns every device allocation, or a runtime that forbids allocation after
 * start-up to keep its memory use fixed.  This call takes the same arguments as
 * wf_paged_decode except the workspace: it uses a file-scope device array of
 * WF_STATIC_SCRATCH_BYTES instead, and it allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library call).
 *
 *   - Arguments are checked as wf_paged_decode checks them, first: an invalid
 *     one returns that call's status.  A valid batch that needs more than
 *     WF_STATIC_SCRATCH_BYTES (compare wf_paged_decode_workspace_size(B,
 *     num_q_heads, max_seq_len, pool)) returns WF_ERR_WORKSPACE.  Either way
 *     nothing is launched.
 *   - The first call on a device looks up the array's device address with that
 *     device current (cudaGetSymbolAddress) and caches it.  Under CUDA's default
 *     lazy module loading that lookup is also what maps the array on the device,
 *     so the device's memory use grows by WF_STATIC_SCRATCH_BYTES at that first
 *     call and not before.  Make that first call before any stream capture.
 *   - A device reset (cudaDeviceReset, or the primary context destroyed and
 *     created again) invalidates the cached address: do not call this entry
 *     point on a device after resetting it.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls that overlap in
 *     time on the same device, e.g. on two streams, race on it and give wrong
 *     results: serialise them.
 */
wf_status wf_paged_decode_static_scratch(void* out, const void* q, const void* k_pool,
                                         const void* v_pool, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                         int32_t B, int32_t max_seq_len, int32_t num_q_heads,
                                         float scale, wf_pool_desc pool, uint32_t* dev_status,
                                         cudaStream_t stream);

/*
 * wf_decode_worker -- a persistent decode worker that takes tasks while it runs.
 * (Awesome System Papers wiki, WEAVER summary, "核心方法": a receiver kernel spins
 *  on a task counter, runs the attention it finds and bumps a completion counter,
 *  so no host launch sits between a request and its attention.)
 *
 * The worker grid (num_workers CTAs of 256 threads) is launched once on `stream`.
 * A feeder outside it -- typically a host thread issuing cudaMemcpyAsync on
 * another non-blocking stream, so the copy engine writes while the worker runs --
 * appends task records to `tasks` and then raises mailbox->posted.  Each CTA
 * claims the next task index (one atomic increment of mailbox->claimed), waits
 * until that task is posted, decodes it and, once its output is written,
 * increments mailbox->done.
 *
 *   tasks      device array of task_capacity records; task t lives in tasks[t].
 *              Write a record before raising `posted` past it (e.g. its copy
 *              earlier on the same stream as the copy of `posted`).
 *   mailbox    device memory (16-byte aligned):
 *                posted   feeder: tasks 0 .. posted-1 are readable (<= task_capacity)
 *                stop     feeder: nonzero = leave once every posted task is claimed;
 *                         write it after the last `posted`
 *                claimed  worker: next task to claim
 *                done     worker: tasks whose outputs are written
 *              The call zeroes `claimed` and `done` on `stream` before the worker
 *              starts; `posted` and `stop` are the feeder's (zero them before).
 *   task       {seq_len, table_row, q_row, out_row}: out[out_row] = decode of
 *              q[q_row] over positions 0 .. seq_len-1 mapped by
 *              block_tables[table_row] (the computation of wf_paged_decode for
 *              one sequence).  Records with an index out of range are skipped
 *              and flagged WF_DEV_BAD_TASK (they still count as done).
 *   out, q     [num_rows, H_q, D] of the pool dtype (float32 or bfloat16 pools)
 *   block_tables [num_table_rows, max_blocks_per_seq] int32
 *   idle_timeout_ns  longest time a CTA waits for its claimed task; past it the
 *              CTA sets WF_DEV_TIMEOUT in *dev_status and returns, leaving its
 *              task unrun.  While a CTA waits it has no copy or tensor-core
 *              operation in flight.
 * The worker holds num_workers CTAs until it stops or times out: anything that
 * waits for the whole device (cudaDeviceSynchronize, cudaMalloc/cudaFree in many
 * allocators) blocks until then, so a feeder must not call such things.
 * fp8 pools: WF_ERR_UNSUPPORTED.
 */
typedef struct wf_worker_mailbox {
    uint32_t posted;
    uint32_t stop;
    uint32_t claimed;
    uint32_t done;
} wf_worker_mailbox;

typedef struct wf_decode_task {
    int32_t seq_len;
    int32_t table_row;
    int32_t q_row;
    int32_t out_row;
} wf_decode_task;

wf_status wf_decode_worker(void* out, const void* q, int32_t num_rows, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, int32_t num_table_rows, int32_t max_blocks_per_seq,
                           int32_t num_q_heads, float scale, wf_pool_desc pool, const wf_decode_task* tasks,
                           int32_t task_capacity, wf_worker_mailbox* mailbox, int32_t num_workers,
                           uint64_t idle_timeout_ns, uint32_t* dev_status, cudaStream_t stream);

/*
 * Which kernel wf_paged_decode / wf_paged_prefill runs for a pool geometry and
 * query-head count (host-only, no CUDA call; for tests and tooling).  Returns a
 * wf_kernel value; WF_KERNEL_NONE when the geometry is invalid or unsupported.
 */
typedef enum wf_kernel {
    WF_KERNEL_NONE = 0,
    WF_KERNEL_CUDA_CORES = 1,            /* decode: split-K kernel on the CUDA cores          */
    WF_KERNEL_TENSOR_CORES = 2,          /* decode: split-K tcgen05 kernel (bf16, or fp8 codes);
                                            prefill: warp-specialised pipelined tcgen05 kernel */
    WF_KERNEL_TENSOR_CORES_SIMPLE = 3    /* prefill: single-stage tcgen05 kernel (any P)       */
} wf_kernel;
int wf_paged_decode_kernel(wf_pool_desc pool, int32_t num_q_heads);
int wf_paged_prefill_kernel(wf_pool_desc pool, int32_t num_q_heads);
/*
 * 1 when wf_paged_prefill runs a batch of B requests of at most max_q_len new tokens
 * as the persistent grid (WF_KERNEL_TENSOR_CORES geometries within the work list's
 * limits: B <= 1024 and B * ceil(max_q_len / query block) <= 4096), 0 when it runs one
 * CTA per query block (or the geometry is not WF_KERNEL_TENSOR_CORES).  Host-only.
 */
int wf_paged_prefill_persistent(wf_pool_desc pool, int32_t num_q_heads, int32_t B, int32_t max_q_len);

/*
 * Wait for `stream`, copy *dev_status to *host_status and, if clear != 0, reset
 * it to zero.  The only call that synchronises.
 */
wf_status wf_device_status_fetch(uint32_t* dev_status, uint32_t* host_status, int clear,
                                 cudaStream_t stream);

/* Static text for a status code. */
const char* wf_status_string(wf_status s);

/* ABI version of this header (major * 100 + minor). */
int wf_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* WF_H */
