// paged_decode_static.cu -- wf_paged_decode for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) at the
// point where they run attention: code inside a custom allocator or memory
// manager that must not re-enter itself, plugins whose host framework owns all
// device allocations, and runtimes that forbid allocation after start-up so that
// memory use stays fixed.  They still own q, the pools and the output; what they
// cannot provide is the decode workspace.  This file gives them one entry point
// whose scratch lives in a fixed, file-scope device array instead.
//
// The array is WF_STATIC_SCRATCH_BYTES large.  Under CUDA's default lazy module
// loading it is mapped on a device when this file's module is first loaded
// there, which the first call on that device does (cudaGetSymbolAddress), and it
// stays until the process exits or the device's context is destroyed.  Host code
// cannot use the array's name as a device address (in host code it names a
// host-side stand-in), so the first call on each device looks up the real
// address with cudaGetSymbolAddress, with that device current, and caches it per
// device.  A device reset (cudaDeviceReset, or the primary context destroyed and
// made again) reloads the module, possibly elsewhere, so the cached address is
// then stale: callers that reset a device must not use this entry point after.
#include <mutex>

#include "wf_internal.h"

namespace {

// Split-K partials (m, l, o) of the decode kernels; nothing in it needs to start
// at zero: every partial the combine kernel reads is written earlier in the same
// call by the split kernel.
static __device__ __align__(256) unsigned char g_decode_scratch[WF_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" wf_status wf_paged_decode_static_scratch(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t B, int32_t max_seq_len, int32_t num_q_heads,
    float scale, wf_pool_desc pool, uint32_t* dev_status, cudaStream_t stream) {
    // Same argument rules as wf_paged_decode, checked first: given no workspace it
    // launches nothing and returns WF_OK (empty batch), an argument error, or
    // WF_ERR_WORKSPACE for a valid batch.
    const wf_status pre = wf_paged_decode(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, B,
                                          max_seq_len, num_q_heads, scale, pool, nullptr, 0, dev_status, stream);
    if (pre != WF_ERR_WORKSPACE) return pre;
    // a valid batch: it must fit the static array
    const size_t need = wf_paged_decode_workspace_size(B, num_q_heads, max_seq_len, pool);
    if (need == 0 || need > (size_t)WF_STATIC_SCRATCH_BYTES) return WF_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return WF_ERR_CUDA;
    return wf_paged_decode(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, B, max_seq_len,
                           num_q_heads, scale, pool, scratch, (size_t)WF_STATIC_SCRATCH_BYTES, dev_status, stream);
}
