// pa_noalloc.cu -- paged decode attention whose split-context scratch lives
// in a statically sized device array, for callers that cannot allocate.
//
// Who needs this: code that must not call cudaMalloc (or any allocating
// routine) on its decode path -- for instance a plugin whose host engine
// owns every device allocation through its own pool and forbids others, a
// latency-critical loop that cannot afford an allocation's implicit device
// synchronisation, or a C interface that only hands over input and output
// buffers and has no way to pass a workspace.  This entry point takes the
// same inputs and outputs as pa_decode_attention and uses the array below as
// its workspace; nothing is allocated by the call.
//
// The array is PA_NOALLOC_WORKSPACE_BYTES long and is created when the
// library's device code is loaded on a GPU; every GPU that loads it keeps
// it until the process exits.
#include <mutex>

#include "pa_common.cuh"

namespace pa {
namespace {

// Scratch shared by every call on a device (one instance per device).
static __device__ __align__(256) unsigned char g_noalloc_workspace[PA_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_workspace_addr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must be looked
// up (once per device, with that device current) before a kernel can use it.
pa_status workspace_address(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return record_cuda(e);
    if (dev < 0 || dev >= kMaxDevices)
        return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_workspace_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess)
            return record_cuda(e);
        g_workspace_addr[dev] = p;
    }
    *addr = g_workspace_addr[dev];
    return PA_OK;
}

} // namespace
} // namespace pa

extern "C" pa_status pa_decode_attention_noalloc(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, int partition_size, pa_dtype dtype,
    int32_t *error_word, void *stream)
{
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads,
                                                  head_dim, max_context_len, partition_size);
    if (need > (size_t)PA_NOALLOC_WORKSPACE_BYTES)
        return PA_ERR_WORKSPACE;  // these sizes need more scratch than the array holds
    void *ws = nullptr;
    if (need > 0) {
        const pa_status st = pa::workspace_address(&ws);
        if (st != PA_OK)
            return st;
    }
    return pa_decode_attention(out, query, key_cache, value_cache, block_tables,
                               max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                               num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                               partition_size, ws, need > 0 ? (size_t)PA_NOALLOC_WORKSPACE_BYTES
                                                            : 0,
                               dtype, error_word, stream);
}
