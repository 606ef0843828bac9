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
#include <cuda.h>

#include <mutex>

#include "pa_decode_common.cuh"

namespace pa {
namespace {

// Scratch shared by every call on a device (one instance per device).
static __device__ __align__(256) unsigned char g_noalloc_workspace[PA_NOALLOC_WORKSPACE_BYTES];

// The array's device address per device, with the unique id of the CUDA
// context it was looked up in: a context created later on that device (after
// a cudaDeviceReset, say) loads the library's device code again, possibly
// elsewhere, and gets its own lookup.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
struct CachedAddress {
    void *addr = nullptr;
    unsigned long long ctx_id = 0;
};
std::mutex g_mutex;
CachedAddress g_workspace_addr[kMaxDevices];

bool current_context_id(unsigned long long *id)
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
           get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must be looked
// up (once per device and context, with that device current) before a
// kernel can use it.
pa_status workspace_address(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return record_cuda(e);
    if (dev < 0 || dev >= kMaxDevices)
        return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    CachedAddress &c = g_workspace_addr[dev];
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (c.addr == nullptr || !have_id || id != c.ctx_id) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess)
            return record_cuda(e);
        // the lookup makes the device's context current if none was
        unsigned long long now = 0;
        c.addr = p;
        c.ctx_id = current_context_id(&now) ? now : 0;
    }
    *addr = c.addr;
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
    // the arguments first, with pa_decode_attention's checks and statuses;
    // only a valid call whose partials do not fit the array is refused for
    // its size
    if (dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_INVALID_ARG;
    pa::DecodeParams prm{};
    const pa_status valid = pa::prepare_decode(
        &prm, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
        context_lens, max_context_len, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
        num_blocks, scale, partition_size, nullptr, 0, error_word);
    if (valid != PA_OK && valid != PA_ERR_WORKSPACE)
        return valid;
    if (num_seqs == 0)
        return PA_OK;
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
