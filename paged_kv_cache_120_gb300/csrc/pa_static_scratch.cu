// pa_decode_static_scratch: pa_decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory: a host framework whose
// allocator owns all of the GPU's memory, a plugin that runs under a fixed
// memory budget, or a latency-critical loop in which an allocation (which
// may synchronise the device) is not allowed. For them this entry point keeps
// pa_decode's split-K scratch in a statically sized device array that is part
// of the library image, so a call allocates nothing.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

// Present on every GPU that loads this library, for the life of the process.
// In host code this name is only a host-side stand-in; the device address is
// obtained below with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once
// per device, with that device current).
int scratch_for_current_device(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pa::set_error(PA_ERR_CUDA, "pa_decode_static_scratch: cudaGetDevice: %s",
                             cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return pa::set_error(PA_ERR_UNSUPPORTED, "pa_decode_static_scratch: device %d >= %d", dev,
                             kMaxDevices);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p)
            return pa::set_error(PA_ERR_CUDA, "pa_decode_static_scratch: cudaGetSymbolAddress: %s",
                                 cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_static_scratch(void *out, const void *query, const void *kv_cache,
                                        const int32_t *block_tables, int max_blocks_per_seq,
                                        const int32_t *seq_lens, int num_seqs, float scale,
                                        int num_q_heads, int num_kv_heads, int head_size,
                                        int num_blocks, int block_size, int dtype,
                                        unsigned flags, pa_stream_t stream)
{
    size_t need = 0;
    int rc = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                      dtype, &need);
    if (rc != PA_OK)
        return rc;
    if (need > kStaticScratchBytes)
        return pa::set_error(PA_ERR_WORKSPACE,
                             "pa_decode_static_scratch: this shape needs %zu bytes of scratch, "
                             "more than the %zu-byte static array; use pa_decode with a workspace",
                             need, kStaticScratchBytes);
    void *scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != PA_OK)
        return rc;
    return pa_decode(out, query, kv_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     scale, num_q_heads, num_kv_heads, head_size, num_blocks, block_size, dtype,
                     scratch, kStaticScratchBytes, flags, stream);
}
