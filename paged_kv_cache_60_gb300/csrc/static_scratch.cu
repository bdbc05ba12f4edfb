// decode_attn_fwd_static_scratch: the decode call for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a scratch buffer: code that
// runs where allocation is forbidden or unavailable -- inside a memory-capped
// or pre-planned arena (an inference server that reserves all device memory at
// start-up and may not call cudaMalloc afterwards), a plug-in loaded into a
// host framework whose allocator it cannot reach, or a real-time path that must
// not risk an allocation stall. For them this entry point keeps the scheduling
// metadata and the split-KV partials in one fixed device array owned by the
// library, so the caller passes only inputs and outputs.
//
// The array is a file-scope static __device__ buffer of DA_STATIC_SCRATCH_BYTES;
// every GPU that loads the library holds it until the process exits. Its device
// address is looked up with cudaGetSymbolAddress the first time the entry point
// runs on a device (with that device current); make that first call before any
// stream capture. All calls share the buffer and it keeps the previous call's
// contents: the scheduling kernel rewrites every field the decode kernels read,
// so nothing needs clearing between calls, but two calls whose work overlaps on
// the GPU (different streams, no ordering) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "decode_attn.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[DA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (set up once per device).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return DA_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return DA_OK;
}

}  // namespace

extern "C" int decode_attn_fwd_static_scratch(const da_desc *desc, const void *q, const void *k_pool,
                                              const void *v_pool, const float *k_scale, const float *v_scale,
                                              const int32_t *block_table, const int32_t *cache_seqlens, void *out,
                                              float *lse, cudaStream_t stream) {
    size_t need = 0;
    int rc = decode_attn_sched_meta_bytes(desc, &need);
    if (rc) return rc;
    if (need > DA_STATIC_SCRATCH_BYTES) return DA_ERR_META_SIZE;  // problem too large for the fixed buffer
    void *scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;
    if ((rc = decode_attn_sched_meta(desc, cache_seqlens, scratch, DA_STATIC_SCRATCH_BYTES, stream))) return rc;
    return decode_attn_fwd(desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, scratch,
                           DA_STATIC_SCRATCH_BYTES, out, lse, stream);
}
