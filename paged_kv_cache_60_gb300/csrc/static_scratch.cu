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
// runs in a CUDA context (with that context's device current); make that first
// call before any stream capture. The address is cached per device together
// with the context's unique id, so after a device reset (a new primary context,
// in which the array may sit elsewhere) the next call looks it up again. All
// calls share the buffer and it keeps the previous call's contents: the
// scheduling kernel rewrites every field the decode kernels read, so nothing
// needs clearing between calls, but two calls whose work overlaps on the GPU
// (different streams, no ordering) race on it. Every argument is checked on
// the host before the first launch, so a rejected call leaves the array as the
// previous call left it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "decode_attn.h"

namespace da {
int check_fwd_args(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                   const float *k_scale, const float *v_scale, const int32_t *block_table,
                   const int32_t *cache_seqlens, const void *out, const float *lse, const da_launch_opts *opts);
}

namespace {

static __device__ __align__(256) unsigned char g_scratch[DA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current CUDA context (0 if there is none
// or the driver cannot say). Ids are never reused within a process.
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) != cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) != cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess)
            return 0;
        get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        get_id = reinterpret_cast<CtxGetIdFn>(q);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_scratch in the current context (looked up once per
// device and context).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = current_ctx_id();
    if (!g_addr[dev] || id == 0 || id != g_ctx_id[dev]) {
        void *p = nullptr;
        // also makes the device's primary context current if nothing had yet
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return DA_ERR_CUDA;
        if (id == 0) id = current_ctx_id();
        g_addr[dev] = p;
        g_ctx_id[dev] = id;
    }
    *out = g_addr[dev];
    return DA_OK;
}

}  // namespace

extern "C" int decode_attn_fwd_static_scratch(const da_desc *desc, const void *q, const void *k_pool,
                                              const void *v_pool, const float *k_scale, const float *v_scale,
                                              const int32_t *block_table, const int32_t *cache_seqlens, void *out,
                                              float *lse, cudaStream_t stream) {
    // sparse decode needs indices, which this call cannot take
    if (desc && desc->topk > 0) return DA_ERR_UNSUPPORTED;
    // every check decode_attn_fwd makes, before anything touches the array
    int rc = da::check_fwd_args(desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, out, lse,
                                nullptr);
    if (rc) return rc;
    size_t need = 0;
    if ((rc = decode_attn_sched_meta_bytes(desc, &need))) return rc;
    if (need > DA_STATIC_SCRATCH_BYTES) return DA_ERR_META_SIZE;  // problem too large for the fixed buffer
    void *scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;
    if ((rc = decode_attn_sched_meta(desc, cache_seqlens, scratch, DA_STATIC_SCRATCH_BYTES, stream))) return rc;
    return decode_attn_fwd(desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, scratch,
                           DA_STATIC_SCRATCH_BYTES, out, lse, stream);
}
