// Host side of the C ABI: argument checks, sched_meta layout, tensor maps,
// kernel launches. No allocation, no synchronisation in the forward path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "decode_attn.h"
#include "layout.h"

namespace da {
cudaError_t launch_sched_meta(const SchedParams &p, cudaStream_t stream, bool pdl);
cudaError_t launch_gqa(int D, bool fp8, const CUtensorMap &tkv, const CUtensorMap &tv, const GqaParams &p,
                       cudaStream_t stream, bool pdl);
cudaError_t launch_mla(const MlaParams &p, cudaStream_t stream, bool pdl);
cudaError_t launch_combine(int DV, const CombineParams &p, cudaStream_t stream, bool pdl);
cudaError_t launch_append(int kv_dtype, const AppendParams &p, cudaStream_t stream, bool pdl);
int mla_ctas_per_part(int s_q);
bool mla_kernel_available();
int mla_max_parts(int s_q);
int gqa_ctas_per_sm(int D, bool fp8, int s_q);
int check_fwd_args(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                   const float *k_scale, const float *v_scale, const int32_t *block_table,
                   const int32_t *cache_seqlens, const void *out, const float *lse, const da_launch_opts *opts);
}  // namespace da

using namespace da;

namespace {

constexpr float kLog2eF = 1.4426950408889634f;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool is_mla(const da_desc *d) { return d->kv_dtype == DA_KV_FP8_MLA656; }

// query tokens per request (0 in the desc means 1)
int sq_of(const da_desc *d) { return d->s_q <= 0 ? 1 : d->s_q; }

// Which kernel serves this desc; returns DA_OK or an error code.
int check_desc(const da_desc *d) {
    if (!d) return DA_ERR_NULL;
    if (d->B < 1 || d->B > (1 << 20) || d->H_kv < 1 || d->H_kv > 4096 || d->G < 1 || d->G > 1024 ||
        d->page_size < 1 || d->max_pages_per_seq < 1 || d->num_pages < 1 || d->D_qk < 1 || d->D_v < 1)
        return DA_ERR_DIMS;
    if ((int64_t)d->max_pages_per_seq * d->page_size > (int64_t)INT32_MAX - 64) return DA_ERR_DIMS;
    if ((int64_t)d->B * d->max_pages_per_seq > (int64_t)INT32_MAX) return DA_ERR_DIMS;
    if (d->splits < 0 || d->splits > 4096) return DA_ERR_SPLITS;
    if (d->num_sms < 0) return DA_ERR_DIMS;
    if (!(d->softmax_scale >= 0.f) || std::isinf(d->softmax_scale)) return DA_ERR_DIMS;
    if (d->s_q < 0 || d->s_q > 64) return DA_ERR_DIMS;
    if (d->window < 0) return DA_ERR_DIMS;
    if (d->topk < 0 || d->topk > (1 << 24)) return DA_ERR_DIMS;
    const int sq = sq_of(d);
    const int P = d->page_size;
    const bool page_ok = (P == 8 || P == 16 || P == 32 || (P % 64) == 0);
    if (!page_ok) return DA_ERR_UNSUPPORTED;
    switch (d->kv_dtype) {
        case DA_KV_BF16:
            if (d->G != 8 || d->D_qk != d->D_v || (d->D_qk != 64 && d->D_qk != 128)) return DA_ERR_UNSUPPORTED;
            if (sq > (d->D_qk == 64 ? kMaxSqD64 : kMaxSqD128) || d->topk != 0) return DA_ERR_UNSUPPORTED;
            break;
        case DA_KV_FP8_PER_TENSOR:
            if (d->G != 8 || d->D_qk != 128 || d->D_v != 128) return DA_ERR_UNSUPPORTED;
            if (sq > kMaxSqD128 || d->topk != 0) return DA_ERR_UNSUPPORTED;
            break;
        case DA_KV_FP8_MLA656:
            if (d->H_kv != 1 || d->D_qk != 576 || d->D_v != 512 || d->G != 128) return DA_ERR_UNSUPPORTED;
            if (sq > kMaxSqMla || d->window != 0 || (d->topk > 0 && sq != 1)) return DA_ERR_UNSUPPORTED;
            if (!mla_kernel_available()) return DA_ERR_UNSUPPORTED;
            break;
        default:
            return DA_ERR_UNSUPPORTED;
    }
    return DA_OK;
}

int resolve_sms(const da_desc *d, int *nsm) {
    if (d->num_sms > 0) {
        *nsm = d->num_sms;
        return DA_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DA_ERR_CUDA;
    if (cudaDeviceGetAttribute(nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DA_ERR_CUDA;
    if (is_mla(d)) {
        // the latent-token kernel runs as clusters of 2 s_q CTAs: count the SMs
        // that can hold them at the same time
        const int cpc = mla_ctas_per_part(sq_of(d));
        const int clusters = mla_max_parts(sq_of(d));
        if (clusters < 1) return DA_ERR_CUDA;
        if (cpc * clusters < *nsm) *nsm = cpc * clusters;
    } else {
        // the GQA builds that run two CTAs per SM count two slots per SM
        *nsm *= gqa_ctas_per_sm(d->D_qk, d->kv_dtype == DA_KV_FP8_PER_TENSOR, sq_of(d));
    }
    return DA_OK;
}

// Page-trace test build: where the kernels record the pool rows they read,
// and an optional shorter limit for every bounded wait.
int32_t *g_page_trace = nullptr;
int32_t g_page_trace_cap = 0;
uint64_t g_wait_limit_ns = 0;  // 0: kWaitLimitNs
int32_t g_debug_stall = 0;

int cpc_of(const da_desc *d) { return is_mla(d) ? mla_ctas_per_part(sq_of(d)) : 1; }

int make_layout(const da_desc *d, MetaLayout *L) {
    int rc = check_desc(d);
    if (rc) return rc;
    int nsm = 0;
    rc = resolve_sms(d, &nsm);
    if (rc) return rc;
    const int cpc = cpc_of(d);
    int64_t num_parts, max_splits;
    if (d->splits > 0) {
        num_parts = (int64_t)d->B * d->splits;
        max_splits = num_parts;
    } else {
        num_parts = nsm / (d->H_kv * cpc);
        if (num_parts < 1) num_parts = 1;
        max_splits = num_parts + d->B;
    }
    if (num_parts > (1 << 24)) return DA_ERR_SPLITS;
    const int64_t H_q = (int64_t)d->H_kv * d->G;
    const int64_t rows = H_q * sq_of(d);  // output rows per request
    size_t off = 0;
    L->header = off;
    off += kHeaderWords * 4;
    L->parts = off;
    off += round_up((size_t)num_parts * sizeof(PartRec), 16);
    L->chunk_offset = off;
    off += round_up((size_t)(d->B + 1) * 4, 16);
    L->split_offset = off;
    off += round_up((size_t)(d->B + 1) * 4, 16);
    L->num_splits = off;
    off += round_up((size_t)d->B * 4, 16);
    off = round_up(off, 256);
    L->lse_part = off;
    off += round_up((size_t)max_splits * rows * 4, 256);
    L->o_part = off;
    off += round_up((size_t)max_splits * rows * d->D_v * 4, 256);
    L->total = off;
    L->num_parts = (int32_t)num_parts;
    L->max_splits = (int32_t)max_splits;
    L->cpc = cpc;
    return DA_OK;
}

MetaView meta_view(void *meta, const MetaLayout &L) {
    uint8_t *base = static_cast<uint8_t *>(meta);
    MetaView v;
    v.header = reinterpret_cast<int32_t *>(base + L.header);
    v.parts = reinterpret_cast<const int4 *>(base + L.parts);
    v.chunk_offset = reinterpret_cast<const int32_t *>(base + L.chunk_offset);
    v.split_offset = reinterpret_cast<const int32_t *>(base + L.split_offset);
    v.num_splits = reinterpret_cast<const int32_t *>(base + L.num_splits);
    v.lse_part = reinterpret_cast<float *>(base + L.lse_part);
    v.o_part = reinterpret_cast<float *>(base + L.o_part);
    v.max_splits = L.max_splits;
    return v;
}

// cuTensorMapEncodeTiled, fetched from the driver at first use.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// The pools are described to the TMA unit as 8-byte elements (16 per 128-byte
// box row): the shared-memory image is the same whatever the KV format.
//
// Both pools as one 5-D map:
//   dim 0: 16 elements = 128 bytes          dim 1: NX halves of a head row (stride 128 B)
//   dim 2: KV head (stride = row)           dim 3: global token = page*P + slot (stride row*H_kv)
//   dim 4: pool, K or V (stride = distance between the two pools)
// and a box {16, NX, 1, box_tok, 2}: one copy brings one page's K and V rows of
// one head, in shared memory as [pool][token][half][128 B]. base is the lower
// of the two pools. With pool = nullptr, a 4-D map of one pool (dims 0-3) and
// a box {16, NX, 1, box_tok}. With half_major the token dimension (1) and the
// half and head dimensions (2, 3) trade places: the box lands as
// [pool][half][token][128 B].
int make_kv_map(CUtensorMap *m, const void *base, uint64_t pool_dist, bool two_pools, const da_desc *d,
                int elem_bytes, int box_tok, bool half_major) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return DA_ERR_CUDA;
    const cuuint64_t row = (cuuint64_t)d->D_qk * elem_bytes;  // bytes of one token's head
    const cuuint64_t nx = row / 128;
    const cuuint64_t ntok = (cuuint64_t)d->page_size * (cuuint64_t)d->num_pages;
    cuuint64_t dims[5] = {128 / kTmaElemBytes, nx, (cuuint64_t)d->H_kv, ntok, 2};
    cuuint64_t strides[4] = {128, row, row * d->H_kv, pool_dist};
    cuuint32_t box[5] = {128 / kTmaElemBytes, (cuuint32_t)nx, 1, (cuuint32_t)box_tok, 2};
    if (half_major) {  // the token dimension inside the half dimension
        dims[1] = ntok;
        dims[2] = nx;
        dims[3] = (cuuint64_t)d->H_kv;
        strides[0] = row * d->H_kv;
        strides[1] = 128;
        strides[2] = row;
        box[1] = (cuuint32_t)box_tok;
        box[2] = (cuuint32_t)nx;
        box[3] = 1;
    }
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, two_pools ? 5 : 4, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

}  // namespace

// Every host-side check of decode_attn_fwd_ex that does not involve the
// sched_meta buffer (desc, pointers, alignment, scales, optional inputs);
// returns DA_OK or the first error. No CUDA call beyond an SM-count query.
int da::check_fwd_args(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                       const float *k_scale, const float *v_scale, const int32_t *block_table,
                       const int32_t *cache_seqlens, const void *out, const float *lse,
                       const da_launch_opts *opts) {
    int rc = check_desc(desc);
    if (rc) return rc;
    const bool mla = is_mla(desc);
    if (!q || !k_pool || !block_table || !cache_seqlens || !out || !lse) return DA_ERR_NULL;
    if (!mla && !v_pool) return DA_ERR_NULL;
    if (mla && v_pool && v_pool != k_pool) return DA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_pool) || (v_pool && !aligned16(v_pool)) || !aligned16(block_table) ||
        !aligned16(cache_seqlens) || !aligned16(out) || !aligned16(lse))
        return DA_ERR_ALIGN;
    if (desc->kv_dtype == DA_KV_FP8_PER_TENSOR) {
        if (!k_scale || !v_scale) return DA_ERR_SCALE;
        if ((reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
            return DA_ERR_ALIGN;
    }
    const float *sinks = opts ? opts->sinks : nullptr;
    if (sinks && mla) return DA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(sinks) & 3u) return DA_ERR_ALIGN;
    const int32_t *indices = opts ? opts->indices : nullptr;
    if (desc->topk > 0 && !indices) return DA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(indices) & 3u) return DA_ERR_ALIGN;
    if ((int64_t)desc->page_size * desc->num_pages > (int64_t)INT32_MAX) return DA_ERR_DIMS;
    return DA_OK;
}

extern "C" {

int decode_attn_sched_meta_bytes(const da_desc *desc, size_t *bytes) {
    if (!bytes) return DA_ERR_NULL;
    MetaLayout L;
    const int rc = make_layout(desc, &L);
    if (rc) return rc;
    *bytes = L.total;
    return DA_OK;
}

int decode_attn_meta_offsets(const da_desc *desc, size_t offs[8]) {
    if (!offs) return DA_ERR_NULL;
    MetaLayout L;
    const int rc = make_layout(desc, &L);
    if (rc) return rc;
    offs[0] = L.header;
    offs[1] = L.parts;
    offs[2] = L.chunk_offset;
    offs[3] = L.split_offset;
    offs[4] = L.num_splits;
    offs[5] = L.lse_part;
    offs[6] = L.o_part;
    offs[7] = L.total;
    return DA_OK;
}

int decode_attn_num_parts(const da_desc *desc, int32_t *num_parts) {
    if (!num_parts) return DA_ERR_NULL;
    MetaLayout L;
    const int rc = make_layout(desc, &L);
    if (rc) return rc;
    *num_parts = L.num_parts;
    return DA_OK;
}

int decode_attn_sched_meta(const da_desc *desc, const int32_t *cache_seqlens, void *sched_meta,
                           size_t sched_meta_bytes, cudaStream_t stream) {
    MetaLayout L;
    int rc = make_layout(desc, &L);
    if (rc) return rc;
    if (!cache_seqlens || !sched_meta) return DA_ERR_NULL;
    if (!aligned16(sched_meta) || (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u)) return DA_ERR_ALIGN;
    if (sched_meta_bytes < L.total) return DA_ERR_META_SIZE;
    int nsm = 0;
    resolve_sms(desc, &nsm);
    uint8_t *base = static_cast<uint8_t *>(sched_meta);
    SchedParams p;
    p.seqlens = cache_seqlens;
    p.meta = reinterpret_cast<int32_t *>(base + L.header);
    p.parts = reinterpret_cast<int32_t *>(base + L.parts);
    p.chunk_offset = reinterpret_cast<int32_t *>(base + L.chunk_offset);
    p.split_offset = reinterpret_cast<int32_t *>(base + L.split_offset);
    p.num_splits = reinterpret_cast<int32_t *>(base + L.num_splits);
    p.B = desc->B;
    p.H_kv = desc->H_kv;
    p.G = desc->G;
    p.splits = desc->splits;
    p.num_parts = L.num_parts;
    p.cpc = L.cpc;
    p.max_len = desc->max_pages_per_seq * desc->page_size;
    p.kv_dtype = desc->kv_dtype;
    p.num_sms = nsm;
    p.s_q = sq_of(desc);
    p.window = desc->window;
    p.topk = desc->topk;
    if (launch_sched_meta(p, stream, true) != cudaSuccess) return DA_ERR_CUDA;
    return DA_OK;
}

int decode_attn_fwd_ex(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                       const float *k_scale, const float *v_scale, const int32_t *block_table,
                       const int32_t *cache_seqlens, void *sched_meta, size_t sched_meta_bytes, void *out,
                       float *lse, const da_launch_opts *opts, cudaStream_t stream) {
    MetaLayout L;
    int rc = make_layout(desc, &L);
    if (rc) return rc;
    const bool mla = is_mla(desc);
    if ((rc = check_fwd_args(desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, out, lse,
                             opts)))
        return rc;
    if (!sched_meta) return DA_ERR_NULL;
    if (!aligned16(sched_meta)) return DA_ERR_ALIGN;
    if (sched_meta_bytes < L.total) return DA_ERR_META_SIZE;
    const float *sinks = opts ? opts->sinks : nullptr;
    const int32_t *indices = opts ? opts->indices : nullptr;
    const bool pdl = opts ? opts->use_pdl != 0 : true;
    const float sigma = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / std::sqrt((float)desc->D_qk);
    const MetaView mv = meta_view(sched_meta, L);
    const int H_q = desc->H_kv * desc->G;

    const cudaEvent_t ev_begin = opts ? opts->main_begin : nullptr;
    if (!mla) {
        const bool fp8 = desc->kv_dtype == DA_KV_FP8_PER_TENSOR;
        const int es = fp8 ? 1 : 2;
        const int P = desc->page_size;
        const int box_tok = P < kChunk ? P : kChunk;
        // one map over both pools when their distance can be a tensor-map
        // stride (a multiple of 16 below 2^40, not overlapping); else one per pool
        const uint64_t pool_bytes = (uint64_t)desc->num_pages * P * desc->H_kv * desc->D_qk * es;
        const uintptr_t ka = reinterpret_cast<uintptr_t>(k_pool), va = reinterpret_cast<uintptr_t>(v_pool);
        const uint64_t dist = ka > va ? (uint64_t)(ka - va) : (uint64_t)(va - ka);
        const bool combined = dist >= pool_bytes && dist < (1ull << 40);
        // the builds with several query tokens or a window read 256-byte rows half-major
        const bool half_major = (sq_of(desc) > 1 || desc->window > 0) && desc->D_qk * es > 128;
        CUtensorMap tkv, tv;
        if (combined) {
            if ((rc = make_kv_map(&tkv, ka < va ? k_pool : v_pool, dist, true, desc, es, box_tok, half_major)))
                return rc;
            tv = tkv;
        } else {
            if ((rc = make_kv_map(&tkv, k_pool, 0, false, desc, es, box_tok, half_major))) return rc;
            if ((rc = make_kv_map(&tv, v_pool, 0, false, desc, es, box_tok, half_major))) return rc;
        }
        GqaParams p;
        p.q = q;
        p.block_table = block_table;
        p.seqlens = cache_seqlens;
        p.k_scale = k_scale;
        p.v_scale = v_scale;
        p.meta = mv;
        p.out = out;
        p.lse = lse;
        p.B = desc->B;
        p.H_kv = desc->H_kv;
        p.G = desc->G;
        p.H_q = H_q;
        p.s_q = sq_of(desc);
        p.window = desc->window;
        p.sinks = sinks;
        // a fixed split count of 2..8: the splits of a (request, KV head) merge
        // inside one thread-block cluster and no combine kernel runs
        p.cluster_merge = (desc->splits >= 2 && desc->splits <= 8) ? 1 : 0;
        p.half_major = half_major ? 1 : 0;
        p.max_pages = desc->max_pages_per_seq;
        p.num_pages = desc->num_pages;
        p.page_size = P;
        p.box_tokens = box_tok;
        p.boxes_per_chunk = kChunk / box_tok;
        p.log2_box_tokens = box_tok == 8 ? 3 : box_tok == 16 ? 4 : box_tok == 32 ? 5 : 6;
        p.kv_swap = (combined && va < ka) ? 1 : 0;
        p.kv_combined = combined ? 1 : 0;
        p.splits = desc->splits;
        p.num_parts = L.num_parts;
        p.scale_log2 = sigma * kLog2eF;
        p.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : kWaitLimitNs;
        p.page_trace = g_page_trace;
        p.page_trace_cap = g_page_trace_cap;
        p.debug_stall = g_debug_stall;
        if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return DA_ERR_CUDA;
        if (launch_gqa(desc->D_qk, fp8, tkv, tv, p, stream, pdl) != cudaSuccess) return DA_ERR_CUDA;
    } else {
        MlaParams p;
        p.q = q;
        p.pool = static_cast<const uint8_t *>(k_pool);
        p.block_table = block_table;
        p.seqlens = cache_seqlens;
        p.meta = mv;
        p.out = out;
        p.lse = lse;
        p.B = desc->B;
        p.H_q = H_q;
        p.max_pages = desc->max_pages_per_seq;
        p.num_pages = desc->num_pages;
        p.page_size = desc->page_size;
        p.splits = desc->splits;
        p.num_parts = L.num_parts;
        p.scale_log2 = sigma * kLog2eF;
        p.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : kWaitLimitNs;
        p.page_trace = g_page_trace;
        p.page_trace_cap = g_page_trace_cap;
        p.indices = desc->topk > 0 ? indices : nullptr;
        p.topk = desc->topk;
        p.s_q = sq_of(desc);
        p.debug_stall = g_debug_stall;
        p.log2_page = -1;
        for (int k = 0; k < 31; ++k)
            if (desc->page_size == (1 << k)) p.log2_page = k;
        if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return DA_ERR_CUDA;
        if (launch_mla(p, stream, pdl) != cudaSuccess) return DA_ERR_CUDA;
    }
    if (opts && opts->main_end && cudaEventRecord(opts->main_end, stream) != cudaSuccess) return DA_ERR_CUDA;
    if (!mla && desc->splits >= 2 && desc->splits <= 8) return DA_OK;  // merged in the split-KV kernel
    CombineParams c;
    c.meta = mv;
    c.out = out;
    c.lse = lse;
    c.B = desc->B;
    c.rows = H_q * sq_of(desc);
    c.s_q = sq_of(desc);
    c.window = desc->window;
    c.topk = desc->topk;
    c.sinks = sinks;
    c.D_v = desc->D_v;
    c.H_kv = desc->H_kv;
    c.G = desc->G;
    c.splits = desc->splits;
    c.num_parts = L.num_parts;
    if (launch_combine(desc->D_v, c, stream, pdl) != cudaSuccess) return DA_ERR_CUDA;
    return DA_OK;
}

int decode_attn_fwd(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                    const float *k_scale, const float *v_scale, const int32_t *block_table,
                    const int32_t *cache_seqlens, void *sched_meta, size_t sched_meta_bytes, void *out, float *lse,
                    cudaStream_t stream) {
    return decode_attn_fwd_ex(desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, sched_meta,
                              sched_meta_bytes, out, lse, nullptr, stream);
}

int decode_attn_append_kv(const da_desc *desc, const void *k_new, const void *v_new, int64_t new_row_stride,
                          const int32_t *positions, const int32_t *block_table, void *k_pool, void *v_pool,
                          const float *k_scale, const float *v_scale, int32_t *device_error, cudaStream_t stream) {
    if (!desc) return DA_ERR_NULL;
    const da_desc *d = desc;
    if (d->B < 1 || d->B > (1 << 24) || d->H_kv < 1 || d->H_kv > 4096 || d->page_size < 1 ||
        d->max_pages_per_seq < 1 || d->num_pages < 1 || d->D_qk < 1 || d->D_v < 1 || d->D_qk > 4096 ||
        d->D_v > 4096)
        return DA_ERR_DIMS;
    if ((int64_t)d->max_pages_per_seq * d->page_size > (int64_t)INT32_MAX) return DA_ERR_DIMS;
    if ((int64_t)d->B * d->max_pages_per_seq > (int64_t)INT32_MAX) return DA_ERR_DIMS;
    const bool mla = is_mla(d);
    int64_t row_len = 0;  // bf16 values of one request's new K (or V) row
    switch (d->kv_dtype) {
        case DA_KV_BF16:
        case DA_KV_FP8_PER_TENSOR:
            if (d->D_qk != d->D_v || (d->D_qk % 8) != 0) return DA_ERR_UNSUPPORTED;
            row_len = (int64_t)d->H_kv * d->D_qk;
            break;
        case DA_KV_FP8_MLA656:
            if (d->H_kv != 1 || d->D_qk != 576 || d->D_v != 512) return DA_ERR_UNSUPPORTED;
            row_len = 576;
            break;
        default:
            return DA_ERR_UNSUPPORTED;
    }
    if (new_row_stride == 0) new_row_stride = row_len;
    if (new_row_stride < row_len || (new_row_stride % 8) != 0 || new_row_stride > ((int64_t)1 << 40))
        return DA_ERR_DIMS;
    if (!k_new || !positions || !block_table || !k_pool) return DA_ERR_NULL;
    if (mla) {
        if (v_new) return DA_ERR_UNSUPPORTED;
        if (v_pool && v_pool != k_pool) return DA_ERR_UNSUPPORTED;
    } else if (!v_new || !v_pool) {
        return DA_ERR_NULL;
    }
    if (!aligned16(k_new) || (v_new && !aligned16(v_new)) || !aligned16(k_pool) || (v_pool && !aligned16(v_pool)) ||
        (reinterpret_cast<uintptr_t>(positions) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(device_error) & 3u))
        return DA_ERR_ALIGN;
    if (d->kv_dtype == DA_KV_FP8_PER_TENSOR) {
        if (!k_scale || !v_scale) return DA_ERR_SCALE;
        if ((reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
            return DA_ERR_ALIGN;
    }
    AppendParams p;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.positions = positions;
    p.block_table = block_table;
    p.k_pool = static_cast<uint8_t *>(k_pool);
    p.v_pool = static_cast<uint8_t *>(mla ? k_pool : v_pool);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.error = device_error;
    p.row_stride = new_row_stride;
    p.B = d->B;
    p.H_kv = d->H_kv;
    p.D = d->D_qk;
    p.page_size = d->page_size;
    p.max_pages = d->max_pages_per_seq;
    p.num_pages = d->num_pages;
    if (launch_append(d->kv_dtype, p, stream, true) != cudaSuccess) return DA_ERR_CUDA;
    return DA_OK;
}

int decode_attn_get_error(const void *sched_meta, int32_t *device_error, cudaStream_t stream) {
    if (!sched_meta || !device_error) return DA_ERR_NULL;
    if (!aligned16(sched_meta)) return DA_ERR_ALIGN;
    const int32_t *w = static_cast<const int32_t *>(sched_meta) + kHError;
    if (cudaMemcpyAsync(device_error, w, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DA_ERR_CUDA;
    return DA_OK;
}

const char *decode_attn_strerror(int code) {
    switch (code) {
        case DA_OK: return "ok";
        case DA_ERR_NULL: return "a required pointer is NULL";
        case DA_ERR_DIMS: return "a size is out of range";
        case DA_ERR_UNSUPPORTED: return "no kernel for this (kv dtype, D_qk, D_v, G, page_size)";
        case DA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case DA_ERR_SPLITS: return "splits out of range";
        case DA_ERR_META_SIZE: return "sched_meta buffer too small";
        case DA_ERR_CUDA: return "a CUDA call failed";
        case DA_ERR_SCALE: return "FP8 KV needs k_scale and v_scale";
        default: return "unknown error code";
    }
}

}  // extern "C"

#ifdef DA_PAGE_TRACE
// Test build only (compiled with -DDA_PAGE_TRACE): record the pool rows every
// later decode_attn_fwd reads into `trace` (device, int32). GQA: per (part, KV
// head) CTA, per chunk, per TMA box: the first pool row of the box (page *
// page_size + offset in the page) or -2 for a box past the sequence. MLA: per
// part, per chunk, per token: the token's pool row or -2. `cap` chunks are kept
// per CTA / part. Pass null to stop recording.
extern "C" int decode_attn_debug_page_trace(int32_t *trace, int32_t cap) {
    if (trace && cap < 1) return DA_ERR_DIMS;
    g_page_trace = trace;
    g_page_trace_cap = trace ? cap : 0;
    return DA_OK;
}

// Test build only: limit every bounded wait of later launches to `ns`
// nanoseconds (0 restores the default of 2 s).
extern "C" int decode_attn_debug_wait_limit(uint64_t ns) {
    g_wait_limit_ns = ns;
    return DA_OK;
}

// Test build only: with `on` != 0, the GQA kernel's consumer warps first wait
// on a barrier that nothing completes, so that wait runs out.
extern "C" int decode_attn_debug_stall(int32_t on) {
    g_debug_stall = on;
    return DA_OK;
}
#endif
