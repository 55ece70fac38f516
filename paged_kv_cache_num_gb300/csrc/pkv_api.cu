// pkv_api.cu -- the extern "C" entry points declared in include/pkv.h:
// argument validation, plan selection and dispatch to the kernel launchers.
// Nothing here touches tensor data; every step of the path runs in kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "pkv_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    g_err[0] = '\0';
    return PKV_OK;
}

int elem_size(int dtype)
{
    switch (dtype) {
    case PKV_DTYPE_F16:
    case PKV_DTYPE_BF16: return 2;
    case PKV_DTYPE_E4M3:
    case PKV_DTYPE_E5M2:
    case PKV_DTYPE_I8:
    case PKV_DTYPE_U3:
    case PKV_DTYPE_U8: return 1;
    case PKV_DTYPE_I32:
    case PKV_DTYPE_F32: return 4;
    case PKV_DTYPE_I64: return 8;
    default: return 0;
    }
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int log2i(int64_t x)
{
    int s = 0;
    while ((int64_t(1) << s) < x) ++s;
    return s;
}

int check_tensor(const pkv_tensor *t, const char *name, int ndim)
{
    if (!t) return fail(PKV_ERR_NULL, "%s: descriptor is NULL", name);
    if (t->ndim != ndim) return fail(PKV_ERR_SHAPE, "%s: expected %d dims, got %d", name, ndim, t->ndim);
    if (elem_size(t->dtype) == 0) return fail(PKV_ERR_DTYPE, "%s: unknown dtype %d", name, t->dtype);
    int64_t numel = 1;
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] < 0) return fail(PKV_ERR_SHAPE, "%s: negative extent", name);
        numel *= t->shape[i];
    }
    if (numel > 0 && !t->data) return fail(PKV_ERR_NULL, "%s: data pointer is NULL", name);
    return PKV_OK;
}

#define TRY(x)                  \
    do {                        \
        int _rc = (x);          \
        if (_rc != PKV_OK) return _rc; \
    } while (0)

struct CacheInfo {
    int kind;
    int64_t num_blocks, block_size, num_kv_heads, head_dim;
    int scale_mode;                       // PKV_SCALE_* (fp8 / int8 caches)
    int64_t gs_blk, gs_slot, gs_head;     // strides of the per-block / per-token scales
    int64_t c_chunk;                      // bytes between the 16-byte pieces of a row
};

// Validate a pkv_cache; head_dim comes from the row length and the dtype.
// `any_block_size`: the append takes any block size (e.g. a contiguous
// [batch, kv_heads, max_seq_len, D] cache seen as one block per request);
// decode needs a power of two <= 256.
int check_cache(const pkv_cache *c, CacheInfo &ci, bool any_block_size = false)
{
    if (!c) return fail(PKV_ERR_NULL, "cache: descriptor is NULL");
    TRY(check_tensor(&c->k_cache, "k_cache", 4));
    TRY(check_tensor(&c->v_cache, "v_cache", 4));
    const pkv_tensor &k = c->k_cache, &v = c->v_cache;
    if (k.dtype != v.dtype) return fail(PKV_ERR_DTYPE, "k_cache and v_cache dtypes differ");
    const int kind = k.dtype;
    if (kind != PKV_DTYPE_F16 && kind != PKV_DTYPE_BF16 && !pkv::is_q8(kind) && kind != PKV_DTYPE_U3)
        return fail(PKV_ERR_DTYPE, "cache dtype %d is not F16, BF16, E4M3, E5M2, I8 or U3", kind);
    for (int i = 0; i < 4; ++i) {
        if (k.shape[i] != v.shape[i]) return fail(PKV_ERR_SHAPE, "k_cache and v_cache shapes differ");
        if (k.stride[i] != v.stride[i]) return fail(PKV_ERR_LAYOUT, "k_cache and v_cache strides differ");
    }
    if (k.stride[3] != 1) return fail(PKV_ERR_LAYOUT, "cache rows must be contiguous (last stride 1)");
    const int es = elem_size(kind);
    // 16-bit and e4m3 rows are whole 16-byte units; packed 3-bit rows
    // (3*head_dim/8 bytes) only need 16-byte aligned blocks
    for (int i = 0; i < (kind == PKV_DTYPE_U3 ? 1 : 3); ++i)
        if ((k.stride[i] * es) % 16 != 0)
            return fail(PKV_ERR_LAYOUT, "cache stride %d is not a multiple of 16 bytes", i);
    if (!aligned(k.data, 16) || !aligned(v.data, 16))
        return fail(PKV_ERR_LAYOUT, "cache base pointers must be 16-byte aligned");
    ci.c_chunk = 16;
    if (c->chunk_stride != 0) {     // x-vectorised rows: pieces of 16 bytes
        if (kind == PKV_DTYPE_U3)
            return fail(PKV_ERR_UNSUPPORTED, "chunk_stride does not apply to U3 caches");
        if (c->chunk_stride < 0 || (c->chunk_stride * es) % 16 != 0)
            return fail(PKV_ERR_LAYOUT, "chunk_stride must be a positive multiple of 16 bytes");
        if ((k.shape[3] * es) % 16 != 0)
            return fail(PKV_ERR_SHAPE, "head_dim must be a multiple of x = 16 bytes / element size");
        ci.c_chunk = c->chunk_stride * es;
    }
    ci.kind = kind;
    ci.num_blocks = k.shape[0];
    ci.block_size = k.shape[1];
    ci.num_kv_heads = k.shape[2];
    ci.head_dim = kind == PKV_DTYPE_U3 ? k.shape[3] * 8 / 3 : k.shape[3];
    if (kind == PKV_DTYPE_U3 && k.shape[3] * 8 != ci.head_dim * 3)
        return fail(PKV_ERR_SHAPE, "U3 cache row of %lld bytes is not 3*head_dim/8", (long long)k.shape[3]);
    if (any_block_size ? ci.block_size < 1 : (!is_pow2(ci.block_size) || ci.block_size > 256))
        return fail(PKV_ERR_UNSUPPORTED, "block_size %lld must be a power of two <= 256",
                    (long long)ci.block_size);
    if (ci.num_blocks * ci.block_size > (int64_t(1) << 31))
        return fail(PKV_ERR_UNSUPPORTED, "pool of more than 2^31 slots");
    ci.scale_mode = c->scale_mode;
    if (c->scale_mode != PKV_SCALE_PER_HEAD && c->scale_mode != PKV_SCALE_PER_BLOCK &&
        c->scale_mode != PKV_SCALE_PER_TOKEN)
        return fail(PKV_ERR_VALUE, "scale_mode %d is not a PKV_SCALE_* value", c->scale_mode);
    if (c->scale_mode != PKV_SCALE_PER_HEAD && !pkv::is_q8(kind))
        return fail(PKV_ERR_UNSUPPORTED, "scale granularities apply to E4M3 / E5M2 / I8 caches");
    if (pkv::is_q8(kind) && c->scale_mode == PKV_SCALE_PER_HEAD && (!c->k_scale || !c->v_scale))
        return fail(PKV_ERR_NULL, "fp8 / int8 cache needs k_scale and v_scale");
    if (c->scale_mode != PKV_SCALE_PER_HEAD) {
        const bool blk = c->scale_mode == PKV_SCALE_PER_BLOCK;
        const int nd = blk ? 2 : 3;
        TRY(check_tensor(&c->k_scales, "k_scales", nd));
        TRY(check_tensor(&c->v_scales, "v_scales", nd));
        if (c->k_scales.dtype != PKV_DTYPE_F32 || c->v_scales.dtype != PKV_DTYPE_F32)
            return fail(PKV_ERR_DTYPE, "k_scales / v_scales must be F32");
        const int64_t want[3] = {ci.num_blocks, blk ? ci.num_kv_heads : ci.block_size, ci.num_kv_heads};
        for (int i = 0; i < nd; ++i) {
            if (c->k_scales.shape[i] != want[i] || c->v_scales.shape[i] != want[i])
                return fail(PKV_ERR_SHAPE, blk ? "per-block scales must be [num_blocks, num_kv_heads]"
                                               : "per-token scales must be [num_blocks, block_size, num_kv_heads]");
            if (c->k_scales.stride[i] != c->v_scales.stride[i])
                return fail(PKV_ERR_LAYOUT, "k_scales and v_scales strides differ");
        }
        ci.gs_blk = c->k_scales.stride[0];
        ci.gs_slot = blk ? 0 : c->k_scales.stride[1];
        ci.gs_head = c->k_scales.stride[blk ? 1 : 2];
    }
    if (kind == PKV_DTYPE_U3) {
        TRY(check_tensor(&c->k_qscale, "k_qscale", 3));
        TRY(check_tensor(&c->k_qzero, "k_qzero", 3));
        TRY(check_tensor(&c->v_qscale, "v_qscale", 3));
        TRY(check_tensor(&c->v_qzero, "v_qzero", 3));
        if (c->k_qscale.dtype != PKV_DTYPE_F16 || c->v_qscale.dtype != PKV_DTYPE_F16)
            return fail(PKV_ERR_DTYPE, "U3 scales must be F16");
        if (c->k_qzero.dtype != PKV_DTYPE_U8 || c->v_qzero.dtype != PKV_DTYPE_U8)
            return fail(PKV_ERR_DTYPE, "U3 zeros must be U8");
        for (int i = 0; i < 3; ++i) {
            const int64_t want = k.shape[i];
            if (c->k_qscale.shape[i] != want || c->v_qscale.shape[i] != want ||
                c->k_qzero.shape[i] != want || c->v_qzero.shape[i] != want)
                return fail(PKV_ERR_SHAPE, "U3 metadata must be [num_blocks, block_size, num_kv_heads]");
            if (c->k_qscale.stride[i] != c->v_qscale.stride[i] || c->k_qzero.stride[i] != c->v_qzero.stride[i])
                return fail(PKV_ERR_LAYOUT, "K and V metadata strides differ");
        }
    }
    return PKV_OK;
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

int launch_status(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

}  // namespace

namespace pkv {
int sm_count_current_device()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

int set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }
}  // namespace pkv

extern "C" {

const char *pkv_version(void) { return "pkv 0.1.0 (sm_103a)"; }
int pkv_abi_version(void) { return PKV_ABI_VERSION; }
const char *pkv_last_error(void) { return g_err; }

// Validation + launch parameters of each entry point, kept apart from the
// launch so that pkv_decode_step can check all three before launching any.
static int prep_slot_mapping(const pkv_tensor *block_tables, const pkv_tensor *req, const pkv_tensor *pos,
                             int block_size, const pkv_tensor *slot_mapping, int32_t *err_flag,
                             pkv::SlotMapParams &p)
{
    TRY(check_tensor(block_tables, "block_tables", 2));
    TRY(check_tensor(req, "req", 1));
    TRY(check_tensor(pos, "pos", 1));
    TRY(check_tensor(slot_mapping, "slot_mapping", 1));
    if (block_tables->dtype != PKV_DTYPE_I32 || req->dtype != PKV_DTYPE_I32 || pos->dtype != PKV_DTYPE_I32)
        return fail(PKV_ERR_DTYPE, "block_tables, req and pos must be I32");
    if (slot_mapping->dtype != PKV_DTYPE_I64) return fail(PKV_ERR_DTYPE, "slot_mapping must be I64");
    const int64_t n = req->shape[0];
    if (pos->shape[0] != n || slot_mapping->shape[0] != n)
        return fail(PKV_ERR_SHAPE, "req, pos and slot_mapping lengths differ");
    if (slot_mapping->stride[0] != 1 && n > 1) return fail(PKV_ERR_LAYOUT, "slot_mapping must be contiguous");
    if (!is_pow2(block_size)) return fail(PKV_ERR_VALUE, "block_size must be a power of two");
    p = pkv::SlotMapParams{};
    p.bt = static_cast<const int32_t *>(block_tables->data);
    p.bt_b = block_tables->stride[0];
    p.bt_j = block_tables->stride[1];
    p.batch = int(block_tables->shape[0]);
    p.max_blocks = int(block_tables->shape[1]);
    p.req = static_cast<const int32_t *>(req->data);
    p.req_stride = req->stride[0];
    p.pos = static_cast<const int32_t *>(pos->data);
    p.pos_stride = pos->stride[0];
    p.n = n;
    p.block_shift = log2i(block_size);
    p.slot_mapping = static_cast<int64_t *>(slot_mapping->data);
    p.err_flag = err_flag;
    return PKV_OK;
}

int pkv_slot_mapping(const pkv_tensor *block_tables, const pkv_tensor *req, const pkv_tensor *pos,
                     int block_size, const pkv_tensor *slot_mapping, int32_t *err_flag, void *stream)
{
    pkv::SlotMapParams p;
    TRY(prep_slot_mapping(block_tables, req, pos, block_size, slot_mapping, err_flag, p));
    return launch_status(pkv::launch_slot_mapping(p, as_stream(stream)), "slot_mapping kernel");
}

static int prep_kv_append(const pkv_tensor *k_new, const pkv_tensor *v_new, const pkv_tensor *slot_mapping,
                          const pkv_cache *cache, int32_t *err_flag, pkv::AppendParams &p, int &kind,
                          bool &vec16, const pkv_tensor *k_new_scale = nullptr,
                          const pkv_tensor *v_new_scale = nullptr)
{
    TRY(check_tensor(k_new, "k_new", 3));
    TRY(check_tensor(v_new, "v_new", 3));
    TRY(check_tensor(slot_mapping, "slot_mapping", 1));
    CacheInfo ci{};
    TRY(check_cache(cache, ci, true));
    if (k_new->dtype != v_new->dtype) return fail(PKV_ERR_DTYPE, "k_new and v_new dtypes differ");
    const int src = k_new->dtype;
    if (src != PKV_DTYPE_F16 && src != PKV_DTYPE_BF16) return fail(PKV_ERR_DTYPE, "k_new must be F16 or BF16");
    if (slot_mapping->dtype != PKV_DTYPE_I64) return fail(PKV_ERR_DTYPE, "slot_mapping must be I64");
    for (int i = 0; i < 3; ++i)
        if (k_new->shape[i] != v_new->shape[i]) return fail(PKV_ERR_SHAPE, "k_new and v_new shapes differ");
    const int64_t T = k_new->shape[0];
    if (slot_mapping->shape[0] != T) return fail(PKV_ERR_SHAPE, "slot_mapping has %lld entries, k_new %lld tokens",
                                                 (long long)slot_mapping->shape[0], (long long)T);
    if (k_new->shape[1] != ci.num_kv_heads) return fail(PKV_ERR_SHAPE, "k_new has %lld heads, cache %lld",
                                                        (long long)k_new->shape[1], (long long)ci.num_kv_heads);
    if (k_new->shape[2] != ci.head_dim) return fail(PKV_ERR_SHAPE, "k_new head_dim %lld, cache %lld",
                                                    (long long)k_new->shape[2], (long long)ci.head_dim);
    if (k_new->stride[2] != 1 || v_new->stride[2] != 1) return fail(PKV_ERR_LAYOUT, "head_dim of k_new/v_new must be contiguous");
    if ((ci.kind == PKV_DTYPE_F16 || ci.kind == PKV_DTYPE_BF16) && ci.kind != src)
        return fail(PKV_ERR_DTYPE, "16-bit cache dtype must equal the source dtype");
    if (pkv::is_q8(ci.kind) && ci.head_dim % 8 != 0)
        return fail(PKV_ERR_UNSUPPORTED, "fp8 / int8 append needs head_dim % 8 == 0");
    if (ci.kind == PKV_DTYPE_U3 && ci.head_dim != 64 && ci.head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "U3 append supports head_dim 64 and 128");
    const int64_t es = 2;
    vec16 = aligned(k_new->data, 16) && aligned(v_new->data, 16) &&
                       (k_new->stride[0] * es) % 16 == 0 && (k_new->stride[1] * es) % 16 == 0 &&
                       (v_new->stride[0] * es) % 16 == 0 && (v_new->stride[1] * es) % 16 == 0 &&
                       (ci.head_dim * 2) % 16 == 0;
    p = pkv::AppendParams{};
    p.k_new = static_cast<const char *>(k_new->data);
    p.v_new = static_cast<const char *>(v_new->data);
    p.k_src_tok = k_new->stride[0] * es;
    p.k_src_head = k_new->stride[1] * es;
    p.v_src_tok = v_new->stride[0] * es;
    p.v_src_head = v_new->stride[1] * es;
    p.slot_mapping = static_cast<const int64_t *>(slot_mapping->data);
    p.slot_stride = slot_mapping->stride[0];
    p.k_cache = static_cast<char *>(cache->k_cache.data);
    p.v_cache = static_cast<char *>(cache->v_cache.data);
    const int ces = elem_size(ci.kind);
    p.c_blk = cache->k_cache.stride[0] * ces;
    p.c_slot = cache->k_cache.stride[1] * ces;
    p.c_head = cache->k_cache.stride[2] * ces;
    p.c_chunk = ci.c_chunk;
    p.k_scale = cache->k_scale;
    p.v_scale = cache->v_scale;
    p.scale_mode = ci.scale_mode;
    if (ci.scale_mode != PKV_SCALE_PER_HEAD) {
        p.k_gs = static_cast<float *>(cache->k_scales.data);
        p.v_gs = static_cast<float *>(cache->v_scales.data);
        p.gs_blk = ci.gs_blk;
        p.gs_slot = ci.gs_slot;
        p.gs_head = ci.gs_head;
    }
    if (ci.scale_mode == PKV_SCALE_PER_TOKEN) {
        if (!k_new_scale || !v_new_scale)
            return fail(PKV_ERR_UNSUPPORTED, "a per-token-scale cache is appended with pkv_kv_append_scaled");
        TRY(check_tensor(k_new_scale, "k_new_scale", 2));
        TRY(check_tensor(v_new_scale, "v_new_scale", 2));
        if (k_new_scale->dtype != PKV_DTYPE_F32 || v_new_scale->dtype != PKV_DTYPE_F32)
            return fail(PKV_ERR_DTYPE, "k_new_scale / v_new_scale must be F32");
        if (k_new_scale->shape[0] != T || v_new_scale->shape[0] != T ||
            k_new_scale->shape[1] != ci.num_kv_heads || v_new_scale->shape[1] != ci.num_kv_heads)
            return fail(PKV_ERR_SHAPE, "new-token scales must be [num_tokens, num_kv_heads]");
        if (k_new_scale->stride[0] != v_new_scale->stride[0] || k_new_scale->stride[1] != v_new_scale->stride[1])
            return fail(PKV_ERR_LAYOUT, "k_new_scale and v_new_scale strides differ");
        p.k_ns = static_cast<const float *>(k_new_scale->data);
        p.v_ns = static_cast<const float *>(v_new_scale->data);
        p.ns_tok = k_new_scale->stride[0];
        p.ns_head = k_new_scale->stride[1];
    } else if (k_new_scale || v_new_scale) {
        return fail(PKV_ERR_VALUE, "new-token scales given for a cache without per-token scales");
    }
    if (ci.kind == PKV_DTYPE_U3) {
        p.k_qs = static_cast<uint16_t *>(cache->k_qscale.data);
        p.v_qs = static_cast<uint16_t *>(cache->v_qscale.data);
        p.k_qz = static_cast<uint8_t *>(cache->k_qzero.data);
        p.v_qz = static_cast<uint8_t *>(cache->v_qzero.data);
        p.m_blk = cache->k_qscale.stride[0];
        p.m_slot = cache->k_qscale.stride[1];
        p.m_head = cache->k_qscale.stride[2];
        p.z_blk = cache->k_qzero.stride[0];
        p.z_slot = cache->k_qzero.stride[1];
        p.z_head = cache->k_qzero.stride[2];
    }
    p.num_tokens = T;
    p.num_kv_heads = int(ci.num_kv_heads);
    p.head_dim = int(ci.head_dim);
    p.block_shift = is_pow2(ci.block_size) ? log2i(ci.block_size) : -1;
    p.block_size = ci.block_size;
    p.num_slots = ci.num_blocks * ci.block_size;
    p.src_kind = src;
    p.err_flag = err_flag;
    kind = ci.kind;
    return PKV_OK;
}

int pkv_kv_append(const pkv_tensor *k_new, const pkv_tensor *v_new, const pkv_tensor *slot_mapping,
                  const pkv_cache *cache, int32_t *err_flag, void *stream)
{
    pkv::AppendParams p;
    int kind = 0;
    bool vec16 = false;
    TRY(prep_kv_append(k_new, v_new, slot_mapping, cache, err_flag, p, kind, vec16));
    return launch_status(pkv::launch_append(p, kind, vec16, as_stream(stream)), "kv_append kernel");
}

int pkv_kv_append_scaled(const pkv_tensor *k_new, const pkv_tensor *v_new, const pkv_tensor *k_new_scale,
                         const pkv_tensor *v_new_scale, const pkv_tensor *slot_mapping, const pkv_cache *cache,
                         int32_t *err_flag, void *stream)
{
    if (!k_new_scale || !v_new_scale) return fail(PKV_ERR_NULL, "k_new_scale / v_new_scale are NULL");
    if (!cache || cache->scale_mode != PKV_SCALE_PER_TOKEN)
        return fail(PKV_ERR_VALUE, "pkv_kv_append_scaled needs a cache with scale_mode PKV_SCALE_PER_TOKEN");
    pkv::AppendParams p;
    int kind = 0;
    bool vec16 = false;
    TRY(prep_kv_append(k_new, v_new, slot_mapping, cache, err_flag, p, kind, vec16, k_new_scale, v_new_scale));
    return launch_status(pkv::launch_append(p, kind, vec16, as_stream(stream)), "kv_append kernel");
}

namespace {

struct DecodeCheck {
    CacheInfo ci;
    int64_t batch, num_heads, max_blocks;
    pkv::DecodeParams p;   // every field known before context_lens / out / workspace
    pkv::DecodePlan plan;
};

// Validate what the workspace query and the decode share, fill the launch
// parameters that follow from it, and choose the kernel: the persistent TMA
// kernel when num_splits == 0 and the shape, dtypes and layout are covered,
// else the general kernel with the requested (or a heuristic) split count.
int check_decode_common(const pkv_tensor *q, const pkv_cache *cache, const pkv_tensor *block_tables,
                        int num_splits, DecodeCheck &dc)
{
    TRY(check_tensor(q, "q", 3));
    TRY(check_cache(cache, dc.ci));
    TRY(check_tensor(block_tables, "block_tables", 2));
    if (q->dtype != PKV_DTYPE_F16 && q->dtype != PKV_DTYPE_BF16) return fail(PKV_ERR_DTYPE, "q must be F16 or BF16");
    if ((dc.ci.kind == PKV_DTYPE_F16 || dc.ci.kind == PKV_DTYPE_BF16) && dc.ci.kind != q->dtype)
        return fail(PKV_ERR_DTYPE, "16-bit cache dtype must equal q's dtype");
    if (block_tables->dtype != PKV_DTYPE_I32) return fail(PKV_ERR_DTYPE, "block_tables must be I32");
    dc.batch = q->shape[0];
    dc.num_heads = q->shape[1];
    if (q->shape[2] != dc.ci.head_dim) return fail(PKV_ERR_SHAPE, "q head_dim %lld, cache %lld",
                                                   (long long)q->shape[2], (long long)dc.ci.head_dim);
    if (dc.ci.head_dim != 64 && dc.ci.head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (q->stride[2] != 1) return fail(PKV_ERR_LAYOUT, "q head_dim must be contiguous");
    if (dc.ci.num_kv_heads <= 0 || dc.num_heads % dc.ci.num_kv_heads != 0)
        return fail(PKV_ERR_SHAPE, "num_heads %lld not a multiple of num_kv_heads %lld",
                    (long long)dc.num_heads, (long long)dc.ci.num_kv_heads);
    if (dc.num_heads / dc.ci.num_kv_heads > 16) return fail(PKV_ERR_UNSUPPORTED, "group of more than 16 q heads");
    if (block_tables->shape[0] != dc.batch) return fail(PKV_ERR_SHAPE, "block_tables has %lld rows, batch %lld",
                                                        (long long)block_tables->shape[0], (long long)dc.batch);
    dc.max_blocks = block_tables->shape[1];
    if (num_splits < 0) return fail(PKV_ERR_VALUE, "num_splits must be >= 0");

    const CacheInfo &ci = dc.ci;
    pkv::DecodeParams &p = dc.p;
    p = pkv::DecodeParams{};
    p.q = static_cast<const char *>(q->data);
    p.q_b = q->stride[0] * 2;
    p.q_h = q->stride[1] * 2;
    p.k_cache = static_cast<const char *>(cache->k_cache.data);
    p.v_cache = static_cast<const char *>(cache->v_cache.data);
    const int ces = elem_size(ci.kind);
    p.c_blk = cache->k_cache.stride[0] * ces;
    p.c_slot = cache->k_cache.stride[1] * ces;
    p.c_head = cache->k_cache.stride[2] * ces;
    p.c_chunk = ci.c_chunk;
    p.k_scale = cache->k_scale;
    p.v_scale = cache->v_scale;
    p.scale_mode = ci.scale_mode;
    if (ci.scale_mode != PKV_SCALE_PER_HEAD) {
        p.k_gs = static_cast<const float *>(cache->k_scales.data);
        p.v_gs = static_cast<const float *>(cache->v_scales.data);
        p.gs_blk = ci.gs_blk;
        p.gs_slot = ci.gs_slot;
        p.gs_head = ci.gs_head;
    }
    if (ci.kind == PKV_DTYPE_U3) {
        p.k_qs = static_cast<const uint16_t *>(cache->k_qscale.data);
        p.v_qs = static_cast<const uint16_t *>(cache->v_qscale.data);
        p.k_qz = static_cast<const uint8_t *>(cache->k_qzero.data);
        p.v_qz = static_cast<const uint8_t *>(cache->v_qzero.data);
        p.m_blk = cache->k_qscale.stride[0];
        p.m_slot = cache->k_qscale.stride[1];
        p.m_head = cache->k_qscale.stride[2];
        p.z_blk = cache->k_qzero.stride[0];
        p.z_slot = cache->k_qzero.stride[1];
        p.z_head = cache->k_qzero.stride[2];
    }
    p.block_tables = static_cast<const int32_t *>(block_tables->data);
    p.bt_b = block_tables->stride[0];
    p.bt_j = block_tables->stride[1];
    p.batch = int(dc.batch);
    p.num_heads = int(dc.num_heads);
    p.num_kv_heads = int(ci.num_kv_heads);
    p.group = int(dc.num_heads / ci.num_kv_heads);
    p.head_dim = int(ci.head_dim);
    p.block_size = int(ci.block_size);
    p.block_shift = log2i(ci.block_size);
    p.max_blocks = int(dc.max_blocks);
    p.num_blocks = int(ci.num_blocks);
    p.q_is_bf16 = q->dtype == PKV_DTYPE_BF16;

    const int sm = pkv::sm_count_current_device();
    dc.plan = pkv::DecodePlan{};
    // fp8 / int8 granular scales take the persistent kernel when each CTA's
    // heads' scales of a block are one 16-byte aligned run: per-block
    // [num_blocks, Hkv] with head stride 1, per-token head-major
    // ([num_blocks, Hkv, block_size] seen as [num_blocks, block_size, Hkv])
    int q8_gs = 0;
    bool gs_ok = ci.scale_mode == PKV_SCALE_PER_HEAD;
    if (ci.scale_mode == PKV_SCALE_PER_BLOCK) {
        q8_gs = 1;
        gs_ok = ci.gs_head == 1 && (ci.gs_blk * 4) % 16 == 0;
    } else if (ci.scale_mode == PKV_SCALE_PER_TOKEN) {
        q8_gs = int(ci.block_size);
        gs_ok = ci.gs_slot == 1 && ci.gs_head == ci.block_size && (ci.gs_blk * 4) % 16 == 0;
    }
    if (ci.scale_mode != PKV_SCALE_PER_HEAD)
        gs_ok = gs_ok && aligned(p.k_gs, 16) && aligned(p.v_gs, 16);
    // x-vectorised caches: the persistent kernel with per-head scales
    if (ci.c_chunk != 16 && ci.scale_mode != PKV_SCALE_PER_HEAD) gs_ok = false;
    if (num_splits == 0 && gs_ok &&
        pkv::fast_decode_supported(ci.kind, p.head_dim, p.block_size, p.group, p.batch)) {
        // q rows are read 16 (3-bit), 8 (fp8) or 4 (16-bit) bytes at a time
        const size_t qa = ci.kind == PKV_DTYPE_U3 ? 16 : (pkv::is_q8(ci.kind) ? 8 : 4);
        const bool q_ok = aligned(q->data, qa) && (p.q_b % qa) == 0 && (p.q_h % qa) == 0;
        // 3-bit: each block's metadata must be one contiguous, 16-byte aligned
        // run per array (staged with bulk copies), either head-major
        // [num_kv_heads][block_size] (a CTA copies its own heads) or
        // slot-major [block_size][num_kv_heads] (a CTA copies all heads)
        bool meta_ok = true, meta_hmaj = false;
        if (ci.kind == PKV_DTYPE_U3) {
            const int64_t hb = ci.block_size * ci.num_kv_heads;
            meta_hmaj = p.m_slot == 1 && p.m_head == ci.block_size && p.z_slot == 1 && p.z_head == ci.block_size;
            const bool smaj = p.m_head == 1 && p.m_slot == ci.num_kv_heads && p.z_head == 1 &&
                              p.z_slot == ci.num_kv_heads;
            meta_ok = (meta_hmaj || smaj) && (p.m_blk * 2) % 16 == 0 && p.z_blk % 16 == 0 && (hb % 16) == 0 &&
                      (ci.block_size % 16) == 0 && aligned(p.k_qs, 16) && aligned(p.v_qs, 16) &&
                      aligned(p.k_qz, 16) && aligned(p.v_qz, 16);
        }
        // 3-bit K / V tiles by one bulk copy each where the CTA's heads'
        // tiles are one run ([block][head][slot][row], the dual-stacked
        // layout); else 4-D tensor copies
        int u3_tiles = 0;
        if (ci.kind == PKV_DTYPE_U3 && aligned(p.k_cache, 16) && aligned(p.v_cache, 16) && p.c_blk % 16 == 0) {
            const int64_t row = 3 * int64_t(p.head_dim) / 8;
            if (p.c_slot == row && p.c_head == row * p.block_size) u3_tiles = 1;
        }
        pkv::FastParams f{};
        size_t ws = 0;
        if (q_ok && meta_ok && pkv::plan_fast(p.batch, p.num_heads, p.num_kv_heads, p.head_dim, p.block_size, p.max_blocks,
                                   ci.kind, meta_hmaj, sm, f, ws, q8_gs, u3_tiles) &&
            pkv::fast_maps_encodable(p, ci.kind, f.nh)) {
            dc.plan.kernel = 1;
            dc.plan.fast = f;
            dc.plan.workspace_bytes = ws;
            dc.plan.num_splits = 0;
            return PKV_OK;
        }
    }
    dc.plan = pkv::plan_decode_general(p.batch, p.num_heads, p.num_kv_heads, p.head_dim, p.block_size,
                                       p.max_blocks, num_splits, sm);
    return PKV_OK;
}

}  // namespace

int pkv_paged_decode_workspace(const pkv_tensor *q, const pkv_cache *cache, const pkv_tensor *block_tables,
                               int num_splits, size_t *bytes)
{
    if (!bytes) return fail(PKV_ERR_NULL, "bytes is NULL");
    DecodeCheck dc{};
    TRY(check_decode_common(q, cache, block_tables, num_splits, dc));
    *bytes = dc.plan.workspace_bytes;
    return ok();
}

int pkv_paged_decode_launches(const pkv_tensor *q, const pkv_cache *cache, const pkv_tensor *block_tables,
                              int num_splits, int32_t *launches)
{
    if (!launches) return fail(PKV_ERR_NULL, "launches is NULL");
    DecodeCheck dc{};
    TRY(check_decode_common(q, cache, block_tables, num_splits, dc));
    // persistent path: decode + merge; general path: decode (+ reduce when split)
    *launches = dc.plan.kernel == 1 ? 2 : (dc.plan.num_splits > 1 ? 2 : 1);
    return ok();
}

static int prep_paged_decode(const pkv_tensor *q, const pkv_cache *cache, const pkv_tensor *block_tables,
                             const pkv_tensor *context_lens, float sm_scale, const pkv_tensor *out,
                             int num_splits, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                             DecodeCheck &dc)
{
    TRY(check_decode_common(q, cache, block_tables, num_splits, dc));
    TRY(check_tensor(context_lens, "context_lens", 1));
    TRY(check_tensor(out, "out", 3));
    if (context_lens->dtype != PKV_DTYPE_I32) return fail(PKV_ERR_DTYPE, "context_lens must be I32");
    if (context_lens->shape[0] != dc.batch) return fail(PKV_ERR_SHAPE, "context_lens length differs from batch");
    if (out->dtype != q->dtype) return fail(PKV_ERR_DTYPE, "out dtype must equal q dtype");
    for (int i = 0; i < 3; ++i)
        if (out->shape[i] != q->shape[i]) return fail(PKV_ERR_SHAPE, "out shape must equal q shape");
    if (out->stride[2] != 1) return fail(PKV_ERR_LAYOUT, "out head_dim must be contiguous");
    if (!std::isfinite(sm_scale)) return fail(PKV_ERR_VALUE, "sm_scale must be finite");
    const pkv::DecodePlan &pl = dc.plan;
    if (pl.workspace_bytes > 0) {
        if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required", pl.workspace_bytes);
        if (workspace_bytes < pl.workspace_bytes)
            return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes given, %zu required", workspace_bytes,
                        pl.workspace_bytes);
        if (!aligned(workspace, 16)) return fail(PKV_ERR_LAYOUT, "workspace must be 16-byte aligned");
    }
    pkv::DecodeParams &p = dc.p;
    p.context_lens = static_cast<const int32_t *>(context_lens->data);
    p.cl_stride = context_lens->stride[0];
    p.out = static_cast<char *>(out->data);
    p.o_b = out->stride[0] * 2;
    p.o_h = out->stride[1] * 2;
    p.out_vec_ok = aligned(out->data, 16) && (p.o_b % 16) == 0 && (p.o_h % 16) == 0;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.err_flag = err_flag;
    if (pl.kernel != 1) {
        p.num_splits = pl.num_splits;
        p.chunk_tokens = pl.chunk_tokens;
        if (pl.num_splits > 1) {
            p.part_acc = static_cast<float *>(workspace);
            p.part_ml = p.part_acc + size_t(dc.batch) * dc.num_heads * pl.num_splits * dc.ci.head_dim;
        }
    }
    return PKV_OK;
}

static int launch_paged_decode(const DecodeCheck &dc, int q_dtype, void *workspace, size_t workspace_bytes,
                               void *stream)
{
    if (dc.plan.kernel == 1)
        return launch_status(pkv::launch_decode_fast(dc.p, dc.plan.fast, dc.ci.kind, workspace, workspace_bytes,
                                                     as_stream(stream)),
                             "paged_decode kernels");
    return launch_status(pkv::launch_decode(dc.p, dc.ci.kind, q_dtype, as_stream(stream)), "paged_decode kernels");
}

int pkv_paged_decode(const pkv_tensor *q, const pkv_cache *cache, const pkv_tensor *block_tables,
                     const pkv_tensor *context_lens, float sm_scale, const pkv_tensor *out, int num_splits,
                     void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream)
{
    DecodeCheck dc{};
    TRY(prep_paged_decode(q, cache, block_tables, context_lens, sm_scale, out, num_splits, workspace,
                          workspace_bytes, err_flag, dc));
    return launch_paged_decode(dc, q->dtype, workspace, workspace_bytes, stream);
}

int pkv_decode_step(const pkv_tensor *k_new, const pkv_tensor *v_new, const pkv_tensor *req,
                    const pkv_tensor *pos, const pkv_tensor *slot_mapping, const pkv_tensor *q,
                    const pkv_cache *cache, const pkv_tensor *block_tables, const pkv_tensor *context_lens,
                    float sm_scale, const pkv_tensor *out, int num_splits, void *workspace,
                    size_t workspace_bytes, int32_t *err_flag, void *stream)
{
    CacheInfo ci{};
    TRY(check_cache(cache, ci));
    pkv::SlotMapParams sp;
    TRY(prep_slot_mapping(block_tables, req, pos, int(ci.block_size), slot_mapping, err_flag, sp));
    pkv::AppendParams ap;
    int kind = 0;
    bool vec16 = false;
    TRY(prep_kv_append(k_new, v_new, slot_mapping, cache, err_flag, ap, kind, vec16));
    DecodeCheck dc{};
    TRY(prep_paged_decode(q, cache, block_tables, context_lens, sm_scale, out, num_splits, workspace,
                          workspace_bytes, err_flag, dc));
    // the append kernel computes each token's slot itself (the slot_mapping
    // kernel's rule) and writes it to slot_mapping: one launch fewer
    ap.from_pos = 1;
    ap.pos_map = sp;
    // the append writes only the cache and slot_mapping, so the decode may
    // read its inputs while the append still runs -- only when the append
    // kernel is launched (it then waits for the stream's earlier kernels
    // before letting the decode start); with no tokens there is none
    dc.p.early_inputs = ap.num_tokens > 0 ? 1 : 0;
    TRY(launch_status(pkv::launch_append(ap, kind, vec16, as_stream(stream)), "kv_append kernel"));
    return launch_paged_decode(dc, q->dtype, workspace, workspace_bytes, stream);
}

int pkv_pack3(const uint8_t *values, uint8_t *packed, int64_t n_octets, void *stream)
{
    if (n_octets < 0) return fail(PKV_ERR_VALUE, "n_octets < 0");
    if (n_octets > 0 && (!values || !packed)) return fail(PKV_ERR_NULL, "NULL pointer");
    if (!aligned(values, 16) || !aligned(packed, 4)) return fail(PKV_ERR_LAYOUT, "values must be 16-byte and packed 4-byte aligned");
    return launch_status(pkv::launch_pack3(values, packed, n_octets, as_stream(stream)), "pack3 kernel");
}

int pkv_unpack3(const uint8_t *packed, uint8_t *values, int64_t n_octets, void *stream)
{
    if (n_octets < 0) return fail(PKV_ERR_VALUE, "n_octets < 0");
    if (n_octets > 0 && (!values || !packed)) return fail(PKV_ERR_NULL, "NULL pointer");
    if (!aligned(values, 16) || !aligned(packed, 4)) return fail(PKV_ERR_LAYOUT, "values must be 16-byte and packed 4-byte aligned");
    return launch_status(pkv::launch_unpack3(packed, values, n_octets, as_stream(stream)), "unpack3 kernel");
}

int pkv_unpack3_words(const uint32_t *words, uint8_t *values, int64_t n_groups, void *stream)
{
    if (n_groups < 0) return fail(PKV_ERR_VALUE, "n_groups < 0");
    if (n_groups > 0 && (!values || !words)) return fail(PKV_ERR_NULL, "NULL pointer");
    if (!aligned(values, 16) || !aligned(words, 4)) return fail(PKV_ERR_LAYOUT, "values must be 16-byte and words 4-byte aligned");
    return launch_status(pkv::launch_unpack3_words(words, values, n_groups, as_stream(stream)), "unpack3_words kernel");
}

int pkv_copy_peak(const void *src, void *dst, size_t bytes, void *stream)
{
    if (bytes % 16 != 0) return fail(PKV_ERR_VALUE, "bytes must be a multiple of 16");
    if (bytes > 0 && (!src || !dst)) return fail(PKV_ERR_NULL, "NULL pointer");
    if (!aligned(src, 16) || !aligned(dst, 16)) return fail(PKV_ERR_LAYOUT, "pointers must be 16-byte aligned");
    return launch_status(pkv::launch_copy_peak(src, dst, bytes, as_stream(stream)), "copy kernel");
}

}  // extern "C"
