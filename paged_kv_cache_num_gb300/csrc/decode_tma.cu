// decode_tma.cu -- host side of the persistent paged-decode path: tensor
// maps, planning, and the launches of the flash-layout instances (the
// x-vectorised ones are in decode_tma_xv.cu).
#include "decode_tma_kernel.cuh"

namespace pkv {
namespace {

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 4-D map over one cache: (row element, slot, kv head, block) with the
// caller's strides; box = one 128-byte swizzled sub-row (16-bit / fp8) or one
// whole packed row (3-bit, no swizzle) x block_size slots x nh heads.
// x-vectorised caches (c_chunk != 16 bytes between a row's 16-byte pieces):
// 5-D map (element in piece, slot, piece, kv head, block), box = the whole
// [nh][head_dim/x][block_size][x] tile, no swizzle.
bool make_map(CUtensorMap *m, const void *base, int ck, int D, int BS, int Hkv, int P, int64_t c_slot,
              int64_t c_head, int64_t c_blk, int64_t c_chunk, int nh)
{
    auto enc = encode_fn();
    if (!enc) return false;
    const bool u3 = ck == kU3;
    const int es = (is_q8(ck) || u3) ? 1 : 2;
    const CUtensorMapDataType dt = (is_q8(ck) || u3) ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : ck == kBF16        ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (c_chunk != 16) {
        if (u3) return false;
        const int x = 16 / es;
        cuuint64_t dims[5] = {cuuint64_t(x), cuuint64_t(BS), cuuint64_t(D / x), cuuint64_t(Hkv), cuuint64_t(P)};
        cuuint64_t strides[4] = {cuuint64_t(c_slot), cuuint64_t(c_chunk), cuuint64_t(c_head), cuuint64_t(c_blk)};
        cuuint32_t box[5] = {cuuint32_t(x), cuuint32_t(BS), cuuint32_t(D / x), cuuint32_t(nh), 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        return enc(m, dt, 5, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const int row_elems = u3 ? 3 * D / 8 : D;
    // 16-bit and one-byte rows: 128-byte swizzled sub-rows, or one 64-byte
    // row with the 64-byte swizzle (one-byte codes at head_dim 64)
    const int sub_bytes = D * es >= 128 ? 128 : D * es;
    cuuint64_t dims[4] = {cuuint64_t(row_elems), cuuint64_t(BS), cuuint64_t(Hkv), cuuint64_t(P)};
    cuuint64_t strides[3] = {cuuint64_t(c_slot), cuuint64_t(c_head), cuuint64_t(c_blk)};
    cuuint32_t box[4] = {cuuint32_t(u3 ? row_elems : sub_bytes / es), cuuint32_t(BS), cuuint32_t(nh), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = u3 ? CU_TENSOR_MAP_SWIZZLE_NONE
                                     : (sub_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    // 3-bit boxes read runs of nh * 48-byte rows that neighbouring head
    // groups (other CTAs, at other times) continue: no L2 promotion, which
    // would fetch up to 256 bytes around each run and read the cache
    // again for the next group
    const CUtensorMapL2promotion l2p = u3 ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    const CUresult r = enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2p, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool fast_decode_supported(int cache_kind, int head_dim, int block_size, int group, int batch)
{
    if (block_size != 16 && block_size != 32 && block_size != 64) return false;
    // groups of up to 16 q heads (two groups of head columns per consumer
    // warp above 8, for blocks of up to 32 slots)
    if (group > 16 || batch > 4096) return false;
    if (group > 8 && block_size > 32) return false;
    if (is_q8(cache_kind)) return head_dim == 128 || head_dim == 64;
    if (cache_kind == kU3) return head_dim == 128;
    return (cache_kind == kF16 || cache_kind == kBF16) && (head_dim == 64 || head_dim == 128);
}

// Choose heads per CTA, stages and grid for the fast kernel.
bool plan_fast(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks,
               int cache_kind, bool meta_head_major, int sm_count, FastParams &f, size_t &workspace,
               int q8_scales_per_head, int u3_tiles)
{
    const bool u3 = cache_kind == kU3;
    const int es = is_q8(cache_kind) ? 1 : 2;
    const int row = u3 ? 3 * head_dim / 8 : head_dim * es;
    const int group = num_heads / num_kv_heads;
    // one consumer warp per kv head (at most 8 per CTA), with two groups of
    // 8 head columns for groups above 8 q heads
    const int ng = group > 8 ? 2 : 1;
    // 3-bit multi-head caches: up to 4 kv heads per consumer warp (a power
    // of two dividing num_kv_heads)
    int hpw = 1;
    if (u3 && group == 1) hpw = num_kv_heads % 4 == 0 ? 4 : (num_kv_heads % 2 == 0 ? 2 : 1);
    int nh = u3 ? (hpw > 1 ? u3_mha_max_heads(hpw) : kU3Heads) : 8;
    while (nh > 1 && (num_kv_heads % nh != 0 || 2 * nh * block_size * row > 65536)) nh >>= 1;
    if (num_kv_heads % nh != 0 || 2 * nh * block_size * row > 65536) return false;
    while (nh % hpw != 0) hpw >>= 1;
    // 3-bit kernels are register-capped so that several CTAs share an SM; the
    // shared memory (228 KB per SM, 1 KB of it reserved per CTA) and the
    // bytes kept in flight are split between them
    const int ctas_per_sm = u3 ? u3_ctas_per_sm(hpw, ng, hpw > 1 ? nh / hpw : nh) : 1;
    const int budget = (228 * 1024) / ctas_per_sm - 1024;
    // ring depth: enough bytes in flight per SM, within the shared memory
    int stages = 8;
    const int meta_heads = meta_head_major ? nh : num_kv_heads;
    // staged fp8 / int8 granular scales: K and V runs of nh * q8_scales_per_head
    // fp32, each a multiple of 16 bytes for the bulk copies
    if (q8_scales_per_head > 0 && (4 * nh * q8_scales_per_head) % 16 != 0) return false;
    // 3-bit: the staged scale / zero runs, and (outside the ring) each
    // consumer warp's fp32 conversion of them; fp8 / int8: the staged
    // granular scales
    const int meta = u3 ? 6 * block_size * meta_heads : 8 * nh * q8_scales_per_head;
    const int ncons = hpw > 1 ? nh / hpw : nh;
    const int conv = u3 ? ncons * u3_conv_bytes_per_warp(hpw, block_size) : 0;
    // bytes a CTA keeps in its ring: at most 192 KB per SM, except for the
    // 3-bit multi-head CTAs, which hold one block per step and use what the
    // shared memory allows
    const int ring_cap = u3 && hpw > 1 ? budget : 192 * 1024 / ctas_per_sm;
    if (!u3) u3_tiles = 0;
    while (stages > 2 && (stages * (2 * nh * block_size * row + meta) > ring_cap ||
                          smem_layout(nh, block_size, row, stages, batch, meta, conv).total > budget))
        --stages;
    const SmemLayout L = smem_layout(nh, block_size, row, stages, batch, meta, conv);
    if (L.total > budget) return false;
    const int n_hg = num_kv_heads / nh;
    const int64_t max_units = int64_t(n_hg) * batch * max_blocks;
    f.nh = nh;
    f.ng = ng;
    f.hpw = hpw;
    f.ncons = ncons;
    f.u3_tiles = u3_tiles;
    f.n_hg = n_hg;
    f.stages = stages;
    const int64_t slots = int64_t(sm_count) * ctas_per_sm;
    f.grid = int(max_units < slots ? (max_units > 0 ? max_units : 1) : slots);
    f.smem_bytes = L.total;
    f.meta_heads = meta_heads;
    f.meta_hmaj = meta_head_major ? 1 : 0;
    const int64_t rows = (int64_t(f.grid) + int64_t(n_hg) * batch) * nh * group;
    const size_t ml_bytes = (size_t(rows) * 2 * 4 + 255) / 256 * 256;
    workspace = ml_bytes + size_t(rows) * head_dim * 4;
    return true;
}

bool fast_maps_encodable(const DecodeParams &p, int cache_kind, int nh)
{
    CUtensorMap mk, mv;
    return make_map(&mk, p.k_cache, cache_kind, p.head_dim, p.block_size, p.num_kv_heads, p.num_blocks, p.c_slot,
                    p.c_head, p.c_blk, p.c_chunk, nh) &&
           make_map(&mv, p.v_cache, cache_kind, p.head_dim, p.block_size, p.num_kv_heads, p.num_blocks, p.c_slot,
                    p.c_head, p.c_blk, p.c_chunk, nh);
}

cudaError_t launch_decode_fast(const DecodeParams &p, FastParams f, int cache_kind, void *ws, size_t ws_bytes,
                               cudaStream_t s)
{
    const int64_t rows = (int64_t(f.grid) + int64_t(f.n_hg) * p.batch) * f.nh * p.group;
    char *c = static_cast<char *>(ws);
    const size_t ml_bytes = (size_t(rows) * 2 * 4 + 255) / 256 * 256;
    (void)ws_bytes;
    f.part_ml = reinterpret_cast<float *>(c);
    f.part_acc = reinterpret_cast<float *>(c + ml_bytes);
    CUtensorMap mk, mv;
    if (!make_map(&mk, p.k_cache, cache_kind, p.head_dim, p.block_size, p.num_kv_heads, p.num_blocks, p.c_slot,
                  p.c_head, p.c_blk, p.c_chunk, f.nh) ||
        !make_map(&mv, p.v_cache, cache_kind, p.head_dim, p.block_size, p.num_kv_heads, p.num_blocks, p.c_slot,
                  p.c_head, p.c_blk, p.c_chunk, f.nh))
        return cudaErrorInvalidValue;
    if (p.c_chunk != 16) {
        const int64_t es = is_q8(cache_kind) ? 1 : 2;
        f.xv_bulk = p.c_slot == 16 && p.c_chunk == 16 * int64_t(p.block_size) &&
                    p.c_head == int64_t(p.block_size) * p.head_dim * es;
        return launch_decode_fast_xv(p, f, cache_kind, &mk, &mv, s);
    }
    if (is_q8(cache_kind) && p.head_dim == 64) return launch_decode_fast_q8_d64(p, f, cache_kind, &mk, &mv, s);
    if (cache_kind == kE4M3) return launch_fast_bs<kE4M3, 128>(p, f, mk, mv, s);
    if (cache_kind == kE5M2) return launch_fast_bs<kE5M2, 128>(p, f, mk, mv, s);
    if (cache_kind == kI8) return launch_fast_bs<kI8, 128>(p, f, mk, mv, s);
    if (cache_kind == kU3) return launch_fast_bs<kU3, 128>(p, f, mk, mv, s);
    if (cache_kind == kBF16)
        return p.head_dim == 128 ? launch_fast_bs<kBF16, 128>(p, f, mk, mv, s) : launch_fast_bs<kBF16, 64>(p, f, mk, mv, s);
    return p.head_dim == 128 ? launch_fast_bs<kF16, 128>(p, f, mk, mv, s) : launch_fast_bs<kF16, 64>(p, f, mk, mv, s);
}

}  // namespace pkv
