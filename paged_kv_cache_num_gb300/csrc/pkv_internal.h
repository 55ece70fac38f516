// pkv_internal.h -- launch parameters shared by the C-ABI layer and the
// kernel translation units (host + device visible, no torch types).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

enum CacheKind : int { kF16 = 1, kBF16 = 2, kE4M3 = 3, kU3 = 4, kE5M2 = 9, kI8 = 10 };

// one-byte codes with a per-kv-head fp32 scale: fp8 e4m3 / e5m2 and int8
constexpr bool is_q8(int ck) { return ck == kE4M3 || ck == kE5M2 || ck == kI8; }

// ---------------------------------------------------------------- append
struct SlotMapParams {
    const int32_t *bt;
    int64_t bt_b, bt_j;
    int batch, max_blocks;
    const int32_t *req;
    int64_t req_stride;
    const int32_t *pos;
    int64_t pos_stride;
    int64_t n;
    int block_shift;
    int64_t *slot_mapping;
    int32_t *err_flag;
};
struct AppendParams {
    const char *k_new;          // source rows (bytes)
    const char *v_new;
    int64_t k_src_tok, k_src_head;  // byte strides
    int64_t v_src_tok, v_src_head;
    const int64_t *slot_mapping;
    int64_t slot_stride;        // elements
    char *k_cache;
    char *v_cache;
    int64_t c_blk, c_slot, c_head;  // byte strides of K and V caches (equal)
    int64_t c_chunk;            // byte stride between the 16-byte pieces of a row (16: contiguous)
    // fp8 / int8 scales: per kv head, or (scale_mode 1 / 2) an array indexed
    // blk * gs_blk + slot * gs_slot + head * gs_head (gs_slot = 0 per block)
    const float *k_scale;
    const float *v_scale;
    int scale_mode;
    float *k_gs;
    float *v_gs;
    int64_t gs_blk, gs_slot, gs_head;
    const float *k_ns;          // per-token mode: the new tokens' scales
    const float *v_ns;
    int64_t ns_tok, ns_head;
    // 3-bit metadata (element strides, same for the four arrays)
    uint16_t *k_qs;
    uint8_t *k_qz;
    uint16_t *v_qs;
    uint8_t *v_qz;
    int64_t m_blk, m_slot, m_head;      // strides of the fp16 scale arrays (elements)
    int64_t z_blk, z_slot, z_head;      // strides of the zero arrays (bytes)
    int64_t num_tokens;
    int num_kv_heads;
    int head_dim;
    int block_shift;            // log2(block_size), or -1 when not a power of two
    int64_t block_size;
    int64_t num_slots;          // num_blocks * block_size
    int src_kind;               // kF16 / kBF16
    int32_t *err_flag;
    // from_pos: slots are computed from (request, position) through the block
    // table (the slot_mapping kernel's rule, fused into the append) and
    // written to pos_map.slot_mapping; slot_mapping above is then unused
    int from_pos;
    SlotMapParams pos_map;
};

cudaError_t launch_append(const AppendParams &p, int cache_kind, bool vec16, cudaStream_t s);

cudaError_t launch_slot_mapping(const SlotMapParams &p, cudaStream_t s);

// ---------------------------------------------------------------- decode
struct DecodeParams {
    const char *q;              // [B, Hq, D] 16-bit
    int64_t q_b, q_h;           // byte strides
    const char *k_cache;
    const char *v_cache;
    int64_t c_blk, c_slot, c_head;  // byte strides (K and V equal)
    int64_t c_chunk;            // byte stride between the 16-byte pieces of a row (16: contiguous)
    const float *k_scale;
    const float *v_scale;
    int scale_mode;             // 0 per kv head, 1 per block, 2 per token (see AppendParams)
    const float *k_gs;
    const float *v_gs;
    int64_t gs_blk, gs_slot, gs_head;
    const uint16_t *k_qs;
    const uint8_t *k_qz;
    const uint16_t *v_qs;
    const uint8_t *v_qz;
    int64_t m_blk, m_slot, m_head;  // fp16 scale strides (elements)
    int64_t z_blk, z_slot, z_head;  // zero strides (bytes)
    const int32_t *block_tables;
    int64_t bt_b, bt_j;         // element strides
    const int32_t *context_lens;
    int64_t cl_stride;
    char *out;                  // [B, Hq, D] 16-bit
    int64_t o_b, o_h;           // byte strides
    int batch, num_heads, num_kv_heads, group, head_dim, block_size, block_shift;
    int max_blocks;
    int num_blocks;
    float scale_log2;           // sm_scale * log2(e)
    int num_splits;             // chunks per sequence (1 = write out directly)
    int chunk_tokens;           // tokens per chunk (multiple of block_size)
    float *part_acc;            // [B, Hq, num_splits, D]   (num_splits > 1)
    float *part_ml;             // [B, Hq, num_splits, 2]  (max in log2 units, sum)
    int q_is_bf16;
    int out_vec_ok;             // out rows 16-byte aligned (vector stores allowed)
    int32_t *err_flag;
    // the stream's previous kernel writes only the cache (the append of
    // pkv_decode_step): the persistent kernel then reads its inputs (q,
    // context_lens, block_tables) and writes out before its dependency wait,
    // which only the cache copies come after
    int early_inputs;
};

// Persistent TMA kernel (16-bit and fp8 caches).
struct FastParams {
    int nh;                     // kv heads per CTA
    int ng;                     // head-column groups of 8 per consumer warp: 2 when the
                                // group has more than 8 q heads (16-bit / one-byte codes)
    int n_hg;                   // head groups = num_kv_heads / nh
    int stages;                 // shared-memory ring depth
    int grid;                   // persistent CTAs
    int smem_bytes;
    int meta_heads;             // 3-bit: kv heads whose scale/zero runs a stage holds
                                // (nh when the arrays are head-major, else all)
    int meta_hmaj;              // 3-bit: 1 when the scale/zero arrays are head-major
                                // ([blocks][kv heads][slots]), 0 when slot-major
    int xv_bulk;                // x-vectorised cache whose nh head tiles of a block are
                                // one contiguous run: staged by 1-D bulk copies
    int hpw;                    // 3-bit multi-head caches: kv heads per consumer warp
                                // (1, 2 or 4); 1 otherwise
    int ncons;                  // consumer warps per CTA
    int u3_tiles;               // 3-bit K / V tiles ([head][slot][row] in shared
                                // memory): 0 by 4-D tensor copies; 1 by one bulk
                                // copy per tile (heads stored [block][head][slot][row])
    float *part_ml;             // [(grid + n_hg*B) * nh * G, 2]
    float *part_acc;            // [(grid + n_hg*B) * nh * G, D]
};

struct DecodePlan {
    int kernel;                 // 0 = general (split-K by chunks), 1 = persistent TMA
    int num_splits;
    int chunk_tokens;
    FastParams fast;
    size_t workspace_bytes;
};

DecodePlan plan_decode_general(int batch, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_blocks, int num_splits, int sm_count);

bool fast_decode_supported(int cache_kind, int head_dim, int block_size, int group, int batch);
bool plan_fast(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
               int max_blocks, int cache_kind, bool meta_head_major, int sm_count, FastParams &f,
               size_t &workspace, int q8_scales_per_head = 0, int u3_tiles = 0);
bool fast_maps_encodable(const DecodeParams &p, int cache_kind, int nh);
// x-vectorised caches (c_chunk != 16): 16-bit or one-byte codes with
// per-head scales, head_dim 128 (16-bit also 64), block size 16 / 32 / 64
// one-byte codes at head_dim 64 (decode_tma_d64.cu)
cudaError_t launch_decode_fast_q8_d64(const DecodeParams &p, const FastParams &f, int cache_kind,
                                      const void *tmk, const void *tmv, cudaStream_t s);
cudaError_t launch_decode_fast_xv(const DecodeParams &p, const FastParams &f, int cache_kind,
                                  const void *tmk, const void *tmv, cudaStream_t s);

cudaError_t launch_decode(const DecodeParams &p, int cache_kind, int q_kind, cudaStream_t s);
cudaError_t launch_decode_fast(const DecodeParams &p, FastParams f, int cache_kind, void *ws,
                               size_t ws_bytes, cudaStream_t s);

// ---------------------------------------------------------------- pack3 / copy
cudaError_t launch_pack3(const uint8_t *values, uint8_t *packed, int64_t n, cudaStream_t s);
cudaError_t launch_unpack3(const uint8_t *packed, uint8_t *values, int64_t n, cudaStream_t s);
cudaError_t launch_unpack3_words(const uint32_t *words, uint8_t *values, int64_t n,
                                 cudaStream_t s);
cudaError_t launch_copy_peak(const void *src, void *dst, size_t bytes, cudaStream_t s);

int sm_count_current_device();

// Launch `kernel` on `s` with programmatic stream serialization: it may
// begin while the stream's previous kernel finishes (see griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Record `msg` as this host thread's pkv_last_error() text; returns `code`.
int set_last_error(int code, const char *msg);

}  // namespace pkv
