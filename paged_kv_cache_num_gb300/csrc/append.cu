// append.cu -- KV-cache append (scatter through slot_mapping) and the
// device slot_mapping builder.
//
// "Write Triton Kv Cache Append Kernel": one writer per (token, kv head) row
// (reasoning step 2), a scalar slot load and an early exit on slot < 0 placed
// before any K/V load (steps 3, design rules), paged destination
// blk = slot / block_size, off = slot % block_size with a power-of-two block
// size done as shift / mask (step 5, design rules), all strides passed in
// (design rules), fp8 quantisation with the scale division in fp32 before
// the cast (step 6).  The 3-bit store follows the "triton-3bit-kv-cache-
// kernel" README section 1.A octet layout.
//
// GB300 mapping: the copy and fp8 kernels give each thread one 16-byte
// chunk of a row, so a warp covers two 256-byte bf16 rows with fully
// coalesced 16-byte loads and stores; the grid is a function of num_tokens
// only (CUDA-graph safe).  The 3-bit kernel gives each warp one row: the
// min / max are warp-shuffle reductions and the packing goes through shared
// memory.  All are programmatic dependent launches, so the launch of each
// overlaps the tail of the previous kernel in the stream.
#include <type_traits>

#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

__device__ __forceinline__ bool resolve_slot(const AppendParams &p, int64_t t, int64_t &blk,
                                             int64_t &off)
{
    const int64_t slot = p.slot_mapping[t * p.slot_stride];
    if (slot < 0) return false;                 // padding token: nothing to read or write
    if (slot >= p.num_slots) {
        raise_err(p.err_flag, PKV_DEVERR_SLOT_RANGE);
        return false;
    }
    if (p.block_shift >= 0) {
        blk = slot >> p.block_shift;
        off = slot & ((int64_t(1) << p.block_shift) - 1);
    } else {                                    // e.g. one block per request of max_seq_len
        blk = slot / p.block_size;
        off = slot - blk * p.block_size;
    }
    return true;
}

// 16-bit copy: one thread per CHUNK-byte piece of one K or V row.
template <int CHUNK>
__global__ void __launch_bounds__(kAppendThreads) append_copy_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    const int chunks_per_row = p.head_dim * 2 / CHUNK;
    const int64_t per_token = int64_t(2) * p.num_kv_heads * chunks_per_row;
    const int64_t total = p.num_tokens * per_token;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = i / per_token;
        int r = int(i - t * per_token);
        const int c = r % chunks_per_row;
        r /= chunks_per_row;
        const int h = r % p.num_kv_heads;
        const int kv = r / p.num_kv_heads;       // 0 = K, 1 = V
        int64_t blk, off;
        if (!resolve_slot(p, t, blk, off)) continue;
        const char *src = kv ? p.v_new + t * p.v_src_tok + h * p.v_src_head
                             : p.k_new + t * p.k_src_tok + h * p.k_src_head;
        char *dst = (kv ? p.v_cache : p.k_cache) + blk * p.c_blk + off * p.c_slot + h * p.c_head;
        // the row's 16-byte pieces are c_chunk bytes apart (16 when contiguous)
        if constexpr (CHUNK == 16) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + c);
            *reinterpret_cast<uint4 *>(dst + c * p.c_chunk) = v;
        } else {
            *reinterpret_cast<uint16_t *>(dst + (c >> 3) * p.c_chunk + 2 * (c & 7)) =
                reinterpret_cast<const uint16_t *>(src)[c];
        }
    }
}

// Two values already divided by the scale -> two one-byte codes (low byte
// first): fp8 satfinite casts, or int8 nearest-even saturated to +-127
// (NaN -> 0).
template <int Q8>
__device__ __forceinline__ uint32_t q8x2_encode(float2 x)
{
    if constexpr (Q8 == kI8) {
        auto one = [](float v) -> uint32_t {
            int c = isnan(v) ? 0 : __float2int_rn(fminf(fmaxf(v, -127.0f), 127.0f));
            return uint32_t(c) & 0xffu;
        };
        return one(x.x) | (one(x.y) << 8);
    } else {
        return __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, Q8 == kE4M3 ? __NV_E4M3 : __NV_E5M2);
    }
}

// One-byte codes (e4m3, e5m2, int8): one thread per 8 elements (16 source
// bytes -> 8 cache bytes).
template <int SRC, bool VEC, int FP8>
__global__ void __launch_bounds__(kAppendThreads) append_fp8_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    const int groups = p.head_dim / 8;
    const int64_t per_token = int64_t(2) * p.num_kv_heads * groups;
    const int64_t total = p.num_tokens * per_token;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = i / per_token;
        int r = int(i - t * per_token);
        const int c = r % groups;
        r /= groups;
        const int h = r % p.num_kv_heads;
        const int kv = r / p.num_kv_heads;
        int64_t blk, off;
        if (!resolve_slot(p, t, blk, off)) continue;
        const uint16_t *src = reinterpret_cast<const uint16_t *>(
            kv ? p.v_new + t * p.v_src_tok + h * p.v_src_head
               : p.k_new + t * p.k_src_tok + h * p.k_src_head) + 8 * c;
        // elements 8c .. 8c+7: half of the row's 16-byte piece c / 2
        uint8_t *dst = reinterpret_cast<uint8_t *>((kv ? p.v_cache : p.k_cache) + blk * p.c_blk +
                                                   off * p.c_slot + h * p.c_head + (c >> 1) * p.c_chunk) +
                       8 * (c & 1);
        float scale;
        if (p.scale_mode == 0) {                // per kv head
            scale = (kv ? p.v_scale : p.k_scale)[h];
        } else if (p.scale_mode == 1) {         // the block's scale for this head
            scale = (kv ? p.v_gs : p.k_gs)[blk * p.gs_blk + h * p.gs_head];
        } else {                                // the token's own, kept at its slot
            scale = (kv ? p.v_ns : p.k_ns)[t * p.ns_tok + h * p.ns_head];
            if (c == 0) (kv ? p.v_gs : p.k_gs)[blk * p.gs_blk + off * p.gs_slot + h * p.gs_head] = scale;
        }
        uint16_t e[8];
        if constexpr (VEC) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
            e[0] = v.x & 0xffff; e[1] = v.x >> 16; e[2] = v.y & 0xffff; e[3] = v.y >> 16;
            e[4] = v.z & 0xffff; e[5] = v.z >> 16; e[6] = v.w & 0xffff; e[7] = v.w >> 16;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = src[j];
        }
        uint32_t packed[2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // scale division in fp32 (IEEE round to nearest), then the cast
            float2 x;
            x.x = __fdiv_rn(h2f<SRC>(e[2 * j]), scale);
            x.y = __fdiv_rn(h2f<SRC>(e[2 * j + 1]), scale);
            const uint32_t two = q8x2_encode<FP8>(x);
            if (j & 1) packed[j >> 1] |= two << 16; else packed[j >> 1] = two;
        }
        if constexpr (VEC) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = uint8_t(packed[j >> 2] >> (8 * (j & 3)));
        }
    }
}

// 3-bit affine quantise + pack: one warp per (token, head, K|V) row.
// Each lane holds head_dim / 32 consecutive elements.
template <int SRC, int EPL>
__global__ void __launch_bounds__(kAppendThreads) append_u3_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int D = EPL * 32;
    constexpr int WARPS = kAppendThreads / 32;
    __shared__ uint8_t codes[WARPS][D];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t rows = p.num_tokens * p.num_kv_heads * 2;
    for (int64_t row = blockIdx.x * int64_t(WARPS) + wid; row < rows;
         row += int64_t(gridDim.x) * WARPS) {
        const int64_t t = row / (2 * p.num_kv_heads);
        const int r = int(row - t * 2 * p.num_kv_heads);
        const int h = r >> 1, kv = r & 1;
        int64_t blk, off;
        if (!resolve_slot(p, t, blk, off)) continue;   // warp-uniform
        const uint16_t *src = reinterpret_cast<const uint16_t *>(
            kv ? p.v_new + t * p.v_src_tok + h * p.v_src_head
               : p.k_new + t * p.k_src_tok + h * p.k_src_head) + EPL * lane;
        float x[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) x[j] = h2f<SRC>(src[j]);
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int j = 1; j < EPL; ++j) { mn = fminf(mn, x[j]); mx = fmaxf(mx, x[j]); }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        // s = fp16_rn((max - min) / 7), saturated to the largest finite fp16
        const float s32 = __fdiv_rn(__fsub_rn(mx, mn), 7.0f);
        uint16_t sbits = __half_as_ushort(__float2half_rn(s32));
        if ((sbits & 0x7fff) == 0x7c00) sbits = 0x7bff;
        const float s = __half2float(__ushort_as_half(sbits));
        float z = 0.0f;
        if (s != 0.0f) z = fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.0f), 7.0f);
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            float q = 0.0f;
            if (s != 0.0f) q = fminf(fmaxf(__fadd_rn(rintf(__fdiv_rn(x[j], s)), z), 0.0f), 7.0f);
            codes[wid][EPL * lane + j] = uint8_t(q);
        }
        __syncwarp();
        uint8_t *dst = reinterpret_cast<uint8_t *>((kv ? p.v_cache : p.k_cache) + blk * p.c_blk +
                                                   off * p.c_slot + h * p.c_head);
        if (lane < D / 8) {            // one octet (8 codes -> 3 bytes) per lane
            const uint8_t *v = &codes[wid][8 * lane];
            uint32_t w24 = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) w24 |= uint32_t(v[i] & 7) << (3 * i);
            dst[3 * lane + 0] = uint8_t(w24);
            dst[3 * lane + 1] = uint8_t(w24 >> 8);
            dst[3 * lane + 2] = uint8_t(w24 >> 16);
        }
        if (lane == 0) {
            uint16_t *qs = kv ? p.v_qs : p.k_qs;
            uint8_t *qz = kv ? p.v_qz : p.k_qz;
            qs[blk * p.m_blk + off * p.m_slot + h * p.m_head] = sbits;
            qz[blk * p.z_blk + off * p.z_slot + h * p.z_head] = uint8_t(z);
        }
        __syncwarp();
    }
}

__global__ void slot_mapping_kernel(SlotMapParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < p.n;
         t += int64_t(gridDim.x) * blockDim.x) {
        const int32_t pos = p.pos[t * p.pos_stride];
        const int32_t req = p.req[t * p.req_stride];
        int64_t slot = -1;
        if (pos >= 0) {
            const int32_t logical = pos >> p.block_shift;
            if (logical >= p.max_blocks || req < 0 || req >= p.batch) {
                raise_err(p.err_flag, PKV_DEVERR_POS_RANGE);
            } else {
                const int64_t blk = p.bt[req * p.bt_b + logical * p.bt_j];
                slot = (blk << p.block_shift) + (pos & ((1 << p.block_shift) - 1));
            }
        }
        p.slot_mapping[t] = slot;
    }
}

int grid_for(int64_t work, int threads)
{
    const int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = int64_t(sm_count_current_device()) * 16;
    return int(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, int cache_kind, bool vec16, cudaStream_t s)
{
    if (p.num_tokens == 0) return cudaSuccess;
    const int T = kAppendThreads;
    if (cache_kind == kF16 || cache_kind == kBF16) {
        if (vec16) {
            const int64_t work = p.num_tokens * 2 * p.num_kv_heads * (p.head_dim * 2 / 16);
            return launch_pdl(append_copy_kernel<16>, grid_for(work, T), T, 0, s, p);
        } else {
            const int64_t work = p.num_tokens * 2 * p.num_kv_heads * p.head_dim;
            return launch_pdl(append_copy_kernel<2>, grid_for(work, T), T, 0, s, p);
        }
    } else if (is_q8(cache_kind)) {
        const int64_t work = p.num_tokens * 2 * p.num_kv_heads * (p.head_dim / 8);
        const int g = grid_for(work, T);
        auto go = [&](auto src_c, auto vec_c) -> cudaError_t {
            constexpr int S = decltype(src_c)::value;
            constexpr bool V = decltype(vec_c)::value;
            if (cache_kind == kE4M3) return launch_pdl(append_fp8_kernel<S, V, kE4M3>, g, T, 0, s, p);
            if (cache_kind == kE5M2) return launch_pdl(append_fp8_kernel<S, V, kE5M2>, g, T, 0, s, p);
            return launch_pdl(append_fp8_kernel<S, V, kI8>, g, T, 0, s, p);
        };
        using BF = std::integral_constant<int, kBF16>;
        using HF = std::integral_constant<int, kF16>;
        if (p.src_kind == kBF16)
            return vec16 ? go(BF{}, std::true_type{}) : go(BF{}, std::false_type{});
        return vec16 ? go(HF{}, std::true_type{}) : go(HF{}, std::false_type{});
    } else {  // kU3
        const int64_t rows = p.num_tokens * 2 * p.num_kv_heads;
        const int g = grid_for(rows * 32, T);
        const bool bf = p.src_kind == kBF16;
        if (p.head_dim == 128) {
            if (bf) return launch_pdl(append_u3_kernel<kBF16, 4>, g, T, 0, s, p);
            else return launch_pdl(append_u3_kernel<kF16, 4>, g, T, 0, s, p);
        } else {
            if (bf) return launch_pdl(append_u3_kernel<kBF16, 2>, g, T, 0, s, p);
            else return launch_pdl(append_u3_kernel<kF16, 2>, g, T, 0, s, p);
        }
    }
    return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const SlotMapParams &p, cudaStream_t s)
{
    if (p.n == 0) return cudaSuccess;
    return launch_pdl(slot_mapping_kernel, grid_for(p.n, 256), 256, 0, s, p);
}

}  // namespace pkv
