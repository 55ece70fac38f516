// decode.cu -- paged flash-decoding over the block pool, and the split-K
// merge kernel.
//
// "10. Triton KV Cache and PagedAttention", reference code TODO 1-5: for each
// logical block of a sequence, look the physical block up in the block table,
// load its K/V rows, score them against the single query token, mask tokens at
// or beyond context_len to -inf, and fold the block into an online softmax
// (running max m, running sum l, accumulator acc rescaled by exp(m_old -
// m_new)); normalise at the end.  Grouped-query heads read kv head
// h / (num_heads / num_kv_heads) ("Write Triton Kv Cache Append Kernel",
// design rules).  A split of the context into chunks writes per-chunk
// (m, l, acc) triples that the merge kernel combines:
//   M = max_i m_i, L = sum_i l_i 2^(m_i - M), out = sum_i acc_i 2^(m_i - M) / L
// (the same rescaling the online softmax applies between blocks).
// Scores are kept in log2 units (the query is pre-scaled by
// sm_scale * log2(e)) so every exponential is one ex2 instruction.
//
// This file holds the general kernel: one CTA of 4 warps per (chunk, kv head,
// sequence); each warp walks steps of a few consecutive tokens of the chunk
// (every 4th step) with its lanes splitting head_dim, and keeps its own
// online-softmax state for all q heads of the group; the four states are
// merged through shared memory.  It serves every cache dtype, head_dim
// 64/128, any block size and any group size up to 16.
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kGenThreads = 128;
constexpr int kGenWarps = kGenThreads / 32;
#define kNegInf (-__int_as_float(0x7f800000))

// Load EPL consecutive elements (starting at element e0) of one cache row
// and dequantise them to float.
template <int CK, int EPL>
__device__ __forceinline__ void load_row(const char *row, int e0, float scale, float qscale,
                                         float qzero, float (&x)[EPL])
{
    if constexpr (CK == kF16 || CK == kBF16) {
        const uint16_t *r = reinterpret_cast<const uint16_t *>(row) + e0;
        if constexpr (EPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(r);
            x[0] = h2f<CK>(u.x & 0xffff); x[1] = h2f<CK>(u.x >> 16);
            x[2] = h2f<CK>(u.y & 0xffff); x[3] = h2f<CK>(u.y >> 16);
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t *>(r);
            x[0] = h2f<CK>(u & 0xffff); x[1] = h2f<CK>(u >> 16);
        }
    } else if constexpr (CK == kI8) {
        const int8_t *r = reinterpret_cast<const int8_t *>(row) + e0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] = float(r[e]) * scale;
    } else if constexpr (is_q8(CK)) {
        const uint8_t *r = reinterpret_cast<const uint8_t *>(row) + e0;
        if constexpr (EPL == 4) {
            const uint32_t u = *reinterpret_cast<const uint32_t *>(r);
            const float2 a = fp8x2_to_float2<CK, 0>(u);
            const float2 b = fp8x2_to_float2<CK, 1>(u);
            x[0] = a.x * scale; x[1] = a.y * scale; x[2] = b.x * scale; x[3] = b.y * scale;
        } else {
            const float2 a = fp8x2_to_float2<CK, 0>(uint32_t(*reinterpret_cast<const uint16_t *>(r)));
            x[0] = a.x * scale; x[1] = a.y * scale;
        }
    } else {  // kU3: element d at bits 3d..3d+2 of the little-endian row
        const uint8_t *r = reinterpret_cast<const uint8_t *>(row);
        const int bit0 = 3 * e0;
        const int byte0 = bit0 >> 3;
        const int last = (bit0 + 3 * EPL - 1) >> 3;   // last byte holding one of our bits
        uint32_t w = r[byte0];
        if (last > byte0) w |= uint32_t(r[byte0 + 1]) << 8;
        if (last > byte0 + 1) w |= uint32_t(r[byte0 + 2]) << 16;
        w >>= (bit0 & 7);
#pragma unroll
        for (int j = 0; j < EPL; ++j) x[j] = (float((w >> (3 * j)) & 7u) - qzero) * qscale;
    }
}

template <int QK, int CK, int D, int GMAX>
__global__ void __launch_bounds__(kGenThreads) decode_general_kernel(DecodeParams p)
{
    constexpr int EPL = D / 32;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = p.group;

    int ctx = p.context_lens[b * p.cl_stride];
    const int cap = p.max_blocks << p.block_shift;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) raise_err(p.err_flag, PKV_DEVERR_CONTEXT_RANGE);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int t0 = split * p.chunk_tokens;
    const int t1 = min(ctx, t0 + p.chunk_tokens);
    if (t0 >= t1) {
        if (p.num_splits == 1) {  // empty context: zero output rows
            for (int i = threadIdx.x; i < G * D; i += kGenThreads) {
                const int g = i / D, d = i % D;
                uint16_t *o = reinterpret_cast<uint16_t *>(p.out + b * p.o_b + (kvh * G + g) * p.o_h);
                o[d] = 0;
            }
        }
        return;
    }

    // query rows of the group, pre-scaled so scores come out in log2 units
    float q[GMAX][EPL];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        if (g < G) {
            const uint16_t *qr =
                reinterpret_cast<const uint16_t *>(p.q + b * p.q_b + (kvh * G + g) * p.q_h) + EPL * lane;
#pragma unroll
            for (int e = 0; e < EPL; ++e) q[g][e] = h2f<QK>(qr[e]) * p.scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) q[g][e] = 0.0f;
        }
    }
    float m[GMAX], l[GMAX], acc[GMAX][EPL];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        m[g] = kNegInf;
        l[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[g][e] = 0.0f;
    }
    const float ks = is_q8(CK) && p.scale_mode == 0 ? p.k_scale[kvh] : 1.0f;
    const float vs = is_q8(CK) && p.scale_mode == 0 ? p.v_scale[kvh] : 1.0f;
    const int bmask = (1 << p.block_shift) - 1;
    // this lane's EPL elements: packed 3-bit rows are addressed by element;
    // the others lie inside one 16-byte piece of the row, the pieces being
    // c_chunk bytes apart (x-vectorised layout) or adjacent
    int64_t eoff = 0;
    int e0 = EPL * lane;
    if constexpr (CK != kU3) {
        constexpr int ES = (CK == kF16 || CK == kBF16) ? 2 : 1;
        eoff = int64_t((EPL * lane * ES) >> 4) * p.c_chunk + ((EPL * lane * ES) & 15);
        e0 = 0;
    }

    // Each warp takes TC consecutive tokens per step (steps strided over the
    // CTA's warps).  Its lanes hold partial dot products for every (q head,
    // token) pair of the step, NV = GMAX * TC values; a transposing butterfly
    // (each xor step swaps half of the values with the partner lane) leaves
    // lane L with the full score of pair index L >> RS, replicated over
    // 2^RS lanes, for NV - 1 shuffles instead of 5 per pair.  The softmax
    // update is then one exponential per lane, and the pairs' P values are
    // broadcast for the V accumulation.
    constexpr int TC = GMAX >= 16 ? 2 : 4;                       // tokens per step
    constexpr int NV = GMAX * TC;                                // (head, token) pairs
    constexpr int LNV = NV == 32 ? 5 : (NV == 16 ? 4 : (NV == 8 ? 3 : 2));   // log2 NV
    constexpr int RS = 5 - LNV;                                  // replication bits
    const int my_pair = lane >> RS;                              // this lane's pair
    const int my_g = my_pair / TC;                               // its head
    float lsum = 0.0f;                                           // sum of P of the lane's pair slot
    for (int tb = t0 + warp * TC; tb < t1; tb += kGenWarps * TC) {
        float part[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) part[i] = 0.0f;
        float vx[TC][EPL];
        bool live[TC];
#pragma unroll
        for (int tt = 0; tt < TC; ++tt) {
            const int t = tb + tt;
            live[tt] = false;
#pragma unroll
            for (int e = 0; e < EPL; ++e) vx[tt][e] = 0.0f;
            if (t >= t1) continue;
            const int j = t >> p.block_shift, off = t & bmask;
            const int pb = p.block_tables[b * p.bt_b + j * p.bt_j];
            if (pb < 0 || pb >= p.num_blocks) {
                if (lane == 0) raise_err(p.err_flag, PKV_DEVERR_BLOCK_RANGE);
                continue;
            }
            live[tt] = true;
            const int64_t roff = pb * p.c_blk + off * p.c_slot + kvh * p.c_head;
            float kq = 1.0f, kz = 0.0f, vq = 1.0f, vz = 0.0f;
            float kst = ks, vst = vs;             // the row's fp8 / int8 scales
            if (is_q8(CK) && p.scale_mode != 0) {
                const int64_t gi = pb * p.gs_blk + off * p.gs_slot + kvh * p.gs_head;
                kst = p.k_gs[gi];
                vst = p.v_gs[gi];
            }
            if constexpr (CK == kU3) {
                kq = __half2float(__ushort_as_half(p.k_qs[pb * p.m_blk + off * p.m_slot + kvh * p.m_head]));
                vq = __half2float(__ushort_as_half(p.v_qs[pb * p.m_blk + off * p.m_slot + kvh * p.m_head]));
                kz = float(p.k_qz[pb * p.z_blk + off * p.z_slot + kvh * p.z_head]);
                vz = float(p.v_qz[pb * p.z_blk + off * p.z_slot + kvh * p.z_head]);
            }
            float kx[EPL];
            load_row<CK, EPL>(p.k_cache + roff + eoff, e0, kst, kq, kz, kx);
            load_row<CK, EPL>(p.v_cache + roff + eoff, e0, vst, vq, vz, vx[tt]);
#pragma unroll
            for (int g = 0; g < GMAX; ++g) {
                float sp = 0.0f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) sp = fmaf(q[g][e], kx[e], sp);
                part[g * TC + tt] = sp;
            }
        }
        // transposing reduction: after the halving steps lane L holds the sum
        // of pair L >> RS over the lanes that share its top LNV bits; the
        // remaining steps sum over those
#pragma unroll
        for (int st = 0; st < 5; ++st) {
            const int o = 16 >> st;
            const int n = NV >> st;                 // values still held
            if (n > 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < n / 2; ++i) {
                    const float send = up ? part[i] : part[i + n / 2];
                    const float keep = up ? part[i + n / 2] : part[i];
                    part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            } else {
                part[0] += __shfl_xor_sync(0xffffffffu, part[0], o);
            }
        }
        // this lane's pair: head my_g, token my_pair % TC
        const int my_t = my_pair % TC;
        float sc = part[0];
        {
            bool lv = false;
#pragma unroll
            for (int tt = 0; tt < TC; ++tt) lv = tt == my_t ? live[tt] : lv;
            if (!lv || my_g >= G) sc = kNegInf;   // masked token, or no such head
        }
        // chunk max per head over its TC lanes, then to every lane
        float cm = sc;
#pragma unroll
        for (int o = 1 << RS; o < (TC << RS); o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        float alpha[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            const float cmg = __shfl_sync(0xffffffffu, cm, (g * TC) << RS);
            const float mn = fmaxf(m[g], cmg);
            alpha[g] = mn == kNegInf ? 1.0f : exp2_approx(m[g] - mn);
            m[g] = mn;
        }
        float mine_m = 0.0f, mine_a = 1.0f;
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
            if (g == my_g) { mine_m = m[g]; mine_a = alpha[g]; }
        const float pe = sc == kNegInf ? 0.0f : exp2_approx(sc - mine_m);
        lsum = lsum * mine_a + pe;
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            if (g < G) {
                float pg[TC];
#pragma unroll
                for (int tt = 0; tt < TC; ++tt) pg[tt] = __shfl_sync(0xffffffffu, pe, (g * TC + tt) << RS);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    float a = acc[g][e] * alpha[g];
#pragma unroll
                    for (int tt = 0; tt < TC; ++tt) a = fmaf(pg[tt], vx[tt][e], a);
                    acc[g][e] = a;
                }
            }
        }
    }
    // the running sums: the lanes of one head hold its token slots (each
    // replicated over 2^RS lanes, which are not summed)
#pragma unroll
    for (int o = 1 << RS; o < (TC << RS); o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
#pragma unroll
    for (int g = 0; g < GMAX; ++g) l[g] = __shfl_sync(0xffffffffu, lsum, (g * TC) << RS);

    // merge the four warps' states
    __shared__ float s_m[kGenWarps][GMAX], s_l[kGenWarps][GMAX];
    __shared__ float s_acc[kGenWarps][GMAX][D];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        if (g < G) {
            if (lane == 0) { s_m[warp][g] = m[g]; s_l[warp][g] = l[g]; }
#pragma unroll
            for (int e = 0; e < EPL; ++e) s_acc[warp][g][EPL * lane + e] = acc[g][e];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += kGenThreads) {
        const int g = i / D, d = i % D;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kGenWarps; ++w) M = fmaxf(M, s_m[w][g]);
        float L = 0.0f, A = 0.0f;
        if (M != kNegInf) {
#pragma unroll
            for (int w = 0; w < kGenWarps; ++w) {
                const float f = exp2_approx(s_m[w][g] - M);
                L += s_l[w][g] * f;
                A += s_acc[w][g][d] * f;
            }
        }
        const int h = kvh * G + g;
        if (p.num_splits == 1) {
            uint16_t *o = reinterpret_cast<uint16_t *>(p.out + b * p.o_b + h * p.o_h);
            o[d] = f2h<QK>(L > 0.0f ? A / L : 0.0f);
        } else {
            const int64_t pi = (int64_t(b) * p.num_heads + h) * p.num_splits + split;
            p.part_acc[pi * D + d] = A;
            if (d == 0) { p.part_ml[2 * pi] = M; p.part_ml[2 * pi + 1] = L; }
        }
    }
}

// Merge the per-chunk partials of one (sequence, q head) per CTA.
template <int QK, int D>
__global__ void __launch_bounds__(D) splitk_reduce_kernel(DecodeParams p)
{
    const int bh = blockIdx.x;
    const int b = bh / p.num_heads, h = bh % p.num_heads;
    const int d = threadIdx.x;
    int ctx = p.context_lens[b * p.cl_stride];
    const int cap = p.max_blocks << p.block_shift;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int n = (ctx + p.chunk_tokens - 1) / p.chunk_tokens;   // chunks that hold tokens
    const int64_t base = int64_t(bh) * p.num_splits;
    float M = kNegInf;
    for (int i = 0; i < n; ++i) M = fmaxf(M, p.part_ml[2 * (base + i)]);
    float L = 0.0f, A = 0.0f;
    if (M != kNegInf) {
        for (int i = 0; i < n; ++i) {
            const float f = exp2_approx(p.part_ml[2 * (base + i)] - M);
            L += p.part_ml[2 * (base + i) + 1] * f;
            A += p.part_acc[(base + i) * D + d] * f;
        }
    }
    uint16_t *o = reinterpret_cast<uint16_t *>(p.out + b * p.o_b + h * p.o_h);
    o[d] = f2h<QK>(L > 0.0f ? A / L : 0.0f);
}

template <int QK, int CK, int D>
cudaError_t launch_general(const DecodeParams &p, cudaStream_t s)
{
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    if (p.group <= 1) decode_general_kernel<QK, CK, D, 1><<<grid, kGenThreads, 0, s>>>(p);
    else if (p.group <= 2) decode_general_kernel<QK, CK, D, 2><<<grid, kGenThreads, 0, s>>>(p);
    else if (p.group <= 4) decode_general_kernel<QK, CK, D, 4><<<grid, kGenThreads, 0, s>>>(p);
    else if (p.group <= 8) decode_general_kernel<QK, CK, D, 8><<<grid, kGenThreads, 0, s>>>(p);
    else decode_general_kernel<QK, CK, D, 16><<<grid, kGenThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.num_splits == 1) return e;
    splitk_reduce_kernel<QK, D><<<p.batch * p.num_heads, D, 0, s>>>(p);
    return cudaGetLastError();
}

template <int QK, int CK>
cudaError_t launch_by_dim(const DecodeParams &p, cudaStream_t s)
{
    return p.head_dim == 128 ? launch_general<QK, CK, 128>(p, s) : launch_general<QK, CK, 64>(p, s);
}

}  // namespace

DecodePlan plan_decode_general(int batch, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_blocks, int num_splits, int sm_count)
{
    DecodePlan pl{};
    pl.kernel = 0;
    const int64_t max_ctx = int64_t(max_blocks) * block_size;
    int64_t chunk;
    if (num_splits > 0) {
        chunk = (max_ctx + num_splits - 1) / num_splits;
    } else {
        const int64_t base = int64_t(batch) * num_kv_heads;
        const int64_t want = int64_t(4) * sm_count;
        const int64_t splits = base >= want ? 1 : (want + base - 1) / base;
        chunk = (max_ctx + splits - 1) / splits;
        if (chunk < 256) chunk = 256;
    }
    chunk = (chunk + block_size - 1) / block_size * block_size;
    if (chunk < block_size) chunk = block_size;
    int64_t splits = max_ctx > 0 ? (max_ctx + chunk - 1) / chunk : 1;
    if (splits < 1) splits = 1;
    pl.num_splits = int(splits);
    pl.chunk_tokens = int(chunk);
    pl.workspace_bytes = splits > 1 ? size_t(batch) * num_heads * splits * (head_dim + 2) * 4 : 0;
    return pl;
}

cudaError_t launch_decode(const DecodeParams &p, int cache_kind, int q_kind, cudaStream_t s)
{
    if (p.batch == 0) return cudaSuccess;
    if (q_kind == kBF16) {
        switch (cache_kind) {
        case kBF16: return launch_by_dim<kBF16, kBF16>(p, s);
        case kE4M3: return launch_by_dim<kBF16, kE4M3>(p, s);
        case kE5M2: return launch_by_dim<kBF16, kE5M2>(p, s);
        case kI8: return launch_by_dim<kBF16, kI8>(p, s);
        case kU3: return launch_by_dim<kBF16, kU3>(p, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (cache_kind) {
    case kF16: return launch_by_dim<kF16, kF16>(p, s);
    case kE4M3: return launch_by_dim<kF16, kE4M3>(p, s);
    case kE5M2: return launch_by_dim<kF16, kE5M2>(p, s);
    case kI8: return launch_by_dim<kF16, kI8>(p, s);
    case kU3: return launch_by_dim<kF16, kU3>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
