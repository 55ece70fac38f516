#pragma once
// decode_tma_kernel.cuh -- the fast paged-decode path for 16-bit, fp8 and 3-bit caches:
// a persistent, load-balanced kernel that streams whole physical blocks into
// shared memory with TMA and runs both products of each block on tensor
// cores, plus the merge kernel for sequences split across CTAs.
//
// What it computes is "10. Triton KV Cache and PagedAttention", reference
// code TODO 1-5 (block-table lookup, masked K/V tile, scores, online softmax,
// V accumulation, final normalisation), with grouped-query heads
// ("Write Triton Kv Cache Append Kernel", design rules) and a split of long
// contexts whose partial (m, l, acc) triples are merged by log-sum-exp
// rescaling.
//
// Work decomposition.  The unit of work is one physical block of one group
// of `nh` kv heads.  All (head group, sequence, logical block) units are laid
// out in one flat index space (head group major, then sequence, then block)
// and CTA i of the persistent grid takes the contiguous range
// [i*N/S, (i+1)*N/S): every CTA streams the same number of blocks, whatever
// the mix of context lengths.  A CTA's range crosses sequence boundaries; each
// maximal run of one (head group, sequence) inside it is a segment.  A segment
// that covers its whole sequence writes the output directly; otherwise it
// writes an fp32 partial in slot (CTA index + unit index), which is unique
// because both grow along the flat order, and the merge kernel combines the
// partials of the CTAs that cover the unit.
//
// CTA layout.  nh consumer warps (one per kv head of the group) and one
// producer warp.  The producer resolves 32 block-table entries at a time
// (one per lane) and issues, per block, TMA tensor copies of the K and V
// tiles [nh heads][block_size tokens][head_dim] (128-byte swizzled rows) into
// a ring of `stages` shared-memory stages guarded by full/empty mbarriers.
// x-vectorised caches ([blocks][kv heads][head_dim/x][block_size][x], x
// elements = 16 bytes) arrive as stored, [nh][head_dim/x][block_size][16 B]:
// the eight rows an ldmatrix phase reads are then 128 consecutive bytes, so
// they need no swizzle.  When the nh heads' tiles of a block are one
// contiguous run (the packed layout), each is staged by a single 1-D bulk
// copy instead of a tensor copy made of 16-byte rows.
// Each consumer warp computes, for its kv head and the G <= 8 query heads
// that share it, with m16n8k16 mma.sync (block tokens on M, q heads on N):
//   S^T = K Q^T (K from shared memory by ldmatrix, or fp8 / 3-bit codes
//   converted to f16 in registers), masking of tokens >= context_len, online
//   softmax per q head in log2 units, O^T = O^T * alpha + V^T P^T (P^T moved
//   from the score accumulators into operand layout by movmatrix; V^T by
//   ldmatrix.trans, or fp8 / 3-bit code pairing + conversion).  3-bit
//   blocks also bring their per-token scale / zero runs with bulk copies.
// Every wait is bounded (about 2 s of wall time) and raises
// PKV_DEVERR_TIMEOUT instead of hanging.
#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxDevices = 64;
#define NEG_INF (-__int_as_float(0x7f800000))

struct SmemLayout {
    int tile_bytes, meta_bytes, stage_bytes, conv_off, bars_off, ok_off, prefix_off, nblk_off, total;
};

// [stages x (K tile, V tile, staged scales / 3-bit metadata of the block)]
// [3-bit: each consumer warp's fp32 conversion of its heads' metadata]
// [mbarriers] [per-stage block ids] [prefix sums] [block counts]
__host__ __device__ inline SmemLayout smem_layout(int nh, int bs, int row_bytes, int stages,
                                                  int batch, int meta_bytes = 0, int conv_bytes = 0)
{
    SmemLayout L;
    L.tile_bytes = nh * bs * row_bytes;
    L.meta_bytes = meta_bytes;
    // TMA writes each tile at a 1024-byte (swizzled tiles: rows of 64, 128
    // or 256 bytes) or 128-byte (unswizzled 3-bit tiles) aligned shared
    // address, so stages are rounded up to that.  (Tiles are multiples of 768
    // bytes (3-bit) or 2048 bytes (others) at block 16+, so only the staged
    // scales / metadata can leave a stage unaligned.)
    const int align = row_bytes % 64 == 0 ? 1024 : 128;
    L.stage_bytes = (2 * L.tile_bytes + meta_bytes + align - 1) / align * align;
    L.conv_off = stages * L.stage_bytes;
    L.bars_off = L.conv_off + (conv_bytes + 15) / 16 * 16;
    L.ok_off = L.bars_off + 2 * stages * 8;
    L.prefix_off = L.ok_off + stages * 4;
    L.nblk_off = L.prefix_off + (batch + 1) * 4;
    L.total = L.nblk_off + batch * 4 + 1024;   // + alignment slack
    return L;
}

// largest b in [0, B) with prefix[b] <= r, for 0 <= r < prefix[B]
__device__ __forceinline__ int find_seq(const int *prefix, int B, int r)
{
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= r) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi, float &rlo, float &rhi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    const float2 r = __bfloat1622float2(v);
    rlo = r.x;
    rhi = r.y;
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi, float &rlo, float &rhi)
{
    const __half2 v = __floats2half2_rn(lo, hi);
    const float2 r = __half22float2(v);
    rlo = r.x;
    rhi = r.y;
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Two one-byte codes of cache kind CK, bytes 2HI and 2HI+1 of w (low byte
// first) -> an f16x2 register, exactly: e4m3 through cvt.rn.f16x2 on the
// 16-bit half of the register (no shift); e5m2 by a byte permute alone (an
// e5m2 code -- sign, 5 exponent bits with the f16 bias, 2 mantissa bits --
// is the high byte of the f16 of the same value, subnormals, infinities and
// NaN included); int8 c as 1152 + c (a byte permute puts c next to the
// exponent of 1024 and an XOR of the byte's top bit adds 128), the 1152
// offset being removed in fp32 after the MMA.
template <int CK, int HI>
__device__ __forceinline__ uint32_t f16x2_from_q8(uint32_t w)
{
    uint32_t r;
    if constexpr (CK == kI8) {
        r = ptx::prmt(w, 0x64646464u, HI ? 0x4342u : 0x4140u) ^ 0x00800080u;
    } else if constexpr (CK == kE4M3) {
        if constexpr (HI)
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}" : "=r"(r) : "r"(w));
        else
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, l;\n}" : "=r"(r) : "r"(w));
    } else {
        r = ptx::prmt(w, 0u, HI ? 0x3424u : 0x1404u);   // codes to the high bytes, zero low bytes
    }
    return r;
}

constexpr float kI8Bias = 1152.0f;

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// ---------------------------------------------------------------- 3-bit
// A 3-bit code v placed at bit x <= 7 of an otherwise zero 16-bit half is
// the f16 subnormal v * 2^(x - 24): exact, and never a NaN or an infinity
// whatever the bits around it.  Products with normal f16 operands are exact
// in the fp32 accumulators, so the factor 2^(x - 24) is folded into q' on
// the K side and into the output on the V side, and no offset has to be
// removed after the MMA.  One LOP3 (mask) makes a pair; the windows the
// masks apply to are the costly part and are shared between pairs.
//
// K side: the A fragments of S^T = K Q'^T pair two codes of one token row.
// A 96-bit group (32 codes, lane i at bits 3i..3i+2) is cut into seven
// 32-bit windows -- its three words and four shifts -- and each window
// gives up to three pairs, lane i at bit x and lane j at bit 16 + y.
struct U3KPair {
    int s, i, j, x, y;   // window = bits s .. s+31 of the group
};
__host__ __device__ constexpr U3KPair u3k_pair_info(int p)
{
    switch (p) {
    case 0: return {0, 0, 7, 0, 5};
    case 1: return {0, 1, 6, 3, 2};
    case 2: return {4, 2, 9, 2, 7};
    case 3: return {4, 3, 8, 5, 4};
    case 4: return {10, 4, 11, 2, 7};
    case 5: return {10, 5, 10, 5, 4};
    case 6: return {32, 12, 17, 4, 3};
    case 7: return {32, 13, 18, 7, 6};
    case 8: return {41, 14, 21, 1, 6};
    case 9: return {41, 15, 20, 4, 3};
    case 10: return {41, 16, 19, 7, 0};
    case 11: return {64, 22, 27, 2, 1};
    case 12: return {64, 23, 28, 5, 4};
    case 13: return {71, 24, 31, 1, 6};
    case 14: return {71, 25, 30, 4, 3};
    default: return {71, 26, 29, 7, 0};
    }
}

// Pair p of the group held in words (w0, w1, w2); p is a constant after
// unrolling, so the window choice folds away (and equal windows are shared).
__device__ __forceinline__ uint32_t u3k_pair(int p, uint32_t w0, uint32_t w1, uint32_t w2)
{
    const U3KPair pr = u3k_pair_info(p);
    uint32_t win;
    if (pr.s == 0) win = w0;
    else if (pr.s < 32) win = __funnelshift_r(w0, w1, pr.s);
    else if (pr.s == 32) win = w1;
    else if (pr.s < 64) win = __funnelshift_r(w1, w2, pr.s - 32);
    else if (pr.s == 64) win = w2;
    else win = w2 >> (pr.s - 64);
    return win & ((7u << pr.x) | (7u << (16 + pr.y)));
}

// V side: the A fragments of O^T = V'^T P'^T pair one code of two tokens.
// A lane owns the 16 codes of bytes 6g .. 6g+5 of a row (g = its group id);
// code c of that slice lies in the 16-bit piece that starts at slice byte
// u3v_win(c), at bit u3v_x(c) of it.  A byte permute puts the piece of
// token A in the low half and that of token B in the high half.
__host__ __device__ constexpr int u3v_win(int c)
{
    return c < 3 ? 0 : c < 6 ? 1 : c < 8 ? 2 : c < 11 ? 3 : c < 14 ? 4 : 5;
}
__host__ __device__ constexpr int u3v_x(int c) { return 3 * c - 8 * u3v_win(c); }

// CK: cache kind (kF16 / kBF16 / kE4M3 / kE5M2 / kU3); D head_dim; BS block size.
// MMA operand type: bf16 for bf16 caches, f16 otherwise (fp8 codes convert
// exactly to f16).
template <int CK, int D, int BS>
struct Tile {
    static constexpr bool kFp8 = is_q8(CK);
    static constexpr bool kIsU3 = CK == pkv::kU3;
    static constexpr bool kBF = CK == kBF16;
    static constexpr int ES = (kFp8 || kIsU3) ? 1 : 2;
    static constexpr int ROW = kIsU3 ? 3 * D / 8 : D * ES;   // bytes per token row
    // swizzled sub-rows: 128 bytes (128-byte swizzle), or the whole 64-byte
    // row of one-byte codes at head_dim 64 (64-byte swizzle)
    static constexpr int SROW = kIsU3 ? ROW : (ROW >= 128 ? 128 : ROW);
    static constexpr int HALVES = kIsU3 ? 1 : ROW / SROW;    // sub-rows per row
    static constexpr int BOX0 = kIsU3 ? ROW : SROW / ES;     // TMA box inner extent (elements)
    static constexpr int KT = BS / 16;              // PV k-steps
    static constexpr int DT = D / 8;                // output n-tiles
    static constexpr int QK = D / 16;               // QK k-steps
};

// 3-bit caches: CTAs of (at most) 4 kv heads, three per SM -- the consumers
// are latency-bound on the unpacking and gain from more warps per SM, and
// 3 x 5 warps keep at most 4 warps (128 registers each) per SM sub-partition.
// The others: CTAs of up to 8 kv heads, one per SM.
constexpr int kU3Heads = 4;
constexpr int kU3CtasPerSm = 3;
// 3-bit multi-head caches with HPW kv heads per consumer warp: CTAs of up to
// 8 HPW kv heads -- eight consumer warps and a producer, one per SM, whose
// per-block copies are then whole runs of the block's heads (with fewer
// heads, four consumer warps or fewer: two CTAs per SM).  Their register
// cap is that of nine warps (three per SM sub-partition: 168).
__host__ __device__ constexpr int u3_mha_max_heads(int hpw) { return 8 * hpw; }
// 3-bit CTAs per SM by kv heads per consumer warp, head-column groups and
// consumer warps (two groups of 8 q heads hold twice the accumulators: two
// CTAs per SM)
__host__ __device__ constexpr int u3_ctas_per_sm(int hpw, int ng, int ncons)
{
    return hpw > 1 ? (ncons <= 4 ? 2 : 1) : (ng == 2 ? 2 : kU3CtasPerSm);
}
// launch bounds: threads per CTA and CTAs per SM the register cap is set for
template <int CK, int U3H, int NG>
constexpr int kCtasPerSm = CK == kU3 && U3H < 2 ? u3_ctas_per_sm(1, NG, kU3Heads) : 1;
template <int CK, int U3H>
constexpr int kMaxThreads = CK == kU3 && U3H < 2 ? 32 * (kU3Heads + 1) : 288;

// fp32 conversion area of a 3-bit consumer warp: (sk, zk, sv, zv) per
// (head, token) of the HPW heads and the tokens of one step (two 16-token
// blocks when one-head warps pair them)
__host__ __device__ constexpr int u3_conv_tokens(int hpw, int bs) { return hpw == 1 && bs == 16 ? 32 : bs; }
__host__ __device__ constexpr int u3_conv_bytes_per_warp(int hpw, int bs) { return 16 * hpw * u3_conv_tokens(hpw, bs); }

// U3H: 3-bit multi-head caches (one q head per kv head).  0: grouped q
// heads (the head columns of a warp are the q heads of one kv head).  1: one
// kv head per consumer warp, whose second head column never exists.  2 or 4:
// HPW = U3H kv heads per consumer warp, column j of the C fragments being
// kv head j of the warp -- K of head j runs through its own MMAs (the other
// columns of those products are dropped), V through block-diagonal MMAs whose
// k range is split between the heads, so that one set of O accumulators,
// one softmax and one walk of the ring serve HPW heads.
// GSC: fp8 / int8 with per-block or per-token scales, staged per block.
// XV: x-vectorised cache layout (16-bit and one-byte codes).
// NG: head-column groups per consumer warp (grouped q heads).  With NG = 2
// a warp serves the up to 16 q heads of its kv head as two groups of 8
// columns: every K / V fragment, loaded and converted once, feeds one MMA
// per group.
template <int CK, int D, int BS, int U3H = 0, bool GSC = false, bool XV = false, int NG = 1>
__global__ void __launch_bounds__((kMaxThreads<CK, U3H>), (kCtasPerSm<CK, U3H, NG>))
decode_tma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  DecodeParams p, FastParams f)
{
    using T = Tile<CK, D, BS>;
    constexpr int NC = U3H == 1 ? 1 : 2;   // head columns (2tig, 2tig+1) that can exist
    constexpr int HPW = U3H >= 2 ? U3H : 1;  // kv heads per consumer warp
    static_assert(HPW == 1 || (T::kIsU3 && (HPW == 2 || HPW == 4)), "heads per warp");
    static_assert(NG == 1 || (NG == 2 && U3H == 0 && BS <= 32), "head-column groups");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nh = f.nh, B = p.batch, G = p.group, stages = f.stages;
    // 3-bit metadata per stage: K scales, V scales (fp16), K zeros, V zeros
    // (u8) for the block's BS slots, of the CTA's nh heads ([nh][BS] runs,
    // head-major arrays) or of all num_kv_heads ([BS][num_kv_heads]).
    // fp8 / int8 with per-block or per-token scales: the K and V scales of
    // the CTA's heads for the block, [nh] or [nh][BS] fp32 each.
    const int GS = p.scale_mode == 2 ? BS : 1;        // staged scales per head
    constexpr bool gscale = T::kFp8 && GSC;
    // 3-bit: the raw metadata as staged (copied); its fp32 conversion
    // (sk, zk, sv, zv per (head, token), written and read by each consumer
    // warp for its own heads) sits after the ring
    const int raw_meta = T::kIsU3 ? 6 * BS * f.meta_heads : (gscale ? 8 * nh * GS : 0);
    const int meta_bytes = raw_meta;
    const int conv_bytes = T::kIsU3 ? f.ncons * u3_conv_bytes_per_warp(HPW, BS) : 0;
    const SmemLayout L = smem_layout(nh, BS, T::ROW, stages, B, meta_bytes, conv_bytes);
    // bytes the copies of one stage bring (tiles + staged scales / metadata)
    const uint32_t stage_tx = uint32_t(2 * L.tile_bytes + raw_meta);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar_full = sbase + L.bars_off, bar_empty = bar_full + 8 * stages;
    volatile int *stage_pb = reinterpret_cast<volatile int *>(smem + L.ok_off);   // block id or -1
    int *prefix = reinterpret_cast<int *>(smem + L.prefix_off);
    int *nblk = reinterpret_cast<int *>(smem + L.nblk_off);
    // the stream's previous kernel is done (with early_inputs: only before
    // the producer's first cache copy, see below)
    if (!p.early_inputs) griddep_wait();

    // ---- per-sequence block counts and their prefix sums
    const int cap = p.max_blocks << p.block_shift;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int ctx = p.context_lens[b * p.cl_stride];
        if (ctx < 0 || ctx > cap) {
            if (blockIdx.x == 0) raise_err(p.err_flag, PKV_DEVERR_CONTEXT_RANGE);
            ctx = ctx < 0 ? 0 : cap;
        }
        nblk[b] = (ctx + BS - 1) / BS;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, f.ncons);   // one arrival per consumer warp
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {               // exclusive scan, 32 sequences per step
        int carry = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int v = (b0 + lane < B) ? nblk[b0 + lane] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (b0 + lane < B) prefix[b0 + lane] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) prefix[B] = carry;
    }
    __syncthreads();

    // the merge kernel may be scheduled now; it waits for this grid to finish
    griddep_launch_dependents();
    const int64_t NBT = prefix[B];                  // blocks per head group
    const int64_t N = NBT * f.n_hg;
    const int64_t lo = int64_t(blockIdx.x) * N / gridDim.x;
    const int64_t hi = int64_t(blockIdx.x + 1) * N / gridDim.x;
    if (lo >= hi) return;

    // ======================================================== producer warp
    if (warp == f.ncons) {
        if (lane == 0) {
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
            // every copy (tiles, 3-bit metadata, granular scales) reads what
            // the previous kernel (the append) may have written
            if (p.early_inputs) griddep_wait();
        }
        // flash-layout 16-bit / one-byte tiles are streamed with an L2
        // evict-first policy (each is read once); measured neutral to
        // slightly worse for 3-bit and x-vectorised tiles, which keep the
        // default policy
        const uint64_t once = ptx::policy_evict_first();
        bool aborted = false;
        int64_t issued = 0;
        int ps = 0;              // next stage to fill
        uint32_t pphase = 0;     // completed-round parity of that stage
        for (int64_t base = lo; base < hi && !aborted; base += 32) {
            const int64_t x = base + lane;
            int pb = -1, hg = 0;
            if (x < hi) {
                hg = int(x / NBT);
                const int r = int(x - int64_t(hg) * NBT);
                const int b = find_seq(prefix, B, r);
                const int j = r - prefix[b];
                pb = p.block_tables[b * p.bt_b + j * p.bt_j];
                if (pb < 0 || pb >= p.num_blocks) {
                    raise_err(p.err_flag, PKV_DEVERR_BLOCK_RANGE);
                    pb = -1;
                }
            }
            const int n = int(hi - base < 32 ? hi - base : 32);
            for (int k = 0; k < n; ++k) {
                const int pbk = __shfl_sync(0xffffffffu, pb, k);
                const int hgk = __shfl_sync(0xffffffffu, hg, k);
                if (lane == 0 && !aborted) {
                    const int s = ps;
                    const bool reuse = issued >= stages;     // stage held a block before
                    const uint32_t par = pphase ^ 1u;
                    if (++ps == stages) {
                        ps = 0;
                        pphase ^= 1u;
                    }
                    if (reuse && !ptx::mbar_wait_bounded(bar_empty + 8 * s, par, kTimeoutNs)) {
                        raise_err(p.err_flag, PKV_DEVERR_TIMEOUT);
                        aborted = true;
                    } else {
                        const uint32_t fb = bar_full + 8 * s;
                        const uint32_t kdst = sbase + s * L.stage_bytes;
                        const uint32_t vdst = kdst + L.tile_bytes;
                        stage_pb[s] = pbk;
                        if (pbk >= 0) {
                            ptx::mbar_arrive_expect_tx(fb, stage_tx);
                            if constexpr (XV) {
                                if (f.xv_bulk) {   // the heads' tiles: one run each of K and V
                                    const int64_t off = int64_t(pbk) * p.c_blk + int64_t(hgk) * nh * p.c_head;
                                    ptx::bulk_load(kdst, p.k_cache + off, uint32_t(L.tile_bytes), fb);
                                    ptx::bulk_load(vdst, p.v_cache + off, uint32_t(L.tile_bytes), fb);
                                } else {           // (x, slot, piece, head, block) boxes
                                    ptx::tma_load_5d(kdst, &tmk, fb, 0, 0, 0, hgk * nh, pbk);
                                    ptx::tma_load_5d(vdst, &tmv, fb, 0, 0, 0, hgk * nh, pbk);
                                }
                            } else {
#pragma unroll
                                for (int h = 0; h < T::HALVES; ++h) {
                                    const int half_bytes = L.tile_bytes / T::HALVES;
                                    if constexpr (T::kIsU3) {
                                        if (f.u3_tiles == 1) {
                                            // the nh heads' tiles are one run
                                            const int64_t off = int64_t(pbk) * p.c_blk + int64_t(hgk) * nh * p.c_head;
                                            ptx::bulk_load(kdst, p.k_cache + off, uint32_t(L.tile_bytes), fb);
                                            ptx::bulk_load(vdst, p.v_cache + off, uint32_t(L.tile_bytes), fb);
                                        } else {
                                            ptx::tma_load_4d(kdst + h * half_bytes, &tmk, fb, h * T::BOX0, 0, hgk * nh, pbk);
                                            ptx::tma_load_4d(vdst + h * half_bytes, &tmv, fb, h * T::BOX0, 0, hgk * nh, pbk);
                                        }
                                    } else {
                                        ptx::tma_load_4d_hint(kdst + h * half_bytes, &tmk, fb, h * T::BOX0, 0,
                                                              hgk * nh, pbk, once);
                                        ptx::tma_load_4d_hint(vdst + h * half_bytes, &tmv, fb, h * T::BOX0, 0,
                                                              hgk * nh, pbk, once);
                                    }
                                }
                            }
                            if constexpr (gscale) {  // the heads' runs of the block's scales
                                const int64_t g0 = int64_t(pbk) * p.gs_blk + int64_t(hgk) * nh * p.gs_head;
                                const uint32_t md = vdst + L.tile_bytes;
                                ptx::bulk_load(md, p.k_gs + g0, uint32_t(4 * nh * GS), fb);
                                ptx::bulk_load(md + 4 * nh * GS, p.v_gs + g0, uint32_t(4 * nh * GS), fb);
                            }
                            if constexpr (T::kIsU3) {
                                const int HB = BS * f.meta_heads;         // entries per stage
                                // head-major: the group's heads are one run at head hgk*nh
                                const int64_t h0 = f.meta_hmaj ? int64_t(hgk) * nh * BS : 0;
                                const uint32_t md = vdst + L.tile_bytes;
                                ptx::bulk_load(md, p.k_qs + int64_t(pbk) * p.m_blk + h0, 2 * HB, fb);
                                ptx::bulk_load(md + 2 * HB, p.v_qs + int64_t(pbk) * p.m_blk + h0, 2 * HB, fb);
                                ptx::bulk_load(md + 4 * HB, p.k_qz + int64_t(pbk) * p.z_blk + h0, HB, fb);
                                ptx::bulk_load(md + 5 * HB, p.v_qz + int64_t(pbk) * p.z_blk + h0, HB, fb);
                            }
                        } else {
                            ptx::mbar_arrive(fb);
                        }
                        ++issued;
                    }
                }
                aborted = __shfl_sync(0xffffffffu, aborted, 0);
            }
        }
        // let the copies in flight land before this warp retires
        if (lane == 0) {
            for (int64_t it = issued > stages ? issued - stages : 0; it < issued; ++it)
                ptx::mbar_wait_bounded(bar_full + 8 * int(it % stages), uint32_t((it / stages) & 1),
                                       kTimeoutNs);   // once per CTA, off the hot loop
        }
        return;
    }

    // ======================================================== consumer warps
    // Consumer warp w serves kv head kvl = w of the CTA's group and its G q
    // heads: head column n of group g (NG groups of 8) is q head 8g + n.
    // With HPW > 1 (3-bit, multi-head) warp w serves kv heads kvl .. kvl +
    // HPW - 1, kvl = HPW w, head column j being kv head kvl + j.
    const int kvl = HPW > 1 ? HPW * warp : warp;
    const int GW = HPW > 1 ? HPW : min(8 * NG, G);   // head columns of this warp
    // Tokens on the MMA's M dimension, this warp's q heads on N (<= 8):
    //   S^T[tok][head] = K[tok][:] . Q[head][:]        (A = K, B = Q^T)
    //   O^T[d][head]  += V^T[d][tok] P^T[tok][head]     (A = V^T, B = P^T)
    // A thread of the C fragments holds heads 2tig, 2tig+1 for tokens
    // (or d) gid and gid+8 of each 16-row tile.
    const int gid = lane >> 2, tig = lane & 3;
    const float log2e_scale = p.scale_log2;
    // walk state
    int64_t x = lo;
    int hg = int(x / NBT);
    int b, j;
    {
        const int r = int(x - int64_t(hg) * NBT);
        b = find_seq(prefix, B, r);
        j = r - prefix[b];
    }
    int64_t seg_start = lo;

    // one-byte codes in 128-byte swizzled rows: 16-byte chunk c of row r sits
    // at r * 128 + ((c ^ r) & 7) * 16; in 64-byte swizzled rows (head_dim 64)
    // at r * 64 + ((c ^ (r >> 1)) & 3) * 16.  The rows a lane reads have a
    // fixed r & 7 (gid for K; 2tig or 2tig + 1 for V), so the chunk offsets
    // are per-lane constants, computed once: K chunk kk, V chunk
    // 2q4 + (gid >> 2) of the even / odd token rows
    uint32_t kswz[8], vswz[2][4];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        kswz[c] = T::SROW == 128 ? uint32_t((c ^ gid) & 7) << 4 : uint32_t((c ^ (gid >> 1)) & 3) << 4;
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            vswz[a][q4] = T::SROW == 128 ? uint32_t(((2 * q4 + (gid >> 2)) ^ ((2 * tig + a) & 7)) & 7) << 4
                                         : uint32_t(((2 * q4 + (gid >> 2)) ^ tig) & 3) << 4;
    uint32_t qb[T::QK][2];        // B fragments of Q^T per k-step
    float o[T::DT / 2][4];        // O^T accumulators: 16-d tiles x (heads 2tig, 2tig+1)
    float m[2], l[2];             // running max / partial sum for heads 2tig, 2tig+1
    float mult = 1.0f, vmul = 1.0f;
    int ctx_b = 0;
    // per head column: 3-bit, sum(q' 2^(x-24)) of the QK operand and the
    // running sum of P' * zero of the PV operand; int8, 1152 sum(q') and the
    // running sum of P' (the operands' 1152 offsets)
    float q1h[2] = {0.0f, 0.0f}, zs[2] = {0.0f, 0.0f};
    // the same for the second group of head columns (NG = 2)
    constexpr int NG1 = NG > 1 ? 1 : 0;
    uint32_t qb1[NG1 ? T::QK : 1][2];
    float o1[NG1 ? T::DT / 2 : 1][4];
    float m1[2], l1[2];
    float q1h1[2] = {0.0f, 0.0f}, zs1[2] = {0.0f, 0.0f};

    auto start_segment = [&]() {
        const int kvh = hg * nh + kvl;
        {
            const int cb = p.context_lens[b * p.cl_stride];
            ctx_b = cb < 0 ? 0 : (cb > cap ? cap : cb);
        }
        const bool hv = gid < GW;  // this lane's B column (q head gid) exists
        const bool hv1 = NG1 && 8 + gid < GW;   // ... and that of the second group
        // column gid: q head gid of kv head kvh, or (HPW > 1) the q head of
        // kv head kvh + gid; second group: q head 8 + gid
        const int qhead = HPW > 1 ? (kvh + gid) * G : kvh * G + gid;
        const uint16_t *qr = reinterpret_cast<const uint16_t *>(p.q + b * p.q_b + qhead * p.q_h);
        const uint16_t *qr1 = reinterpret_cast<const uint16_t *>(p.q + b * p.q_b + (qhead + 8) * p.q_h);
        if constexpr (T::kIsU3) {
            // q' = q qs 2^(1-x) (f16, exact) in the pair order of the K
            // fragments: k-step kk, lane tig holds pair 2kk (k = 2tig, 2tig+1)
            // and pair 2kk+1 (k = 2tig+8, 2tig+9) of 96-bit group tig, so that
            // q' k' = qs 2^-23 q v for every code.  One power-of-two qs
            // serves all the warp's head columns (both groups).
            auto load_q = [&](const uint16_t *qrow, bool has, float (&qv)[32]) -> float {
                float amax = 0.0f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint4 u = make_uint4(0, 0, 0, 0);
                    if (has) u = *reinterpret_cast<const uint4 *>(qrow + 32 * tig + 8 * c4);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float a, c;
                        if (p.q_is_bf16) {
                            a = __uint_as_float(w[e] << 16);
                            c = __uint_as_float(w[e] & 0xffff0000u);
                        } else {
                            const float2 t2 = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
                            a = t2.x;
                            c = t2.y;
                        }
                        qv[8 * c4 + 2 * e] = a;
                        qv[8 * c4 + 2 * e + 1] = c;
                        amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(c)));
                    }
                }
                return amax;
            };
            float qv[32];
            float amax = load_q(qr, hv, qv);
            if constexpr (NG1) {
                float qv1[32];
                amax = fmaxf(amax, load_q(qr1, hv1, qv1));
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
            float qs = 1.0f;
            while (amax * qs > 16384.0f) qs *= 0.5f;
            // the fragments of one group and, per head column 2tig + c, the
            // sum of q' 2^(x-24) over head_dim
            auto convert_q = [&](const float (&qv)[32], uint32_t (*qbg)[2], float *q1g) {
                float q1 = 0.0f;
#pragma unroll
                for (int pp = 0; pp < 16; ++pp) {
                    const U3KPair pr = u3k_pair_info(pp);
                    float ra, rb;
                    const uint32_t w = pack_f16(qv[pr.i] * qs * (2.0f / float(1 << pr.x)),
                                                qv[pr.j] * qs * (2.0f / float(1 << pr.y)), ra, rb);
                    qbg[pp >> 1][pp & 1] = w;
                    q1 += ra * (float(1 << pr.x) * 0x1p-24f) + rb * (float(1 << pr.y) * 0x1p-24f);
                }
                q1 += __shfl_xor_sync(0xffffffffu, q1, 1);
                q1 += __shfl_xor_sync(0xffffffffu, q1, 2);
#pragma unroll
                for (int c = 0; c < 2; ++c) q1g[c] = __shfl_sync(0xffffffffu, q1, 4 * (2 * tig + c));
            };
            convert_q(qv, qb, q1h);
            zs[0] = zs[1] = 0.0f;
            if constexpr (NG1) {
                float qv1[32];
                load_q(qr1, hv1, qv1);     // (read again: fewer live registers)
                convert_q(qv1, qb1, q1h1);
                zs1[0] = zs1[1] = 0.0f;
            }
            mult = log2e_scale * 0x1p23f / qs;
            vmul = 1.0f;
        } else if constexpr (!T::kFp8) {
#pragma unroll
            for (int kk = 0; kk < T::QK; ++kk) {
                const int d = 16 * kk + 2 * tig;
                qb[kk][0] = hv ? *reinterpret_cast<const uint32_t *>(qr + d) : 0u;
                qb[kk][1] = hv ? *reinterpret_cast<const uint32_t *>(qr + d + 8) : 0u;
                if constexpr (NG1) {
                    qb1[kk][0] = hv1 ? *reinterpret_cast<const uint32_t *>(qr1 + d) : 0u;
                    qb1[kk][1] = hv1 ? *reinterpret_cast<const uint32_t *>(qr1 + d + 8) : 0u;
                }
            }
            mult = log2e_scale;
            vmul = 1.0f;
        } else {
            // q (16-bit) -> f16 operands in the element order of the fp8 K
            // fragments: k-step kk, lane tig holds d = 16kk + 4tig + {0,1}
            // (k = 2tig, 2tig+1) and + {2,3} (k = 2tig+8, 2tig+9).  A
            // power-of-two pre-scale keeps every element inside f16 range.
            float f[NG][T::QK][4];
            float amax = 0.0f;
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
                for (int kk = 0; kk < T::QK; ++kk) {
                    uint2 u = make_uint2(0, 0);
                    if (g == 0 ? hv : hv1) u = *reinterpret_cast<const uint2 *>((g == 0 ? qr : qr1) + 16 * kk + 4 * tig);
                    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (p.q_is_bf16) {
                            f[g][kk][2 * e] = __uint_as_float(w[e] << 16);
                            f[g][kk][2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                        } else {
                            const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
                            f[g][kk][2 * e] = t.x;
                            f[g][kk][2 * e + 1] = t.y;
                        }
                        amax = fmaxf(amax, fmaxf(fabsf(f[g][kk][2 * e]), fabsf(f[g][kk][2 * e + 1])));
                    }
                }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
            float qs = 1.0f;
            while (amax * qs > 16384.0f) qs *= 0.5f;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                float d0, d1, d2, d3, c0 = 0.0f;
                uint32_t (*qg)[2] = g == 0 ? qb : qb1;
#pragma unroll
                for (int kk = 0; kk < T::QK; ++kk) {
                    qg[kk][0] = pack_f16(f[g][kk][0] * qs, f[g][kk][1] * qs, d0, d1);
                    qg[kk][1] = pack_f16(f[g][kk][2] * qs, f[g][kk][3] * qs, d2, d3);
                    c0 += (d0 + d1) + (d2 + d3);
                }
                if constexpr (CK == kI8) {     // sum of q' over head_dim, per q head gid
                    c0 += __shfl_xor_sync(0xffffffffu, c0, 1);
                    c0 += __shfl_xor_sync(0xffffffffu, c0, 2);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {   // head columns 2tig, 2tig+1
                        (g == 0 ? q1h : q1h1)[c] = kI8Bias * __shfl_sync(0xffffffffu, c0, 4 * (2 * tig + c));
                        (g == 0 ? zs : zs1)[c] = 0.0f;
                    }
                }
            }
            // per-block / per-token scales are applied per row (scores and P')
            mult = log2e_scale * (gscale ? 1.0f : p.k_scale[kvh]) / qs;
            vmul = gscale ? 1.0f : p.v_scale[kvh];
        }
#pragma unroll
        for (int t = 0; t < T::DT / 2; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.0f;
        m[0] = m[1] = NEG_INF;
        l[0] = l[1] = 0.0f;
        if constexpr (NG1) {
#pragma unroll
            for (int t = 0; t < T::DT / 2; ++t) o1[t][0] = o1[t][1] = o1[t][2] = o1[t][3] = 0.0f;
            m1[0] = m1[1] = NEG_INF;
            l1[0] = l1[1] = 0.0f;
        }
    };

    // d held by this lane for accumulator tile t, row half r (0: gid, 1: gid+8)
    auto d_of = [&](int t, int r) -> int {
        if constexpr (T::kIsU3) {
            return 16 * gid + 2 * t + r;                     // slice code 2t + r
        } else if constexpr (!T::kFp8) {
            return 16 * t + 8 * r + gid;
        } else {
            return 32 * (t >> 1) + 4 * gid + 2 * (t & 1) + r;
        }
    };

    // Write the segment's result of one group of head columns (accumulators
    // og, running max mg, sums lg, P' * zero / P' sums zsg), columns
    // 8 g0 + 2tig + c.
    auto finish_group = [&](int64_t seg_end, int g0, float (*og)[4], const float *mg, const float *lg,
                            const float *zsg) {
        const int64_t unit_first = int64_t(hg) * NBT + prefix[b];
        const int64_t unit_last = unit_first + nblk[b] - 1;
        float lt[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {       // sum the partial sums over the 8 token rows (gid)
            float v = lg[c];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            lt[c] = v;
        }
        float zt[2] = {0.0f, 0.0f};
        if constexpr (T::kIsU3 || CK == kI8) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float z = zsg[c];
#pragma unroll
                for (int o2 = 4; o2 < 32; o2 <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o2);
                zt[c] = CK == kI8 ? kI8Bias * z : z;
            }
        }
        // accumulator entry (t, r, c) -> value of the segment's unnormalised output
        auto oval = [&](int t, int r, int c) -> float {
            if constexpr (T::kIsU3) {
                return og[t][2 * r + c] * float(1 << (24 - u3v_x(2 * t + r))) - zt[c];
            } else if constexpr (CK == kI8) {
                return og[t][2 * r + c] - zt[c];
            } else {
                return og[t][2 * r + c];
            }
        };
        const bool whole = seg_start == unit_first && seg_end == unit_last;
        const int64_t key = int64_t(blockIdx.x) + int64_t(hg) * B + b;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int g = 8 * g0 + 2 * tig + c;
            if (g >= GW) continue;
            // q head of column g, within the head group and overall
            const int local = HPW > 1 ? (kvl + g) * G : kvl * G + g;
            const int h = hg * nh * G + local;
            if (whole) {
                const float inv = lt[c] > 0.0f ? vmul / lt[c] : 0.0f;
                uint16_t *orow = reinterpret_cast<uint16_t *>(p.out + b * p.o_b + h * p.o_h);
#pragma unroll
                for (int t = 0; t < T::DT / 2; ++t)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float v = oval(t, r, c) * inv;
                        orow[d_of(t, r)] = p.q_is_bf16 ? f2h<kBF16>(v) : f2h<kF16>(v);
                    }
            } else {
                const int64_t row = key * (int64_t(nh) * G) + local;
                float *acc = f.part_acc + row * D;
                if (gid == 0) {
                    f.part_ml[2 * row] = mg[c];
                    f.part_ml[2 * row + 1] = lt[c];
                }
#pragma unroll
                for (int t = 0; t < T::DT / 2; ++t)
#pragma unroll
                    for (int r = 0; r < 2; ++r) acc[d_of(t, r)] = oval(t, r, c) * vmul;
            }
        }
    };
    auto finish_segment = [&](int64_t seg_end) {
        finish_group(seg_end, 0, o, m, l, zs);
        if constexpr (NG1) finish_group(seg_end, 1, o1, m1, l1, zs1);
    };

    // 3-bit blocks: NB (1, or 2 for 16-token blocks) consecutive blocks of
    // one sequence, held in stages s0 (and s1), as NB * KT tiles of 16
    // tokens; `valid` counts the live tokens of all NB blocks (only the last
    // block of a sequence can be partial).  The warp serves HPW kv heads
    // (kvl ..): with HPW = 1 its head columns are q heads of kv head kvl,
    // with HPW > 1 column j is kv head kvl + j.
    auto u3_body = [&](auto nb_c, int s0, int s1, int valid) {
        constexpr int NB = decltype(nb_c)::value;
        constexpr int KTT = NB * T::KT;          // 16-token tiles of the NB blocks
        constexpr int NT = NB * BS;              // tokens of the NB blocks
        const int kvh = hg * nh + kvl;
        const bool partial = valid < NT;
        // shared-memory strides of the staged rows ([head][slot][row]):
        // between heads and between slots
        constexpr int hs = BS * T::ROW, ts = T::ROW;
        // stage of tile t, and the tile's first row within its block
        auto tile_stage = [&](int t) { return t < T::KT ? s0 : s1; };
        auto tile_row = [&](int t) { return 16 * (t % T::KT); };
        // packed K rows of tile t of the warp's head hh (shared address)
        auto kpk = [&](int t, int hh) {
            return sbase + tile_stage(t) * L.stage_bytes + (kvl + hh) * hs + tile_row(t) * ts;
        };
        // ---- metadata: the warp converts each (head, token) of its HPW
        // heads and the NB blocks to fp32 (sk, zk, sv, zv) in the stage's
        // conversion area -- one entry per lane and step instead of four 16-
        // / 8-bit loads and conversions per score row in every lane -- and
        // each lane then reads its score rows' entries.  Staged as [nh][BS]
        // runs (head-major) or [BS][num_kv_heads] arrays.
        const int MH = f.meta_heads;
        const bool hmaj = f.meta_hmaj != 0;
        // this warp's conversion area: entry (head hh, token tk of the NB
        // blocks) at hh * NTM + tk
        constexpr int NTM = u3_conv_tokens(HPW, BS);
        static_assert(NT <= NTM, "conversion area");
        float4 *cw = reinterpret_cast<float4 *>(smem + L.conv_off) + warp * HPW * NTM;
        __syncwarp();    // the previous step's reads of the area are done
        if (HPW > 1 && hmaj) {
            // head-major runs of multi-head warps: a lane takes two
            // consecutive tokens of one head (an even slot, both in one
            // stage), loading their two scales and two zeros of K and of V
            // at once
            constexpr int NP2 = HPW * NT / 2;
#pragma unroll
            for (int i0 = 0; i0 < NP2; i0 += 32) {
                const int i = i0 + lane;
                if (i < NP2) {
                    const int hh = i / (NT / 2), tk = 2 * (i % (NT / 2));
                    const int st = tk < BS ? s0 : s1, slot = tk & (BS - 1);
                    const unsigned char *raw = smem + (st * L.stage_bytes + 2 * L.tile_bytes);
                    const int k = (kvl + hh) * BS + slot;
                    const float2 ks = __half22float2(*reinterpret_cast<const __half2 *>(raw + 2 * k));
                    const float2 vs = __half22float2(*reinterpret_cast<const __half2 *>(raw + 2 * BS * MH + 2 * k));
                    const uint32_t kz = *reinterpret_cast<const uint16_t *>(raw + 4 * BS * MH + k);
                    const uint32_t vz = *reinterpret_cast<const uint16_t *>(raw + 5 * BS * MH + k);
                    cw[hh * NTM + tk] = make_float4(ks.x, float(kz & 0xffu), vs.x, float(vz & 0xffu));
                    cw[hh * NTM + tk + 1] = make_float4(ks.y, float(kz >> 8), vs.y, float(vz >> 8));
                }
            }
        } else {
#pragma unroll
        for (int i0 = 0; i0 < HPW * NT; i0 += 32) {
            const int i = i0 + lane;
            if (i < HPW * NT) {
                const int hh = i / NT, tk = i % NT;
                const int st = tk < BS ? s0 : s1, slot = tk & (BS - 1);
                const unsigned char *raw = smem + (st * L.stage_bytes + 2 * L.tile_bytes);
                const __half *mks = reinterpret_cast<const __half *>(raw);
                const __half *mvs = mks + BS * MH;
                const uint8_t *mkz = raw + 4 * BS * MH;
                const uint8_t *mvz = mkz + BS * MH;
                const int k = hmaj ? (kvl + hh) * BS + slot : slot * MH + kvh + hh;
                cw[hh * NTM + tk] =
                    make_float4(__half2float(mks[k]), float(mkz[k]), __half2float(mvs[k]), float(mvz[k]));
            }
        }
        }
        __syncwarp();
        // conversion entry of score row (tile t, row half r) and head column c
        auto meta_of = [&](int t, int r, int c) -> const float4 * {
            // HPW 4: lanes tig 0, 1 hold columns 0-3; lanes tig 2, 3 hold
            // none and read an in-range entry
            const int hc = HPW == 1 ? 0 : (HPW == 2 ? c : ((2 * tig + c) & 3));
            return cw + hc * NTM + 16 * t + gid + 8 * r;
        };
        // ---- S^T = K Q'^T with K converted straight into A fragments:
        // lane (gid, tig) takes group tig of token rows gid and gid+8.  With
        // HPW > 1 each head's product keeps only its own column: heads 2i
        // and 2i+1 fill columns (0, 1) of lanes tig = i.
        float sc[KTT][4];
        [[maybe_unused]] float sc1[NG1 ? KTT : 1][4];
#pragma unroll
        for (int mt = 0; mt < KTT; ++mt) {
            float colp[HPW > 1 ? HPW / 2 : 1][4];
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) {
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float sx[4] = {0.0f, 0.0f, 0.0f, 0.0f};     // second chain (odd k-steps)
                [[maybe_unused]] float acc1[NG1 ? 4 : 1] = {}, sx1[NG1 ? 4 : 1] = {};   // second group
                const uint32_t a0 = kpk(mt, hh) + gid * ts + 12 * tig;
                const uint32_t a1 = a0 + 8 * ts;
                const uint32_t x0 = ld_shared_u32(a0), x1 = ld_shared_u32(a0 + 4), x2 = ld_shared_u32(a0 + 8);
                const uint32_t y0 = ld_shared_u32(a1), y1 = ld_shared_u32(a1 + 4), y2 = ld_shared_u32(a1 + 8);
#pragma unroll
                for (int kk = 0; kk < T::QK; ++kk) {
                    uint32_t a[4];
                    a[0] = u3k_pair(2 * kk, x0, x1, x2);
                    a[1] = u3k_pair(2 * kk, y0, y1, y2);
                    a[2] = u3k_pair(2 * kk + 1, x0, x1, x2);
                    a[3] = u3k_pair(2 * kk + 1, y0, y1, y2);
                    ptx::mma16816<false>((kk & 1) ? sx : acc, a, qb[kk][0], qb[kk][1]);
                    if constexpr (NG1) ptx::mma16816<false>((kk & 1) ? sx1 : acc1, a, qb1[kk][0], qb1[kk][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (NG1) sc1[mt][e] = acc1[e] + sx1[e];
                    if (HPW == 1)
                        colp[0][e] = acc[e] + sx[e];
                    else if ((e & 1) == (hh & 1))
                        colp[hh >> 1][e] = acc[e] + sx[e];
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[mt][e] = HPW == 4 ? (tig == 0 ? colp[0][e] : colp[HPW > 2 ? 1 : 0][e]) : colp[0][e];
        }
        // ---- scores: remove the zero point, apply the per-token
        // scale, mask; online softmax per head column.  One group of head
        // columns: scores scg, running max mg / sums lg / P' * zero sums zsg,
        // q' sums q1g, accumulators og; P'^T (B operand of the PV product)
        // in ptg: pt[t][r] gives lane (gid, tig) the P' of tokens 8r + 2tig,
        // +1 of tile t in head column gid
        auto u3_softmax = [&](float (*scg)[4], float *mg, float *lg, float *zsg, const float *q1g,
                              uint32_t (*ptg)[2], float (*og)[4]) {
            float mx[2] = {NEG_INF, NEG_INF};
#pragma unroll
            for (int t = 0; t < KTT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = e >> 1, c = e & 1;
                    if (c >= NC) continue;
                    const float2 kz = *reinterpret_cast<const float2 *>(meta_of(t, r, c));   // (sk, zk)
                    float v = mult * kz.x * (scg[t][e] - kz.y * q1g[c]);
                    if (partial) v = (16 * t + gid + 8 * r) < valid ? v : NEG_INF;
                    scg[t][e] = v;
                    mx[c] = fmaxf(mx[c], v);
                }
            // (a block that raises no running max skips the reductions and
            // the rescale, as in the other caches' softmax)
            float alpha[2] = {1.0f, 1.0f};
            const bool raise = __any_sync(0xffffffffu, mx[0] > mg[0] || (NC > 1 && mx[1] > mg[1]));
            if (raise) {
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 4));
                    mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 8));
                    mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 16));
                    const float mn = fmaxf(mg[c], mx[c]);
                    alpha[c] = mn == NEG_INF ? 1.0f : exp2_approx(mg[c] - mn);
                    mg[c] = mn;
                    lg[c] *= alpha[c];
                    zsg[c] *= alpha[c];
                }
            }
            // P' = p * v_scale (0 for masked tokens), transposed by movmatrix
#pragma unroll
            for (int t = 0; t < KTT; ++t)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const bool ok = !partial || (16 * t + gid + 8 * r) < valid;
                    const float2 vz0 = *reinterpret_cast<const float2 *>(&meta_of(t, r, 0)->z);   // (sv, zv)
                    const float2 vz1 = HPW > 1 ? *reinterpret_cast<const float2 *>(&meta_of(t, r, 1)->z) : vz0;
                    const float p0 = exp2_approx(scg[t][2 * r] - mg[0]);
                    const float p1 = NC > 1 ? exp2_approx(scg[t][2 * r + 1] - mg[1]) : 0.0f;
                    lg[0] += p0;
                    if (NC > 1) lg[1] += p1;
                    float q0, q1;
                    const uint32_t w = pack_f16(ok ? p0 * vz0.x : 0.0f, ok ? p1 * vz1.x : 0.0f, q0, q1);
                    zsg[0] += q0 * vz0.y;
                    if (NC > 1) zsg[1] += q1 * vz1.y;
                    ptg[t][r] = ptx::movmatrix_trans(w);
                }
            if (raise && __any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
                for (int t = 0; t < T::DT / 2; ++t) {
                    og[t][0] *= alpha[0];
                    og[t][2] *= alpha[0];
                    if (NC > 1) {
                        og[t][1] *= alpha[1];
                        og[t][3] *= alpha[1];
                    }
                }
            }
        };
        uint32_t pt[KTT][2];
        [[maybe_unused]] uint32_t pt1[NG1 ? KTT : 1][2];
        u3_softmax(sc, m, l, zs, q1h, pt, o);
        if constexpr (NG1) u3_softmax(sc1, m1, l1, zs1, q1h1, pt1, o1);
        // ---- O^T += V'^T P'^T with V converted straight into A fragments:
        // lane (gid, tig) owns codes 16gid .. 16gid+15 (row bytes 6gid ..
        // 6gid+5) of two token rows ra0, ra0+1 of head ha (k = 2tig, 2tig+1)
        // and two rows rb0, rb0+1 of head hb (k = 2tig+8, 2tig+9); tile md
        // holds codes 2md (row gid) and 2md+1 (row gid+8) of the slices.
        // X / Y are slice bytes 0-3 / 2-5.  One pass per 16 tokens (HPW 1:
        // one head, tokens 2tig.. and 2tig+8..), else block-diagonal passes
        // in which the k range is split between heads: HPW 2, pass r: k < 8
        // head 0, k >= 8 head 1, tokens 8r + 2tig, +1; HPW 4, pass (r, j):
        // quarter i of k (4 tokens) is head (i ^ j) for i < 2, 2 + ((i-2) ^ j)
        // above, tokens 8r + 2tig, +1.  The B operand of a pass is pt[t][r]
        // kept only in the columns of the heads it pairs with each k.
        const int sxy = 16 * (gid & 1);
        constexpr int NP = HPW == 1 ? 1 : HPW;   // passes per 16-token tile
#pragma unroll
        for (int kt = 0; kt < KTT; ++kt) {
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                [[maybe_unused]] const int r = HPW == 4 ? (ps >> 1) : ps;
                [[maybe_unused]] const int j = HPW == 4 ? (ps & 1) : 0;
                int ha = 0, hb = 0, ra0 = 2 * tig, rb0 = 2 * tig + 8;
                uint32_t b0 = pt[kt][0], b1 = pt[kt][1];
                if constexpr (HPW > 1) {
                    ha = HPW == 2 ? 0 : ((tig >> 1) ^ j);
                    hb = HPW == 2 ? 1 : 2 + ((tig >> 1) ^ j);
                    ra0 = rb0 = 8 * r + 2 * tig;
                    b0 = gid == ha ? pt[kt][r] : 0u;
                    b1 = gid == hb ? pt[kt][r] : 0u;
                }
                const uint32_t va = kpk(kt, ha) + L.tile_bytes + ((6 * gid) & ~3);   // packed V rows
                const uint32_t vb = kpk(kt, hb) + L.tile_bytes + ((6 * gid) & ~3);
                uint32_t X[4], Y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t ra = (i < 2 ? va + ra0 * ts : vb + rb0 * ts) + (i & 1) * ts;
                    const uint32_t w0 = ld_shared_u32(ra);
                    const uint32_t w1 = ld_shared_u32(ra + 4);
                    X[i] = __funnelshift_r(w0, w1, sxy);
                    Y[i] = __funnelshift_rc(w0, w1, sxy + 16);
                }
                uint32_t win[2][6];
#pragma unroll
                for (int tp = 0; tp < 2; ++tp) {
                    win[tp][0] = ptx::prmt(X[2 * tp], X[2 * tp + 1], 0x5410u);
                    win[tp][1] = ptx::prmt(X[2 * tp], X[2 * tp + 1], 0x6521u);
                    win[tp][2] = ptx::prmt(X[2 * tp], X[2 * tp + 1], 0x7632u);
                    win[tp][3] = ptx::prmt(Y[2 * tp], Y[2 * tp + 1], 0x6521u);
                    win[tp][4] = ptx::prmt(Y[2 * tp], Y[2 * tp + 1], 0x7632u);
                    win[tp][5] = ptx::prmt(Y[2 * tp], Y[2 * tp + 1], 0x7733u);
                }
#pragma unroll
                for (int md = 0; md < T::DT / 2; ++md) {
                    constexpr uint32_t kMask3 = 0x00070007u;
                    uint32_t a[4];
                    a[0] = win[0][u3v_win(2 * md)] & (kMask3 << u3v_x(2 * md));
                    a[1] = win[0][u3v_win(2 * md + 1)] & (kMask3 << u3v_x(2 * md + 1));
                    a[2] = win[1][u3v_win(2 * md)] & (kMask3 << u3v_x(2 * md));
                    a[3] = win[1][u3v_win(2 * md + 1)] & (kMask3 << u3v_x(2 * md + 1));
                    ptx::mma16816<false>(o[md], a, b0, b1);
                    if constexpr (NG1) ptx::mma16816<false>(o1[md], a, pt1[kt][0], pt1[kt][1]);
                }
            }
        }
    };

    start_segment();
    int cs = 0;                  // stage of the current block
    uint32_t cphase = 0;         // parity of its fill round
    for (; x < hi; ++x) {
        const int s = cs;
        if (!ptx::mbar_wait_bounded(bar_full + 8 * s, cphase, kTimeoutNs)) {
            raise_err(p.err_flag, PKV_DEVERR_TIMEOUT);
            return;
        }
        if (++cs == stages) {
            cs = 0;
            cphase ^= 1u;
        }
        // valid tokens of this block (only the last block of a sequence is partial)
        const int valid = min(BS, ctx_b - j * BS);
        const int spb = stage_pb[s];
        if (spb >= 0 && !T::kIsU3) {
            // fp8 / int8 per-block or per-token scales of this warp's head,
            // staged with the block: [nh][GS] K scales, then V scales
            const float *gsk = reinterpret_cast<const float *>(smem + s * L.stage_bytes + 2 * L.tile_bytes) +
                               kvl * GS;
            const float *gsv = gsk + nh * GS;
            auto row_ks = [&](int tok) { return gsk[GS == 1 ? 0 : tok]; };
            auto row_vs = [&](int tok) { return gsv[GS == 1 ? 0 : tok]; };
            // this warp's head: rows of swizzled sub-rows per half, or (XV)
            // one [head_dim/x][BS][16 B] run; piece c of token t at
            // (c * BS + t) * 16
            const uint32_t ktile = sbase + s * L.stage_bytes + kvl * BS * (XV ? T::ROW : T::SROW);
            const uint32_t vtile = ktile + L.tile_bytes;
            const int half_bytes = L.tile_bytes / T::HALVES;
            const int mi = lane >> 3;    // ldmatrix: which 8x8 matrix this lane addresses
            // ---------------- S^T = K Q^T
            float sc[T::KT][4], sc1[NG1 ? T::KT : 1][4];
#pragma unroll
            for (int t = 0; t < T::KT; ++t) {
                sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.0f;
                if constexpr (NG1) sc1[t][0] = sc1[t][1] = sc1[t][2] = sc1[t][3] = 0.0f;
            }
#pragma unroll
            for (int kk = 0; kk < T::QK; ++kk) {
#pragma unroll
                for (int mt = 0; mt < T::KT; ++mt) {
                    uint32_t a[4];
                    if constexpr (!T::kFp8) {
                        // matrices: (tok 0-7 | 8-15) x (d chunk 2kk | 2kk+1)
                        const int tok = 16 * mt + 8 * (mi & 1) + (lane & 7);
                        const int chunk = 2 * kk + (mi >> 1);
                        ptx::ldmatrix_x4(XV ? ktile + (chunk * BS + tok) * 16
                                            : ktile + (chunk >> 3) * half_bytes + tok * 128 +
                                                  (((chunk & 7) ^ (tok & 7)) << 4),
                                         a[0], a[1], a[2], a[3]);
                    } else {
                        uint32_t w0, w1;
                        if constexpr (XV) {   // piece kk of rows 16mt+gid and +8
                            const uint32_t kb = ktile + (kk * BS + 16 * mt + gid) * 16 + 4 * tig;
                            w0 = ld_shared_u32(kb);
                            w1 = ld_shared_u32(kb + 8 * 16);
                        } else {   // chunk kk of rows 16mt+gid and +8 (both r & 7 = gid)
                            const uint32_t kb = ktile + gid * T::SROW + 4 * tig + kswz[kk & (T::SROW / 16 - 1)] +
                                                mt * 16 * T::SROW;
                            w0 = ld_shared_u32(kb);
                            w1 = ld_shared_u32(kb + 8 * T::SROW);
                        }
                        a[0] = f16x2_from_q8<CK, 0>(w0);
                        a[1] = f16x2_from_q8<CK, 0>(w1);
                        a[2] = f16x2_from_q8<CK, 1>(w0);
                        a[3] = f16x2_from_q8<CK, 1>(w1);
                    }
                    ptx::mma16816<T::kBF>(sc[mt], a, qb[kk][0], qb[kk][1]);
                    if constexpr (NG1) ptx::mma16816<T::kBF>(sc1[mt], a, qb1[kk][0], qb1[kk][1]);
                }
            }
            // ---------------- online softmax per q head (columns), log2 units
            const bool partial = valid < BS;   // only a sequence's last block
            // one group of head columns: scores scg, running max mg / sums lg,
            // int8 offsets zsg / q1g, accumulators og; P^T as the B operand of
            // the PV product in pbg: each 8-token half of a tile (rows =
            // tokens, cols = heads) packed and transposed in registers, giving
            // lane (gid, tig) tokens 2tig, 2tig+1 of head gid
            auto softmax_group = [&](float (*scg)[4], float *mg, float *lg, float *zsg, const float *q1g,
                                     uint32_t (*pbg)[2], float (*og)[4]) {
                float mx[2] = {NEG_INF, NEG_INF};
#pragma unroll
                for (int t = 0; t < T::KT; ++t) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float v = (CK == kI8 ? scg[t][e] - q1g[e & 1] : scg[t][e]) * mult;
                        if (T::kFp8 && gscale) v *= row_ks(16 * t + gid + 8 * (e >> 1));
                        if (partial) {
                            const int tok = 16 * t + gid + 8 * (e >> 1);
                            v = tok < valid ? v : NEG_INF;
                        }
                        scg[t][e] = v;
                        mx[e & 1] = fmaxf(mx[e & 1], v);
                    }
                }
                // A block none of whose scores passes the running max leaves
                // it (and the sums) as they are: the warp then skips the
                // reductions and the rescale.  (The first block of a segment
                // always raises it from -inf.)
                float alpha[2] = {1.0f, 1.0f};
                const bool raise = __any_sync(0xffffffffu, mx[0] > mg[0] || mx[1] > mg[1]);
                if (raise) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 4));
                        mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 8));
                        mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 16));
                        const float mn = fmaxf(mg[c], mx[c]);
                        alpha[c] = mn == NEG_INF ? 1.0f : exp2_approx(mg[c] - mn);
                        mg[c] = mn;
                        lg[c] *= alpha[c];
                        if constexpr (CK == kI8) zsg[c] *= alpha[c];
                    }
                }
#pragma unroll
                for (int t = 0; t < T::KT; ++t) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float p0 = exp2_approx(scg[t][2 * r] - mg[0]);
                        const float p1 = exp2_approx(scg[t][2 * r + 1] - mg[1]);
                        lg[0] += p0;
                        lg[1] += p1;
                        // per-block / per-token V scales fold into P' = p * scale
                        const float vsr = T::kFp8 && gscale ? row_vs(16 * t + gid + 8 * r) : 1.0f;
                        float q0, q1;
                        const uint32_t w = T::kBF ? pack_bf16(p0, p1, q0, q1) : pack_f16(p0 * vsr, p1 * vsr, q0, q1);
                        if constexpr (CK == kI8) {   // the PV operand's offset: sum of P' as rounded
                            zsg[0] += q0;
                            zsg[1] += q1;
                        }
                        pbg[t][r] = ptx::movmatrix_trans(w);
                    }
                }
                if (raise && __any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
                    for (int t = 0; t < T::DT / 2; ++t) {
                        og[t][0] *= alpha[0];
                        og[t][1] *= alpha[1];
                        og[t][2] *= alpha[0];
                        og[t][3] *= alpha[1];
                    }
                }
            };
            uint32_t pb[T::KT][2], pb1[NG1 ? T::KT : 1][2];
            softmax_group(sc, m, l, zs, q1h, pb, o);
            if constexpr (NG1) softmax_group(sc1, m1, l1, zs1, q1h1, pb1, o1);
            // ---------------- O^T += V^T P^T
#pragma unroll
            for (int kt = 0; kt < T::KT; ++kt) {
                if constexpr (!T::kFp8) {
                    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                    if (partial) {  // zero V of masked tokens (0 * NaN would poison O)
                        const int t0 = 16 * kt + 2 * tig;
                        mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
                        mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int md = 0; md < T::DT / 2; ++md) {
                        // matrices: (tok 0-7 | 8-15) x (d chunk 2md | 2md+1), transposed
                        const int tok = 16 * kt + 8 * (mi >> 1) + (lane & 7);
                        const int chunk = 2 * md + (mi & 1);
                        uint32_t a[4];
                        ptx::ldmatrix_x4_trans(XV ? vtile + (chunk * BS + tok) * 16
                                                  : vtile + (chunk >> 3) * half_bytes + tok * 128 +
                                                        (((chunk & 7) ^ (tok & 7)) << 4),
                                               a[0], a[1], a[2], a[3]);
                        a[0] &= mlo;
                        a[1] &= mlo;
                        a[2] &= mhi;
                        a[3] &= mhi;
                        ptx::mma16816<T::kBF>(o[md], a, pb[kt][0], pb[kt][1]);
                        if constexpr (NG1) ptx::mma16816<T::kBF>(o1[md], a, pb1[kt][0], pb1[kt][1]);
                    }
                } else {
                    const int t0 = 16 * kt + 2 * tig;
                    // XV: lanes of the odd piece (gid >= 4) load each row pair
                    // swapped, so that a load's 32 lanes hit 32 banks; the
                    // byte permutes below undo the swap
                    const int sw = XV ? (gid >> 2) : 0;
                    const int rows[4] = {t0 + sw, t0 + 1 - sw, t0 + 8 + sw, t0 + 9 - sw};
                    const uint32_t swsel = sw ? 0x4444u : 0u;
                    uint32_t vb[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if constexpr (XV)   // piece 2q4 + (gid >> 2) of row i
                            vb[i] = vtile + ((gid >> 2) * BS + rows[i]) * 16 + (gid & 3) * 4;
                        else                // row i; its chunk offset is vswz[i & 1][q4]
                            vb[i] = vtile + rows[i] * T::SROW + (gid & 3) * 4;
                    }
#pragma unroll
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        // bytes d = 32q4 + 4gid .. +3 of the four token rows;
                        // tile 2q4 takes bytes 0 (rows gid) and 1 (rows gid+8),
                        // tile 2q4+1 bytes 2 and 3
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            w[i] = ld_shared_u32(XV ? vb[i] + q4 * 2 * BS * 16 : vb[i] + vswz[i & 1][q4 & 3]);
                            if (partial && rows[i] >= valid) w[i] = 0u;
                        }
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {
                            const uint32_t sel = ((2 * hb) | ((2 * hb + 4) << 4) | ((2 * hb + 1) << 8) |
                                                  ((2 * hb + 5) << 12)) ^ swsel;
                            const uint32_t x01 = ptx::prmt(w[0], w[1], sel);
                            const uint32_t x23 = ptx::prmt(w[2], w[3], sel);
                            uint32_t a[4];
                            a[0] = f16x2_from_q8<CK, 0>(x01);
                            a[1] = f16x2_from_q8<CK, 1>(x01);
                            a[2] = f16x2_from_q8<CK, 0>(x23);
                            a[3] = f16x2_from_q8<CK, 1>(x23);
                            ptx::mma16816<false>(o[2 * q4 + hb], a, pb[kt][0], pb[kt][1]);
                            if constexpr (NG1) ptx::mma16816<false>(o1[2 * q4 + hb], a, pb1[kt][0], pb1[kt][1]);
                        }
                    }
                }
            }
        }
        if constexpr (T::kIsU3) {
            // 16-token blocks of one kv head per warp go two at a time when
            // the next unit continues the sequence: the per-block softmax,
            // barrier and walk work is then shared by 32 tokens (warps of
            // several heads share it between their heads instead, and keep
            // one block per step so that more of the ring is in flight)
            const bool pair = BS == 16 && HPW == 1 && NG == 1 && x + 1 < hi && j + 1 < nblk[b];
            if (pair) {
                const int s1 = cs;
                if (!ptx::mbar_wait_bounded(bar_full + 8 * s1, cphase, kTimeoutNs)) {
                    raise_err(p.err_flag, PKV_DEVERR_TIMEOUT);
                    return;
                }
                if (++cs == stages) {
                    cs = 0;
                    cphase ^= 1u;
                }
                const int spb1 = stage_pb[s1];
                const int valid1 = min(BS, ctx_b - (j + 1) * BS);
                if (spb >= 0 && spb1 >= 0) {
                    // (only one-head warps pair blocks, of 16 tokens)
                    u3_body(std::integral_constant<int, HPW == 1 && BS == 16 && NG == 1 ? 2 : 1>{}, s, s1, BS + valid1);
                } else {
                    if (spb >= 0) u3_body(std::integral_constant<int, 1>{}, s, s, valid);
                    if (spb1 >= 0) u3_body(std::integral_constant<int, 1>{}, s1, s1, valid1);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s1);
                ++j;             // the pair's first block is never its sequence's last
                ++x;
            } else if (spb >= 0) {
                u3_body(std::integral_constant<int, 1>{}, s, s, valid);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
        // advance the walk; close the segment at a unit boundary
        if (x + 1 < hi) {
            if (++j == nblk[b]) {
                finish_segment(x);
                j = 0;
                do {
                    if (++b == B) {
                        b = 0;
                        ++hg;
                    }
                } while (nblk[b] == 0);
                seg_start = x + 1;
                start_segment();
            }
        } else {
            finish_segment(x);
        }
    }
}

// floor(a / n) for 0 <= a < 2^62, 0 < n < 2^31: a float estimate corrected
// by exact integer comparisons (cheaper than a 64-bit division).
__device__ __forceinline__ int64_t floordiv_i64(int64_t a, int64_t n)
{
    int64_t q = int64_t(__fdividef(float(a), float(n)));
    while (q > 0 && q * n > a) --q;
    while ((q + 1) * n <= a) ++q;
    return q;
}

// Merge the partials of units split across CTAs (one warp per (sequence,
// q head)); units held whole by one CTA were written by it, units with an
// empty context get zeros.
constexpr int kMergeBatch = 16;  // partials a row combines in one round trip
// 4 warps a CTA: small enough in registers to sit beside a decode CTA on its
// SM, where it computes its prologue before the decode grid completes
constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(DecodeParams p, FastParams f)
{
    // Blocks per sequence and their prefix sums, from context_lens (an input
    // of the call, clamped as the decode kernel clamps it): computed while
    // the decode kernel still runs, this kernel being its programmatic
    // dependent, so that only the partials are read after the wait.
    extern __shared__ int sprefix[];            // [batch + 1]
    __shared__ int wsum[kMergeWarps];
    const int B = p.batch, tid = threadIdx.x, lane = tid & 31;
    {
        const int cap = p.max_blocks << p.block_shift;
        const int per = (B + 32 * kMergeWarps - 1) / (32 * kMergeWarps);
        const int lo = min(B, tid * per), hi = min(B, lo + per);
        int sum = 0;
        for (int b = lo; b < hi; ++b) {
            int ctx = p.context_lens[b * p.cl_stride];
            ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
            const int nb = (ctx + p.block_size - 1) >> p.block_shift;
            sprefix[b] = nb;
            sum += nb;
        }
        int incl = sum;             // block-wide exclusive scan of the sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) wsum[tid >> 5] = incl;
        __syncthreads();
        int run = incl - sum, total = 0;
#pragma unroll
        for (int w4 = 0; w4 < kMergeWarps; ++w4) {
            if (w4 < (tid >> 5)) run += wsum[w4];
            total += wsum[w4];
        }
        for (int b = lo; b < hi; ++b) {
            const int c = sprefix[b];
            sprefix[b] = run;
            run += c;
        }
        if (tid == 0) sprefix[B] = total;
        __syncthreads();
    }
    // wait until the decode grid has completed and its writes are visible
    griddep_wait();
    const int w = blockIdx.x * kMergeWarps + (tid >> 5);
    if (w >= B * p.num_heads) return;
    const int b = w / p.num_heads, h = w % p.num_heads;
    const int G = p.group, nh = f.nh;
    const int kvh = h / G, hg = kvh / nh;
    const int local = h - hg * nh * G;
    const int64_t NBT = sprefix[B];
    const int64_t N = NBT * f.n_hg;
    const int n = sprefix[b + 1] - sprefix[b];
    constexpr int EPL = D / 32;
    uint16_t *orow = reinterpret_cast<uint16_t *>(p.out + b * p.o_b + h * p.o_h);
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.0f;
    if (n > 0) {
        const int64_t S = f.grid;
        const int64_t first = int64_t(hg) * NBT + sprefix[b];
        // CTA i streams [i*N/S, (i+1)*N/S): the owner of flat index x is
        // floor(((x+1)*S - 1) / N)
        const int64_t i0 = floordiv_i64((first + 1) * S - 1, N);
        const int64_t i1 = floordiv_i64((first + n) * S - 1, N);
        if (i0 == i1) return;                         // written whole by CTA i0
        const int64_t unit = int64_t(hg) * p.batch + b;
        const int64_t stride = int64_t(nh) * G;      // partial rows per CTA slot
        // with fewer blocks than CTAs some CTAs have an empty range and wrote
        // nothing (never the case when N >= S)
        auto live = [&](int64_t i) { return !(N < S && (i * N) / S == ((i + 1) * N) / S); };
        const int64_t np = i1 - i0 + 1;               // partials (CTA slots) to combine
        float M = NEG_INF, Lsum = 0.0f;
        if (np <= kMergeBatch) {
            // one round trip: lane k loads (m, l) of partial k while every
            // lane loads its head_dim slice of all partials
            float v[kMergeBatch][EPL];
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                const bool ok = k < np && live(i0 + k);
                const float *pa = f.part_acc + ((i0 + k + unit) * stride + local) * D + EPL * lane;
                if constexpr (EPL == 4) {
                    const float4 t = ok ? *reinterpret_cast<const float4 *>(pa) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[k][0] = t.x;
                    v[k][1] = t.y;
                    v[k][2] = t.z;
                    v[k][3] = t.w;
                } else {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) v[k][e] = ok ? pa[e] : 0.0f;
                }
            }
            float mi = NEG_INF, li = 0.0f;
            if (lane < np && live(i0 + lane)) {
                const int64_t row = (i0 + lane + unit) * stride + local;
                mi = f.part_ml[2 * row];
                li = f.part_ml[2 * row + 1];
            }
            M = mi;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float wgt = mi == NEG_INF ? 0.0f : exp2_approx(mi - M);
            Lsum = li * wgt;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                const float wk = __shfl_sync(0xffffffffu, wgt, k);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[e] += v[k][e] * wk;
            }
        } else {
            // many partials (a long sequence over many CTAs): lanes over the
            // partials for the maximum and the weights, then lanes over
            // head_dim for the accumulation, 32 partials at a time
            for (int64_t c = i0; c <= i1; c += 32) {
                const int64_t i = c + lane;
                if (i <= i1 && live(i)) M = fmaxf(M, f.part_ml[2 * ((i + unit) * stride + local)]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            for (int64_t c = i0; c <= i1; c += 32) {
                const int64_t i = c + lane;
                float wgt = 0.0f;
                if (i <= i1 && live(i)) {
                    const int64_t row = (i + unit) * stride + local;
                    const float mi = f.part_ml[2 * row];
                    wgt = mi == NEG_INF ? 0.0f : exp2_approx(mi - M);
                    Lsum += f.part_ml[2 * row + 1] * wgt;
                }
                const int cnt = int(i1 - c + 1 < 32 ? i1 - c + 1 : 32);
                for (int k = 0; k < cnt; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, wgt, k);
                    if (wk == 0.0f) continue;       // uniform; also skips unwritten slots
                    const float *pa = f.part_acc + ((c + k + unit) * stride + local) * D + EPL * lane;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] += pa[e] * wk;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
        }
        const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= inv;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e)
        orow[EPL * lane + e] = p.q_is_bf16 ? f2h<kBF16>(acc[e]) : f2h<kF16>(acc[e]);
}

template <int CK, int D, int BS, int U3H = 0, bool GSC = false, bool XV = false, int NG = 1>
cudaError_t launch_fast_t(const DecodeParams &p, const FastParams &f, const CUtensorMap &mk,
                          const CUtensorMap &mv, cudaStream_t s)
{
    auto kern = decode_tma_kernel<CK, D, BS, U3H, GSC, XV, NG>;
    // dynamic shared memory limit, raised once per device as needed
    static std::atomic<int> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (configured[dev].load(std::memory_order_relaxed) < f.smem_bytes) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, f.smem_bytes);
        if (e != cudaSuccess) return e;
        configured[dev].store(f.smem_bytes, std::memory_order_relaxed);
    }
    e = launch_pdl(kern, dim3(f.grid), dim3((f.ncons + 1) * 32), f.smem_bytes, s, mk, mv, p, f);
    if (e != cudaSuccess) return e;
    const int rows = p.batch * p.num_heads;
    return launch_pdl(merge_kernel<D>, dim3((rows + kMergeWarps - 1) / kMergeWarps), dim3(32 * kMergeWarps),
                      size_t(p.batch + 1) * 4, s, p, f);
}

// The instances of one cache kind and head_dim: block size, 3-bit kv heads
// per consumer warp, staged granular scales and head-column groups.
template <int CK, int D>
cudaError_t launch_fast_bs(const DecodeParams &p, const FastParams &f, const CUtensorMap &mk,
                           const CUtensorMap &mv, cudaStream_t s)
{
    if constexpr (CK == kU3) {      // MHA caches: f.hpw kv heads per consumer warp
        if (p.group == 1) {
            if (p.block_size == 16) {
                if (f.hpw == 4) return launch_fast_t<CK, D, 16, 4>(p, f, mk, mv, s);
                if (f.hpw == 2) return launch_fast_t<CK, D, 16, 2>(p, f, mk, mv, s);
                return launch_fast_t<CK, D, 16, 1>(p, f, mk, mv, s);
            }
            if (p.block_size == 32) {
                if (f.hpw == 4) return launch_fast_t<CK, D, 32, 4>(p, f, mk, mv, s);
                if (f.hpw == 2) return launch_fast_t<CK, D, 32, 2>(p, f, mk, mv, s);
                return launch_fast_t<CK, D, 32, 1>(p, f, mk, mv, s);
            }
            if (p.block_size == 64) {
                if (f.hpw == 4) return launch_fast_t<CK, D, 64, 4>(p, f, mk, mv, s);
                if (f.hpw == 2) return launch_fast_t<CK, D, 64, 2>(p, f, mk, mv, s);
                return launch_fast_t<CK, D, 64, 1>(p, f, mk, mv, s);
            }
        }
    }
    if constexpr (is_q8(CK)) {      // per-block / per-token scales staged with the tiles
        if (p.scale_mode != 0) {
            switch (p.block_size) {
            case 16:
                return f.ng == 2 ? launch_fast_t<CK, D, 16, 0, true, false, 2>(p, f, mk, mv, s)
                                 : launch_fast_t<CK, D, 16, 0, true>(p, f, mk, mv, s);
            case 32:
                return f.ng == 2 ? launch_fast_t<CK, D, 32, 0, true, false, 2>(p, f, mk, mv, s)
                                 : launch_fast_t<CK, D, 32, 0, true>(p, f, mk, mv, s);
            case 64: return launch_fast_t<CK, D, 64, 0, true>(p, f, mk, mv, s);
            default: return cudaErrorInvalidValue;
            }
        }
    }
    switch (p.block_size) {
    case 16:
        if (f.ng == 2) return launch_fast_t<CK, D, 16, 0, false, false, 2>(p, f, mk, mv, s);
        return launch_fast_t<CK, D, 16>(p, f, mk, mv, s);
    case 32:
        if (f.ng == 2) return launch_fast_t<CK, D, 32, 0, false, false, 2>(p, f, mk, mv, s);
        return launch_fast_t<CK, D, 32>(p, f, mk, mv, s);
    case 64: return launch_fast_t<CK, D, 64>(p, f, mk, mv, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace pkv
