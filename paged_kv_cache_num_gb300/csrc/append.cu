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
// GB300 mapping: the copy and fp8 kernels give each (token, K|V) to one
// warp whose lanes take the token's 16-byte pieces across its kv heads (one
// slot lookup per warp, 32-bit index arithmetic, four 16-byte loads in
// flight per lane, fully coalesced loads and stores); the grid is a
// function of num_tokens only (CUDA-graph safe).  The 3-bit kernel gives
// each row eight lanes (four rows per warp): the min / max are shuffle
// reductions among them and the packed 12-byte runs are assembled by
// shuffles.  Work items are walked by additions, without a 64-bit division
// per item.  Large batches with contiguous head rows move by TMA bulk
// copies instead (append_bulk_kernel).  All are programmatic dependent
// launches, so the launch of each overlaps the tail of the previous kernel
// in the stream.
#include <algorithm>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

// slot of token t from its (request, position) through the block table:
// blk = block_tables[req][pos >> log2(BS)], slot = blk * BS + (pos & (BS-1));
// -1 for pos < 0 (padding), and for positions outside the table (raising
// PKV_DEVERR_POS_RANGE)
__device__ __forceinline__ int64_t slot_from_position(const SlotMapParams &p, int64_t t)
{
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
    return slot;
}

// the slot of token t; `first`: this caller writes a computed slot out
// (from_pos)
__device__ __forceinline__ int64_t fetch_slot(const AppendParams &p, int64_t t, bool first)
{
    if (p.from_pos) {
        const int64_t slot = slot_from_position(p.pos_map, t);
        if (first) p.pos_map.slot_mapping[t] = slot;
        return slot;
    }
    return p.slot_mapping[t * p.slot_stride];
}

// (block, offset) of a slot; false for a padding token (slot < 0) and for a
// slot outside the pool (raising PKV_DEVERR_SLOT_RANGE)
__device__ __forceinline__ bool place_slot(const AppendParams &p, int64_t slot, int64_t &blk, int64_t &off)
{
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

// `first`: this caller writes the token's computed slot out (from_pos)
__device__ __forceinline__ bool resolve_slot(const AppendParams &p, int64_t t, int64_t &blk,
                                             int64_t &off, bool first = false)
{
    return place_slot(p, fetch_slot(p, t, first), blk, off);
}

// A grid-stride walk over items i = major * n + minor (0 <= minor < n)
// that keeps (major, minor) current by additions: two 32-bit divisions per
// warp at the start, none per item (a 64-bit division by a runtime value
// costs about a hundred instructions).  The first item and the stride are
// warp counts of grids capped at a few thousand blocks, far below 2^32.
struct Walk2 {
    int64_t major, step_major;
    int minor, step_minor, n;
    __device__ __forceinline__ Walk2(int64_t first, int64_t step, int n_) : n(n_)
    {
        const uint32_t f = uint32_t(first), s = uint32_t(step), un = uint32_t(n_);
        const uint32_t fq = f / un, sq = s / un;
        major = fq;
        minor = int(f - fq * un);
        step_major = sq;
        step_minor = int(s - sq * un);
    }
    __device__ __forceinline__ void next()
    {
        major += step_major;
        minor += step_minor;
        if (minor >= n) {
            minor -= n;
            ++major;
        }
    }
};

// Work items of the copy and one-byte append kernels: a (token, K|V) row
// split into parts of 32 * U pieces, one warp per item.  U = 4 (four loads
// in flight per lane) for large batches, U = 1 for small ones, which then
// spread over more warps.
__host__ __device__ inline int append_parts(int per, int U) { return (per + 32 * U - 1) / (32 * U); }

// 16-bit copy: one warp per (token, K|V, part), its lanes over the part's
// (kv head, CHUNK-byte piece) pieces.  The slot is resolved once per warp;
// the index arithmetic is 32-bit.
template <int CHUNK, int U>
__global__ void __launch_bounds__(kAppendThreads) append_copy_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    using V = std::conditional_t<CHUNK == 16, uint4, uint16_t>;
    const int lane = threadIdx.x & 31;
    const int cph = p.head_dim * 2 / CHUNK;        // pieces per head row
    const int per = p.num_kv_heads * cph;          // pieces per (token, K|V)
    const int parts = append_parts(per, U);
    const int64_t wstep = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (Walk2 w((blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5, wstep, parts);
         w.major < p.num_tokens * 2; w.next()) {
        const int64_t row = w.major;          // (token, K|V)
        const int part = w.minor;
        const int64_t t = row >> 1;
        const int kv = int(row & 1);
        int64_t blk, off;
        if (!resolve_slot(p, t, blk, off, kv == 0 && part == 0 && lane == 0)) continue;   // warp-uniform
        const char *src = kv ? p.v_new + t * p.v_src_tok : p.k_new + t * p.k_src_tok;
        const int64_t src_head = kv ? p.v_src_head : p.k_src_head;
        char *dst = (kv ? p.v_cache : p.k_cache) + blk * p.c_blk + off * p.c_slot;
        {
            const int i0 = part * 32 * U + lane;
            constexpr int kU = U;
            V v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + 32 * u;
                if (i < per) {
                    const int h = i / cph, c = i - h * cph;
                    v[u] = __ldg(reinterpret_cast<const V *>(src + h * src_head) + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + 32 * u;
                if (i < per) {
                    const int h = i / cph, c = i - h * cph;
                    // the row's 16-byte pieces are c_chunk bytes apart (16 when contiguous)
                    char *d = dst + h * p.c_head;
                    if constexpr (CHUNK == 16)
                        *reinterpret_cast<uint4 *>(d + c * p.c_chunk) = v[u];
                    else
                        *reinterpret_cast<uint16_t *>(d + (c >> 3) * p.c_chunk + 2 * (c & 7)) = v[u];
                }
            }
        }
    }
}

// 16-bit rows whose kv heads are contiguous in the source and in the cache
// (the flash layout): each (token, K|V) row is one run of Hkv * head_dim
// elements on both sides and moves with two TMA bulk copies, global ->
// shared -> global, without passing through registers.  One thread per CTA
// issues them through a ring of kBulkSlots shared-memory rows: the load of
// row k is issued kBulkLag rows ahead of its store, and a slot is reloaded
// only once the store issued from it has read it.  The warp's lanes fetch
// the slots of the next 32 rows at once.  Every wait is bounded.
constexpr int kBulkSlots = 8;
constexpr int64_t kBulkMinTokens = 1024;   // below this the warp kernel is as fast
constexpr int kBulkLag = 4;
constexpr uint64_t kBulkTimeoutNs = 2000000000ull;

__global__ void __launch_bounds__(32) append_bulk_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ __align__(128) unsigned char bulk_buf[];
    __shared__ __align__(8) uint64_t bars[kBulkSlots];
    __shared__ char *dsts[kBulkSlots];
    const int lane = threadIdx.x;
    const uint32_t row_bytes = uint32_t(p.num_kv_heads) * uint32_t(p.head_dim) * 2u;
    const uint32_t buf = ptx::smem_u32(bulk_buf);
    const uint32_t bar0 = ptx::smem_u32(bars);
    if (lane == 0) {
        for (int i = 0; i < kBulkSlots; ++i) ptx::mbar_init(bar0 + 8 * i, 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    const int64_t rows = p.num_tokens * 2;
    const int64_t n = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t k = 0;                  // rows of this CTA with a copy issued (lane 0)
    bool aborted = false;
    // store of the row in ring position j (its load issued earlier)
    auto store = [&](int64_t j) {
        const int sl = int(j % kBulkSlots);
        if (!ptx::mbar_wait_bounded(bar0 + 8 * sl, uint32_t((j / kBulkSlots) & 1), kBulkTimeoutNs)) {
            raise_err(p.err_flag, PKV_DEVERR_TIMEOUT);
            aborted = true;
            return;
        }
        ptx::fence_proxy_async_smem();
        ptx::bulk_store(dsts[sl], buf + sl * row_bytes, row_bytes);
        ptx::bulk_commit();
    };
    for (int64_t i0 = 0; i0 < n; i0 += 32) {
        int64_t mine = -1;          // lane l: the slot of this CTA's row i0 + l
        if (i0 + lane < n) {
            const int64_t r = blockIdx.x + (i0 + lane) * gridDim.x;
            mine = fetch_slot(p, r >> 1, (r & 1) == 0);
        }
        for (int jj = 0; jj < 32 && i0 + jj < n; ++jj) {
            const int64_t slot = __shfl_sync(0xffffffffu, mine, jj);
            if (lane != 0 || aborted) continue;
            int64_t blk, off;
            if (!place_slot(p, slot, blk, off)) continue;      // padding / out of range
            const int64_t r = blockIdx.x + (i0 + jj) * gridDim.x;
            const int64_t t = r >> 1;
            const int kv = int(r & 1);
            const int sl = int(k % kBulkSlots);
            // the store issued from this slot kBulkSlots rows ago has read it:
            // stores of rows <= k - kBulkLag - 1 are committed, at most
            // kBulkSlots - kBulkLag - 1 of them may still be reading
            if (k >= kBulkSlots) ptx::bulk_wait_read<kBulkSlots - kBulkLag - 1>();
            dsts[sl] = (kv ? p.v_cache : p.k_cache) + blk * p.c_blk + off * p.c_slot;
            const char *src = kv ? p.v_new + t * p.v_src_tok : p.k_new + t * p.k_src_tok;
            ptx::mbar_arrive_expect_tx(bar0 + 8 * sl, row_bytes);
            ptx::bulk_load(buf + sl * row_bytes, src, row_bytes, bar0 + 8 * sl);
            if (k >= kBulkLag) store(k - kBulkLag);
            ++k;
        }
    }
    if (lane == 0) {
        for (int64_t j = k > kBulkLag ? k - kBulkLag : 0; j < k && !aborted; ++j) store(j);
        // copies still in flight (an aborted wait) land before the CTA exits
        for (int64_t j = k > kBulkLag ? k - kBulkLag : 0; aborted && j < k; ++j)
            ptx::mbar_wait_bounded(bar0 + 8 * int(j % kBulkSlots), uint32_t((j / kBulkSlots) & 1), kBulkTimeoutNs);
        ptx::bulk_wait_all();
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

// One-byte codes (e4m3, e5m2, int8): one warp per (token, K|V, part), its
// lanes over the part's (kv head, 8-element group) pieces (16 source bytes
// -> 8 cache bytes each).
template <int SRC, bool VEC, int FP8, int U>
__global__ void __launch_bounds__(kAppendThreads) append_fp8_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int kU = U;
    const int lane = threadIdx.x & 31;
    const int groups = p.head_dim / 8;             // pieces per head row
    const int gsh = (groups & (groups - 1)) == 0 ? __ffs(groups) - 1 : -1;   // log2(groups), if a power of 2
    const int per = p.num_kv_heads * groups;       // pieces per (token, K|V)
    const int parts = append_parts(per, U);
    const int64_t wstep = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (Walk2 w((blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5, wstep, parts);
         w.major < p.num_tokens * 2; w.next()) {
        const int64_t row = w.major;          // (token, K|V)
        const int part = w.minor;
        const int64_t t = row >> 1;
        const int kv = int(row & 1);
        int64_t blk, off;
        if (!resolve_slot(p, t, blk, off, kv == 0 && part == 0 && lane == 0)) continue;   // warp-uniform
        const char *src_row = kv ? p.v_new + t * p.v_src_tok : p.k_new + t * p.k_src_tok;
        const int64_t src_head = kv ? p.v_src_head : p.k_src_head;
        char *dst_row = (kv ? p.v_cache : p.k_cache) + blk * p.c_blk + off * p.c_slot;
        {
            const int i0 = part * 32 * U + lane;
            uint16_t e[kU][8];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + 32 * u;
                if (i >= per) continue;
                const int h = gsh >= 0 ? i >> gsh : i / groups, c = i - h * groups;
                const uint16_t *src = reinterpret_cast<const uint16_t *>(src_row + h * src_head) + 8 * c;
                if constexpr (VEC) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
                    e[u][0] = v.x & 0xffff; e[u][1] = v.x >> 16; e[u][2] = v.y & 0xffff; e[u][3] = v.y >> 16;
                    e[u][4] = v.z & 0xffff; e[u][5] = v.z >> 16; e[u][6] = v.w & 0xffff; e[u][7] = v.w >> 16;
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) e[u][j] = src[j];
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + 32 * u;
                if (i >= per) continue;
                const int h = gsh >= 0 ? i >> gsh : i / groups, c = i - h * groups;
                // elements 8c .. 8c+7: half of the row's 16-byte piece c / 2
                uint8_t *dst = reinterpret_cast<uint8_t *>(dst_row + h * p.c_head + (c >> 1) * p.c_chunk) +
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
                uint32_t packed[2];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // scale division in fp32 (IEEE round to nearest), then the cast
                    float2 x;
                    x.x = __fdiv_rn(h2f<SRC>(e[u][2 * j]), scale);
                    x.y = __fdiv_rn(h2f<SRC>(e[u][2 * j + 1]), scale);
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
    }
}

// RN(x / s) for 16-bit float x and fp16 s > 0, through the correctly
// rounded reciprocal rs = RN(1 / s): with y1 = RN(x rs) and the exact
// residual e = x - y1 s (one FMA), RN(y1 + e rs) is within far less than
// half an ulp of x / s (Markstein's refinement), so it equals x / s
// wherever x / s is an fp32 value -- at every half-integer in particular.
// Off the half-integers rint of it is rint(fl(x / s)) in the codes' range:
// x and s have at most 11 significant bits, so an x / s with |x / s| < 2^10
// that is not a half-integer lies at least 2^-13 away from one.
__device__ __forceinline__ float u3_quotient(float x, float s, float rs)
{
    const float y1 = __fmul_rn(x, rs);
    return __fmaf_rn(__fmaf_rn(-y1, s, x), rs, y1);
}

// min / max of two pairs of 16-bit floats (non-NaN operand wins, as fminf /
// fmaxf); exact, the values being 16-bit floats
template <int SRC>
__device__ __forceinline__ uint32_t min2_16(uint32_t a, uint32_t b)
{
    uint32_t r;
    if constexpr (SRC == kBF16) asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else asm("min.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <int SRC>
__device__ __forceinline__ uint32_t max2_16(uint32_t a, uint32_t b)
{
    uint32_t r;
    if constexpr (SRC == kBF16) asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 3-bit affine quantise + pack: LPR = 4 lanes per (token, head, K|V) row,
// eight rows per warp.  Each lane holds EPL = head_dim / 4 consecutive
// elements; a row's min / max are two-step shuffle reductions among its
// lanes, which then each derive the row's scale (one IEEE division) and
// zero point.  A lane's codes make EPL / 8 fields of 24 bits (8 codes each;
// code d sits at bit 3d of the packed row); four consecutive fields -- 96
// bits -- fill one 12-byte run, which is a lane's own at head_dim 128 and
// is gathered from two lanes by shuffles at head_dim 64.
template <int SRC, int EPL, int LPR>
__global__ void __launch_bounds__(kAppendThreads) append_u3_kernel(AppendParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int RPW = 32 / LPR;        // rows per warp
    constexpr int WARPS = kAppendThreads / 32;
    constexpr int NF = EPL / 8;          // 24-bit fields per lane
    constexpr int LR = NF >= 4 ? 1 : 4 / NF;   // lanes per 12-byte run
    constexpr int RUNS = NF >= 4 ? NF / 4 : 1;  // runs a storing lane writes
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int grp = lane / LPR, sub = lane % LPR;   // the warp's row, the lane within it
    Walk2 w((blockIdx.x * int64_t(WARPS) + wid) * RPW + grp, int64_t(gridDim.x) * WARPS * RPW,
            2 * p.num_kv_heads);
    while (__any_sync(0xffffffffu, w.major < p.num_tokens)) {
        const int64_t t = w.major;
        const int r = w.minor;               // (kv head, K|V)
        const int h = r >> 1, kv = r & 1;
        int64_t blk = 0, off = 0;
        const bool live = t < p.num_tokens && resolve_slot(p, t, blk, off, r == 0 && sub == 0);
        // the lane's EPL source values as pairs of 16-bit floats
        uint32_t wv[EPL / 2];
#pragma unroll
        for (int j = 0; j < EPL / 2; ++j) wv[j] = 0u;
        if (live) {
            const uint16_t *src = reinterpret_cast<const uint16_t *>(
                kv ? p.v_new + t * p.v_src_tok + h * p.v_src_head
                   : p.k_new + t * p.k_src_tok + h * p.k_src_head) + EPL * sub;
            if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {       // 16-byte vector loads
#pragma unroll
                for (int v = 0; v < EPL / 8; ++v) {
                    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src) + v);
                    wv[4 * v] = u.x;
                    wv[4 * v + 1] = u.y;
                    wv[4 * v + 2] = u.z;
                    wv[4 * v + 3] = u.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < EPL / 2; ++j) wv[j] = uint32_t(src[2 * j]) | (uint32_t(src[2 * j + 1]) << 16);
            }
        }
        float x[EPL];
#pragma unroll
        for (int j = 0; j < EPL / 2; ++j) {
            x[2 * j] = h2f<SRC>(uint16_t(wv[j]));
            x[2 * j + 1] = h2f<SRC>(uint16_t(wv[j] >> 16));
        }
        // the lane's min / max: pairwise in 16 bits, then its two halves
        uint32_t mn2 = wv[0], mx2 = wv[0];
#pragma unroll
        for (int j = 1; j < EPL / 2; ++j) {
            mn2 = min2_16<SRC>(mn2, wv[j]);
            mx2 = max2_16<SRC>(mx2, wv[j]);
        }
        float mn = fminf(h2f<SRC>(uint16_t(mn2)), h2f<SRC>(uint16_t(mn2 >> 16)));
        float mx = fmaxf(h2f<SRC>(uint16_t(mx2)), h2f<SRC>(uint16_t(mx2 >> 16)));
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) {   // within the row's lanes
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        // s = fp16_rn((max - min) / 7), saturated to the largest finite fp16
        uint16_t sbits = __half_as_ushort(__float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 7.0f)));
        if ((sbits & 0x7fff) == 0x7c00) sbits = 0x7bff;
        const float s = __half2float(__ushort_as_half(sbits));
        const float rs = s != 0.0f ? __frcp_rn(s) : 0.0f;
        // z = clamp(rint(fl(-min / s)), 0, 7); -min is one of the row's
        // 16-bit values, so u3_quotient gives the same rint
        float z = 0.0f;
        if (s != 0.0f) z = fminf(fmaxf(rintf(u3_quotient(-mn, s, rs)), 0.0f), 7.0f);
        // fields: codes q_j = clamp(rint(fl(x_j / s)) + z, 0, 7) at bits 3j
        // (small integers, exact in fp32).  A constant row (s = 0: every x_j
        // equal and finite) has rs = 0 and z = 0, so its quotients are 0 and
        // its codes 0 without a test per element.
        uint32_t f[NF];
#pragma unroll
        for (int fi = 0; fi < NF; ++fi) {
            float fv = 0.0f;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                const float q = fminf(fmaxf(__fadd_rn(rintf(u3_quotient(x[8 * fi + j], s, rs)), z), 0.0f), 7.0f);
                fv = fmaf(fv, 8.0f, q);
            }
            f[fi] = uint32_t(fv);
        }
        // each run's four fields, in order (gathered by its first lane when
        // a lane holds fewer than four)
        uint32_t F[RUNS][4];
#pragma unroll
        for (int ru = 0; ru < RUNS; ++ru)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                F[ru][k] = LR == 1 ? f[4 * ru + k] : __shfl_sync(0xffffffffu, f[k % NF], lane + k / NF);
        if (live && sub % LR == 0) {
            uint8_t *row = reinterpret_cast<uint8_t *>((kv ? p.v_cache : p.k_cache) + blk * p.c_blk +
                                                       off * p.c_slot + h * p.c_head);
#pragma unroll
            for (int ru = 0; ru < RUNS; ++ru) {
                const uint32_t w0 = F[ru][0] | (F[ru][1] << 24);
                const uint32_t w1 = (F[ru][1] >> 8) | (F[ru][2] << 16);
                const uint32_t w2 = (F[ru][2] >> 16) | (F[ru][3] << 8);
                uint8_t *dst = row + 12 * (RUNS * sub / LR + ru);
                if ((reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
                    uint32_t *d32 = reinterpret_cast<uint32_t *>(dst);
                    d32[0] = w0;
                    d32[1] = w1;
                    d32[2] = w2;
                } else {                // rows at strides that are not multiples of 4 bytes
                    const uint32_t run[3] = {w0, w1, w2};
#pragma unroll
                    for (int b = 0; b < 12; ++b) dst[b] = uint8_t(run[b >> 2] >> (8 * (b & 3)));
                }
            }
        }
        if (live && sub == 0) {
            uint16_t *qs = kv ? p.v_qs : p.k_qs;
            uint8_t *qz = kv ? p.v_qz : p.k_qz;
            qs[blk * p.m_blk + off * p.m_slot + h * p.m_head] = sbits;
            qz[blk * p.z_blk + off * p.z_slot + h * p.z_head] = uint8_t(z);
        }
        w.next();
    }
}

__global__ void slot_mapping_kernel(SlotMapParams p)
{
    griddep_wait();
    griddep_launch_dependents();
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < p.n;
         t += int64_t(gridDim.x) * blockDim.x)
        p.slot_mapping[t] = slot_from_position(p, t);
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
    // one warp per (token, K|V, part): four pieces per lane when that still
    // gives every SM several warps, else one (more, shorter warps)
    auto small = [&](int per) {
        return p.num_tokens * 2 * append_parts(per, 4) < int64_t(sm_count_current_device()) * 8;
    };
    auto grid = [&](int per, int U) { return grid_for(p.num_tokens * 2 * append_parts(per, U) * 32, T); };
    if (cache_kind == kF16 || cache_kind == kBF16) {
        // large batches with contiguous head rows on both sides: TMA bulk copies
        const int64_t row_bytes = int64_t(p.num_kv_heads) * p.head_dim * 2;
        if (vec16 && p.num_tokens >= kBulkMinTokens && p.k_src_head == p.head_dim * 2 &&
            p.v_src_head == p.head_dim * 2 && p.c_head == p.head_dim * 2 && p.c_chunk == 16 &&
            row_bytes % 16 == 0 && kBulkSlots * row_bytes <= 48 * 1024) {
            const int g = int(std::min<int64_t>(p.num_tokens * 2, int64_t(sm_count_current_device()) * 8));
            return launch_pdl(append_bulk_kernel, g, 32, size_t(kBulkSlots * row_bytes), s, p);
        }
        const int per = p.num_kv_heads * (vec16 ? p.head_dim * 2 / 16 : p.head_dim);
        const bool one = small(per);
        const int g = grid(per, one ? 1 : 4);
        if (vec16) return one ? launch_pdl(append_copy_kernel<16, 1>, g, T, 0, s, p)
                              : launch_pdl(append_copy_kernel<16, 4>, g, T, 0, s, p);
        return one ? launch_pdl(append_copy_kernel<2, 1>, g, T, 0, s, p)
                   : launch_pdl(append_copy_kernel<2, 4>, g, T, 0, s, p);
    } else if (is_q8(cache_kind)) {
        const int per = p.num_kv_heads * (p.head_dim / 8);
        const bool one = small(per);
        const int g = grid(per, one ? 1 : 4);
        auto go = [&](auto src_c, auto vec_c, auto u_c) -> cudaError_t {
            constexpr int S = decltype(src_c)::value;
            constexpr bool V = decltype(vec_c)::value;
            constexpr int U = decltype(u_c)::value;
            if (cache_kind == kE4M3) return launch_pdl(append_fp8_kernel<S, V, kE4M3, U>, g, T, 0, s, p);
            if (cache_kind == kE5M2) return launch_pdl(append_fp8_kernel<S, V, kE5M2, U>, g, T, 0, s, p);
            return launch_pdl(append_fp8_kernel<S, V, kI8, U>, g, T, 0, s, p);
        };
        auto go_u = [&](auto src_c, auto vec_c) -> cudaError_t {
            return one ? go(src_c, vec_c, std::integral_constant<int, 1>{})
                       : go(src_c, vec_c, std::integral_constant<int, 4>{});
        };
        using BF = std::integral_constant<int, kBF16>;
        using HF = std::integral_constant<int, kF16>;
        if (p.src_kind == kBF16)
            return vec16 ? go_u(BF{}, std::true_type{}) : go_u(BF{}, std::false_type{});
        return vec16 ? go_u(HF{}, std::true_type{}) : go_u(HF{}, std::false_type{});
    } else {  // kU3
        const int64_t rows = p.num_tokens * 2 * p.num_kv_heads;
        constexpr int LPR = 4;                      // lanes per row (two: slower)
        const int g = grid_for(rows * LPR, T);
        const bool bf = p.src_kind == kBF16;
        if (p.head_dim == 128) {
            if (bf) return launch_pdl(append_u3_kernel<kBF16, 128 / LPR, LPR>, g, T, 0, s, p);
            else return launch_pdl(append_u3_kernel<kF16, 128 / LPR, LPR>, g, T, 0, s, p);
        } else {
            if (bf) return launch_pdl(append_u3_kernel<kBF16, 64 / LPR, LPR>, g, T, 0, s, p);
            else return launch_pdl(append_u3_kernel<kF16, 64 / LPR, LPR>, g, T, 0, s, p);
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
