// pack3.cu -- standalone 3-bit packing / unpacking and the copy kernel used
// as the HBM bandwidth yardstick.
//
// "triton-3bit-kv-cache-kernel" README, section 1.A: an octet of 8 three-bit
// lanes occupies 24 bits, lane i at bits 3i..3i+2 of
// word24 = b0 | b1 << 8 | b2 << 16, so every lane (including v2 and v5, which
// straddle bytes) is one shift and mask of word24.  Section 1.B: in a 96-bit
// group of three little-endian uint32 words, lane i starts at bit 3i, in word
// 3i/32 at shift 3i%32; lanes 10 and 21 take their high bits from the next
// word.
//
// GB300 mapping: each thread handles 4 octets (32 value bytes <-> 12 packed
// bytes) so both sides move with aligned 16-byte / 4-byte vector accesses;
// the unpacking moves four codes at a time from their 3-bit to their byte
// positions in two halving steps (spread4), a few ALU operations each;
// the unpacking kernels exchange halves between lanes so that each store
// instruction of a warp is one contiguous 512-byte run.  The kernels are
// pure HBM streams.
#include <atomic>

#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;

// Blocks of kernel K (kThreads threads each, no dynamic shared memory) that
// one SM holds at once, at least 1; queried once per device.  The
// grid-stride kernels below size their grids to SMs x this, one wave:
// blocks beyond it would start only after a first wave had finished its
// share.
template <auto K>
int resident_blocks()
{
    constexpr int kDevices = 64;
    static std::atomic<int> cache[kDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return 1;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K, kThreads, 0) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();     // not left pending for the launch's own check
            n = 1;
        }
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Four codes at bits 0-11 (code i at bit 3i) -> bytes 0-3, in two halving
// steps instead of one shift and mask per code: codes 0-1 and 2-3 first
// move apart as 6-bit pairs to bits 0-5 and 16-21, then each pair opens
// out into its two bytes.  u < 2^12.
__device__ __forceinline__ uint32_t spread4(uint32_t u)
{
    const uint32_t t = (u | (u << 10)) & 0x003F003Fu;
    return (t | (t << 5)) & 0x07070707u;
}

__device__ __forceinline__ uint32_t pack_octet(uint32_t lo4, uint32_t hi4)
{
    // lo4 / hi4 hold lanes 0-3 / 4-7 as bytes; keep 3 bits of each
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w |= ((lo4 >> (8 * i)) & 7u) << (3 * i);
        w |= ((hi4 >> (8 * i)) & 7u) << (3 * (i + 4));
    }
    return w;  // 24 significant bits
}

// w24 < 2^24
__device__ __forceinline__ void unpack_octet(uint32_t w24, uint32_t &lo4, uint32_t &hi4)
{
    lo4 = spread4(w24 & 0xFFFu);
    hi4 = spread4(w24 >> 12);
}

// 4 octets per thread: 32 value bytes (two 16-byte loads) -> 12 bytes.
__global__ void __launch_bounds__(kThreads) pack3_kernel(const uint8_t *__restrict__ values,
                                                         uint8_t *__restrict__ packed, int64_t n)
{
    const int64_t n4 = n / 4;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(values) + 2 * i);
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(values) + 2 * i + 1);
        const uint32_t w0 = pack_octet(a.x, a.y), w1 = pack_octet(a.z, a.w);
        const uint32_t w2 = pack_octet(b.x, b.y), w3 = pack_octet(b.z, b.w);
        // 4 x 24 bits -> 3 little-endian words
        uint32_t *dst = reinterpret_cast<uint32_t *>(packed + 12 * i);
        dst[0] = w0 | (w1 << 24);
        dst[1] = (w1 >> 8) | (w2 << 16);
        dst[2] = (w2 >> 16) | (w3 << 8);
    }
    // tail octets (n % 4), one thread each
    const int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (t < n - 4 * n4) {
        const int64_t o = 4 * n4 + t;
        uint32_t lo = 0, hi = 0;
        for (int j = 0; j < 4; ++j) {
            lo |= uint32_t(values[8 * o + j]) << (8 * j);
            hi |= uint32_t(values[8 * o + 4 + j]) << (8 * j);
        }
        const uint32_t w = pack_octet(lo, hi);
        packed[3 * o] = uint8_t(w);
        packed[3 * o + 1] = uint8_t(w >> 8);
        packed[3 * o + 2] = uint8_t(w >> 16);
    }
}

// 96 packed bits w0 | w1 << 32 | w2 << 64 as 32 value bytes: code i (bit
// 3i) lies in 12-bit field i/4 at bit 3(i%4), and each field spreads into
// 4 bytes.  Fields 2 and 5 span two words -- they hold codes 10 and 21, the
// two codes whose high bits come from the next word -- and are cut with
// funnel shifts.  Four octets (12 bytes, octet j = bits 24j..24j+23) and a
// 96-bit group of three little-endian words are the same bits, so both
// unpacking kernels use this.
__device__ __forceinline__ void unpack96(uint32_t w0, uint32_t w1, uint32_t w2, uint4 &x, uint4 &y)
{
    x.x = spread4(w0 & 0xFFFu);
    x.y = spread4((w0 >> 12) & 0xFFFu);
    x.z = spread4(__funnelshift_r(w0, w1, 24) & 0xFFFu);
    x.w = spread4((w1 >> 4) & 0xFFFu);
    y.x = spread4((w1 >> 16) & 0xFFFu);
    y.y = spread4(__funnelshift_r(w1, w2, 28) & 0xFFFu);
    y.z = spread4((w2 >> 8) & 0xFFFu);
    y.w = spread4(w2 >> 20);
}

// Quad (4 octets, 12 packed bytes) i of the input as 32 value bytes: x holds
// octets 0-1, y octets 2-3 (zeros past the end).
__device__ __forceinline__ void unpack_quad(const uint8_t *__restrict__ packed, int64_t i, int64_t n4, uint4 &x,
                                            uint4 &y)
{
    x = make_uint4(0, 0, 0, 0);
    y = make_uint4(0, 0, 0, 0);
    if (i < n4) {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(packed + 12 * i);
        unpack96(__ldg(src), __ldg(src + 1), __ldg(src + 2), x, y);
    }
}

// The warp's 32 units (x, y: 32 value bytes each, unit `lane` in lane
// `lane`) of chunk wc, written as 16-byte pieces 32k + lane of the chunk's
// kilobyte: piece 32k + lane is half (lane & 1) of unit 16k + (lane >> 1),
// moved between lanes by shuffles, so that each store instruction is one
// contiguous 512-byte run.  Every lane takes part in both shuffles, then
// keeps its half.
__device__ __forceinline__ void store_chunk(uint8_t *__restrict__ values, int64_t wc, int64_t units, int lane,
                                            const uint4 &x, const uint4 &y)
{
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int srcl = 16 * k + (lane >> 1);
        const bool hi = lane & 1;
        const uint32_t a0 = __shfl_sync(0xffffffffu, x.x, srcl), b0 = __shfl_sync(0xffffffffu, y.x, srcl);
        const uint32_t a1 = __shfl_sync(0xffffffffu, x.y, srcl), b1 = __shfl_sync(0xffffffffu, y.y, srcl);
        const uint32_t a2 = __shfl_sync(0xffffffffu, x.z, srcl), b2 = __shfl_sync(0xffffffffu, y.z, srcl);
        const uint32_t a3 = __shfl_sync(0xffffffffu, x.w, srcl), b3 = __shfl_sync(0xffffffffu, y.w, srcl);
        const uint4 o = hi ? make_uint4(b0, b1, b2, b3) : make_uint4(a0, a1, a2, a3);
        if (wc * 32 + srcl < units) reinterpret_cast<uint4 *>(values)[2 * (wc * 32) + 32 * k + lane] = o;
    }
}

// A warp unpacks chunks of 32 consecutive 4-octet quads (384 packed bytes ->
// 1 KB of values), lane l quad l; two chunks per pass, both loads issued
// before either is unpacked, so that each warp keeps two reads in flight.
__global__ void __launch_bounds__(kThreads) unpack3_kernel(const uint8_t *__restrict__ packed,
                                                           uint8_t *__restrict__ values, int64_t n)
{
    const int64_t n4 = n / 4;
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (n4 + 31) / 32;
    const int64_t wstep = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wc = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; wc < chunks; wc += 2 * wstep) {
        const int64_t wc2 = wc + wstep;
        uint4 x0, y0, x1, y1;
        unpack_quad(packed, wc * 32 + lane, n4, x0, y0);
        unpack_quad(packed, wc2 * 32 + lane, n4, x1, y1);
        store_chunk(values, wc, n4, lane, x0, y0);
        if (wc2 < chunks) store_chunk(values, wc2, n4, lane, x1, y1);
    }
    const int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (t < n - 4 * n4) {
        const int64_t o = 4 * n4 + t;
        const uint32_t w = uint32_t(packed[3 * o]) | uint32_t(packed[3 * o + 1]) << 8 |
                           uint32_t(packed[3 * o + 2]) << 16;
        uint32_t lo, hi;
        unpack_octet(w, lo, hi);
        for (int j = 0; j < 4; ++j) {
            values[8 * o + j] = uint8_t(lo >> (8 * j));
            values[8 * o + 4 + j] = uint8_t(hi >> (8 * j));
        }
    }
}

// 96-bit group g as 32 value bytes, lane i = bits 3i..3i+2 of the group
// (zeros past the end).
__device__ __forceinline__ void unpack_group(const uint32_t *__restrict__ words, int64_t g, int64_t m, uint4 &x,
                                             uint4 &y)
{
    x = make_uint4(0, 0, 0, 0);
    y = make_uint4(0, 0, 0, 0);
    if (g < m) unpack96(__ldg(words + 3 * g), __ldg(words + 3 * g + 1), __ldg(words + 3 * g + 2), x, y);
}

// One 96-bit group per lane, chunks of 32 consecutive groups (a kilobyte of
// values) per warp, two chunks per pass as in unpack3_kernel.
__global__ void __launch_bounds__(kThreads) unpack3_words_kernel(
    const uint32_t *__restrict__ words, uint8_t *__restrict__ values, int64_t m)
{
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (m + 31) / 32;
    const int64_t wstep = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wc = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; wc < chunks; wc += 2 * wstep) {
        const int64_t wc2 = wc + wstep;
        uint4 x0, y0, x1, y1;
        unpack_group(words, wc * 32 + lane, m, x0, y0);
        unpack_group(words, wc2 * 32 + lane, m, x1, y1);
        store_chunk(values, wc, m, lane, x0, y0);
        if (wc2 < chunks) store_chunk(values, wc2, m, lane, x1, y1);
    }
}

// Streaming copy: each thread moves 4 x 16 bytes per iteration with all
// loads issued before the stores.
__global__ void __launch_bounds__(kThreads) copy_kernel(const uint4 *__restrict__ src,
                                                        uint4 *__restrict__ dst, int64_t n16)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// blocks for `work` threads of kernel K, at most one resident wave
template <auto K>
int grid_for(int64_t work)
{
    const int64_t blocks = (work + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(sm_count_current_device()) * resident_blocks<K>();
    return int(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_pack3(const uint8_t *values, uint8_t *packed, int64_t n, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    pack3_kernel<<<grid_for<pack3_kernel>(n / 4 + 4), kThreads, 0, s>>>(values, packed, n);
    return cudaGetLastError();
}

cudaError_t launch_unpack3(const uint8_t *packed, uint8_t *values, int64_t n, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    unpack3_kernel<<<grid_for<unpack3_kernel>(n / 4 + 4), kThreads, 0, s>>>(packed, values, n);
    return cudaGetLastError();
}

cudaError_t launch_unpack3_words(const uint32_t *words, uint8_t *values, int64_t m,
                                 cudaStream_t s)
{
    if (m == 0) return cudaSuccess;
    unpack3_words_kernel<<<grid_for<unpack3_words_kernel>(m), kThreads, 0, s>>>(words, values, m);
    return cudaGetLastError();
}

cudaError_t launch_copy_peak(const void *src, void *dst, size_t bytes, cudaStream_t s)
{
    const int64_t n16 = int64_t(bytes / 16);
    if (n16 == 0) return cudaSuccess;
    const int blocks = sm_count_current_device() * resident_blocks<copy_kernel>();
    copy_kernel<<<blocks, kThreads, 0, s>>>(reinterpret_cast<const uint4 *>(src),
                                            reinterpret_cast<uint4 *>(dst), n16);
    return cudaGetLastError();
}

}  // namespace pkv
