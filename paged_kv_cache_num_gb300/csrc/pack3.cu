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
// the unpacking kernels exchange halves between lanes so that each store
// instruction of a warp is one contiguous 512-byte run.  The kernels are
// pure HBM streams.
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;

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

__device__ __forceinline__ void unpack_octet(uint32_t w24, uint32_t &lo4, uint32_t &hi4)
{
    lo4 = 0;
    hi4 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lo4 |= ((w24 >> (3 * i)) & 7u) << (8 * i);
        hi4 |= ((w24 >> (3 * (i + 4))) & 7u) << (8 * i);
    }
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

// A warp unpacks 32 consecutive 4-octet quads (384 packed bytes -> 1 KB of
// values): lane l unpacks quad l, then the two store instructions write
// 16-byte units l and 32 + l of the warp's kilobyte, the halves moved
// between lanes by shuffles, so that every store instruction is one
// contiguous 512-byte run.
__global__ void __launch_bounds__(kThreads) unpack3_kernel(const uint8_t *__restrict__ packed,
                                                           uint8_t *__restrict__ values, int64_t n)
{
    const int64_t n4 = n / 4;
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (n4 + 31) / 32;
    const int64_t wstep = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wc = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; wc < chunks; wc += wstep) {
        const int64_t i = wc * 32 + lane;
        uint4 x = make_uint4(0, 0, 0, 0), y = make_uint4(0, 0, 0, 0);
        if (i < n4) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(packed + 12 * i);
            const uint32_t a = __ldg(src), b = __ldg(src + 1), c = __ldg(src + 2);
            const uint32_t w0 = a & 0xffffffu;
            const uint32_t w1 = (a >> 24) | ((b & 0xffffu) << 8);
            const uint32_t w2 = (b >> 16) | ((c & 0xffu) << 16);
            const uint32_t w3 = c >> 8;
            unpack_octet(w0, x.x, x.y);
            unpack_octet(w1, x.z, x.w);
            unpack_octet(w2, y.x, y.y);
            unpack_octet(w3, y.z, y.w);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            // unit 32k + lane = half (lane & 1) of quad 16k + (lane >> 1)
            const int srcl = 16 * k + (lane >> 1);
            // every lane takes part in both shuffles, then keeps its half
            const bool hi = lane & 1;
            const uint32_t a0 = __shfl_sync(0xffffffffu, x.x, srcl), b0 = __shfl_sync(0xffffffffu, y.x, srcl);
            const uint32_t a1 = __shfl_sync(0xffffffffu, x.y, srcl), b1 = __shfl_sync(0xffffffffu, y.y, srcl);
            const uint32_t a2 = __shfl_sync(0xffffffffu, x.z, srcl), b2 = __shfl_sync(0xffffffffu, y.z, srcl);
            const uint32_t a3 = __shfl_sync(0xffffffffu, x.w, srcl), b3 = __shfl_sync(0xffffffffu, y.w, srcl);
            const uint4 o = hi ? make_uint4(b0, b1, b2, b3) : make_uint4(a0, a1, a2, a3);
            const int64_t q = wc * 32 + srcl;
            if (q < n4) reinterpret_cast<uint4 *>(values)[2 * (wc * 32) + 32 * k + lane] = o;
        }
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

// One 96-bit group per lane: lane i = (W[w] >> s | W[w+1] << (32-s)) & 7
// with w = 3i/32, s = 3i%32, the second term only for s > 29.  A warp takes
// 32 consecutive groups and writes their kilobyte of values with two
// contiguous store instructions (halves exchanged by shuffles, as in
// unpack3_kernel).
__global__ void __launch_bounds__(kThreads) unpack3_words_kernel(
    const uint32_t *__restrict__ words, uint8_t *__restrict__ values, int64_t m)
{
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (m + 31) / 32;
    const int64_t wstep = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wc = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; wc < chunks; wc += wstep) {
        const int64_t g = wc * 32 + lane;
        uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (g < m) {
            uint32_t W[3];
            W[0] = __ldg(words + 3 * g);
            W[1] = __ldg(words + 3 * g + 1);
            W[2] = __ldg(words + 3 * g + 2);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int w = (3 * i) >> 5, s = (3 * i) & 31;
                uint32_t v = W[w] >> s;
                if (s > 29) v |= W[w + 1] << (32 - s);   // compile-time lanes 10, 21
                v &= 7u;
                if ((i & 3) == 0) out[i >> 2] = v; else out[i >> 2] |= v << (8 * (i & 3));
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            // unit 32k + lane = half (lane & 1) of group 16k + (lane >> 1)
            const int srcl = 16 * k + (lane >> 1);
            const bool hi = lane & 1;
            uint32_t a[4], b[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // every lane takes part in both shuffles
                a[j] = __shfl_sync(0xffffffffu, out[j], srcl);
                b[j] = __shfl_sync(0xffffffffu, out[4 + j], srcl);
            }
            const uint4 o = hi ? make_uint4(b[0], b[1], b[2], b[3]) : make_uint4(a[0], a[1], a[2], a[3]);
            if (wc * 32 + srcl < m) reinterpret_cast<uint4 *>(values)[2 * (wc * 32) + 32 * k + lane] = o;
        }
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

int grid_for(int64_t work)
{
    const int64_t blocks = (work + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(sm_count_current_device()) * 8;
    return int(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_pack3(const uint8_t *values, uint8_t *packed, int64_t n, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    pack3_kernel<<<grid_for(n / 4 + 4), kThreads, 0, s>>>(values, packed, n);
    return cudaGetLastError();
}

cudaError_t launch_unpack3(const uint8_t *packed, uint8_t *values, int64_t n, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    unpack3_kernel<<<grid_for(n / 4 + 4), kThreads, 0, s>>>(packed, values, n);
    return cudaGetLastError();
}

cudaError_t launch_unpack3_words(const uint32_t *words, uint8_t *values, int64_t m,
                                 cudaStream_t s)
{
    if (m == 0) return cudaSuccess;
    unpack3_words_kernel<<<grid_for(m), kThreads, 0, s>>>(words, values, m);
    return cudaGetLastError();
}

cudaError_t launch_copy_peak(const void *src, void *dst, size_t bytes, cudaStream_t s)
{
    const int64_t n16 = int64_t(bytes / 16);
    if (n16 == 0) return cudaSuccess;
    const int blocks = sm_count_current_device() * 8;
    copy_kernel<<<blocks, kThreads, 0, s>>>(reinterpret_cast<const uint4 *>(src),
                                            reinterpret_cast<uint4 *>(dst), n16);
    return cudaGetLastError();
}

}  // namespace pkv
