// decode_tma_xv.cu -- the persistent paged-decode kernel instantiated for
// x-vectorised caches ([num_blocks][num_kv_heads][head_dim/x][block_size][x],
// x = 16 bytes / element size): 16-bit and one-byte codes (one-byte with
// per-kv-head scales), head_dim 64 / 128, block sizes 16, 32 and 64.
#include "decode_tma_kernel.cuh"

namespace pkv {
namespace {

template <int CK, int D>
cudaError_t launch_xv_bs(const DecodeParams &p, const FastParams &f, const CUtensorMap &mk,
                         const CUtensorMap &mv, cudaStream_t s)
{
    switch (p.block_size) {
    case 16:
        return f.ng == 2 ? launch_fast_t<CK, D, 16, 0, false, true, 2>(p, f, mk, mv, s)
                         : launch_fast_t<CK, D, 16, 0, false, true>(p, f, mk, mv, s);
    case 32:
        return f.ng == 2 ? launch_fast_t<CK, D, 32, 0, false, true, 2>(p, f, mk, mv, s)
                         : launch_fast_t<CK, D, 32, 0, false, true>(p, f, mk, mv, s);
    case 64: return launch_fast_t<CK, D, 64, 0, false, true>(p, f, mk, mv, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_fast_xv(const DecodeParams &p, const FastParams &f, int cache_kind, const void *tmk,
                                  const void *tmv, cudaStream_t s)
{
    const CUtensorMap &mk = *static_cast<const CUtensorMap *>(tmk);
    const CUtensorMap &mv = *static_cast<const CUtensorMap *>(tmv);
    if (p.scale_mode != 0) return cudaErrorInvalidValue;
    switch (cache_kind) {
    case kE4M3:
        return p.head_dim == 128 ? launch_xv_bs<kE4M3, 128>(p, f, mk, mv, s) : launch_xv_bs<kE4M3, 64>(p, f, mk, mv, s);
    case kE5M2:
        return p.head_dim == 128 ? launch_xv_bs<kE5M2, 128>(p, f, mk, mv, s) : launch_xv_bs<kE5M2, 64>(p, f, mk, mv, s);
    case kI8:
        return p.head_dim == 128 ? launch_xv_bs<kI8, 128>(p, f, mk, mv, s) : launch_xv_bs<kI8, 64>(p, f, mk, mv, s);
    case kBF16:
        return p.head_dim == 128 ? launch_xv_bs<kBF16, 128>(p, f, mk, mv, s) : launch_xv_bs<kBF16, 64>(p, f, mk, mv, s);
    case kF16:
        return p.head_dim == 128 ? launch_xv_bs<kF16, 128>(p, f, mk, mv, s) : launch_xv_bs<kF16, 64>(p, f, mk, mv, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
