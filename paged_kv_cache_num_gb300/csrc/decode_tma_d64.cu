// decode_tma_d64.cu -- the persistent paged-decode kernel instantiated for
// one-byte caches (e4m3, e5m2, int8) at head_dim 64: 64-byte rows staged
// with the 64-byte swizzle, block sizes 16, 32 and 64, per-kv-head and
// granular scales, groups of up to 16 q heads.  (A translation unit of its
// own, so that the build compiles it beside the head_dim 128 instances.)
#include "decode_tma_kernel.cuh"

namespace pkv {

cudaError_t launch_decode_fast_q8_d64(const DecodeParams &p, const FastParams &f, int cache_kind,
                                      const void *tmk, const void *tmv, cudaStream_t s)
{
    const CUtensorMap &mk = *static_cast<const CUtensorMap *>(tmk);
    const CUtensorMap &mv = *static_cast<const CUtensorMap *>(tmv);
    switch (cache_kind) {
    case kE4M3: return launch_fast_bs<kE4M3, 64>(p, f, mk, mv, s);
    case kE5M2: return launch_fast_bs<kE5M2, 64>(p, f, mk, mv, s);
    case kI8: return launch_fast_bs<kI8, 64>(p, f, mk, mv, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
