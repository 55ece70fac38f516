/*
 * pkv.h -- C ABI of the paged KV-cache kernels for NVIDIA GB300 (sm_103a).
 *
 * Three operations make up the path:
 *   - kv_append: scatter new K/V rows into a paged block pool through a
 *     slot_mapping, optionally quantising them to fp8 e4m3 (per-kv-head
 *     fp32 scales) or to 3-bit affine codes packed 8 values per 3 bytes;
 *   - paged_decode: one-query-token attention over that pool, indirected by
 *     block tables, with grouped-query heads, online softmax, a split over
 *     the context merged by log-sum-exp rescaling, and the fp8 / int8 /
 *     3-bit dequantisation done in registers;
 *   - pack3 / unpack3: the bit-exact 3-bit packing on its own.
 *
 * Conventions shared by every call
 *   - All data pointers are DEVICE pointers unless a call says otherwise.
 *     The caller owns every buffer (inputs, outputs, caches, metadata,
 *     workspace); the library never allocates device memory and never
 *     synchronises the stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; results are visible to later
 *     work on the same stream.  Ordering against other streams is the
 *     caller's job.
 *   - Return value: PKV_OK (0) or a negative PKV_ERR_* code.  On an error
 *     nothing is launched, and pkv_last_error() (per host thread) holds a
 *     one-line message.
 *   - `err_flag` (optional, may be NULL): a device int32 into which kernels
 *     atomically OR PKV_DEVERR_* bits when they meet data they cannot use
 *     (an out-of-range slot or block id, ...).  The offending access is
 *     skipped; kernels never trap.  The caller zeroes and reads it.
 *   - Shapes and strides are given with pkv_tensor; strides count elements
 *     of the tensor's dtype (bytes for the 8-bit and packed dtypes).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 3

/* Element types. */
enum {
    PKV_DTYPE_F16 = 1,  /* IEEE binary16 */
    PKV_DTYPE_BF16 = 2, /* bfloat16 */
    PKV_DTYPE_E4M3 = 3, /* OCP fp8 e4m3 ("fn": max 448, no inf) */
    PKV_DTYPE_U3 = 4,   /* 3-bit codes packed 8 per 3 bytes (see kv_append) */
    PKV_DTYPE_U8 = 5,
    PKV_DTYPE_I32 = 6,
    PKV_DTYPE_I64 = 7,
    PKV_DTYPE_F32 = 8,
    PKV_DTYPE_E5M2 = 9, /* OCP fp8 e5m2 (max 57344, with inf / NaN codes) */
    PKV_DTYPE_I8 = 10   /* int8 codes (scaled, symmetric range +-127) */
};

/* Host-side status codes. */
enum {
    PKV_OK = 0,
    PKV_ERR_NULL = -1,        /* a required pointer is NULL */
    PKV_ERR_DTYPE = -2,       /* unsupported or mismatched dtype */
    PKV_ERR_SHAPE = -3,       /* shapes disagree with each other */
    PKV_ERR_LAYOUT = -4,      /* stride / alignment requirement not met */
    PKV_ERR_UNSUPPORTED = -5, /* head_dim, block_size or group size not built */
    PKV_ERR_WORKSPACE = -6,   /* workspace missing or too small */
    PKV_ERR_VALUE = -7,       /* an argument value is out of its range */
    PKV_ERR_CUDA = -8         /* a CUDA runtime call or launch failed */
};

/* Device-side error bits OR-ed into *err_flag. */
enum {
    PKV_DEVERR_SLOT_RANGE = 1,    /* append: slot >= num_blocks * block_size */
    PKV_DEVERR_BLOCK_RANGE = 2,   /* decode: block id outside [0, num_blocks) */
    PKV_DEVERR_CONTEXT_RANGE = 4, /* decode: context_len < 0 or > table capacity */
    PKV_DEVERR_POS_RANGE = 8,     /* slot_mapping: position outside the table */
    PKV_DEVERR_TIMEOUT = 16       /* a bounded in-kernel wait gave up */
};

/* A strided view of device memory (up to 4 dimensions). */
typedef struct pkv_tensor {
    void *data;
    int32_t dtype;     /* PKV_DTYPE_* */
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4]; /* in elements of dtype (bytes for U8/E4M3/U3) */
} pkv_tensor;

/*
 * A paged KV cache ("Write Triton Kv Cache Append Kernel", "Inputs the agent
 * should gather first" item 1, vLLM v1 flash layout; "10. Triton KV Cache
 * and PagedAttention", Step 1):
 *
 *   k_cache, v_cache : [num_blocks, block_size, num_kv_heads, row]
 *       F16 / BF16 / E4M3 / E5M2 / I8 : row = head_dim elements;
 *       U3                : row = 3 * head_dim / 8 bytes; element d of a
 *                           head row is bits 3d..3d+2 of the row read as one
 *                           little-endian bit string, i.e. octet j holds
 *                           elements 8j..8j+7 in the layout of the
 *                           "triton-3bit-kv-cache-kernel" README, section 1.A.
 *     The last dimension must be contiguous (stride 1) and the base 16-byte
 *     aligned; the block stride must be a multiple of 16 bytes, and for
 *     F16/BF16/E4M3 also the slot and head strides.  K and V must have the
 *     same dtype, shape and strides.
 *   k_scale, v_scale : E4M3, E5M2 and I8 with scale_mode PER_HEAD, device
 *     fp32 [num_kv_heads], > 0.  A stored code c means fp8(c) * scale, or
 *     c * scale for I8, with the scale of the row's granularity (see
 *     PKV_SCALE_*).
 *   k_qscale, v_qscale (F16) and k_qzero, v_qzero (U8), U3 only:
 *     [num_blocks, block_size, num_kv_heads]; a stored code u means
 *     (u - zero) * scale for its (slot, head) row.  Any strides are
 *     accepted (the two scale arrays alike, the two zero arrays alike).
 *     Decode reads them fastest head-major (slot stride 1, head stride
 *     block_size: a [num_blocks, num_kv_heads, block_size] array seen through
 *     a transposed view), where each CTA stages only its own heads' runs;
 *     slot-major (head stride 1, slot stride num_kv_heads) also takes the
 *     persistent kernel; other layouts take the general one.
 */
/* Scale granularity of E4M3 / E5M2 / I8 caches ("Write Triton Kv Cache
 * Append Kernel", inputs items 4 and 8: per tensor, per token, per head or
 * per block; a per-tensor scale is a per-head scale equal for every head). */
enum {
    PKV_SCALE_PER_HEAD = 0,  /* k_scale / v_scale: fp32 [num_kv_heads] */
    PKV_SCALE_PER_BLOCK = 1, /* k_scales / v_scales: F32 [num_blocks, num_kv_heads] */
    PKV_SCALE_PER_TOKEN = 2  /* k_scales / v_scales: F32 [num_blocks, block_size,
                                num_kv_heads], one per cached row; written by
                                pkv_kv_append_scaled from the new tokens' scales */
};

typedef struct pkv_cache {
    pkv_tensor k_cache;
    pkv_tensor v_cache;
    const float *k_scale;
    const float *v_scale;
    pkv_tensor k_qscale;
    pkv_tensor k_qzero;
    pkv_tensor v_qscale;
    pkv_tensor v_qzero;
    /* ABI 2: scale granularity of E4M3 / E5M2 / I8 caches (PKV_SCALE_*; 0 =
     * per head, the ABI-1 behaviour) and the per-block / per-token scale
     * arrays (any strides, the same for K and V; positive values). */
    int32_t scale_mode;
    pkv_tensor k_scales;
    pkv_tensor v_scales;
    /* ABI 3: F16 / BF16 / E4M3 / E5M2 / I8 only -- stride, in elements,
     * between consecutive pieces of x elements of a head row, x = 16 bytes /
     * element size (8 for 16-bit, 16 for one-byte codes); 0 means x (the
     * row is contiguous).  A non-zero value selects the x-vectorised layout
     * of older vLLM ("Write Triton Kv Cache Append Kernel", "Inputs the
     * agent should gather first" item 1):
     *   storage [num_blocks, num_kv_heads, head_dim / x, block_size, x],
     * described by k_cache / v_cache as [num_blocks, block_size,
     * num_kv_heads, head_dim] with strides [Hkv*D*BS, x, D*BS, 1] and
     * chunk_stride = block_size * x (element (b, s, h, d) at
     * b*stride0 + s*stride1 + h*stride2 + (d/x)*chunk_stride + d%x).
     * head_dim must be a multiple of x and chunk_stride a multiple of 16
     * bytes.  Both caches use it. */
    int64_t chunk_stride;
} pkv_cache;

/* Library version string and ABI version. */
const char *pkv_version(void);
int pkv_abi_version(void);

/* Message for the last non-OK status returned on this host thread. */
const char *pkv_last_error(void);

/*
 * pkv_slot_mapping -- the launcher's slot computation, on the device
 * ("Write Triton Kv Cache Append Kernel", reasoning step 9 and "Common
 * failure modes": the new token's slot comes from its position through the
 * block table).
 *
 *   block_tables : I32 [batch, max_blocks_per_seq] (any strides)
 *   req, pos     : I32 [n]: request index and position of each new token;
 *                  pos < 0 marks a padding token.
 *   slot_mapping : I64 [n] output, contiguous:
 *                  slot = block_tables[req][pos / block_size] * block_size
 *                         + pos % block_size, or -1 for padding.
 *   A position at or beyond max_blocks_per_seq * block_size, or a request
 *   index outside [0, batch), yields -1 and PKV_DEVERR_POS_RANGE.
 *   Note: a decode step's new token sits at position context_len - 1 when
 *   context_lens counts the tokens attended including the new one (the
 *   convention of pkv_paged_decode), which is the same slot as position
 *   context_len taken before the increment.
 */
int pkv_slot_mapping(const pkv_tensor *block_tables, const pkv_tensor *req,
                     const pkv_tensor *pos, int block_size, const pkv_tensor *slot_mapping,
                     int32_t *err_flag, void *stream);

/*
 * pkv_kv_append -- scatter new K/V rows into the cache ("Write Triton Kv
 * Cache Append Kernel", reasoning steps 1-8 and "Kernel design rules").
 *
 *   k_new, v_new : F16 or BF16 [num_tokens, num_kv_heads, head_dim]; any
 *                  token and head strides, head_dim contiguous.
 *   slot_mapping : I64 [num_tokens]; slot = block_id * block_size +
 *                  slot_in_block.  slot < 0 is a no-op token (CUDA-graph
 *                  padding): its rows are neither read nor written.
 *   cache        : see pkv_cache.  The cache dtype selects the store:
 *     F16/BF16 : bit copy; the cache dtype must equal the source dtype.
 *     E4M3     : code = e4m3_rn_satfinite(x / scale[h]) with x / scale taken
 *                in fp32 before the cast (design rules: scale before the
 *                cast); finite overflow and infinities saturate to +-448,
 *                NaN stores 0x7F.
 *     E5M2     : the same with e5m2_rn_satfinite (overflow and infinities
 *                to +-57344, NaN stores 0x7F).
 *     I8       : code = clamp(rint(x / scale), -127, 127), x / scale in fp32,
 *                rint rounding half to even; NaN stores 0.
 *     U3       : per (token, head) row, all in fp32 with IEEE rounding:
 *                s = fp16_rn((max - min) / 7) (65504 if that overflows),
 *                z = clamp(rint(-min / s), 0, 7),
 *                q_d = clamp(rint(x_d / s) + z, 0, 7), packed along head_dim;
 *                s == 0 stores z = 0 and all q = 0.  head_dim % 8 == 0.
 *                Rows must be finite.
 *   block_size may be any positive number here (decode needs a power of two
 *   <= 256): a contiguous per-request cache [batch, num_kv_heads,
 *   max_seq_len, D] ("Write Triton Kv Cache Append Kernel", inputs item 1,
 *   the contiguous layout with slot = req * max_seq_len + pos) is passed as
 *   the view [batch, max_seq_len, num_kv_heads, D] with strides
 *   (num_kv_heads * max_seq_len * D, D, max_seq_len * D, 1), i.e. one block
 *   of max_seq_len slots per request.
 *   The grid depends only on num_tokens and num_kv_heads (graph safe).  A
 *   slot >= num_blocks * block_size is skipped and raises
 *   PKV_DEVERR_SLOT_RANGE.  Two tokens with the same slot race (undefined
 *   which one lands) unless their rows are equal.
 */
int pkv_kv_append(const pkv_tensor *k_new, const pkv_tensor *v_new,
                  const pkv_tensor *slot_mapping, const pkv_cache *cache, int32_t *err_flag,
                  void *stream);

/*
 * pkv_kv_append_scaled -- pkv_kv_append for caches with per-token scales
 * (scale_mode PKV_SCALE_PER_TOKEN; "load the appropriate scalar first",
 * reasoning step 6): each new row is divided by its own scale, and the
 * scale is stored at the token's slot in cache->k_scales / v_scales for
 * decode.
 *   k_new_scale, v_new_scale : F32 [num_tokens, num_kv_heads], > 0, any
 *                              strides; rows of padding tokens are not read.
 * Everything else as pkv_kv_append (which rejects per-token caches).
 */
int pkv_kv_append_scaled(const pkv_tensor *k_new, const pkv_tensor *v_new,
                         const pkv_tensor *k_new_scale, const pkv_tensor *v_new_scale,
                         const pkv_tensor *slot_mapping, const pkv_cache *cache, int32_t *err_flag,
                         void *stream);

/*
 * pkv_paged_decode -- paged attention for one query token per sequence
 * ("10. Triton KV Cache and PagedAttention", Steps 1 and 3 and the
 * reference code TODO 1-5), extended with grouped-query heads ("Write Triton
 * Kv Cache Append Kernel", design rules: replication happens in the
 * attention kernel by index arithmetic) and a split of each context into
 * chunks whose partial (max, sum, accumulator) triples a second kernel
 * merges by log-sum-exp rescaling (pkv_paged_decode_launches tells how
 * many kernels a call launches).
 *
 *   q            : F16 or BF16 [batch, num_heads, head_dim], head_dim
 *                  contiguous, 16-byte aligned rows.
 *   cache        : see pkv_cache; for F16/BF16 caches the dtype equals q's.
 *   block_tables : I32 [batch, max_blocks_per_seq]; entry j of row b is the
 *                  physical block of logical block j.  Entries at or beyond
 *                  ceil(context_len / block_size) are never read.
 *   context_lens : I32 [batch]: tokens to attend for each sequence, the
 *                  newest (just appended) token included.  0 gives an
 *                  all-zero output row.
 *   sm_scale     : softmax scale, usually 1 / sqrt(head_dim).
 *   out          : [batch, num_heads, head_dim], same dtype as q, head_dim
 *                  contiguous.
 *   num_splits   : context chunks per sequence; 0 = chosen by the library
 *                  from the shapes and the SM count (no device data read).
 *   workspace    : device scratch of at least the size returned by
 *                  pkv_paged_decode_workspace for the same arguments (may be
 *                  NULL when that size is 0); its contents need no
 *                  initialisation and are dead after the call's kernels.
 *                  Calls whose kernels may overlap must not share one.
 *
 *   Grouped-query mapping: q head h reads kv head h / (num_heads /
 *   num_kv_heads).  Output = softmax(sm_scale * q . K^T) V over the first
 *   context_len tokens, with the dequantised K/V for E4M3 and U3 caches,
 *   accumulated in fp32 and rounded once to the output dtype.  Cache
 *   contents beyond context_len (the tail of the last block) never affect
 *   the output, whatever they hold.
 *   Supported: head_dim in {64, 128}, block_size in {8, 16, 32, 64},
 *   num_heads % num_kv_heads == 0 with a group of at most 16 q heads.
 *   Bad table data never faults: a block id outside [0, num_blocks) is
 *   skipped (its tokens are left out) and raises PKV_DEVERR_BLOCK_RANGE; a
 *   context length below 0 is taken as 0 and one above the table's capacity
 *   (max_blocks_per_seq * block_size) as that capacity, raising
 *   PKV_DEVERR_CONTEXT_RANGE.  The affected rows are then not meaningful.
 */
int pkv_paged_decode_workspace(const pkv_tensor *q, const pkv_cache *cache,
                               const pkv_tensor *block_tables, int num_splits, size_t *bytes);

/* Kernel launches a pkv_paged_decode call with these arguments makes (1 or
 * 2), written to *launches; validation as pkv_paged_decode_workspace. */
int pkv_paged_decode_launches(const pkv_tensor *q, const pkv_cache *cache,
                              const pkv_tensor *block_tables, int num_splits, int32_t *launches);

int pkv_paged_decode(const pkv_tensor *q, const pkv_cache *cache, const pkv_tensor *block_tables,
                     const pkv_tensor *context_lens, float sm_scale, const pkv_tensor *out,
                     int num_splits, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                     void *stream);

/*
 * pkv_decode_step -- one decode step of a serving loop in one call:
 * pkv_slot_mapping of the step's tokens (block size from the cache), then
 * pkv_kv_append of their K/V rows through that mapping, then
 * pkv_paged_decode over every sequence ("Write Triton Kv Cache Append
 * Kernel", reasoning step 9, followed by the decode of "10. Triton KV Cache
 * and PagedAttention").  The arguments are those of the three calls, with
 * the same meaning, layouts and rules; slot_mapping (I64 [num_tokens],
 * caller-owned) receives the computed slots.  Every argument of all three
 * is validated before the first launch, so an error status means nothing
 * was enqueued.  The slot computation runs inside the append kernel (same
 * rule and error bits as pkv_slot_mapping; the slots are still written to
 * slot_mapping), then the decode kernels follow on `stream` as programmatic
 * dependents.  An addition of this library: it saves two host-side calls
 * and one kernel launch per step.
 */
int pkv_decode_step(const pkv_tensor *k_new, const pkv_tensor *v_new, const pkv_tensor *req,
                    const pkv_tensor *pos, const pkv_tensor *slot_mapping, const pkv_tensor *q,
                    const pkv_cache *cache, const pkv_tensor *block_tables, const pkv_tensor *context_lens,
                    float sm_scale, const pkv_tensor *out, int num_splits, void *workspace,
                    size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * pkv_paged_decode_noalloc -- pkv_paged_decode for callers that cannot
 * allocate device memory at call time: plugin or custom-op hooks of
 * inference engines that may not allocate while enqueueing, runtimes whose
 * device memory all belongs to their own pool allocator, and serving loops
 * that cannot afford the device-wide synchronisation of cudaMalloc.  The
 * pages have no counterpart; it is an addition of this library.
 *
 * Same arguments and result as pkv_paged_decode without the workspace: the
 * split-K scratch is a fixed array inside the library
 * (pkv_noalloc_scratch_bytes(), 8 MiB), reserved on a GPU when the CUDA
 * runtime loads the library's device code there (with lazy module loading,
 * the CUDA default, at the first use of the library on that GPU -- at the
 * latest, the first call of this function) and held until the process
 * exits.  The call itself allocates nothing and calls nothing that does.
 *   - num_splits 0: the automatic plan when its scratch fits the array,
 *     else the largest explicit split count (16 down to 1) that fits; one
 *     split needs no scratch, so num_splits 0 always finds a plan.
 *   - An explicit num_splits whose scratch need (pkv_paged_decode_workspace)
 *     exceeds the array is rejected with PKV_ERR_WORKSPACE before any
 *     launch.  num_splits 1 needs no scratch.
 *   - The first call on a device looks the array's device address up with
 *     cudaGetSymbolAddress (once per device, with that device current);
 *     make that first call before any stream capture.  The address is
 *     cached per device ordinal: only the device's primary context (the
 *     runtime API's) is supported, and not across a cudaDeviceReset.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose kernels overlap
 *     on the GPU (different streams, or concurrent host threads) race on
 *     it: serialise them, e.g. on one stream.
 */
size_t pkv_noalloc_scratch_bytes(void);

int pkv_paged_decode_noalloc(const pkv_tensor *q, const pkv_cache *cache,
                             const pkv_tensor *block_tables, const pkv_tensor *context_lens,
                             float sm_scale, const pkv_tensor *out, int num_splits,
                             int32_t *err_flag, void *stream);

/*
 * pkv_pack3 / pkv_unpack3 -- 8 x uint3 <-> 3 bytes per octet
 * ("triton-3bit-kv-cache-kernel" README, section 1.A, packing and
 * explicit unpacking formulas).
 *   values : U8 [n_octets * 8], contiguous, 16-byte aligned; only the low
 *            3 bits are used.
 *   packed : U8 [n_octets * 3], contiguous, 4-byte aligned.
 *   A misaligned pointer is rejected with PKV_ERR_LAYOUT.
 *   Bit exact: packing the lanes v_i of octet state n = sum v_i * 8^i gives
 *   the three little-endian bytes of n.
 */
int pkv_pack3(const uint8_t *values, uint8_t *packed, int64_t n_octets, void *stream);
int pkv_unpack3(const uint8_t *packed, uint8_t *values, int64_t n_octets, void *stream);

/*
 * pkv_unpack3_words -- 3 x uint32 -> 32 x uint3 per 96-bit group
 * ("triton-3bit-kv-cache-kernel" README, section 1.B: lane i at bit 3i,
 * word 3i/32, shift 3i%32; lanes 10 and 21 straddle words).
 *   words  : device uint32 [n_groups * 3], 4-byte aligned.  The same bytes
 *            as 4 packed octets read as little-endian words.
 *   values : U8 [n_groups * 32], 16-byte aligned.
 *   A misaligned pointer is rejected with PKV_ERR_LAYOUT.
 */
int pkv_unpack3_words(const uint32_t *words, uint8_t *values, int64_t n_groups, void *stream);

/*
 * pkv_copy_peak -- a 16-byte-vectorised device-to-device copy of `bytes`
 * bytes (a multiple of 16, both pointers 16-byte aligned), used to measure
 * the HBM bandwidth the decode kernels are compared against.
 */
int pkv_copy_peak(const void *src, void *dst, size_t bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
