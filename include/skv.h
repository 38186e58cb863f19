/*
 * skv.h -- C ABI of the GB300 speculative-KV-coding library (libskv.so).
 *
 * What it computes.  Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍"
 * (Speculative KV coding, lpnh.cn/news/878951):
 *   - section "什么能预测 KV 缓存" (what can predict the KV cache): an
 *     arithmetic coder turns (KV_full, mu, sigma) into a bitstream on the
 *     encoding side and (bits, mu, sigma) back into KV_full on the decoding side;
 *   - section "q 应是什么样的" (what q should look like): each scalar is coded
 *     under a Gaussian centred on its prediction mu with calibrated sigma^2;
 *   - section "早期结果" (early results): bf16 caches use the mixture
 *     q = 0.95 N(mu, sigma^2) + 0.03 N(mu, (3 sigma)^2) + 0.02 p-hat_bf16,
 *     with sigma per (kv, head, channel) and p-hat the empirical bf16 symbol
 *     distribution measured on calibration data;
 *   - section "原生 FP8 KV 缓存" (native FP8 cache): e4m3 caches use the
 *     bin-integrated N(mu, sigma^2);
 *   - section "下一步计划" (next steps): both ends must derive bit-identical
 *     probabilities, so the model is evaluated in integer fixed point.
 *   - section "KV 缓存并非真正随机" (the cache is not random): the coded size
 *     is the cross-entropy -sum log2 q(x); skv_ideal_bits reports it.
 *
 * Format (spec v1; the pages fix no coder details).  Every symbol r (its rank
 * in value order) gets cum(r) = floor((2^M - |S|) F(lo(r))) + r, M = 28 for
 * bf16 (|S| = 65282 non-NaN patterns) and 16 for e4m3 (|S| = 254), where lo(r)
 * is the lower edge of the symbol's round-to-nearest bin and F the model CDF
 * built from an integer-interpolated Phi table and the integer p-hat prefix
 * table.  The coder is interleaved rANS with a 64-bit state, L = 2^31 and
 * 32-bit words.  A chunk is one (layer, kv, head, token block); scalar p of a
 * chunk belongs to lane (p / 8) mod G.  The container is a 64-byte header,
 * u64 offsets[num_chunks + 1] and the chunk payloads; see skv_encode.
 *
 * Conventions for every call below.
 *   - Pointers are DEVICE pointers unless marked "host": device memory, or
 *     pinned host memory mapped into the device's address space, which the
 *     kernels then read or write over the CPU-GPU link.  The caller owns every
 *     buffer; no call allocates memory.
 *   - Tensors are row-major [layers][2][heads][tokens][head_dim]: KV is bf16
 *     bit patterns (uint16) or e4m3 codes (uint8); mu is always bf16.
 *   - Work is issued on `stream` (a cudaStream_t; NULL = legacy default).
 *     Calls that return a status or a host value synchronize that stream.
 *   - Return value: SKV_OK (0) or a negative skv_status.  Kernel-side errors
 *     (bad symbols, parameters or streams) are gathered in a device flag in
 *     the workspace and reported at the end of the call; the library never
 *     traps the GPU.
 *   - The first call on a device uploads the model constants to that device
 *     (a synchronous copy), so make one call before any stream capture.  The
 *     library remembers per device that this was done (and, for
 *     skv_ideal_bits_noalloc, where its scratch array lives), so it must not
 *     be used across a cudaDeviceReset of a device it has already run on.
 *   - Calls on different streams must use different workspaces.
 */
#ifndef SKV_H
#define SKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *skv_stream_t; /* cudaStream_t */

typedef enum { SKV_BF16 = 0, SKV_E4M3 = 1 } skv_dtype;

typedef enum {
  SKV_OK = 0,
  SKV_ERR_ARG = -1,       /* bad shape, token block, lanes, or a NULL pointer */
  SKV_ERR_CAPACITY = -2,  /* output buffer or workspace too small */
  SKV_ERR_SYMBOL = -3,    /* a NaN bit pattern in the KV input */
  SKV_ERR_PARAM = -4,     /* invalid sigma (not finite, < FLT_MIN, 3 sigma overflows),
                             non-finite mu, or an ill-formed p-hat table */
  SKV_ERR_CORRUPT = -5,   /* bad header, offsets, model fingerprint, stream overrun,
                             or a lane that does not end in the initial state */
  SKV_ERR_CUDA = -6       /* a CUDA runtime error */
} skv_status;

typedef enum {
  SKV_OP_ENCODE = 0,
  SKV_OP_DECODE = 1,
  SKV_OP_IDEAL_BITS = 2,
  SKV_OP_MODEL_BITS = 3
} skv_op;

/* Tensor shape.  kv must be 2 (keys and values); head_dim a multiple of 8. */
typedef struct {
  int32_t layers, kv, heads, tokens, head_dim;
} skv_shape;

/* Coding model and chunking.
 *   dtype        SKV_BF16 or SKV_E4M3.
 *   token_block  tokens per chunk (Tb >= 1); chunk = Tb * head_dim scalars.
 *   lanes        rANS lanes per chunk, G in {1, 2, 4, 8, 16, 32}.
 *   flags        SKV_FLAG_* bits; 0 for the default behaviour.
 *   sigma        device, fp32 [layers][2][heads][head_dim]; per (layer, kv,
 *                head, channel) standard deviation of the narrow component.
 *   ecdf         device, bf16 only: u32 E_q[0..65282], E_q[r] =
 *                floor(2^26 S[r] / S_tot), S[r] = sum over ranks j < r of
 *                (count_j + 1); built by skv_build_ecdf.  Unused for e4m3.
 *   phat         device, bf16 only: fp32 p-hat[0..65281] by rank, the
 *                smoothed empirical probability (count + 1) / S_tot.  Read by
 *                skv_ideal_bits only; NULL is allowed for encode and decode.
 */
/* skv_params.flags bits (all others must be 0). */
#define SKV_FLAG_DECODE_BISECT 1 /* decode by plain bisection over ranks (reference
                                    search; the output is identical, only slower) */
/* Per-block sigma scales (the pages' section "下一步计划": the error scale moves
 * with prompt and position).  Every (chunk, 8-channel group) codes with
 * sigma_eff = fp32(sigma * m(s)), m(s) = fp32(2^((s - 128) / 32)), s one byte
 * chosen by the encoder: b + C, b the median over the group's residuals of
 * the bin (bits(|x - mu| / sigma) >> 18) - 127*32 + 128 clamped to [0, 255]
 * (0 for a zero or NaN residual, 255 for infinity), C = 18 (bf16) or 21
 * (e4m3); 128 if sigma_eff would be invalid for a channel of the group.  The
 * bytes travel in the container (header feature bit 0, ceil(head_dim / 32)
 * words at the start of each chunk).  Requires head_dim <= 2048.  Encode,
 * decode and ideal bits must all be given the flag; skv_ideal_bits_noalloc
 * rejects it (SKV_ERR_ARG). */
#define SKV_FLAG_BLOCK_SCALE 2
/* Order-0 baseline (the pages' introduction: an entropy coder over the bf16
 * symbols alone reaches about 11 bits per value): the same coder with q =
 * p-hat, i.e. cum(r) = floor(K * E_q[r] / 2^26) + r, without prediction.
 * bf16 only, not with SKV_FLAG_BLOCK_SCALE.  mu and sigma are not read and
 * may be NULL; sigma is not part of the model fingerprint; header feature
 * bit 1.  Ideal bits are -log2 p-hat.  skv_ideal_bits_noalloc rejects it. */
#define SKV_FLAG_ORDER0 4
/* Adaptive counts (the entropy-estimation page's virtual sliding window:
 * decayed counts C = 0.97 C + delta per token, smoothed updates P = 0.9 P +
 * 0.1 C / sum C): with SKV_FLAG_ORDER0, one model per (layer, kv, head) row,
 * updated after every chunk from the row's earlier token blocks, so the token
 * block is the update period.  Integer arithmetic throughout, the prior is
 * E_q.  The coder then runs one phase per token block (rows in parallel,
 * blocks of a row in order).  Requires head_dim <= 512 and token_block <=
 * 65536; header feature bit 2;
 * skv_decode_range and skv_ideal_bits_noalloc reject it (SKV_ERR_ARG). */
#define SKV_FLAG_ADAPTIVE 8

typedef struct {
  int32_t dtype;
  int32_t token_block;
  int32_t lanes;
  int32_t flags;    /* SKV_FLAG_* bits */
  const float *sigma;
  const uint32_t *ecdf;
  const float *phat;
} skv_params;

/* Upper bound on the container size in bytes for this shape (worst case:
 * every symbol costs one 32-bit word).  Returns 0 if the arguments are invalid. */
size_t skv_max_encoded_bytes(const skv_params *params, const skv_shape *shape);

/* Workspace bytes needed by `op` (an skv_op) for this shape; 0 if invalid.
 * The encoder's workspace holds one word stack per chunk (about M/8 bytes per
 * scalar), the chunk sizes and offsets, the per-channel reciprocals and the
 * error flags; decode and ideal-bits need only small tables.  The workspace
 * must be 256-byte aligned (cudaMalloc memory is). */
size_t skv_workspace_bytes(const skv_params *params, const skv_shape *shape, int op);

/* Encode a whole cache into one container.
 *   kv, mu        device inputs as above.
 *   out           device output, out_capacity bytes (skv_max_encoded_bytes is
 *                 always enough).
 *   out_bytes     host; receives the container size.
 * Container v1 (little-endian): a 64-byte header {u32 magic "SKV1", u16 version
 * 1, u8 dtype, u8 M, u32 layers, u32 2, u32 heads, u32 tokens, u32 head_dim,
 * u32 token_block, u16 lanes, u8 8, u8 9, u16 8, u16 features (bit 0:
 * SKV_FLAG_BLOCK_SCALE, bit 1: SKV_FLAG_ORDER0, bit 2: SKV_FLAG_ADAPTIVE), u64 num_chunks, u64 payload_bytes, u64 model
 * fingerprint of sigma (and E_q for bf16)}, then u64 offsets[num_chunks + 1]
 * (byte offsets from the payload start, multiples of 4), then the payload:
 * chunk c (index ((l*2 + kv)*heads + h)*ceil(tokens/Tb) + tb) is u32 words in
 * decoder order -- with per-block scales first ceil(head_dim / 32) words
 * holding the scale bytes (group g in word g / 4, byte g % 4, low byte first;
 * unused bytes 0), then the lane states (lo, hi) for lanes 0..G-1, then the
 * renormalisation words.  Errors: SKV_ERR_ARG, SKV_ERR_CAPACITY (out or
 * workspace too small; nothing useful is written), SKV_ERR_SYMBOL,
 * SKV_ERR_PARAM, SKV_ERR_CUDA.  Synchronizes `stream`. */
int skv_encode(const skv_params *params, const skv_shape *shape, const void *kv,
               const uint16_t *mu, void *out, size_t out_capacity, size_t *out_bytes,
               void *workspace, size_t workspace_bytes, skv_stream_t stream);

/* Decode a container produced by skv_encode with the same params, shape and mu.
 *   in, in_bytes  device container and its exact size.
 *   kv_out        device output tensor (2 or 1 bytes per scalar).
 * The header must match params and shape, and its model fingerprint must match
 * sigma (and E_q); every offset, every stream read and every lane's final
 * state are checked.  Errors: SKV_ERR_ARG, SKV_ERR_CAPACITY (workspace),
 * SKV_ERR_PARAM, SKV_ERR_CORRUPT (kv_out is then unspecified), SKV_ERR_CUDA.
 * Synchronizes `stream`. */
int skv_decode(const skv_params *params, const skv_shape *shape, const void *in,
               size_t in_bytes, const uint16_t *mu, void *kv_out, void *workspace,
               size_t workspace_bytes, skv_stream_t stream);

/* Decode part of a container, asynchronously, into a contiguous or a paged
 * layout: the decoder fused with its consumer (the pages' section "该方法的用途":
 * caches offloaded to host memory over a slow link are streamed back and
 * decoded where they are needed; section "下一步计划": the decoder must keep up
 * with the fast side).
 *   in, in_bytes    the whole container as skv_encode wrote it.  It may sit in
 *                   pinned host memory (the kernels then stream the payload
 *                   over the CPU-GPU link) or in device memory; only the
 *                   header, the offset table and the payload of the chunks
 *                   being decoded are read, so a caller may copy a device
 *                   buffer's chunk ranges in just before decoding them.
 *   chunk_begin, chunk_end   chunks [chunk_begin, chunk_end) in container order.
 *   mu, kv_out      device.  Without a page table: the [L][2][H][T][D] tensors
 *                   of skv_decode.  With page_of_chunk (device, u32 per chunk
 *                   of the container, num_pages > 0): page pools of num_pages
 *                   pages of token_block * head_dim scalars each, chunk c's
 *                   scalars in page page_of_chunk[c] in their contiguous order
 *                   (a short last token block fills the start of its page).
 *                   A page index >= num_pages is reported as SKV_ERR_ARG by
 *                   skv_decode_status and that chunk is not written.
 *   range_flags     SKV_RANGE_FIRST on the first call for a container: clears
 *                   the status, prepares the model tables in the workspace and
 *                   checks the header and the model fingerprint.  Later calls
 *                   for the same container reuse them and must be ordered
 *                   after it (same stream, or caller-made ordering).
 *                   SKV_RANGE_PARTIAL (with or without FIRST): the container is
 *                   still being written by skv_encode_commit, so FIRST skips
 *                   the header check; in_bytes is then the buffer's capacity
 *                   (every offset read is bounded by it) and only committed
 *                   chunks may be decoded, after their commit in stream order.
 *                   The header and model fingerprint are not checked in this
 *                   mode: it is for a container this process is writing.
 * Argument errors (SKV_ERR_ARG, SKV_ERR_CAPACITY, a container shorter than its
 * offset table: SKV_ERR_CORRUPT) return at once; data errors accumulate in the
 * workspace until skv_decode_status.  Does not synchronize. */
#define SKV_RANGE_FIRST 1
#define SKV_RANGE_PARTIAL 2
#define SKV_RANGE_BITS 4   /* skv_encode_range only: see there */
int skv_decode_range(const skv_params *params, const skv_shape *shape, const void *in,
                     size_t in_bytes, uint64_t chunk_begin, uint64_t chunk_end,
                     const uint16_t *mu, void *kv_out, const uint32_t *page_of_chunk,
                     uint64_t num_pages, int range_flags, void *workspace,
                     size_t workspace_bytes, skv_stream_t stream);

/* Status accumulated by skv_decode_range calls on this decode workspace since
 * the last SKV_RANGE_FIRST: SKV_OK, SKV_ERR_ARG (a page index), SKV_ERR_PARAM,
 * SKV_ERR_CORRUPT.  Synchronizes `stream`. */
int skv_decode_status(const void *workspace, skv_stream_t stream);

/* skv_encode and skv_ideal_bits in one call: the container (byte for byte the
 * one skv_encode writes) and the ideal code length of the cache -- the
 * per-scalar values and the total skv_ideal_bits gives, within its tolerance
 * (1e-3 relative + 1e-6 bits per scalar) -- so that a caller gets a coder's
 * cost and the cross-entropy it should reach side by side (the pages' section
 * "KV 缓存并非真正随机").  On bf16 mixture caches (with or without per-block
 * scales) the encoder computes the bits itself from the symbols, mu and
 * reciprocals in its registers, one read of the inputs for both; on e4m3 and
 * with SKV_FLAG_ORDER0 the ideal-bits pass runs behind the encoder on the
 * same stream.  The total
 * is summed in fp64 in a fixed order for a given device and shape.
 *   per_scalar    device fp32 [N] output, or NULL.
 *   total         host; receives the ideal bits.
 * Requires params->phat for bf16; workspace: skv_workspace_bytes(...,
 * SKV_OP_ENCODE).  Rejects SKV_FLAG_ADAPTIVE (SKV_ERR_ARG).  Other errors as
 * skv_encode.  Synchronizes. */
int skv_encode_with_bits(const skv_params *params, const skv_shape *shape, const void *kv,
                         const uint16_t *mu, void *out, size_t out_capacity, size_t *out_bytes,
                         float *per_scalar, double *total, void *workspace,
                         size_t workspace_bytes, skv_stream_t stream);

/* Whether skv_encode_with_bits computes the ideal bits inside the encoder
 * (*fused = 1: one kernel over the inputs) or runs the ideal-bits pass behind
 * it (*fused = 0) for this model and shape on the current device.  fused:
 * host.  Errors: SKV_ERR_ARG (NULL fused, bad params or shape,
 * SKV_FLAG_ADAPTIVE), SKV_ERR_CUDA (no device). */
int skv_encode_with_bits_fused(const skv_params *params, const skv_shape *shape, int *fused);

/* Encode part of a cache, asynchronously: chunks [chunk_begin, chunk_end) in
 * container order go into the workspace's per-chunk stacks, and a later
 * skv_encode_finish turns the stacks into the container.  A caller can so
 * start encoding the layers that have arrived while the rest of the cache is
 * still being copied in (the pages' section "该方法的用途": caches move between
 * tiers over links slower than HBM; section "下一步计划": coding must keep up with
 * the fast side).  The container is byte for byte the one skv_encode writes.
 *   kv, mu          device, the whole [L][2][H][T][D] tensors; only the range's
 *                   chunks are read, so the rest may still be in flight.
 *   range_flags     SKV_RANGE_FIRST on the first call for a container: clears
 *                   the status, the chunk count and the ideal-bits total and
 *                   prepares the model tables.  Later calls must be ordered
 *                   after it (same stream, or caller-made ordering) and use the
 *                   same workspace.
 *                   SKV_RANGE_BITS: the encoder also evaluates the ideal code
 *                   length of the range's scalars (the per-scalar values
 *                   skv_ideal_bits gives, within its tolerance) as it codes
 *                   them, and adds their sum to the
 *                   workspace's total, in call order; skv_encode_range_bits
 *                   reads it.  bf16 mixture model only, with or without
 *                   per-block scales (not e4m3, not SKV_FLAG_ORDER0:
 *                   SKV_ERR_ARG), with params->phat.  Calls with this flag share
 *                   the workspace's partial sums: order them one after the
 *                   other (same stream, or caller-made ordering).
 * Every chunk must be encoded exactly once before skv_encode_finish.  Rejects
 * SKV_FLAG_ADAPTIVE (its tables depend on a row's earlier blocks).  Argument
 * errors (SKV_ERR_ARG, SKV_ERR_CAPACITY) return at once; data errors
 * (SKV_ERR_SYMBOL, SKV_ERR_PARAM) are reported by skv_encode_finish.  Does not
 * synchronize. */
int skv_encode_range(const skv_params *params, const skv_shape *shape, const void *kv,
                     const uint16_t *mu, uint64_t chunk_begin, uint64_t chunk_end,
                     int range_flags, void *workspace, size_t workspace_bytes,
                     skv_stream_t stream);

/* Size scan, compaction and header after skv_encode_range calls have coded
 * every chunk once: writes the container to `out` (device) and its size to
 * *out_bytes (host).  Checks the number of chunks coded since SKV_RANGE_FIRST
 * before reading any stack: a different count is SKV_ERR_ARG and nothing is
 * written.  Other errors as skv_encode.  Synchronizes `stream`. */
int skv_encode_finish(const skv_params *params, const skv_shape *shape, void *out,
                      size_t out_capacity, size_t *out_bytes, void *workspace,
                      size_t workspace_bytes, skv_stream_t stream);

/* The ideal bits of the chunks encoded with SKV_RANGE_BITS since the last
 * SKV_RANGE_FIRST on this workspace (each range's fixed-order sum, added in
 * call order) into *total (host); 0 if none.  Reads the workspace's status
 * first: a data error of the ranges encoded so far (SKV_ERR_SYMBOL,
 * SKV_ERR_PARAM) is returned instead.  Synchronizes `stream`. */
int skv_encode_range_bits(const skv_params *params, const skv_shape *shape, double *total,
                          void *workspace, size_t workspace_bytes, skv_stream_t stream);

/* Place encoded chunks in the container while later ones are still being
 * encoded: chunks [chunk_begin, chunk_end), the next in container order after
 * those committed before (chunk_begin = 0 on the first call since
 * SKV_RANGE_FIRST, then the previous chunk_end), whose skv_encode_range calls
 * were enqueued before this one (same stream, or caller-made ordering), get
 * their offsets and payload in `out`, right after the committed prefix.  The
 * chunk after the range gets its offset too, so the range can be decoded
 * (skv_decode_range with SKV_RANGE_PARTIAL) or its bytes copied out before the
 * rest of the cache is encoded (the pages' section "该方法的用途": caches move
 * to a slower tier as they are produced).  skv_encode_finish then writes the
 * header; it requires every chunk committed, to the same `out`.
 *   out, out_capacity   device buffer of the container (8-byte aligned), at
 *                       least skv_max_encoded_bytes for a whole cache.
 *   end_bytes       optional (NULL: none): receives, when the commit runs (in
 *                   stream order), the container's size so far -- header,
 *                   offset table and the committed payload -- so that a caller
 *                   can copy the new bytes out without a synchronisation.
 *                   Device memory, or pinned host memory the device can write.
 * Argument errors return at once (SKV_ERR_ARG; SKV_ERR_CAPACITY for a buffer
 * without room for the offset table).  A range that does not start where the
 * committed prefix ends, or with a chunk not encoded since SKV_RANGE_FIRST, is
 * reported by skv_encode_finish as SKV_ERR_ARG, a container that outgrows
 * out_capacity as SKV_ERR_CAPACITY; such a range places nothing.  Does not
 * synchronize. */
int skv_encode_commit(const skv_params *params, const skv_shape *shape, uint64_t chunk_begin,
                      uint64_t chunk_end, void *out, size_t out_capacity, uint64_t *end_bytes,
                      void *workspace, size_t workspace_bytes, skv_stream_t stream);

/* The model fingerprint a container of this cache carries in its header (a
 * sum of SplitMix64 terms over sigma's and E_q's 32-bit words, so a decoder
 * with a different model refuses the container).  For skv_merge_parts.
 *   fingerprint   host; receives the value.
 *   workspace     any operation's workspace for this shape.
 * Errors: SKV_ERR_ARG, SKV_ERR_CAPACITY, SKV_ERR_PARAM (sigma or E_q
 * invalid), SKV_ERR_CUDA.  Synchronizes. */
int skv_model_fingerprint(const skv_params *params, const skv_shape *shape,
                          uint64_t *fingerprint, void *workspace, size_t workspace_bytes,
                          skv_stream_t stream);

/* One container from the containers of consecutive layer ranges of a cache,
 * host memory only (no GPU call): the multi-GPU path, where each GPU codes
 * its own contiguous layer range -- a contiguous chunk range, since chunks are
 * independent -- and one exclusive scan of the parts' payload sizes places
 * them.  parts[i] (host, part_bytes[i] bytes) must be a container written by
 * skv_encode (or skv_encode_finish) for layers [l_i, l_i + n_i) of the cache
 * described by params and shape, with sigma's rows of those layers, in layer
 * order and covering every layer.  The result, written to out (host,
 * out_capacity bytes; *out_bytes receives its size), is byte for byte the
 * container skv_encode writes for the whole cache, given the whole cache's
 * fingerprint (skv_model_fingerprint).  Errors: SKV_ERR_ARG (shape, count of
 * layers), SKV_ERR_CORRUPT (a part's header does not belong to this cache
 * or its offsets are malformed), SKV_ERR_CAPACITY. */
int skv_merge_parts(const skv_params *params, const skv_shape *shape, uint64_t fingerprint,
                    const void *const *parts, const size_t *part_bytes, int nparts, void *out,
                    size_t out_capacity, size_t *out_bytes);

/* Ideal code length: the cross-entropy -log2 q(x) of every scalar under the
 * continuous model (bin mass of the mixture, or of N(mu, sigma^2) for e4m3),
 * evaluated in tail-safe fp32 and summed in fp64 in a fixed order.  Every
 * per-scalar value is within 1e-3 relative + 1e-6 bits of the exact binary64
 * value; the total is the same on every call with the same inputs and grid.
 *   per_scalar    device fp32 [N] output, or NULL.
 *   total         host; receives the sum in bits.
 * Requires params->phat for bf16.  Errors: SKV_ERR_ARG, SKV_ERR_CAPACITY
 * (workspace), SKV_ERR_SYMBOL, SKV_ERR_PARAM, SKV_ERR_CUDA.  Synchronizes. */
int skv_ideal_bits(const skv_params *params, const skv_shape *shape, const void *kv,
                   const uint16_t *mu, float *per_scalar, double *total, void *workspace,
                   size_t workspace_bytes, skv_stream_t stream);

/* Model cost: the code length the coder's own integer frequencies give,
 * sum over scalars of M - log2(freq), freq = cum(r + 1) - cum(r) exactly as
 * skv_encode computes it (with per-block scales, under the scales the
 * encoder would choose).  This is what an ideal arithmetic coder with these
 * frequencies would write; the rANS payload of a chunk exceeds it by 32 to 64
 * bits per lane (initial state and flush), the container adds its header and
 * offsets.  It differs from skv_ideal_bits where the continuous model gives a
 * scalar less mass than the 1-in-2^M floor of the frequencies (e4m3 outliers
 * far beyond 9 sigma), and by the rounding of the fixed-point model
 * elsewhere.  (The pages' section "KV 缓存并非真正随机": the code length of a
 * symbol is -log2 of its probability.)
 *   per_scalar    device fp32 [N] output, or NULL.
 *   total         host; receives the sum in bits (fp64, fixed order).
 * Per-scalar values are fp32: costs below one bit through log1p of the exact
 * complement, others as M - log2(freq), within 4e-6 bits of exact.
 * Workspace: skv_workspace_bytes(..., SKV_OP_MODEL_BITS).  Rejects
 * SKV_FLAG_ADAPTIVE (SKV_ERR_ARG).  Errors: SKV_ERR_ARG, SKV_ERR_CAPACITY
 * (workspace), SKV_ERR_SYMBOL, SKV_ERR_PARAM, SKV_ERR_CUDA.  Synchronizes. */
int skv_model_bits(const skv_params *params, const skv_shape *shape, const void *kv,
                   const uint16_t *mu, float *per_scalar, double *total, void *workspace,
                   size_t workspace_bytes, skv_stream_t stream);

/* skv_ideal_bits without a caller workspace.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory, such
 * as serving engines that reserve all free HBM for their KV-cache pool at
 * start-up (a later cudaMalloc fails or forces cache eviction) and plugins
 * running inside such an engine without access to its allocator.
 *
 * Same arguments, results and errors as skv_ideal_bits minus the workspace.
 * Its scratch is a fixed 2 MiB device array inside libskv.so, held by every
 * device that loads the library until the process exits; the call allocates
 * nothing.  Shapes whose (layers * 2 * heads * head_dim) sigma entries exceed
 * skv_ideal_bits_noalloc_max_channels() are rejected with SKV_ERR_CAPACITY.
 * SKV_FLAG_BLOCK_SCALE is rejected with SKV_ERR_ARG: its per-(chunk, channel)
 * table grows with the cache and has no fixed bound.  So is SKV_FLAG_ORDER0.
 * Every call shares that one array, so calls that may overlap on the GPU (on
 * different streams, or from different host threads) race; serialise them.
 * The first call on a device looks up the array's device address and uploads
 * the model constants (synchronous copies): make it before any stream capture. */
int skv_ideal_bits_noalloc(const skv_params *params, const skv_shape *shape, const void *kv,
                           const uint16_t *mu, float *per_scalar, double *total,
                           skv_stream_t stream);

/* Largest number of sigma entries skv_ideal_bits_noalloc accepts. */
size_t skv_ideal_bits_noalloc_max_channels(void);

/* Host helper: p-hat tables from a calibration histogram.
 *   counts   host, u64[65536], occurrences of each bf16 bit pattern (NaN
 *            patterns are ignored).
 *   ecdf     host output, u32[65283] (E_q, see skv_params).
 *   phat     host output, fp32[65282] by rank, or NULL.
 * Add-one smoothing over the 65282 non-NaN symbols.  Errors: SKV_ERR_ARG
 * (NULL pointer, or a total count >= 2^37). */
int skv_build_ecdf(const uint64_t *counts, uint32_t *ecdf, float *phat);

/* Host helper: the Phi table of the model, u32[8193] with
 * T[i] = RNE(2^26 Phi(-8 + i/512)), T[0] = 0, T[8192] = 2^26. */
int skv_phi_table(uint32_t *table);

/* Static description of a status code. */
const char *skv_strerror(int status);

/* Library format version (1). */
int skv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SKV_H */
