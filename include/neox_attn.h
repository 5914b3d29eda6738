/*
 * neox_attn.h -- C ABI of the B300 (sm_103a) causal NeoX-rotary self-attention
 * forward.
 *
 * The operation (defined from these pages):
 *   - "GPT-NeoX on FasterTransformer" guide, section "背景": GPT-NeoX uses the
 *     Neox-style rotary embedding (neox_rotary_style_ = true) and the context
 *     attention accumulates Q.K^T in fp32 by default (is_context_qk_buf_float_).
 *   - same guide, section "模型配置（config.ini）": rotary_embedding=24 of
 *     size_per_head=96, with the rotation applied to both Query and Key.
 *   - same guide, section "从 HuggingFace 检查点部署": the fused
 *     query_key_value weight is laid out [hidden, num_heads, 3, head_hidden], so a
 *     token's projection output is packed [H, 3, D]; this op reads that packed
 *     tensor directly.
 *   - "gpt-neox - 模型与框架" hub page, section "问题二：注意力计算太慢": the
 *     attention is exact (Flash Attention 2 changes memory traffic, not results).
 *
 * For every batch b, head h and query position i (0-based; positions are the
 * token indices 0..S-1, identical for Q and K):
 *   q' = R(i) q_i,  k'_j = R(j) k_j, where R(p) rotates each pair (d, d + r/2),
 *        d < r/2, by the angle p * rotary_base^(-2d/r) ("rotate-half"):
 *        y_d = x_d cos - x_{d+r/2} sin,  y_{d+r/2} = x_{d+r/2} cos + x_d sin;
 *        dims >= r pass through.  V is not rotated.
 *   s_ij = q'.k'_j / sqrt(D) for j <= i (causal, diagonal kept),
 *   out_i = sum_j softmax_j(s_ij) v_j,   lse_i = ln sum_j exp(s_ij).
 *
 * Threading: every entry point may be called from any host thread.  All work is
 * stream-ordered on the caller's stream and asynchronous unless stated.
 * No entry point throws across the ABI; errors come back as neox_status codes.
 */
#ifndef NEOX_ATTN_H_
#define NEOX_ATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NEOX_OK = 0,
  NEOX_ERR_INVALID_ARG = -1,          /* null pointer, bad size, overlap of out/lse with qkv */
  NEOX_ERR_UNSUPPORTED_HEAD_DIM = -2, /* D not in {64, 96, 128} */
  NEOX_ERR_MISALIGNED = -3,           /* qkv/out not 16-byte aligned, lse not 4-byte aligned */
  NEOX_ERR_CUDA = -4,                 /* a CUDA runtime/driver call failed (see neox_attn_last_cuda_error) */
  NEOX_ERR_DEVICE_TIMEOUT = -5,       /* a kernel's bounded wait ran out; results are not valid */
  NEOX_ERR_NO_DEVICE_SUPPORT = -6,    /* current device is not compute capability 10.3 (B300) */
  NEOX_ERR_TOO_LARGE = -7,            /* neox_attn_fwd_noalloc: S * rotary_dim/2 > 1048576 */
  NEOX_ERR_DEVICE_BAD_POSITION = -8,  /* neox_attn_decode: a pos[b] was outside [0, Smax) */
  NEOX_ERR_DEVICE_RANGE = -9          /* forward: a rotated q/k value exceeded 65504 (see neox_attn_fwd) */
} neox_status;

/*
 * Causal NeoX-rotary self-attention forward.
 *
 *   qkv          device pointer, bf16 [B, S, H, 3, D], contiguous, slot 0 = Q,
 *                1 = K, 2 = V; 16-byte aligned; read only (never rotated in place).
 *   B, S, H      batch, sequence length, heads; each >= 1; B*S*H*3*D < 2^40.
 *                Any S is accepted (ragged tails are masked).
 *   D            head dim, one of 64, 96, 128.
 *   rotary_dim   even, 0 <= rotary_dim <= D (0 = no rotary embedding).
 *   rotary_base  > 0 and finite (10000 for GPT-NeoX).
 *   out          device pointer, bf16 [B, S, H, D], contiguous, 16-byte aligned;
 *                must not overlap qkv or lse.  Written, never read.
 *   lse          device pointer, fp32 [B, H, S], contiguous, 4-byte aligned;
 *                natural-log logsumexp of the scaled scores of each row.
 *   stream       a cudaStream_t (NULL = legacy default stream).
 *
 * Ownership: the caller owns qkv/out/lse; the library neither frees nor keeps
 * them.  The library owns one cached fp32 cos/sin table per (device, rotary_dim,
 * rotary_base), grown on demand; the call that builds or grows it synchronizes
 * `stream` once, later calls do not.  neox_attn_release() frees the cache.  When
 * the rotation is placed in a separate pass (see neox_attn_fwd_ex), the rotated copy
 * lives in the library's per-device scratch.
 *
 * Numerics: scores and outputs accumulate in fp32.  The rotated dims of Q and K are
 * computed in fp32 and enter the score MMA rounded once to fp16 when the rotation runs in
 * the attention kernel at rotary_dim 16, 24 or 32 (those 16-column chunks, including dims
 * 24..31 at rotary_dim 24, are fp16 x fp16, the rest bf16 x bf16); at any other
 * rotary_dim, or with the separate pre-rotation pass, as an exact two-term bf16 split
 * (hi + lo, three products).  fp16 holds |v| <= 65504: a larger rotated value (or
 * dim 24..31 value at rotary_dim 24) makes the results invalid and is reported as
 * NEOX_ERR_DEVICE_RANGE; NEOX_ROTATION_PRE (neox_attn_fwd_ex, rotary_dim 16/24/32)
 * accepts the whole bf16 range.
 *
 * Errors: every argument is validated before any CUDA call; on error nothing is
 * launched and nothing is written.  NEOX_ERR_CUDA means a launch or allocation
 * failed.  A device-side wait timeout, and a value beyond the fp16 range (above), is
 * reported only by neox_attn_get_device_error() after the stream has been synchronized.
 */
int neox_attn_fwd(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base,
                  void* out, float* lse, void* stream);

/*
 * Where the rotary embedding of Q and K is computed (bit-identical results, except that
 * the in-kernel rotation at rotary_dim 16, 24 and 32 rounds the rotated chunks to fp16
 * where the pass keeps the hi/lo split; see neox_attn_fwd):
 *   NEOX_ROTATION_FUSED  inside the attention kernel, in shared memory, on every K tile
 *                        each query unit streams (no extra HBM traffic; the K tile of a
 *                        head is rotated once per query unit that reads it);
 *   NEOX_ROTATION_PRE    by a separate pass that writes q' and k' (split hi/lo) once into
 *                        the library's per-device scratch, 4*B*S*H*D bf16 values, which the
 *                        attention kernel then loads instead of Q and K (needs
 *                        rotary_dim > 0 and rotary_dim % 16 == 0 or rotary_dim == 24);
 *   NEOX_ROTATION_AUTO   PRE when rotary_dim >= 64 and rotary_dim % 16 == 0, else FUSED
 *                        (the choice measured faster on B300 for the GPT-NeoX shapes).
 */
enum { NEOX_ROTATION_AUTO = 0, NEOX_ROTATION_FUSED = 1, NEOX_ROTATION_PRE = 2 };

/*
 * neox_attn_fwd with the rotation placement chosen by the caller (one of the
 * NEOX_ROTATION_* values; anything else, or PRE with rotary_dim == 0 or a rotary_dim
 * that is neither a multiple of 16 nor 24, gives NEOX_ERR_INVALID_ARG before any CUDA
 * call).
 * neox_attn_fwd(...) is neox_attn_fwd_ex(..., NEOX_ROTATION_AUTO, stream).
 *
 * The PRE placement uses the library's per-device scratch (allocated or grown on
 * demand; growing synchronizes the device), which neox_attn_decode and neox_attn_bwd
 * use too: calls that use it must not overlap on the GPU (order them on one stream).
 */
int neox_attn_fwd_ex(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base,
                     void* out, float* lse, int rotation, void* stream);

/*
 * ALiBi variant of the forward: the other positional scheme GPT-NeoX supports ("gpt-neox -
 * 模型与框架" hub page, sections "架构创新" and "位置编码"; GPT-NeoX library summary, "Key
 * capabilities": rotary and ALiBi position embeddings).  No rotation; instead each score
 * gets a linear bias by query-key distance:
 *   s_ij = q_i.k_j / sqrt(D) - m_h (i - j)   for j <= i,
 * with the head slopes of the published ALiBi method (the pages name the scheme but print
 * no formula): for the n = largest power of two <= H heads m_h = 2^(-8(h+1)/n), h < n;
 * the remaining heads take 2^(-8k/(2n)) for odd k = 1, 3, 5, ... in order.
 * out_i = sum_j softmax_j(s_ij) v_j and lse_i = ln sum_j exp(s_ij), as in neox_attn_fwd.
 * Arguments, layouts, ownership and errors are those of neox_attn_fwd (no rotary
 * arguments; no table is built).
 */
int neox_attn_fwd_alibi(const void* qkv, int B, int S, int H, int D, void* out, float* lse, void* stream);

/*
 * The fused query_key_value projection that produces the packed qkv, with its bias and,
 * when rotary_dim > 0, the NeoX rotary embedding of the query and key slots applied on the
 * way out ("GPT-NeoX on FasterTransformer" guide: section "从 HuggingFace 检查点部署" gives
 * the weight layout [hidden_size, num_heads, 3, head_hidden], the layer list in
 * "从 EleutherAI 检查点部署" gives attention.query_key_value's weight and bias, and
 * "模型配置（config.ini）" the 20B shape: hidden 6144 = 64 heads x 96, rotary_embedding 24).
 *
 *   x     device, bf16 [B*S, hidden] row-major: token t = b*S + s is at position s.
 *   w     device, bf16 [hidden, H, 3, D] row-major (= [hidden, N], N = 3*H*D).
 *   bias  device, bf16 [N], or NULL for none.
 *   qkv   device, bf16 [B, S, H, 3, D] (= [B*S, N]), written:
 *           y[t, n] = bf16( sum_k x[t,k] * w[k,n] + bias[n] )   (fp32 accumulation)
 *         and then, if rotary_dim > 0, for every head's query and key slot and each
 *         i < rotary_dim/2, with a = y[.., i], b = y[.., i + rotary_dim/2] and
 *         theta = s * rotary_base^(-2i/rotary_dim):
 *           y[.., i] = bf16(a cos(theta) - b sin(theta)),
 *           y[.., i + rotary_dim/2] = bf16(b cos(theta) + a sin(theta)),
 *         (rotation in fp32 of the bf16 projection, rounded once more); value slots and
 *         dims >= rotary_dim are the plain projection.  A qkv written with rotary_dim > 0
 *         is already rotated: give it to neox_attn_fwd with rotary_dim 0.
 * Sizes: hidden a multiple of 8 (>= 8); D in {64, 96, 128}; 0 <= rotary_dim <= D, even;
 * B*S and N below 2^31.  All pointers 16-byte aligned; qkv may not overlap x, w or bias.
 * Errors as neox_attn_fwd: NEOX_ERR_INVALID_ARG / _UNSUPPORTED_HEAD_DIM / _MISALIGNED
 * before any CUDA call; NEOX_ERR_CUDA if a launch or the cos/sin table (cached per device,
 * rotary_dim and base, shared with the attention calls) fails; a device-side timeout shows
 * in neox_attn_get_device_error().  Asynchronous on `stream`; the caller owns all buffers.
 */
int neox_attn_qkv_proj(const void* x, const void* w, const void* bias, int B, int S, int hidden, int H, int D,
                       int rotary_dim, float rotary_base, void* qkv, void* stream);

/*
 * Same contract as neox_attn_fwd, computed by the plain single-warpgroup tcgen05 kernel
 * (one CTA per 128-row query tile, every stage in sequence).  Slower; kept as an
 * independent second implementation of the same tile layouts for cross-checking.
 * Limits: B <= 65535 and H <= 65535 (grid dimensions), else NEOX_ERR_INVALID_ARG.
 */
int neox_attn_fwd_simple(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base,
                         void* out, float* lse, void* stream);

/*
 * The same computation as neox_attn_fwd, for callers that cannot let a library
 * allocate device memory.  The pages have no counterpart to this entry point.
 *
 * Who needs it: a framework or inference server whose own caching allocator has
 * already reserved nearly all of the GPU's memory (a cudaMalloc from a library would
 * then fail, or carve a block out of memory the caller has accounted for), and
 * request paths that must not call cudaMalloc/cudaFree at all because those calls can
 * synchronize the device.  neox_attn_fwd allocates its cos/sin table on first use;
 * this entry point never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Instead the cos/sin table lives in one fixed device array compiled into the library
 * (8 MiB, 1048576 entries; every GPU that loads the library holds it until the process
 * exits).  Limit: S * rotary_dim/2 <= 1048576 (e.g. S = 16384 with rotary_dim = 128),
 * else NEOX_ERR_TOO_LARGE and nothing is launched.
 *
 * Each call rebuilds rows [0, S) of the table on `stream` and then runs the attention
 * kernel on the same stream; the array keeps the last call's contents.  All calls share
 * the one array, so calls that overlap on the GPU (different streams, no ordering
 * between them) race on it and may read another call's table: order them.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 * before any stream capture.  The CUDA driver may place the library's device code and
 * this array on a device only when the library is first used there (lazy module
 * loading), so make the first call on each device -- or any earlier call into the library
 * there -- before the caller's allocator takes up the rest of the device's memory.
 * Arguments, layouts, ownership and the other errors are those of neox_attn_fwd
 * (the rotation is always computed inside the attention kernel).
 */
int neox_attn_fwd_noalloc(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base,
                          void* out, float* lse, void* stream);

/*
 * Incremental decode: one new token per sequence against a key/value cache.
 *
 * GPT-NeoX serving runs a per-token decoder that extends a growing context
 * ("GPT-NeoX on FasterTransformer" guide, section "背景"); the pages print no
 * interface, so this one is the library's own.  Sequence b already holds pos[b]
 * tokens; the new token sits at position pos[b].  Its query, rotated at pos[b],
 * attends to keys 0..pos[b] (itself included), each rotated at its own position
 * exactly as in neox_attn_fwd, scaled by 1/sqrt(D): the result equals row pos[b]
 * of neox_attn_fwd over the whole sequence.  The new key and value are then part
 * of the cache (row pos[b] is written).
 *
 *   qkv_new      device, bf16 [B, H, 3, D], contiguous (the new token's packed
 *                projection, slot 0 = Q, 1 = K, 2 = V); 16-byte aligned; read only.
 *   k_cache,     device, bf16 [B, H, Smax, D] each, contiguous, 16-byte aligned,
 *   v_cache      not overlapping each other or any other argument.  Keys are stored
 *                as projected, NOT rotated.  Rows p < pos[b] are read; row pos[b] is
 *                overwritten with the new token's k / v (raw bf16, bit for bit);
 *                rows > pos[b] are neither read nor written.
 *   pos          device, int32 [B], 4-byte aligned: tokens already cached per
 *                sequence, 0 <= pos[b] < Smax.  Read on the device only, so a value
 *                out of range cannot be rejected before launch: that sequence's out
 *                and lse are left undefined, its cache is not written, and
 *                neox_attn_get_device_error() reports NEOX_ERR_DEVICE_BAD_POSITION.
 *   B, H, Smax   each >= 1, B and H <= 65535, B*H*Smax*D < 2^40.
 *   D, rotary_dim, rotary_base   as for neox_attn_fwd.
 *   out          device, bf16 [B, H, D], 16-byte aligned, written.
 *   lse          device, fp32 [B, H], 4-byte aligned, natural-log logsumexp.
 *   stream       a cudaStream_t (NULL = legacy default stream).
 *
 * Ownership and errors as for neox_attn_fwd.  Besides the cos/sin table the library
 * owns a per-device scratch: fp32 partial results of heads whose keys are split
 * between several CTAs, and one int32 arrival counter per head that every call
 * leaves at zero (grown on demand like the table; the call that grows it
 * synchronizes the device once; neox_attn_release() frees it).  Calls share the
 * scratch, so decode calls must not overlap on the GPU (different streams with no
 * ordering between them).  After a NEOX_ERR_DEVICE_TIMEOUT report,
 * neox_attn_get_device_error() re-zeroes the counters.
 */
int neox_attn_decode(const void* qkv_new, void* k_cache, void* v_cache, const int* pos, int B, int H, int Smax,
                     int D, int rotary_dim, float rotary_base, void* out, float* lse, void* stream);

/*
 * Backward of neox_attn_fwd: the gradients of sum(dout * out) with respect to the
 * packed projection.
 *
 * GPT-NeoX is a training framework that runs its attention as the exact, tiled
 * Flash Attention ("gpt-neox - 模型与框架" page, section "问题二：注意力计算太慢");
 * the pages print no backward, so the interface is the library's own and follows the
 * chain rule through the forward: with p_ij = exp(s_ij - lse_i) over keys j <= i,
 * dv_j = sum_i p_ij dout_i, ds_ij = p_ij (dout_i.v_j - dout_i.out_i),
 * dq'_i = sum_j ds_ij k'_j / sqrt(D), dk'_j = sum_i ds_ij q'_i / sqrt(D), and dq, dk are
 * dq', dk' rotated back (rotation by -theta on the first rotary_dim dims).
 *
 *   qkv          device, bf16 [B, S, H, 3, D], the forward's input; read only.
 *   out, lse     device, the forward's outputs for this qkv (bf16 [B, S, H, D], 16-byte
 *                aligned; fp32 [B, H, S], natural log, 4-byte aligned); read only.
 *   dout         device, bf16 [B, S, H, D], 16-byte aligned; read only.
 *   B, S, H, D, rotary_dim, rotary_base   as for neox_attn_fwd.
 *   dqkv         device, bf16 [B, S, H, 3, D] (slot 0 = dq, 1 = dk, 2 = dv), 16-byte
 *                aligned, written completely; may not overlap any input.
 *   stream       a cudaStream_t (NULL = legacy default stream).
 *
 * Arithmetic: rotated q', k', the probabilities and ds enter the tensor cores as bf16,
 * everything accumulates in fp32.  Ownership and errors as for neox_attn_fwd.  The
 * library's per-device scratch (shared with neox_attn_decode, grown on demand, freed by
 * neox_attn_release) holds an fp32 dq' accumulator of B*S*H*D floats, B*H*S floats of
 * dout.out, and a bf16 copy of qkv's shape holding the rotated q', k' (about 10 bytes
 * per element of out in all), so backward and decode calls must not overlap on the GPU;
 * two backward calls must not overlap either (they also share the device's work counter
 * of the main kernel, which is persistent: one CTA per SM).  dk and dv are identical from
 * call to call; dq can differ by one bf16 rounding, since its fp32 sums are added in the
 * order the key blocks' partial results arrive.
 */
int neox_attn_bwd(const void* qkv, const void* out, const float* lse, const void* dout, int B, int S, int H, int D,
                  int rotary_dim, float rotary_base, void* dqkv, void* stream);

/*
 * Reads and clears the current device's error word written by the kernels' bounded
 * waits and input checks.  Call after synchronizing the streams that ran the kernels.
 * Returns NEOX_OK, NEOX_ERR_DEVICE_TIMEOUT, NEOX_ERR_DEVICE_RANGE (forward with in-kernel
 * rotation at rotary_dim 16, 24 or 32), NEOX_ERR_DEVICE_BAD_POSITION (decode only), or
 * NEOX_ERR_CUDA if the read failed; a timeout is reported before the others.
 */
int neox_attn_get_device_error(void);

/* A static, human-readable name for a neox_status value. */
const char* neox_attn_status_string(int status);

/* The last CUDA error code the library saw on this host thread (0 = none). */
int neox_attn_last_cuda_error(void);

/* Frees the library-owned cos/sin tables and decode scratch buffers on every device.
 * Waits for the device first; not to be called while work is being enqueued elsewhere. */
void neox_attn_release(void);

/*
 * Self-test of the bounded-wait machinery: launches one tiny kernel that waits on
 * a shared-memory barrier nothing arrives on, with a limit of `timeout_ns`
 * nanoseconds (1e3 .. 1e9).  After the stream is synchronized,
 * neox_attn_get_device_error() must return NEOX_ERR_DEVICE_TIMEOUT.  Nothing
 * faults and nothing hangs; the context stays usable.
 */
int neox_attn_selftest_wait_timeout(int64_t timeout_ns, void* stream);

/* ABI version: major * 10000 + minor * 100 + patch. */
int neox_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NEOX_ATTN_H_ */
