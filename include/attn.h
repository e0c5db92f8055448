/*
 * exact_attention_43_gb300 -- fused exact attention for one NVIDIA GB300 (sm_103a).
 *
 * C ABI: plain pointers and sizes, no C++ or framework types.  Every entry
 * point returns an attn_status_t code, never aborts and never traps on the
 * device.  Work is enqueued asynchronously on the caller's CUDA stream; the
 * library keeps no pointer after a call returns and the caller owns every
 * buffer.  All tensors are dense, row-major, with the head dimension
 * innermost.  Workspaces are allocated and freed on the caller's stream, so a
 * call may be captured into a CUDA graph (the backward's kernels are chained by
 * programmatic launches, recorded as programmatic edges).
 *
 * Sources of what is computed (page title and the part of the page):
 *   - abaddon 0.2.0-rc.2, src/cuda_inference/kernels/attention.rs: module doc
 *     "Algorithm" (tiled exact attention, online softmax, final divide by the
 *     sum), kernels flash_attention_f16 (layouts [batch, heads, seq, head_dim]
 *     and [batch, kv_heads, seq, head_dim], GQA kv_head = head * kv_heads /
 *     heads, causal masking) and flash_attention_cached_f16 /
 *     FlashAttentionKernel::forward_cached (single-query decode against a
 *     cache [batch, kv_heads, cache_len, head_dim], scale 1/sqrt(head_dim)),
 *     and the Shape / Kernel error returns of FlashAttentionKernel::forward;
 *   - rustytorch flash_attention_forward.cu: kernel flash_attention_forward_kernel
 *     (arguments q, k, v, o, lse, softmax_scale, causal; LSE laid out
 *     [batch * heads, seq_len]) and OnlineSoftmaxState::get_log_sum_exp
 *     (LSE = m + log l, natural log);
 *   - aprender-gpu 0.32.0, kernels/attention/paged/flash_decoding/reduce_kernel.rs:
 *     FlashDecodingReduceKernel (per-sequence seq_lens, chunk partials
 *     [M, num_heads, max_chunks, head_dim + 2], LSE-rescaling merge).
 */
#ifndef EXACT_ATTENTION_43_GB300_ATTN_H
#define EXACT_ATTENTION_43_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* cudaStream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null or misaligned pointer, negative size, Hq % Hkv != 0, ... */
  ATTN_ERR_UNSUPPORTED = 2,    /* head dim not 64/128, unknown dtype, device is not sm_103 */
  ATTN_ERR_CUDA = 3,           /* a CUDA call or kernel launch failed */
  ATTN_ERR_DEVICE_TIMEOUT = 4  /* a kernel's bounded wait ran out (read by attn_check_device_status) */
} attn_status_t;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype_t;

/*
 * attn_fwd -- prefill attention with per-row log-sum-exp.
 *
 *   O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,g,j,:] + mask) V[b,g,j,:],
 *   LSE[b,h,i] = ln sum_j exp(scale * Q[b,h,i,:] . K[b,g,j,:] + mask),
 *   g = h / (Hq / Hkv)  (consecutive query heads share a KV head).
 *
 * q, o   device, [B, Hq, Sq, D], dtype `dtype`, 16-byte aligned.
 * k, v   device, [B, Hkv, Skv, D], dtype `dtype`, 16-byte aligned.
 * lse    device, [B, Hq, Sq] float32, 4-byte aligned, or NULL to skip it.
 * causal 0: every key visible.  1: key j visible to query i iff
 *        j <= i + (Skv - Sq) (aligned bottom-right; j <= i when Sq == Skv).
 *        A row that sees no key gets O = 0 and LSE = -inf.
 * scale  any finite float (the softmax temperature, typically 1/sqrt(D)).
 * D      64 or 128.  dtype: ATTN_BF16 or ATTN_FP16 (O has the dtype of q).
 * Sizes  B, Hq, Hkv >= 1 unless B*Hq*Sq == 0 (then nothing is done);
 *        Sq, Skv >= 0; Hq % Hkv == 0; B, Hq <= 65535.
 * Returns ATTN_OK once the work is enqueued on `stream`; validation errors
 * are returned before any CUDA call.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Skv, int D, int causal, float scale, int dtype,
             cudaStream_t stream);

/*
 * attn_fwd_varlen -- attn_fwd over a packed batch of sequences of different
 * lengths, with an optional sliding window.
 *
 * The flash-attention backward page names `Varlen` and `Is_local` switches
 * without defining them; the readings here:
 *   sequence b has query tokens [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key
 *   tokens [cu_seqlens_k[b], cu_seqlens_k[b+1]), attended on their own; with
 *   d = (its keys) - (its queries), its query i keeps key j iff
 *   j <= i + d (causal) and i + d - window_left <= j <= i + d + window_right,
 *   a bound of -1 being absent (causal makes the right bound 0).
 *
 * q, o        device, [total_q, Hq, D], dtype `dtype`, 16-byte aligned.
 * k, v        device, [total_k, Hkv, D], 16-byte aligned (unused if total_k == 0).
 * lse         device, [Hq, total_q] float32, 4-byte aligned, or NULL.
 * cu_seqlens_q, cu_seqlens_k  device, [B + 1] int32, non-decreasing offsets
 *             within [0, total_q] / [0, total_k]; a sequence's lengths must not
 *             exceed max_seqlen_q / max_seqlen_k.  Offsets or lengths outside
 *             those ranges are clamped on the device (no access leaves the
 *             arrays) and reported by attn_check_device_status as
 *             ATTN_ERR_INVALID_ARG.  Rows outside every sequence are not written.
 * A row that keeps no key gets O = 0 and LSE = -inf.  Every element of k and v
 * must be finite: a tile that ends inside a sequence also reads the next
 * sequence's keys, whose probabilities are exactly 0.
 * window_left, window_right >= -1; max_seqlen_q + max_seqlen_k < 2^30;
 * B, Hq <= 65535; D 64 or 128; scale finite; Hq % Hkv == 0.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int D, int causal,
                    int window_left, int window_right, float scale, int dtype, cudaStream_t stream);

/*
 * attn_fwd_qkvpacked -- attn_fwd reading Q, K and V in place from one packed
 * projection (the llm.c attention page's (B, N, 3, NH, d) QKV tensor, which it
 * permutes into three (B, NH, N, d) arrays first; here no copy is made).
 *
 * qkv   device, [B, S, 3, H, D], dtype `dtype`, 16-byte aligned.
 * o     device, [B, S, H, D] (the llm.c page's unpermuted output layout).
 * lse   device, [H, B, S] float32 or NULL.
 * causal, window_left, window_right, scale as in attn_fwd_varlen (every
 * sequence has S queries and S keys).  B * S < 2^31, 2 S < 2^30.
 */
int attn_fwd_qkvpacked(const void* qkv, void* o, float* lse, int B, int S, int H, int D, int causal,
                       int window_left, int window_right, float scale, int dtype,
                       cudaStream_t stream);

/*
 * attn_bwd -- gradients of attn_fwd: dQ, dK, dV for an incoming dO.
 *
 * As the llm.c attention page's attention_backward computes them:
 *   dP = dO V^T, dV = P^T dO, dS = scale * P * (dP - rowsum(P * dP)),
 *   dQ = dS K, dK = dS^T Q,
 * P being the forward's probabilities, re-formed here from its LSE
 * (P = e^(scale Q K^T - LSE) on the visible keys), and rowsum(P * dP) taken as
 * rowsum(dO * O).  A KV head's dK and dV are summed over the query heads that
 * share it.  Same layouts, causal rule and head mapping as attn_fwd.
 *
 * q, o, dout, dq   device, [B, Hq, Sq, D], dtype `dtype`, 16-byte aligned.
 * k, v, dk, dv     device, [B, Hkv, Skv, D], 16-byte aligned.
 * lse              device, [B, Hq, Sq] float32, the forward's (natural log).
 * o, lse must be attn_fwd's outputs for these q, k, v, causal and scale.
 * A workspace of attn_bwd_workspace_bytes(B, Hq, Sq, D) bytes (the fp32 row
 * terms and the persistent kernels' two work counters) is taken from the
 * library's stream-ordered pool.  No gradient is
 * accumulated with atomics: two calls give identical bits.
 * D 64 or 128; B, Hq, Hkv <= 65535; scale finite.  With Skv == 0, dq = 0.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Skv,
             int D, int causal, float scale, int dtype, cudaStream_t stream);

/* Bytes of workspace attn_bwd allocates for these sizes; 0 on invalid sizes.  The
 * token-major entry points below allocate the same for B = 1, Sq = total_q. */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq, int D);

/*
 * attn_bwd_varlen -- attn_bwd for attn_fwd_varlen: packed sequences of different
 * lengths and sliding windows, in the token-major layout.
 *
 * The flash-attention backward page's kernel class takes the same `Varlen` and
 * `Is_local` switches as the forward; the readings are attn_fwd_varlen's: each
 * sequence's gradients are those of its own rows, with its own bottom-right
 * alignment and the window's bounds.
 *
 * q, o, dout, dq   device, [total_q, Hq, D], dtype `dtype`, 16-byte aligned.
 * k, v, dk, dv     device, [total_k, Hkv, D], 16-byte aligned.
 * lse              device, [Hq, total_q] float32: attn_fwd_varlen's, for the same
 *                  inputs, offsets, causal flag, window and scale (as is o).
 * cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, window_left,
 * window_right, scale, D, dtype, B, Hq, Hkv: as in attn_fwd_varlen (offsets
 * outside their ranges are clamped on the device and reported by
 * attn_check_device_status as ATTN_ERR_INVALID_ARG).  Gradient rows of tokens
 * outside every sequence are not written; a sequence's keys that no query sees
 * get dK = dV = 0, its queries that see no key dQ = 0.  Every element of q, k, v
 * and dout must be finite (a tile that ends inside a sequence also reads the
 * next sequence's rows, with weight exactly 0).
 */
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k,
                    int max_seqlen_q, int max_seqlen_k, int D, int causal, int window_left,
                    int window_right, float scale, int dtype, cudaStream_t stream);

/*
 * attn_bwd_qkvpacked -- attn_bwd for attn_fwd_qkvpacked: the gradient of one packed
 * projection, written in place into the same layout.
 *
 * qkv    device, [B, S, 3, H, D] (attn_fwd_qkvpacked's input), 16-byte aligned.
 * o      device, [B, S, H, D], lse [H, B, S] float32: attn_fwd_qkvpacked's outputs.
 * dout   device, [B, S, H, D].
 * dqkv   device, [B, S, 3, H, D]: dQ, dK, dV at the places of Q, K, V.
 * causal, window_left, window_right, scale as in attn_fwd_qkvpacked.
 */
int attn_bwd_qkvpacked(const void* qkv, const void* o, const float* lse, const void* dout, void* dqkv,
                       int B, int S, int H, int D, int causal, int window_left, int window_right,
                       float scale, int dtype, cudaStream_t stream);

/*
 * attn_decode -- flash-decoding: one query token per sequence against a KV cache.
 *
 *   O[b,h,:] = softmax_j(Q[b,h,:] . K[b,g,j,:] / sqrt(D)) V[b,g,j,:],  0 <= j < seq_lens[b].
 *
 * The keys of every sequence are split into chunks of
 * chunk = ceil(max_S / num_splits) positions (512 when num_splits == 0); a
 * split kernel writes per-chunk partials (o, m, l) to a stream-ordered fp32
 * workspace of attn_decode_workspace_bytes(...) bytes and a reduce kernel
 * merges them by LSE rescaling.
 *
 * q, o      device, [B, Hq, D], dtype `dtype`, 16-byte aligned.
 * k_cache,  device, [B, Hkv, max_S, D], dtype `dtype`, 16-byte aligned;
 * v_cache   only positions [0, seq_lens[b]) are read.
 * seq_lens  device, [B] int32, 0 <= seq_lens[b] <= max_S.  A value outside
 *           that range is clamped on the device and reported by
 *           attn_check_device_status as ATTN_ERR_INVALID_ARG.  A sequence
 *           of length 0 gets O = 0.
 * D 64 or 128; Hq % Hkv == 0; num_splits >= 0; B, Hkv <= 65535.
 * The workspace is taken from a library-owned CUDA memory pool with
 * cudaMallocFromPoolAsync / cudaFreeAsync on `stream`.
 */
int attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                void* o, int B, int Hq, int Hkv, int max_S, int D, int num_splits, int dtype,
                cudaStream_t stream);

/*
 * attn_decode_fused -- attn_decode in one kernel launch.
 *
 * Same arguments, layouts, chunking, partials workspace and status codes as
 * attn_decode; the result agrees with it to fp32 rounding (the merge adds the
 * chunk terms in another order).  Instead of a second (reduce) kernel, each
 * split-kernel CTA takes a ticket from a counter of its (sequence, head group)
 * when its partials are written, and the CTA that takes the last ticket merges
 * that group's partials by the same LSE rescaling and writes O.  The counters
 * are a library-owned device array, zeroed once per device by a memset that
 * the first call enqueues on its stream (make that first call before any
 * stream capture begins) and left at zero by every call.  Calls whose kernels
 * may overlap on the GPU (two streams with no ordering between them) share
 * the counters: order them on one stream or with events.
 * B * Hq <= 1048576, else ATTN_ERR_UNSUPPORTED before any CUDA call.
 */
int attn_decode_fused(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* seq_lens, void* o, int B, int Hq, int Hkv, int max_S, int D,
                      int num_splits, int dtype, cudaStream_t stream);

/*
 * attn_decode_paged -- attn_decode over a paged KV cache.
 *
 * Same computation, chunking, partials and merge as attn_decode; only where
 * the keys and values live differs.  The pages place the flash-decoding code
 * under a paged-cache directory but give no page layout; the layout here keeps
 * one page of one KV head contiguous, so a page is read with one bulk copy:
 *
 * k_pages,    device, [num_pages, Hkv, page_size, D], dtype `dtype`, 16-byte
 * v_pages     aligned; a page holds page_size consecutive positions of one
 *             sequence, for every KV head.
 * block_table device, [B, max_pages] int32, 4-byte aligned: position j of
 *             sequence b is row j % page_size of page block_table[b, j / page_size].
 *             Only the first ceil(seq_lens[b] / page_size) entries of a row are
 *             read.  An entry outside [0, num_pages) is replaced by page 0 (no
 *             read leaves the pool) and reported by attn_check_device_status as
 *             ATTN_ERR_INVALID_ARG.
 * seq_lens    device, [B] int32, 0 <= seq_lens[b] <= max_pages * page_size
 *             (clamped and reported as in attn_decode).
 * page_size >= 1; num_pages, max_pages >= 0 (num_pages >= 1 when max_pages > 0);
 * max_pages * page_size plays the role of max_S for the chunking and for
 * attn_decode_workspace_bytes.  Other arguments, the workspace and the status
 * codes are those of attn_decode.
 */
int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* block_table, const int32_t* seq_lens, void* o, int B, int Hq,
                      int Hkv, int num_pages, int page_size, int max_pages, int D, int num_splits,
                      int dtype, cudaStream_t stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that must not allocate GPU memory.
 *
 * Some callers cannot allocate device memory while they run: a plugin whose
 * host application owns the whole device memory budget, a serving loop that
 * must not risk an allocator call that waits on the device or fails under
 * memory pressure, or code running where the CUDA allocator is off limits.
 * This entry point computes exactly what attn_decode computes, with the same
 * arguments, layouts and status codes, but keeps the per-chunk partials in a
 * fixed scratch array that the library reserves on every device that loads
 * it, for the life of the process.  It calls no allocator.  (No counterpart
 * on the pages: the reduce kernel there simply receives a partials pointer.)
 *
 * Limit: attn_decode_workspace_bytes(B, Hq, max_S, D, num_splits) must not
 * exceed ATTN_DECODE_NOALLOC_MAX_BYTES (16 MiB, e.g. B = 8, Hq = 32,
 * max_S = 32768, D = 128, 64 splits); larger problems return
 * ATTN_ERR_UNSUPPORTED before any CUDA call, and nothing is launched.
 *
 * The first call on each device looks up the device address of the scratch
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture begins.  All calls share the one scratch array:
 * calls whose kernels may overlap on the GPU (for instance on two streams
 * with no ordering between them) race on it, so order them on one stream or
 * with events.  The array keeps the last call's partials; no call depends on
 * its earlier contents.
 */
#define ATTN_DECODE_NOALLOC_MAX_BYTES ((size_t)16 << 20)
int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seq_lens, void* o, int B, int Hq, int Hkv, int max_S, int D,
                        int num_splits, int dtype, cudaStream_t stream);

/* Bytes of fp32 partials attn_decode allocates for these sizes
 * (B * Hq * ceil(max_S / chunk) * (D + 2) * 4); 0 on invalid sizes. */
size_t attn_decode_workspace_bytes(int B, int Hq, int max_S, int D, int num_splits);

/* Chunk length attn_decode uses for (max_S, num_splits); 0 on invalid sizes. */
int attn_decode_chunk(int max_S, int num_splits);

/*
 * Synchronise `stream`, then read and clear the library's device status
 * words.  Returns ATTN_ERR_DEVICE_TIMEOUT if any kernel gave up a bounded
 * wait, ATTN_ERR_INVALID_ARG if a decode seq_len was clamped, ATTN_ERR_CUDA
 * if the stream reported an error, else ATTN_OK.
 */
int attn_check_device_status(cudaStream_t stream);

/* Test hooks for the bounded waits.  wait_limit_us sets how long any wait
 * may run before the kernel gives up (0 restores the default of 2 s).  A
 * fault value makes later launches withhold one copy so that the waits on it
 * run out: 1, attn_fwd withholds its first V tile; 2, the decode split kernel
 * (attn_decode, attn_decode_fused, attn_decode_paged, attn_decode_noalloc)
 * withholds the first V sub-tile of its CTA (0, 0, 0); 3, attn_bwd withholds
 * the second Q/dO tile pair of its first work item (the dK/dV kernel's key tile
 * 0 of the first head).  0 turns the fault off.
 * Returns ATTN_OK or ATTN_ERR_INVALID_ARG. */
int attn_debug_set(int fault, unsigned wait_limit_us);

/* Static description of a status code. */
const char* attn_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_43_GB300_ATTN_H */
