// Host-side interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ea {

// Arguments of one prefill launch, already validated by the C-ABI layer.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, Sq, Skv, D;
  int causal;
  float scale;
  int bf16;
  uint64_t wait_limit_ns;
  int debug_fault;  // 1: the loader withholds the first V tile (bounded-wait test only)
  int num_sms;      // multiprocessors of the current device (persistent grid size)
  int* work_counter;  // device int, zero when the kernel starts (work-item claims)
  // token-major layouts (attn_fwd_varlen, attn_fwd_qkvpacked): vl = 1; q, k, v, o
  // are [tokens, heads, D] with the token strides below (elements); sequence b's
  // offsets come from cu_q / cu_k ([B + 1]), or are b * Sq / b * Skv when cu_q is
  // null; Sq and Skv are the longest lengths; LSE is [Hq, total_q]
  int vl;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  long long q_rstride, k_rstride, o_rstride;
  int win_left, win_right;  // sliding-window bounds, -1: none
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* seq_lens;
  void* o;
  float* partials;  // [B, Hq, max_chunks, D + 2] fp32 workspace
  int B, Hq, Hkv, max_S, D, chunk, max_chunks;
  int num_sms;      // multiprocessors of the device
  // paged cache: block_table != nullptr, see attn_decode_paged
  const int32_t* block_table;
  int page_size, max_pages, num_pages;
  // single launch (attn_decode_fused): zeroed counters, one per (sequence, head
  // group); nullptr selects the split kernel + reduce kernel pair
  unsigned* tickets;
  float scale;
  int bf16;
  uint64_t wait_limit_ns;
  int debug_fault;  // 2: split-kernel CTA (0, 0, 0) withholds its first V sub-tile (test only)
};

// Arguments of one backward call (attn_bwd), already validated.
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;  // [B, Hq, Sq] natural log, from the forward pass
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* delta;   // [B, Hq, Sq] fp32 workspace (the row terms)
  int* work_counter;  // two ints of workspace: the persistent kernels' work-item counters
  int B, Hq, Hkv, Sq, Skv, D;
  int causal;
  float scale;
  int bf16;
  uint64_t wait_limit_ns;
  int num_sms;  // multiprocessors of the device (persistent grids)
  int debug_fault;  // 3: the dK/dV CTA of work item 0 withholds its second Q/dO pair (test only)
  int win_left, win_right;  // sliding-window bounds, -1: none (causal: the right bound is 0)
  // token-major layouts (attn_bwd_varlen, attn_bwd_qkvpacked): vl = 1; q, o, dout, dq are
  // [tokens, Hq, D] and k, v, dk, dv [tokens, Hkv, D] with the token strides below
  // (elements); sequence b's offsets come from cu_q / cu_k ([B + 1]), or are b * Sq /
  // b * Skv when cu_q is null; Sq and Skv are the longest lengths; LSE is [Hq, total_q]
  int vl;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  long long q_rstride, k_rstride, do_rstride, dq_rstride, dk_rstride;
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Returns the driver's cuTensorMapEncodeTiled, or nullptr.
EncodeTiledFn encode_tiled_fn();

// Each returns a CUDA error (cudaSuccess on a clean launch) or, for a failed
// tensor-map encoding, cudaErrorInvalidValue.
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_empty_keys(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);

// Read and clear the device status word of each kernel file.
cudaError_t read_fwd_status(unsigned* out, cudaStream_t stream);
cudaError_t read_decode_status(unsigned* out, cudaStream_t stream);
cudaError_t read_bwd_status(unsigned* out, cudaStream_t stream);

// Size of the fixed device scratch behind attn_decode_noalloc (see attn.h).
constexpr size_t kNoallocPartialsBytes = 16u << 20;
// Device address of that scratch on `device`, which must be the current device;
// resolved with cudaGetSymbolAddress on the first request per device.
cudaError_t noalloc_partials(int device, float** out);

// Counters of the single-launch decode: at least B * Hq of them are needed.
constexpr size_t kDecodeTickets = 1u << 20;
// Device address of those counters on `device` (the current device); the first
// request per device zeroes them with a memset enqueued on `stream`.
cudaError_t decode_tickets(int device, unsigned** out, cudaStream_t stream);

}  // namespace ea
