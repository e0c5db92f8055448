// C-ABI entry points: argument validation, device checks, the decode
// workspace pool and the device status words.  Declared in include/attn.h.
#include "../../include/attn.h"
#include "internal.h"

#include <nvtx3/nvToolsExt.h>

#include <math.h>
#include <mutex>

static_assert(ATTN_DECODE_NOALLOC_MAX_BYTES == ea::kNoallocPartialsBytes,
              "header limit and device scratch size must agree");

namespace {

constexpr int kVersion = 100;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr int kDefaultChunk = 512;
constexpr int kMaxDevices = 64;

uint64_t g_wait_limit_ns = kDefaultWaitNs;
int g_fault = 0;

std::mutex g_mu;
int g_arch_ok[kMaxDevices];              // 0 unknown, 1 sm_103, -1 other
int g_num_sms[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// An NVTX range named after the entry point around its validation and launches, so a
// profiler's timeline shows which call enqueued which kernels (the llm.c attention page
// wraps attention_forward and attention_backward the same way).  Without an attached
// tool the push and pop return at once.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

int check_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_num_sms[dev] = sms;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (dev_out) *dev_out = dev;
  return g_arch_ok[dev] == 1 ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

// Library-owned stream-ordered pool for the decode partials; it keeps up to
// 1 GiB cached between calls so repeated decodes do not remap memory.
int pool_for(int dev, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    uint64_t keep = 1ull << 30;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return ATTN_OK;
}

int chunk_for(int max_S, int num_splits) {
  if (max_S < 0 || num_splits < 0) return 0;
  if (num_splits == 0) return kDefaultChunk;
  int c = (max_S + num_splits - 1) / num_splits;
  return c < 1 ? 1 : c;
}

int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  cudaGetLastError();
  return ATTN_ERR_CUDA;
}

}  // namespace

namespace ea {

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

}  // namespace ea

// The persistent prefill kernel with its zeroed work-item counter.
static int run_fwd(ea::FwdArgs& a, int dev, cudaStream_t stream) {
  int st;
  // the persistent kernel's work-item counter: 256 stream-ordered bytes, zeroed
  cudaMemPool_t pool;
  if ((st = pool_for(dev, &pool)) != ATTN_OK) return st;
  void* counter = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&counter, 256, pool, stream);
  if (e != cudaSuccess) return from_cuda(e);
  e = cudaMemsetAsync(counter, 0, sizeof(int), stream);
  if (e == cudaSuccess) {
    a.work_counter = static_cast<int*>(counter);
    e = ea::launch_fwd(a, stream);
  }
  cudaError_t f = cudaFreeAsync(counter, stream);
  if (e == cudaErrorInvalidValue && !ea::encode_tiled_fn()) return ATTN_ERR_UNSUPPORTED;
  if (e == cudaSuccess) e = f;
  return from_cuda(e);
}

// Token-major prefill (attn_fwd_varlen, attn_fwd_qkvpacked): the checks of the
// window and the longest lengths, then the launch.
static int run_fwd_tm(ea::FwdArgs& a, int max_q, int max_k, int window_left, int window_right,
                      cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return ATTN_ERR_INVALID_ARG;
  if (!isfinite(a.scale)) return ATTN_ERR_INVALID_ARG;
  // keeps every key index of the masks inside an int
  if ((long long)max_q + max_k > 0x3fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (((long long)max_q + 255) / 256 * a.Hq * a.B > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  int dev = 0;
  int st = check_device(&dev);
  if (st != ATTN_OK) return st;
  a.vl = 1;
  a.Sq = max_q;
  a.Skv = max_k;
  // a bound at least max_q + max_k away from every diagonal excludes no key
  a.win_left = window_left > max_q + max_k ? -1 : window_left;
  a.win_right = window_right > max_q + max_k ? -1 : window_right;
  a.wait_limit_ns = g_wait_limit_ns;
  a.debug_fault = 0;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  return run_fwd(a, dev, stream);
}

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Skv, int D, int causal, float scale, int dtype,
             cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Skv < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq * Sq == 0) return ATTN_OK;  // nothing to compute
  if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (((long long)Sq + 255) / 256 * Hq * B > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (!q || !o || (Skv > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
      (lse && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  int st = check_device(&dev);
  if (st != ATTN_OK) return st;

  ea::FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Skv = Skv;
  a.D = D;
  a.causal = causal != 0;
  a.scale = scale;
  a.bf16 = dtype == ATTN_BF16;
  a.wait_limit_ns = g_wait_limit_ns;
  a.debug_fault = g_fault;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  if (Skv == 0) return from_cuda(ea::launch_fwd_empty_keys(a, stream));
  return run_fwd(a, dev, stream);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int D, int causal,
                    int window_left, int window_right, float scale, int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || Hq < 0 || Hkv < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
      max_seqlen_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Hq == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_OK;  // no query row
  if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!q || !o || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
      (lse && !aligned(lse, 4)) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return ATTN_ERR_INVALID_ARG;
  ea::FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.causal = causal != 0;
  a.scale = scale;
  a.bf16 = dtype == ATTN_BF16;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.total_q = total_q;
  a.total_k = total_k;
  a.q_rstride = (long long)Hq * D;
  a.k_rstride = (long long)Hkv * D;
  a.o_rstride = (long long)Hq * D;
  return run_fwd_tm(a, max_seqlen_q, max_seqlen_k, window_left, window_right, stream);
}

int attn_fwd_qkvpacked(const void* qkv, void* o, float* lse, int B, int S, int H, int D, int causal,
                       int window_left, int window_right, float scale, int dtype,
                       cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || S < 0 || H < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * S * H == 0) return ATTN_OK;
  if (B > 65535 || H > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * S > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (!qkv || !o || !aligned(qkv, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  const size_t plane = (size_t)H * D;  // elements of one of Q, K, V of one token
  ea::FwdArgs a{};
  a.q = qkv;
  a.k = static_cast<const uint16_t*>(qkv) + plane;
  a.v = static_cast<const uint16_t*>(qkv) + 2 * plane;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = H;
  a.Hkv = H;
  a.D = D;
  a.causal = causal != 0;
  a.scale = scale;
  a.bf16 = dtype == ATTN_BF16;
  a.cu_q = nullptr;  // sequence b starts at token b * S
  a.cu_k = nullptr;
  a.total_q = B * S;
  a.total_k = B * S;
  a.q_rstride = 3 * (long long)plane;
  a.k_rstride = 3 * (long long)plane;
  a.o_rstride = (long long)plane;
  return run_fwd_tm(a, S, S, window_left, window_right, stream);
}

}  // extern "C"

// The backward's row-term workspace from the library pool, stream-ordered around the
// kernels.  rows: (query token, head) pairs.
static int run_bwd(ea::BwdArgs& a, int dev, size_t rows, cudaStream_t stream) {
  int st;
  void* ws = nullptr;
  cudaMemPool_t pool;
  if ((st = pool_for(dev, &pool)) != ATTN_OK) return st;
  // the row terms, then (16-byte aligned) the two work-item counters
  const size_t vec_bytes = (rows * sizeof(float) + 15) / 16 * 16;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, rows * sizeof(float) + 256, pool, stream);
  if (e != cudaSuccess) return from_cuda(e);
  a.delta = static_cast<float*>(ws);
  a.work_counter = reinterpret_cast<int*>(static_cast<char*>(ws) + vec_bytes);
  e = ea::launch_bwd(a, stream);
  cudaError_t f = cudaFreeAsync(ws, stream);
  if (e == cudaSuccess) e = f;
  if (e == cudaErrorInvalidValue && !ea::encode_tiled_fn()) return ATTN_ERR_UNSUPPORTED;
  return from_cuda(e);
}

// Token-major backward (attn_bwd_varlen, attn_bwd_qkvpacked): the checks of the
// window and the longest lengths, then the launch.
static int run_bwd_tm(ea::BwdArgs& a, int max_q, int max_k, int window_left, int window_right,
                      cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return ATTN_ERR_INVALID_ARG;
  if (!isfinite(a.scale)) return ATTN_ERR_INVALID_ARG;
  if ((long long)max_q + max_k > 0x3fffffffLL) return ATTN_ERR_UNSUPPORTED;
  int dev = 0;
  int st = check_device(&dev);
  if (st != ATTN_OK) return st;
  a.vl = 1;
  a.Sq = max_q;
  a.Skv = max_k;
  // a bound at least max_q + max_k away from every diagonal excludes no key
  a.win_left = window_left > max_q + max_k ? -1 : window_left;
  a.win_right = window_right > max_q + max_k ? -1 : window_right;
  a.wait_limit_ns = g_wait_limit_ns;
  a.debug_fault = 0;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  return run_bwd(a, dev, (size_t)a.total_q * a.Hq, stream);
}

extern "C" {

size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq, int D) {
  if (B < 0 || Hq < 0 || Sq < 0 || D <= 0) return 0;
  const size_t rows = (size_t)B * Hq * Sq;
  return rows * sizeof(float) + 256;  // row terms, then (16-byte aligned) two work counters
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Skv,
             int D, int causal, float scale, int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Skv < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Hq == 0 || (Sq == 0 && Skv == 0)) return ATTN_OK;  // nothing to compute
  if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hkv > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (Sq > 0 && (!q || !o || !lse || !dout || !dq)) return ATTN_ERR_INVALID_ARG;
  if (Skv > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_INVALID_ARG;
  const void* a16[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* ptr : a16)
    if (ptr && !aligned(ptr, 16)) return ATTN_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  int st = check_device(&dev);
  if (st != ATTN_OK) return st;

  ea::BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Skv = Skv;
  a.D = D;
  a.causal = causal != 0;
  a.scale = scale;
  a.bf16 = dtype == ATTN_BF16;
  a.wait_limit_ns = g_wait_limit_ns;
  a.debug_fault = g_fault;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  a.win_left = -1;
  a.win_right = -1;
  const size_t rows = (size_t)B * Hq * Sq;
  if (Skv == 0) {
    // no key: O was 0 whatever Q, K, V were, so every gradient is 0 (dK, dV are empty)
    cudaError_t e = cudaMemsetAsync(dq, 0, rows * D * 2, stream);
    return from_cuda(e);
  }
  return run_bwd(a, dev, rows, stream);
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k,
                    int max_seqlen_q, int max_seqlen_k, int D, int causal, int window_left,
                    int window_right, float scale, int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || Hq < 0 || Hkv < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
      max_seqlen_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Hq == 0 || ((total_q == 0 || max_seqlen_q == 0) && (total_k == 0 || max_seqlen_k == 0)))
    return ATTN_OK;  // no query and no key: nothing to compute
  if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!cu_seqlens_q || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
  if (total_q > 0 && (!q || !o || !lse || !dout || !dq)) return ATTN_ERR_INVALID_ARG;
  if (total_k > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_INVALID_ARG;
  const void* a16[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* ptr : a16)
    if (ptr && !aligned(ptr, 16)) return ATTN_ERR_INVALID_ARG;
  if ((lse && !aligned(lse, 4)) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return ATTN_ERR_INVALID_ARG;
  ea::BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.causal = causal != 0;
  a.scale = scale;
  a.bf16 = dtype == ATTN_BF16;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.total_q = total_q;
  a.total_k = total_k;
  a.q_rstride = a.do_rstride = a.dq_rstride = (long long)Hq * D;
  a.k_rstride = a.dk_rstride = (long long)Hkv * D;
  return run_bwd_tm(a, max_seqlen_q, max_seqlen_k, window_left, window_right, stream);
}

int attn_bwd_qkvpacked(const void* qkv, const void* o, const float* lse, const void* dout, void* dqkv,
                       int B, int S, int H, int D, int causal, int window_left, int window_right,
                       float scale, int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || S < 0 || H < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * S * H == 0) return ATTN_OK;
  if (B > 65535 || H > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * S > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (!qkv || !o || !lse || !dout || !dqkv) return ATTN_ERR_INVALID_ARG;
  if (!aligned(qkv, 16) || !aligned(o, 16) || !aligned(dout, 16) || !aligned(dqkv, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  const size_t plane = (size_t)H * D;  // elements of one of Q, K, V of one token
  ea::BwdArgs a{};
  a.q = qkv;
  a.k = static_cast<const uint16_t*>(qkv) + plane;
  a.v = static_cast<const uint16_t*>(qkv) + 2 * plane;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dqkv;
  a.dk = static_cast<uint16_t*>(dqkv) + plane;
  a.dv = static_cast<uint16_t*>(dqkv) + 2 * plane;
  a.B = B;
  a.Hq = H;
  a.Hkv = H;
  a.D = D;
  a.causal = causal != 0;
  a.scale = scale;
  a.bf16 = dtype == ATTN_BF16;
  a.cu_q = nullptr;  // sequence b starts at token b * S
  a.cu_k = nullptr;
  a.total_q = B * S;
  a.total_k = B * S;
  a.q_rstride = a.k_rstride = a.dq_rstride = a.dk_rstride = 3 * (long long)plane;
  a.do_rstride = (long long)plane;
  return run_bwd_tm(a, S, S, window_left, window_right, stream);
}

int attn_decode_chunk(int max_S, int num_splits) { return chunk_for(max_S, num_splits); }

size_t attn_decode_workspace_bytes(int B, int Hq, int max_S, int D, int num_splits) {
  if (B < 0 || Hq < 0 || max_S < 0 || D <= 0 || num_splits < 0) return 0;
  const int chunk = chunk_for(max_S, num_splits);
  const size_t max_chunks = chunk > 0 ? ((size_t)max_S + chunk - 1) / chunk : 0;
  return (size_t)B * Hq * max_chunks * (D + 2) * sizeof(float);
}

// Partials workspace from the library pool, stream-ordered around the two kernels.
static int decode_with_pool(ea::DecodeArgs& a, int dev, size_t bytes, cudaStream_t stream) {
  void* ws = nullptr;
  if (bytes > 0) {
    cudaMemPool_t pool;
    const int st = pool_for(dev, &pool);
    if (st != ATTN_OK) return st;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  a.partials = static_cast<float*>(ws);
  cudaError_t e = ea::launch_decode(a, stream);
  if (ws) {
    cudaError_t f = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

// Checks of the contiguous-cache decode entry points that need no CUDA call,
// and their arguments.  Returns ATTN_OK with *empty set when B * Hq == 0.
static int decode_contiguous_args(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* seq_lens, void* o, int B, int Hq, int Hkv,
                                  int max_S, int D, int num_splits, int dtype, ea::DecodeArgs* a,
                                  bool* empty) {
  *empty = false;
  if (B < 0 || Hq < 0 || Hkv < 0 || max_S < 0 || num_splits < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hkv > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!q || !o || !seq_lens || (max_S > 0 && (!k_cache || !v_cache))) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(seq_lens, 4) ||
      (k_cache && !aligned(k_cache, 16)) || (v_cache && !aligned(v_cache, 16)))
    return ATTN_ERR_INVALID_ARG;
  *a = ea::DecodeArgs{};
  a->q = q;
  a->k = k_cache;
  a->v = v_cache;
  a->seq_lens = seq_lens;
  a->o = o;
  a->B = B;
  a->Hq = Hq;
  a->Hkv = Hkv;
  a->max_S = max_S;
  a->D = D;
  a->chunk = chunk_for(max_S, num_splits);
  a->max_chunks = max_S > 0 ? (max_S + a->chunk - 1) / a->chunk : 0;
  // the split kernel numbers its (chunk, head group, sequence) items with an int
  if ((long long)B * Hq * a->max_chunks > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  a->scale = 1.0f / sqrtf((float)D);
  a->bf16 = dtype == ATTN_BF16;
  a->wait_limit_ns = g_wait_limit_ns;
  a->debug_fault = g_fault;
  return ATTN_OK;
}

int attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                void* o, int B, int Hq, int Hkv, int max_S, int D, int num_splits, int dtype,
                cudaStream_t stream) {
  NvtxRange range_(__func__);
  ea::DecodeArgs a;
  bool empty;
  int st = decode_contiguous_args(q, k_cache, v_cache, seq_lens, o, B, Hq, Hkv, max_S, D,
                                  num_splits, dtype, &a, &empty);
  if (st != ATTN_OK || empty) return st;
  int dev = 0;
  if ((st = check_device(&dev)) != ATTN_OK) return st;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  return decode_with_pool(a, dev, attn_decode_workspace_bytes(B, Hq, max_S, D, num_splits), stream);
}

int attn_decode_fused(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* seq_lens, void* o, int B, int Hq, int Hkv, int max_S, int D,
                      int num_splits, int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  ea::DecodeArgs a;
  bool empty;
  int st = decode_contiguous_args(q, k_cache, v_cache, seq_lens, o, B, Hq, Hkv, max_S, D,
                                  num_splits, dtype, &a, &empty);
  if (st != ATTN_OK || empty) return st;
  if ((size_t)B * Hq > ea::kDecodeTickets) return ATTN_ERR_UNSUPPORTED;
  int dev = 0;
  if ((st = check_device(&dev)) != ATTN_OK) return st;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  cudaError_t e = ea::decode_tickets(dev, &a.tickets, stream);
  if (e != cudaSuccess) return from_cuda(e);
  return decode_with_pool(a, dev, attn_decode_workspace_bytes(B, Hq, max_S, D, num_splits), stream);
}

int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* block_table, const int32_t* seq_lens, void* o, int B, int Hq,
                      int Hkv, int num_pages, int page_size, int max_pages, int D, int num_splits,
                      int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  if (B < 0 || Hq < 0 || Hkv < 0 || num_pages < 0 || page_size < 1 || max_pages < 0 || num_splits < 0)
    return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)max_pages * page_size > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const int max_S = max_pages * page_size;  // logical positions per sequence
  if ((long long)B * Hq == 0) return ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hkv > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!q || !o || !seq_lens) return ATTN_ERR_INVALID_ARG;
  if (max_S > 0 && (!k_pages || !v_pages || !block_table || num_pages == 0)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(seq_lens, 4) ||
      (k_pages && !aligned(k_pages, 16)) || (v_pages && !aligned(v_pages, 16)) ||
      (block_table && !aligned(block_table, 4)))
    return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  int st = check_device(&dev);
  if (st != ATTN_OK) return st;

  ea::DecodeArgs a{};
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.seq_lens = seq_lens;
  a.o = o;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.max_S = max_S;
  a.D = D;
  a.chunk = chunk_for(max_S, num_splits);
  a.max_chunks = max_S > 0 ? (max_S + a.chunk - 1) / a.chunk : 0;
  if ((long long)B * Hq * a.max_chunks > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  a.scale = 1.0f / sqrtf((float)D);
  a.bf16 = dtype == ATTN_BF16;
  a.wait_limit_ns = g_wait_limit_ns;
  a.debug_fault = g_fault;
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  a.block_table = max_S > 0 ? block_table : nullptr;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  return decode_with_pool(a, dev, attn_decode_workspace_bytes(B, Hq, max_S, D, num_splits), stream);
}

int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seq_lens, void* o, int B, int Hq, int Hkv, int max_S, int D,
                        int num_splits, int dtype, cudaStream_t stream) {
  NvtxRange range_(__func__);
  ea::DecodeArgs a;
  bool empty;
  int st = decode_contiguous_args(q, k_cache, v_cache, seq_lens, o, B, Hq, Hkv, max_S, D,
                                  num_splits, dtype, &a, &empty);
  if (st != ATTN_OK || empty) return st;
  // the partials must fit the fixed scratch: larger problems are refused, never allocated
  const size_t bytes = attn_decode_workspace_bytes(B, Hq, max_S, D, num_splits);
  if (bytes > ea::kNoallocPartialsBytes) return ATTN_ERR_UNSUPPORTED;
  int dev = 0;
  if ((st = check_device(&dev)) != ATTN_OK) return st;
  cudaError_t e = ea::noalloc_partials(dev, &a.partials);
  if (e != cudaSuccess) return from_cuda(e);
  a.num_sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 1;
  return from_cuda(ea::launch_decode(a, stream));
}

int attn_check_device_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return from_cuda(e);
  unsigned f = 0, d = 0, g = 0;
  if ((e = ea::read_fwd_status(&f, stream)) != cudaSuccess) return from_cuda(e);
  if ((e = ea::read_decode_status(&d, stream)) != cudaSuccess) return from_cuda(e);
  if ((e = ea::read_bwd_status(&g, stream)) != cudaSuccess) return from_cuda(e);
  const unsigned all = f | d | g;
  if (all & 1u) return ATTN_ERR_DEVICE_TIMEOUT;
  if (all & 6u) return ATTN_ERR_INVALID_ARG;  // a seq_len clamped, a page index replaced
  return ATTN_OK;
}

int attn_debug_set(int fault, unsigned wait_limit_us) {
  if (fault < 0 || fault > 3) return ATTN_ERR_INVALID_ARG;
  g_fault = fault;
  g_wait_limit_ns = wait_limit_us ? (uint64_t)wait_limit_us * 1000ull : kDefaultWaitNs;
  return ATTN_OK;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int attn_version(void) { return kVersion; }

}  // extern "C"
