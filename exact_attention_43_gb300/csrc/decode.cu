// Flash-decoding: one query token per (sequence, query head) against a KV cache,
// split over chunks of the sequence and merged by an LSE-rescaling reduce.
//
// What is computed follows aprender-gpu reduce_kernel.rs
// (FlashDecodingReduceKernel): each chunk c of sequence b stores a partial
// [o_c (D floats), m_c, l_c] with o_c unnormalised (sum of e^(s - m_c) v),
// m_c the chunk's max scaled score (natural log units) and l_c its exp-sum,
// in a [B, Hq, max_chunks, D + 2] fp32 buffer; the reduce takes
// M = max_c m_c and returns sum_c o_c e^(m_c - M) / sum_c l_c e^(m_c - M),
// skipping empty chunks.  The single-query role, the GQA head mapping and the
// scale 1/sqrt(D) are those of abaddon attention.rs (flash_attention_cached_f16,
// FlashAttentionKernel::forward_cached).
//
// GB300 design: the split kernel is bandwidth-bound (about 4 flops per cache
// byte), so it moves K/V with contiguous bulk copies (cp.async.bulk, a chunk's
// rows of one KV head are contiguous) through a 3-stage shared-memory ring of
// 128-key sub-tiles (32 KB each; 2 CTAs per SM)
// and reads every byte once for all query heads of the GQA group: the group's
// query vectors live in registers, scores are formed with 8 lanes per key
// (16-byte loads, 3 shuffle levels), the online max/sum run per 128-key
// sub-tile, and P V uses one lane per 4 output columns.  No tensor cores: the
// contraction is too thin to pay for them and the bound is HBM.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

#include <mutex>

namespace ea {
namespace dec {

__device__ unsigned g_status;

constexpr int SUB = 128;       // keys per staged sub-tile (a multiple of 32)
constexpr int NST = 3;         // ring stages (each holds a K or a V sub-tile)
constexpr int THREADS = 256;   // 8 warps
constexpr int WARPS = THREADS / 32;
constexpr int KEYS_PER_WARP = SUB / WARPS;  // 16

struct Params {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* seq_lens;
  float* part;
  uint16_t* o;
  int Hq, Hkv, max_S, chunk, max_chunks, group, heads_per_cta;
  float c2;  // scale * log2(e)
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ int clamp_len(const Params& p, int b) {
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_S) {
    L = L < 0 ? 0 : p.max_S;
    if (threadIdx.x == 0) atomicOr(&g_status, kStatusSeqLenClamped);
  }
  return L;
}

template <int D, int G>
struct SplitLayout {
  static constexpr int STAGE = SUB * D * 2;
  static constexpr int RING_OFF = 0;
  static constexpr int SC_OFF = RING_OFF + NST * STAGE;      // scores / probabilities [SUB][G]
  static constexpr int STAT_OFF = SC_OFF + SUB * G * 4;      // m, l, alpha per head
  static constexpr int BAR_OFF = (STAT_OFF + 3 * G * 4 + 15) / 16 * 16;  // NST barriers
  static constexpr int ABORT_OFF = BAR_OFF + NST * 8;
  static constexpr int BYTES = ABORT_OFF + 16;
  static_assert(WARPS * G * D * 4 <= NST * STAGE, "cross-warp reduction aliases the ring");
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(STAGE % 16 == 0 && RING_OFF % 16 == 0, "bulk copies need 16-byte alignment");
};

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(THREADS) decode_split_kernel(const Params p) {
  using L = SplitLayout<D, G>;
  constexpr int EPL = D / 8;   // key elements per lane when 8 lanes share a key
  constexpr int DPL = D / 32;  // output columns per lane in P V
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  float* sc = reinterpret_cast<float*>(smem + L::SC_OFF);
  float* m_run = reinterpret_cast<float*>(smem + L::STAT_OFF);
  float* l_run = m_run + G;
  float* alpha_s = l_run + G;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT_OFF);

  const int c = blockIdx.x;
  const int kvh = blockIdx.y / (p.group / G);
  const int h0 = kvh * p.group + (blockIdx.y % (p.group / G)) * G;  // first query head of this CTA
  const int b = blockIdx.z;
  const int len = clamp_len(p, b);
  const int n_chunks = (len + p.chunk - 1) / p.chunk;
  if (c >= n_chunks) return;
  const int k0 = c * p.chunk;
  const int n = min(p.chunk, len - k0);
  const int nsub = (n + SUB - 1) / SUB;
  const int nload = 2 * nsub;  // K_0, V_0, K_1, V_1, ...
  const size_t row0 = ((size_t)b * p.Hkv + kvh) * p.max_S + k0;
  const uint16_t* kg = p.k + row0 * D;
  const uint16_t* vg = p.v + row0 * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int issued = 0;  // loads issued so far (thread 0 only)
  auto issue = [&](int i, uint64_t pol) {  // called by thread 0 only, in increasing i
    const int st = i % NST;
    issued = i + 1;
    const int sub = i >> 1;
    const int rows = min(SUB, n - sub * SUB);
    const uint16_t* src = ((i & 1) ? vg : kg) + (size_t)sub * SUB * D;
    const uint32_t bar = sb + L::BAR_OFF + 8 * st;
    mbar_expect_tx(bar, rows * D * 2);
    bulk_load(sb + L::RING_OFF + st * L::STAGE, src, rows * D * 2, bar, pol);
  };

  uint64_t pol = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(sb + L::BAR_OFF + 8 * i, 1);
    *abort_flag = 0;
    fence_barrier_init();
    pol = policy_evict_first();
    for (int i = 0; i < min(NST, nload); ++i) issue(i, pol);
  }
  if (threadIdx.x < G) {
    m_run[threadIdx.x] = -INFINITY;
    l_run[threadIdx.x] = 0.f;
  }

  // query vectors of the group, pre-multiplied by scale * log2 e, for this lane's key slice
  // (8 lanes share a key; lane slice s owns elements [8 (8 v + s), 8 (8 v + s) + 8) for v < D / 64)
  const int slice = lane & 7;
  float qr[G][EPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4* qs = reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.Hq + h0 + g) * D);
#pragma unroll
    for (int v4 = 0; v4 < EPL / 8; ++v4) {
      const uint4 w = qs[v4 * 8 + slice];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<BF16>(ws[i]);
        qr[g][v4 * 8 + 2 * i] = f.x * p.c2;
        qr[g][v4 * 8 + 2 * i + 1] = f.y * p.c2;
      }
    }
  }
  float acc[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[g][e] = 0.f;
  __syncthreads();

  bool ok = true;
  for (int sub = 0; sub < nsub && ok; ++sub) {
    const int rows = min(SUB, n - sub * SUB);
    // ---------------------------------------------------------------- scores
    {
      const int i = 2 * sub, st = i % NST;
      ok = mbar_wait(sb + L::BAR_OFF + 8 * st, (i / NST) & 1, abort_flag, &g_status, p.wait_limit_ns);
      if (__syncthreads_or(!ok)) { ok = false; break; }
      const uint8_t* tile = smem + L::RING_OFF + st * L::STAGE;
#pragma unroll
      for (int step = 0; step < KEYS_PER_WARP / 4; ++step) {
        const int key = warp * KEYS_PER_WARP + step * 4 + (lane >> 3);
        float dot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) dot[g] = 0.f;
        if (key < rows) {
          // lane slice s reads 16-byte chunks s, s + 8, ...: a quarter-warp covers 128
          // contiguous bytes of one row, so the loads are free of bank conflicts
          const uint4* kr = reinterpret_cast<const uint4*>(tile + key * D * 2);
#pragma unroll
          for (int v4 = 0; v4 < EPL / 8; ++v4) {
            const uint4 w = kr[v4 * 8 + slice];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
              const float2 f = unpack2<BF16>(ws[i2]);
#pragma unroll
              for (int g = 0; g < G; ++g)
                dot[g] = fmaf(qr[g][v4 * 8 + 2 * i2], f.x, fmaf(qr[g][v4 * 8 + 2 * i2 + 1], f.y, dot[g]));
            }
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 1);
          dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 2);
          dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 4);
        }
        if (slice == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) sc[key * G + g] = key < rows ? dot[g] : -INFINITY;
        }
      }
      __syncthreads();  // scores visible; every read of this stage done
      if (threadIdx.x == 0 && i + NST < nload) issue(i + NST, pol);
      // online max / sum per head over this sub-tile (log2 units), one warp per head
      for (int g = warp; g < G; g += WARPS) {
        constexpr int PER_LANE = SUB / 32;
        float sv[PER_LANE];
#pragma unroll
        for (int u = 0; u < PER_LANE; ++u) sv[u] = sc[(lane + 32 * u) * G + g];
        float mx = sv[0];
#pragma unroll
        for (int u = 1; u < PER_LANE; ++u) mx = fmaxf(mx, sv[u]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = m_run[g];
        const float m_new = fmaxf(m_old, mx);  // finite: key 0 of the sub-tile is valid
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < PER_LANE; ++u) {
          const float e = ex2(sv[u] - m_new);
          sc[(lane + 32 * u) * G + g] = e;
          sum += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        __syncwarp();
        if (lane == 0) {
          const float alpha = ex2(m_old - m_new);  // 0 on the first sub-tile
          alpha_s[g] = alpha;
          l_run[g] = l_run[g] * alpha + sum;
          m_run[g] = m_new;
        }
      }
      __syncthreads();
    }
    // ---------------------------------------------------------------- P V
    {
      const int i = 2 * sub + 1, st = i % NST;
      ok = mbar_wait(sb + L::BAR_OFF + 8 * st, (i / NST) & 1, abort_flag, &g_status, p.wait_limit_ns);
      if (__syncthreads_or(!ok)) { ok = false; break; }
      const uint8_t* tile = smem + L::RING_OFF + st * L::STAGE;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float a = alpha_s[g];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[g][e] *= a;
      }
#pragma unroll
      for (int kk = 0; kk < KEYS_PER_WARP; ++kk) {
        const int key = warp * KEYS_PER_WARP + kk;
        if (key < rows) {
          float vv[DPL];
          if constexpr (DPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(tile + key * D * 2 + lane * 8);
            const float2 f0 = unpack2<BF16>(w.x), f1 = unpack2<BF16>(w.y);
            vv[0] = f0.x; vv[1] = f0.y; vv[2] = f1.x; vv[3] = f1.y;
          } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + key * D * 2 + lane * 4);
            const float2 f0 = unpack2<BF16>(w);
            vv[0] = f0.x; vv[1] = f0.y;
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pr = sc[key * G + g];
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(pr, vv[e], acc[g][e]);
          }
        }
      }
      __syncthreads();  // every read of this stage done
      if (threadIdx.x == 0 && i + NST < nload) issue(i + NST, pol);
    }
  }

  if (!ok) {
    // unwind: wait (bounded) for the copies still in flight, then leave
    if (threadIdx.x == 0) {
      const uint64_t t0 = global_timer_ns();
      for (int i = max(0, issued - NST); i < issued; ++i) {
        const uint32_t bar = sb + L::BAR_OFF + 8 * (i % NST);
        while (!mbar_try_wait(bar, (i / NST) & 1)) {
          if (global_timer_ns() - t0 > p.wait_limit_ns) break;
        }
      }
    }
    __syncthreads();
    return;
  }

  // cross-warp sum of the P V partials (aliases the ring: every copy has been consumed)
  float* red = reinterpret_cast<float*>(smem + L::RING_OFF);
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < DPL; ++e) red[(warp * G + g) * D + lane * DPL + e] = acc[g][e];
  __syncthreads();
  const size_t pbase = (((size_t)b * p.Hq + h0) * p.max_chunks + c) * (D + 2);
  const size_t hstride = (size_t)p.max_chunks * (D + 2);
  for (int idx = threadIdx.x; idx < G * D; idx += THREADS) {
    const int g = idx / D, d = idx % D;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) s += red[(w * G + g) * D + d];
    p.part[pbase + g * hstride + d] = s;
  }
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    p.part[pbase + g * hstride + D] = m_run[g] * 0.69314718055994531f;  // natural-log units
    p.part[pbase + g * hstride + D + 1] = l_run[g];
  }
}

// One warp per (query head, sequence): M = max_c m_c, then the rescaled sums.
template <int D, bool BF16>
__global__ void __launch_bounds__(32) decode_reduce_kernel(const Params p) {
  constexpr int DPL = D / 32;
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const int len = clamp_len(p, b);
  const int n = (len + p.chunk - 1) / p.chunk;
  const float* base = p.part + ((size_t)b * p.Hq + h) * p.max_chunks * (D + 2);
  float M = -INFINITY;
  for (int c = lane; c < n; c += 32) M = fmaxf(M, base[(size_t)c * (D + 2) + D]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float total = 0.f;
  for (int c = 0; c < n; ++c) {
    const float* pc = base + (size_t)c * (D + 2);
    const float m_c = pc[D];
    if (!(m_c > -1e30f)) continue;  // empty chunk
    const float w = ex2((m_c - M) * 1.4426950408889634f);
    total = fmaf(pc[D + 1], w, total);
    if constexpr (DPL == 4) {
      const float2 a = *reinterpret_cast<const float2*>(pc + lane * 4);
      const float2 bb = *reinterpret_cast<const float2*>(pc + lane * 4 + 2);
      acc[0] = fmaf(a.x, w, acc[0]);
      acc[1] = fmaf(a.y, w, acc[1]);
      acc[2] = fmaf(bb.x, w, acc[2]);
      acc[3] = fmaf(bb.y, w, acc[3]);
    } else {
      const float2 a = *reinterpret_cast<const float2*>(pc + lane * 2);
      acc[0] = fmaf(a.x, w, acc[0]);
      acc[1] = fmaf(a.y, w, acc[1]);
    }
  }
  const float inv = total > 0.f ? 1.f / total : 0.f;  // no chunk (len 0): O = 0
  uint16_t* out = p.o + ((size_t)b * p.Hq + h) * D + lane * DPL;
  if constexpr (DPL == 4) {
    *reinterpret_cast<uint2*>(out) = make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv),
                                                pack2<BF16>(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(out) = pack2<BF16>(acc[0] * inv, acc[1] * inv);
  }
}

template <int D, int G, bool BF16>
static cudaError_t launch_t(const DecodeArgs& a, const Params& p, cudaStream_t stream) {
  using L = SplitLayout<D, G>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G, BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  if (e != cudaSuccess) return e;
  if (a.max_chunks > 0) {
    dim3 grid(a.max_chunks, a.Hkv * (p.group / G), a.B);
    decode_split_kernel<D, G, BF16><<<grid, THREADS, L::BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  decode_reduce_kernel<D, BF16><<<dim3(a.Hq, a.B), 32, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_d(const DecodeArgs& a, Params& p, cudaStream_t stream) {
  const int G = p.group;
  // heads per CTA: the largest of 8, 4, 2, 1 dividing the group
  p.heads_per_cta = (G % 8 == 0) ? 8 : (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
  switch (p.heads_per_cta) {
    case 8: return launch_t<D, 8, BF16>(a, p, stream);
    case 4: return launch_t<D, 4, BF16>(a, p, stream);
    case 2: return launch_t<D, 2, BF16>(a, p, stream);
    default: return launch_t<D, 1, BF16>(a, p, stream);
  }
}

}  // namespace dec

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  dec::Params p{};
  p.q = static_cast<const uint16_t*>(a.q);
  p.k = static_cast<const uint16_t*>(a.k);
  p.v = static_cast<const uint16_t*>(a.v);
  p.seq_lens = a.seq_lens;
  p.part = a.partials;
  p.o = static_cast<uint16_t*>(a.o);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.max_S = a.max_S;
  p.chunk = a.chunk;
  p.max_chunks = a.max_chunks;
  p.group = a.Hq / a.Hkv;
  p.c2 = a.scale * 1.4426950408889634f;
  p.wait_limit_ns = a.wait_limit_ns;
  if (a.D == 64) return a.bf16 ? dec::launch_d<64, true>(a, p, stream) : dec::launch_d<64, false>(a, p, stream);
  return a.bf16 ? dec::launch_d<128, true>(a, p, stream) : dec::launch_d<128, false>(a, p, stream);
}

// ---------------------------------------------------------------------------
// Fixed scratch for attn_decode_noalloc: the chunk partials live in this
// file-scope device array instead of memory allocated per call.  Its size is
// fixed at build time and every device that loads the library keeps it for the
// life of the process.  All calls share it: two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) overwrite each other's
// partials.  Nothing in it has to start at zero: each call's split kernel
// writes every partial that the same call's reduce kernel reads.
static __device__ __align__(256) float g_noalloc_partials[kNoallocPartialsBytes / sizeof(float)];

namespace {
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[64];  // device address of the array, per device ordinal
}  // namespace

cudaError_t noalloc_partials(int device, float** out) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[device]) {
    // On the host, g_noalloc_partials names a host-side stand-in, not device
    // memory: the kernels must be given the address the runtime reports for
    // the current device.
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_partials);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[device] = static_cast<float*>(ptr);
  }
  *out = g_noalloc_ptr[device];
  return cudaSuccess;
}

cudaError_t read_decode_status(unsigned* out, cudaStream_t stream) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, dec::g_status, sizeof(unsigned), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(dec::g_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace ea
