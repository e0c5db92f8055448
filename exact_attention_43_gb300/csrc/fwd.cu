// Prefill: fused exact attention O = softmax(scale * Q K^T [+ causal mask]) V
// with the per-row log-sum-exp, for sm_103a.
//
// What is computed follows the pages' algorithm (abaddon attention.rs, module
// doc "Algorithm": load a Q tile, for each K/V tile form S = Q K^T, mask,
// update the running max and sum, rescale and accumulate O += P V, divide by
// the sum at the end; rustytorch flash_attention_forward.cu,
// OnlineSoftmaxState: LSE = m + log(l)).  How it is computed is GB300-native:
//
//  * one CTA owns a 128-row Q tile of one (batch, query head); KV head =
//    query head / (Hq / Hkv) (abaddon flash_attention_f16, GQA mapping);
//  * warp 4 streams Q once and K/V 128-key tiles through two-stage rings with
//    TMA (3-D tensor maps, 128-byte swizzle, mbarrier transaction counts);
//  * warp 5 issues tcgen05.mma: S_t = Q K_t^T into one of two TMEM buffers,
//    then O += P_t V_t with P read from TMEM and V from shared memory;
//  * warps 0-3 own one query row per thread (TMEM lane = row): load S_t,
//    mask, row max, exponentiate with exp2 (scale * log2 e folded into one
//    FMA), accumulate the row sum, write P_t (16-bit) to TMEM, and rescale the
//    O row in TMEM only when the running max grew by more than 2^8 (exact:
//    O and l always share the same stale max);
//  * causal: KV tiles wholly after the tile's last query row are never
//    loaded (abaddon flash_attention_f16, causal `break`); only tiles that
//    cross the diagonal or the end of the keys are masked element-wise.
//    Causal alignment is bottom-right: key j is visible to row i iff
//    j <= i + (Skv - Sq);
//  * epilogue: O / l rounded to the input dtype, LSE = ln 2 * (m + log2 l);
//    a row with no visible key gets O = 0, LSE = -inf.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace ea {
namespace fwd {

__device__ unsigned g_status;

constexpr int BM = 128;            // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;            // keys per KV tile
constexpr int NUM_THREADS = 192;   // warps 0-3 softmax/epilogue, 4 loader, 5 MMA
constexpr int LOADER_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr float RESCALE_LOG2 = 8.0f;  // rescale O when the max grows by more than 2^8
constexpr uint32_t TMEM_COLS = 512;
// TMEM column map (fp32 columns): S double buffer, O accumulator, P double buffer
constexpr uint32_t COL_S = 0;      // S_0 [0,128), S_1 [128,256)
constexpr uint32_t COL_O = 256;    // O   [256, 256 + D)
constexpr uint32_t COL_P = 384;    // P_0 [384,448), P_1 [448,512): 128 16-bit values packed in 64 columns

struct Params {
  void* o;
  float* lse;
  int Hq, Hkv, Sq, Skv, group, num_m_tiles, causal, neg, zero;
  float c2;  // scale * log2(e); 1 when scale == 0 (then every visible score is set to 0)
  uint64_t wait_limit_ns;
  int debug_fault;
};

template <int D>
struct Layout {
  static constexpr int REGION = 128 * 128;  // one 128-row x 128-byte swizzle region (64 columns)
  static constexpr int NREG = D / 64;
  static constexpr int TILE = NREG * REGION;  // a 128 x D 16-bit tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;
  static constexpr int V_OFF = K_OFF + 2 * TILE;
  static constexpr int BAR_OFF = V_OFF + 2 * TILE;
  enum {
    Q_FULL, K_FULL, K_EMPTY = K_FULL + 2, V_FULL = K_EMPTY + 2, V_EMPTY = V_FULL + 2,
    S_FULL = V_EMPTY + 2, P_FULL = S_FULL + 2, O_DONE = P_FULL + 2, DRAIN = O_DONE + 2, NUM_BARS
  };
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 bytes
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(REGION % 1024 == 0 && K_OFF % 1024 == 0 && V_OFF % 1024 == 0,
                "128-byte-swizzled tiles need 1024-byte alignment");
};

// Wait with no abort short-cut: used only while unwinding, for copies and MMAs in flight.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(&g_status, kStatusTimeout);
      return;
    }
  }
}

template <int D, bool BF16>
__device__ __forceinline__ void store_row(const Params& p, int bh, int row, float inv_l,
                                          uint32_t o_taddr) {
  using T = uint4;
  T* dst = reinterpret_cast<T*>(static_cast<uint16_t*>(p.o) + ((size_t)bh * p.Sq + row) * D);
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(o_taddr + c * 32, r);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
    if (row < p.Sq) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[c * 4 + i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const Params p) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = p.num_m_tiles - 1 - (int)blockIdx.x;  // longest causal rows first
  const int hq = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.Hq + hq;
  const int kvh = hq / p.group;
  const int m0 = mt * BM;
  const int last_row = min(m0 + BM, p.Sq) - 1;
  const int delta = p.Skv - p.Sq;
  int n_keys = p.Skv;
  if (p.causal) n_keys = max(0, min(p.Skv, last_row + delta + 1));
  const int n_tiles = (n_keys + BN - 1) / BN;
  // first KV tile whose keys may be invisible to some row of this tile
  int mask_from = p.Skv / BN;
  if (p.causal) mask_from = min(mask_from, max(0, m0 + delta + 1) / BN);

  if (n_tiles == 0) {  // no row of this tile sees a key: O = 0, LSE = -inf
    if (threadIdx.x < BM) {
      const int row = m0 + threadIdx.x;
      if (row < p.Sq) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)bh * p.Sq + row) * D);
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        if (p.lse) p.lse[(size_t)bh * p.Sq + row] = -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(L::Q_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::K_FULL + i), 1);
      mbar_init(bar(L::K_EMPTY + i), 1);
      mbar_init(bar(L::V_FULL + i), 1);
      mbar_init(bar(L::V_EMPTY + i), 1);
      mbar_init(bar(L::S_FULL + i), 1);
      mbar_init(bar(L::P_FULL + i), BM);
      mbar_init(bar(L::O_DONE + i), 1);
    }
    mbar_init(bar(L::DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == LOADER_WARP && lane == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(misc), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint64_t lim = p.wait_limit_ns;

  if (warp == LOADER_WARP) {
    // ------------------------------------------------------------ TMA loader
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      const int kv_z = b * p.Hkv + kvh;
      mbar_expect_tx(bar(L::Q_FULL), L::TILE);
      for (int r = 0; r < L::NREG; ++r)
        tma_load_3d(sb + L::Q_OFF + r * L::REGION, &tmq, bar(L::Q_FULL), r * 64, m0, bh, pol_q);
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t & 1;
        const uint32_t ph = ((t >> 1) & 1) ^ 1;
        if (!mbar_wait(bar(L::K_EMPTY + s), ph, abort_flag, &g_status, lim)) break;
        mbar_expect_tx(bar(L::K_FULL + s), L::TILE);
        for (int r = 0; r < L::NREG; ++r)
          tma_load_3d(sb + L::K_OFF + s * L::TILE + r * L::REGION, &tmk, bar(L::K_FULL + s), r * 64,
                      t * BN, kv_z, pol_kv);
        last_k[s] = t;
        if (p.debug_fault == 1 && t == 0) continue;  // withhold V_0: consumers must time out
        if (!mbar_wait(bar(L::V_EMPTY + s), ph, abort_flag, &g_status, lim)) break;
        mbar_expect_tx(bar(L::V_FULL + s), L::TILE);
        for (int r = 0; r < L::NREG; ++r)
          tma_load_3d(sb + L::V_OFF + s * L::TILE + r * L::REGION, &tmv, bar(L::V_FULL + s), r * 64,
                      t * BN, kv_z, pol_kv);
        last_v[s] = t;
      }
      // every copy issued must have landed before the CTA may exit
      drain_wait(bar(L::Q_FULL), 0, lim);
      for (int s = 0; s < 2; ++s) {
        if (last_k[s] >= 0) drain_wait(bar(L::K_FULL + s), (last_k[s] >> 1) & 1, lim);
        if (last_v[s] >= 0) drain_wait(bar(L::V_FULL + s), (last_v[s] >> 1) & 1, lim);
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_f16(BF16, BM, BN, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_f16(BF16, BM, D, false, true);
      const uint32_t tO = tmem + COL_O;
      auto issue_pv = [&](int u) -> bool {
        const int s = u & 1;
        const uint32_t ph = (u >> 1) & 1;
        if (!mbar_wait(bar(L::P_FULL + s), ph, abort_flag, &g_status, lim)) return false;
        if (!mbar_wait(bar(L::V_FULL + s), ph, abort_flag, &g_status, lim)) return false;
        tc_fence_after();
        const uint32_t v_base = sb + L::V_OFF + s * L::TILE;
        const uint32_t tP = tmem + COL_P + 64u * s;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // V is [key][d] (d contiguous): MN-major B, 16 keys = 2 swizzle atoms of 8 rows;
          // LBO steps to the next 64-column block of d, SBO to the next 8 keys.
          const uint64_t bdesc = sdesc_sw128(v_base + kk * 16 * 128, L::REGION, 1024);
          umma_ts(tO, tP + kk * 8, bdesc, idesc_pv, (u > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(L::O_DONE + s));
        umma_commit(bar(L::V_EMPTY + s));
        return true;
      };
      bool ok = mbar_wait(bar(L::Q_FULL), 0, abort_flag, &g_status, lim);
      int t = 0;
      for (; ok && t < n_tiles; ++t) {
        const int s = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!(ok = mbar_wait(bar(L::K_FULL + s), ph, abort_flag, &g_status, lim))) break;
        tc_fence_after();
        const uint32_t k_base = sb + L::K_OFF + s * L::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major operands: 16 columns = 32 bytes inside a 128-byte swizzled row
          const uint32_t off = (kk >> 2) * L::REGION + (kk & 3) * 32;
          const uint64_t adesc = sdesc_sw128(sb + L::Q_OFF + off, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(k_base + off, 16, 1024);
          umma_ss(tmem + COL_S + 128u * s, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(L::S_FULL + s));
        umma_commit(bar(L::K_EMPTY + s));
        if (t > 0 && !(ok = issue_pv(t - 1))) break;
      }
      if (ok) issue_pv(n_tiles - 1);
      umma_commit(bar(L::DRAIN));  // fires once every MMA issued above has completed
      drain_wait(bar(L::DRAIN), 0, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax + epilogue (rows)
    const int r = threadIdx.x;  // TMEM lane == tile row
    const int row = m0 + r;
    const uint32_t lane_t = tmem + ((uint32_t)(warp * 32) << 16);
    const int lim_key = p.causal ? row + delta : 0x7fffffff;
    const float mval = p.neg ? INFINITY : -INFINITY;
    const float c2 = p.c2;
    float m_used = -INFINITY, l_sum = 0.f;
    // tcgen05.ld/st are warp-collective: every wait outcome and every rescale
    // decision below is made uniform across the warp before TMEM is touched.
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b_, ph_, abort_flag, &g_status, lim));
    };
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      if (!(ok = wait_warp(bar(L::S_FULL + s), ph))) break;
      tc_fence_after();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_t + COL_S + 128u * s + 32u * c, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(rr[i]);
      }
      if (p.zero) {
#pragma unroll
        for (int j = 0; j < BN; ++j) x[j] = 0.f;
      }
      if (t >= mask_from) {
        const int kbase = t * BN;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const int key = kbase + j;
          if (key > lim_key || key >= p.Skv) x[j] = mval;
        }
      }
      float red;
      if (!p.neg) {
        float a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
#pragma unroll
        for (int j = 4; j < BN; j += 4) {
          a0 = fmaxf(a0, x[j]);
          a1 = fmaxf(a1, x[j + 1]);
          a2 = fmaxf(a2, x[j + 2]);
          a3 = fmaxf(a3, x[j + 3]);
        }
        red = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      } else {
        float a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
#pragma unroll
        for (int j = 4; j < BN; j += 4) {
          a0 = fminf(a0, x[j]);
          a1 = fminf(a1, x[j + 1]);
          a2 = fminf(a2, x[j + 2]);
          a3 = fminf(a3, x[j + 3]);
        }
        red = fminf(fminf(a0, a1), fminf(a2, a3));
      }
      const float m_tile = red * c2;  // -inf when every key of the tile is masked
      const float m_new = fmaxf(m_used, m_tile);
      const bool grow = m_new > m_used + RESCALE_LOG2;
      // O needs the factor only once it holds P V of an earlier tile with a finite max
      const bool o_scale = grow && t > 0 && m_used != -INFINITY;
      float alpha_o = 1.f;
      if (grow) {
        const float alpha = ex2(m_used - m_new);  // 0 while nothing was visible yet
        l_sum *= alpha;
        if (o_scale) alpha_o = alpha;
        m_used = m_new;
      }
      if (__any_sync(0xffffffffu, o_scale)) {
        // O holds P V up to tile t-1: wait for that MMA, then rescale the rows in place
        const int u = t - 1;
        if (!(ok = wait_warp(bar(L::O_DONE + (u & 1)), (u >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(lane_t + COL_O + 32u * c, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha_o);
          tmem_st32(lane_t + COL_O + 32u * c, rr);
        }
      }
      if (t >= 2) {  // P_s was read by the MMA of tile t-2: wait until it completed
        const int u = t - 2;
        if (!(ok = wait_warp(bar(L::O_DONE + s), (u >> 1) & 1))) break;
      }
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float e0 = ex2(fmaf(x[h * 64 + 2 * i], c2, -mu));
          const float e1 = ex2(fmaf(x[h * 64 + 2 * i + 1], c2, -mu));
          ls0 += e0;
          ls1 += e1;
          pk[i] = pack2<BF16>(e0, e1);
        }
        tmem_st32(lane_t + COL_P + 64u * s + 32u * h, pk);
      }
      l_sum += ls0 + ls1;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::P_FULL + s));
    }
    if (ok) {
      const int u = n_tiles - 1;
      ok = wait_warp(bar(L::O_DONE + (u & 1)), (u >> 1) & 1);
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      store_row<D, BF16>(p, bh, row, inv_l, lane_t + COL_O);
      if (p.lse && row < p.Sq)
        p.lse[(size_t)bh * p.Sq + row] =
            l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Every row sees no key (Skv == 0): O = 0, LSE = -inf.
__global__ void fill_empty_kernel(uint16_t* o, float* lse, size_t rows, int D) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < rows;
       i += (size_t)gridDim.x * blockDim.x) {
    uint4* dst = reinterpret_cast<uint4*>(o + i * D);
    for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    if (lse) lse[i] = -INFINITY;
  }
}

static bool make_map(CUtensorMap* map, const void* base, int D, int S, int BH, bool bf16) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool BF16>
static cudaError_t launch_t(const FwdArgs& a, cudaStream_t stream) {
  using L = Layout<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, D, a.Sq, a.B * a.Hq, BF16) ||
      !make_map(&tk, a.k, D, a.Skv, a.B * a.Hkv, BF16) ||
      !make_map(&tv, a.v, D, a.Skv, a.B * a.Hkv, BF16))
    return cudaErrorInvalidValue;
  Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.group = a.Hq / a.Hkv;
  p.num_m_tiles = (a.Sq + BM - 1) / BM;
  p.causal = a.causal ? 1 : 0;
  const float c2 = a.scale * 1.4426950408889634f;
  p.zero = (c2 == 0.f) ? 1 : 0;
  p.neg = (c2 < 0.f) ? 1 : 0;
  p.c2 = p.zero ? 1.f : c2;
  p.wait_limit_ns = a.wait_limit_ns;
  p.debug_fault = a.debug_fault;
  dim3 grid(p.num_m_tiles, a.Hq, a.B);
  attn_fwd_kernel<D, BF16><<<grid, NUM_THREADS, L::ALLOC, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return a.bf16 ? fwd::launch_t<64, true>(a, stream) : fwd::launch_t<64, false>(a, stream);
  return a.bf16 ? fwd::launch_t<128, true>(a, stream) : fwd::launch_t<128, false>(a, stream);
}

cudaError_t launch_fwd_empty_keys(const FwdArgs& a, cudaStream_t stream) {
  const size_t rows = (size_t)a.B * a.Hq * a.Sq;
  const int blocks = (int)((rows + 255) / 256 < 4096 ? (rows + 255) / 256 : 4096);
  fwd::fill_empty_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint16_t*>(a.o), a.lse, rows, a.D);
  return cudaGetLastError();
}

cudaError_t read_fwd_status(unsigned* out, cudaStream_t stream) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, fwd::g_status, sizeof(unsigned), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(fwd::g_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace ea
