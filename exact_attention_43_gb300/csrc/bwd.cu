// Backward of fused exact attention: dQ, dK, dV from Q, K, V, O, the forward's
// per-row LSE and dO, for sm_103a.
//
// What is computed follows llm.c attention.cuh (attention_backward with
// softmax_autoregressive_backward_inplace_kernel): dP = dO V^T, dV = P^T dO,
// dS = scale * P * (dP - sum_j P dP) per row, dQ = dS K, dK = dS^T Q, with P the
// probabilities of the forward pass (here re-formed from its LSE, P = e^(S - LSE),
// rather than stored) and the row term taken as sum_d dO O, equal to
// sum_j P dP because O = P V.  A K/V head shared by several query heads (GQA)
// receives the sum of their gradients.
//
// GB300 design:
//  * a prep kernel forms the row term delta_i = sum_d dO_id O_id;
//  * the main kernel keeps one 128-key tile of one KV head per CTA: K and V stay
//    in shared memory, and dK, dV accumulate in TMEM over every query head of the
//    GQA group and every Q tile that sees the keys (causal tiles that see none are
//    skipped), so K/V gradients need no atomics;
//  * per Q tile one thread issues the tcgen05 MMAs: S^T = K Q^T and
//    dP^T = V dO^T into TMEM; four compute warps (one key row per thread, TMEM
//    lane = key) form P^T = 2^(S^T c - LSE_2) and dS^T = P^T (dP^T - delta), write
//    both to TMEM as 16-bit (over the columns they came from) and dS^T also to a
//    128-byte-swizzled shared-memory tile; then dV += P^T dO and dK += dS^T Q (A
//    from TMEM) and dQ_part = dS K (A: the dS^T tile read M-major) over S^T's
//    columns; the compute warps add scale * dQ_part (TMEM lane = query row) into
//    an fp32 accumulator with 16-byte vector atomics;
//  * a last kernel rounds the dQ accumulator to the input type.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace ea {
namespace bwd {

__device__ unsigned g_status;

constexpr int BM = 128;  // queries per Q tile
constexpr int BN = 128;  // keys per K/V tile (= TMEM lanes)
constexpr int THREADS = 160;  // warps 0-3 compute, warp 4 loads and issues
constexpr int ISSUER_WARP = 4;
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: S^T at 0 (P^T over its first 64; dQ_part over its first D once
// dV has read P^T), dP^T at 128 (dS^T over its first 64), dV at 256, dK at 256 + D

struct Params {
  const float* lse;    // [B, Hq, Sq], natural log
  const float* delta;  // [B, Hq, Sq]
  float* dq_acc;       // [B, Hq, Sq, D], zero at launch
  uint16_t* dk;        // [B, Hkv, Skv, D]
  uint16_t* dv;
  int B, Hq, Hkv, Sq, Skv, group, causal;
  float c2;     // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
};

template <int D>
struct Layout {
  static constexpr int REGION = 128 * 128;  // 128 rows x 64 16-bit columns, 128-byte swizzle
  static constexpr int NREG = D / 64;
  static constexpr int TILE = NREG * REGION;  // 128 x D
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE;
  static constexpr int Q_OFF = 2 * TILE;
  static constexpr int DO_OFF = 3 * TILE;
  static constexpr int DS_OFF = 4 * TILE;               // dS^T: 128 keys x 128 queries
  static constexpr int VEC_OFF = DS_OFF + 2 * REGION;   // LSE (log2 units), delta of the Q tile
  static constexpr int BAR_OFF = VEC_OFF + 2 * BM * 4;
  enum { KV_FULL, QD_FULL, S_FULL, P_FULL, DQ_FULL, DQ_FREE, VEC_READY, NUM_BARS };
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 bytes
  static_assert(TILE % 1024 == 0 && DS_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

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

// Eight consecutive fp32 values of a TMEM row, times f, as 16-bit values in one uint4.
template <bool BF16>
__device__ __forceinline__ uint4 pack8(const uint32_t* r, float f) {
  return make_uint4(pack2<BF16>(__uint_as_float(r[0]) * f, __uint_as_float(r[1]) * f),
                    pack2<BF16>(__uint_as_float(r[2]) * f, __uint_as_float(r[3]) * f),
                    pack2<BF16>(__uint_as_float(r[4]) * f, __uint_as_float(r[5]) * f),
                    pack2<BF16>(__uint_as_float(r[6]) * f, __uint_as_float(r[7]) * f));
}

// delta_i = sum_d dO_id O_id, one warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* o, const uint16_t* dout,
                                                        float* delta, long long rows) {
  constexpr int EPL = D / 32;  // elements per lane
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const uint16_t* a = o + row * D + lane * EPL;
  const uint16_t* g = dout + row * D + lane * EPL;
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    const float2 x = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(a + e));
    const float2 y = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(g + e));
    s = fmaf(x.x, y.x, s);
    s = fmaf(x.y, y.y, s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[row] = s;
}

// dq = dq_acc rounded to the input type, eight elements per thread.
template <bool BF16>
__global__ void bwd_dq_convert_kernel(const float* acc, uint16_t* dq, long long n8) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 c = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w),
                                                 pack2<BF16>(c.x, c.y), pack2<BF16>(c.z, c.w));
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const Params p) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;

  const int n0 = blockIdx.x * BN, hk = blockIdx.y, b = blockIdx.z;
  const int dlen = p.Skv - p.Sq;  // key j is visible to query i iff j <= i + dlen (causal)
  const int n_mt = (p.Sq + BM - 1) / BM;
  int m_lo = 0;  // first Q tile with a row that sees a key of this tile
  if (p.causal) {
    const long long lo = (long long)n0 - dlen - (BM - 1);
    m_lo = lo <= 0 ? 0 : (int)min((lo + BM - 1) / BM, (long long)n_mt);
  }
  const int per_head = n_mt - m_lo;
  const int n_iter = p.group * per_head;  // (query head, Q tile) pairs of this CTA

  if (threadIdx.x == 0) {
    mbar_init(bar(L::KV_FULL), 1);
    mbar_init(bar(L::QD_FULL), 1);
    mbar_init(bar(L::S_FULL), 1);
    mbar_init(bar(L::P_FULL), BM);
    mbar_init(bar(L::DQ_FULL), 1);
    mbar_init(bar(L::DQ_FREE), BM);
    mbar_init(bar(L::VEC_READY), BM);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(misc), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == ISSUER_WARP) {
    // ------------------------------------------------ loads and MMAs (one thread)
    if (lane == 0 && n_iter > 0) {
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      prefetch_tmap(&tmdo);
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      const int kv_z = b * p.Hkv + hk;
      mbar_expect_tx(bar(L::KV_FULL), 2 * L::TILE);
      for (int rr = 0; rr < L::NREG; ++rr) {
        tma_load_3d(sb + L::K_OFF + rr * L::REGION, &tmk, bar(L::KV_FULL), rr * 64, n0, kv_z, pol_kv);
        tma_load_3d(sb + L::V_OFF + rr * L::REGION, &tmv, bar(L::KV_FULL), rr * 64, n0, kv_z, pol_kv);
      }
      // K-major operands (S^T = K Q^T, dP^T = V dO^T): 16 columns = 32 bytes of a
      // 128-byte swizzled row; M/N-major operands (dO, Q, K as B and dS^T as A):
      // rows are the K dimension, LBO steps to the next 64 columns, SBO to the next 8 rows
      const uint64_t k_km = sdesc_sw128(sb + L::K_OFF, 16, 1024);
      const uint64_t v_km = sdesc_sw128(sb + L::V_OFF, 16, 1024);
      const uint64_t q_km = sdesc_sw128(sb + L::Q_OFF, 16, 1024);
      const uint64_t do_km = sdesc_sw128(sb + L::DO_OFF, 16, 1024);
      const uint64_t k_mn = sdesc_sw128(sb + L::K_OFF, L::REGION, 1024);
      const uint64_t q_mn = sdesc_sw128(sb + L::Q_OFF, L::REGION, 1024);
      const uint64_t do_mn = sdesc_sw128(sb + L::DO_OFF, L::REGION, 1024);
      const uint64_t ds_mn = sdesc_sw128(sb + L::DS_OFF, L::REGION, 1024);
      constexpr uint32_t idesc_s = umma_idesc_f16(BF16, BN, BM, false, false);
      constexpr uint32_t idesc_kv = umma_idesc_f16(BF16, BN, D, false, true);
      constexpr uint32_t idesc_dq = umma_idesc_f16(BF16, BM, D, true, true);
      const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 256 + D;
      int n_qd = 0, n_s = 0, n_dq = 0;  // phases of QD_FULL, S_FULL, DQ_FULL started
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        const int h = hk * p.group + it / per_head, m = m_lo + it % per_head;
        // Q, dO of this tile may overwrite the last ones once its MMAs are done
        if (it > 0 && !(ok = mbar_wait(bar(L::DQ_FULL), (it - 1) & 1, abort_flag, &g_status, lim)))
          break;
        mbar_expect_tx(bar(L::QD_FULL), 2 * L::TILE);
        for (int rr = 0; rr < L::NREG; ++rr) {
          tma_load_3d(sb + L::Q_OFF + rr * L::REGION, &tmq, bar(L::QD_FULL), rr * 64, m * BM,
                      b * p.Hq + h, pol_q);
          tma_load_3d(sb + L::DO_OFF + rr * L::REGION, &tmdo, bar(L::QD_FULL), rr * 64, m * BM,
                      b * p.Hq + h, pol_q);
        }
        ++n_qd;
        if (!(ok = mbar_wait(bar(L::QD_FULL), it & 1, abort_flag, &g_status, lim))) break;
        if (it == 0 && !(ok = mbar_wait(bar(L::KV_FULL), 0, abort_flag, &g_status, lim))) break;
        // S^T's columns held the last dQ_part: the compute warps must have read it
        if (it > 0 && !(ok = mbar_wait(bar(L::DQ_FREE), (it - 1) & 1, abort_flag, &g_status, lim)))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::REGION + (kk & 3) * 32) >> 4;
          umma_ss(t_s, k_km + off, q_km + off, idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::REGION + (kk & 3) * 32) >> 4;
          umma_ss(t_dp, v_km + off, do_km + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(L::S_FULL));
        ++n_s;
        if (!(ok = mbar_wait(bar(L::P_FULL), it & 1, abort_flag, &g_status, lim))) break;
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q over the tile's 128 queries, 16 per MMA
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_ts(t_dv, t_s + kk * 8, do_mn + kk * 128, idesc_kv, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_ts(t_dk, t_dp + kk * 8, q_mn + kk * 128, idesc_kv, (it > 0 || kk > 0) ? 1u : 0u);
        // dQ_part = dS K over the tile's 128 keys, into S^T's columns (after dV read P^T)
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ss(t_s, ds_mn + kk * 128, k_mn + kk * 128, idesc_dq, kk > 0 ? 1u : 0u);
        umma_commit(bar(L::DQ_FULL));
        ++n_dq;
      }
      // nothing may be in flight when the CTA exits: wait for the last phase of each
      // barrier this thread started (no later phase follows, so none is missed)
      drain_wait(bar(L::KV_FULL), 0, lim);
      if (n_qd > 0) drain_wait(bar(L::QD_FULL), (n_qd - 1) & 1, lim);
      if (n_s > 0) drain_wait(bar(L::S_FULL), (n_s - 1) & 1, lim);
      if (n_dq > 0) drain_wait(bar(L::DQ_FULL), (n_dq - 1) & 1, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ compute warps: one key row per thread
    const int r = threadIdx.x;  // TMEM lane: key n0 + r (S^T, dP^T, dK, dV), query m0 + r (dQ_part)
    const uint32_t lane_t = tmem + ((uint32_t)(warp * 32) << 16);
    float* v_lse = reinterpret_cast<float*>(smem + L::VEC_OFF);
    float* v_dl = v_lse + BM;
    const int key = n0 + r;
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b_, ph_, abort_flag, &g_status, lim));
    };
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      const int h = hk * p.group + it / per_head, m = m_lo + it % per_head;
      const int m0 = m * BM;
      const size_t bh = (size_t)b * p.Hq + h;
      // the row vectors of this Q tile: every thread read the last ones before P_FULL
      // completed, which the last DQ_FULL implies
      {
        const int qi = m0 + r;
        v_lse[r] = qi < p.Sq ? p.lse[bh * p.Sq + qi] * 1.4426950408889634f : INFINITY;
        v_dl[r] = qi < p.Sq ? p.delta[bh * p.Sq + qi] : 0.f;
        mbar_arrive(bar(L::VEC_READY));
      }
      if (!(ok = wait_warp(bar(L::VEC_READY), it & 1))) break;
      if (!(ok = wait_warp(bar(L::S_FULL), it & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < BM; c0 += 64) {
        uint32_t sr[64], dr[64];
        tmem_ld(lane_t + c0, sr);
        tmem_ld(lane_t + 128 + c0, dr);
        uint32_t pp[32], dd[32];
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          float pv[2], dsv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int q = m0 + c0 + j + u;
            const bool vis = q < p.Sq && key < p.Skv && (!p.causal || key <= q + dlen);
            const float x = fmaf(__uint_as_float(sr[j + u]), p.c2, -v_lse[c0 + j + u]);
            pv[u] = vis ? ex2(x) : 0.f;
            dsv[u] = pv[u] * (__uint_as_float(dr[j + u]) - v_dl[c0 + j + u]);
          }
          pp[j >> 1] = pack2<BF16>(pv[0], pv[1]);
          dd[j >> 1] = pack2<BF16>(dsv[0], dsv[1]);
        }
        tmem_st32(lane_t + (c0 >> 1), pp);        // P^T over S^T's columns
        tmem_st32(lane_t + 128 + (c0 >> 1), dd);  // dS^T over dP^T's columns
        // dS^T row r, queries c0 .. c0 + 63: 16-byte chunk c at chunk c ^ (r mod 8)
        const uint32_t reg = sb + L::DS_OFF + (c0 / 64) * L::REGION + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(reg + ((c ^ (r & 7)) << 4),
                       make_uint4(dd[4 * c], dd[4 * c + 1], dd[4 * c + 2], dd[4 * c + 3]));
      }
      tmem_wait_st();
      fence_proxy_async_smem();  // dS^T in shared memory, for the MMA that reads it
      tc_fence_before();
      mbar_arrive(bar(L::P_FULL));
      if (!(ok = wait_warp(bar(L::DQ_FULL), it & 1))) break;
      tc_fence_after();
      // dQ_part row r (query m0 + r) into the fp32 accumulator
      const bool live = m0 + r < p.Sq;
      float* dst = p.dq_acc + (bh * p.Sq + (live ? m0 + r : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_t + 32 * c, v);
        if (live) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            atomicAdd(reinterpret_cast<float4*>(dst + 32 * c + 4 * i),
                      make_float4(__uint_as_float(v[4 * i]) * p.scale,
                                  __uint_as_float(v[4 * i + 1]) * p.scale,
                                  __uint_as_float(v[4 * i + 2]) * p.scale,
                                  __uint_as_float(v[4 * i + 3]) * p.scale));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::DQ_FREE));
    }
    // dV and dK rows of this tile's keys (zero when no query sees them)
    if (ok && key < p.Skv) {
      uint4* dvr = reinterpret_cast<uint4*>(p.dv + (((size_t)b * p.Hkv + hk) * p.Skv + key) * D);
      uint4* dkr = reinterpret_cast<uint4*>(p.dk + (((size_t)b * p.Hkv + hk) * p.Skv + key) * D);
      if (n_iter == 0) {
        for (int i = 0; i < D / 8; ++i) dvr[i] = dkr[i] = make_uint4(0, 0, 0, 0);
      }
    }
    if (ok && n_iter > 0) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32], w[32];
        tmem_ld32(lane_t + 256 + 32 * c, v);
        tmem_ld32(lane_t + 256 + D + 32 * c, w);
        if (key < p.Skv) {
          uint4* dvr = reinterpret_cast<uint4*>(p.dv + (((size_t)b * p.Hkv + hk) * p.Skv + key) * D);
          uint4* dkr = reinterpret_cast<uint4*>(p.dk + (((size_t)b * p.Hkv + hk) * p.Skv + key) * D);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dvr[4 * c + i] = pack8<BF16>(v + 8 * i, 1.f);
            dkr[4 * c + i] = pack8<BF16>(w + 8 * i, p.scale);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

static bool make_map(CUtensorMap* map, const void* base, int D, int S, long long planes, bool bf16) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BF16>
static cudaError_t launch_t(const BwdArgs& a, cudaStream_t stream) {
  using L = Layout<D>;
  const long long rows = (long long)a.B * a.Hq * a.Sq;
  if (rows > 0) {
    bwd_delta_kernel<D, BF16><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.delta, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.Skv > 0) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    // with no query rows the maps cover one (never read) row of k
    const int sq_map = a.Sq > 0 ? a.Sq : 1;
    const void* qb = a.Sq > 0 ? a.q : a.k;
    const void* gb = a.Sq > 0 ? a.dout : a.k;
    CUtensorMap tq, tk, tv, tg;
    if (!make_map(&tq, qb, D, sq_map, a.Sq > 0 ? (long long)a.B * a.Hq : 1, BF16) ||
        !make_map(&tg, gb, D, sq_map, a.Sq > 0 ? (long long)a.B * a.Hq : 1, BF16) ||
        !make_map(&tk, a.k, D, a.Skv, (long long)a.B * a.Hkv, BF16) ||
        !make_map(&tv, a.v, D, a.Skv, (long long)a.B * a.Hkv, BF16))
      return cudaErrorInvalidValue;
    Params p{};
    p.lse = a.lse;
    p.delta = a.delta;
    p.dq_acc = a.dq_acc;
    p.dk = static_cast<uint16_t*>(a.dk);
    p.dv = static_cast<uint16_t*>(a.dv);
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.Sq = a.Sq;
    p.Skv = a.Skv;
    p.group = a.Hq / a.Hkv;
    p.causal = a.causal ? 1 : 0;
    p.scale = a.scale;
    p.c2 = a.scale * 1.4426950408889634f;
    p.wait_limit_ns = a.wait_limit_ns;
    dim3 grid((a.Skv + BN - 1) / BN, a.Hkv, a.B);
    attn_bwd_kernel<D, BF16><<<grid, THREADS, L::ALLOC, stream>>>(tq, tk, tv, tg, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (rows > 0) {
    const long long n8 = rows * D / 8;
    const long long blocks = (n8 + 255) / 256 < 4096 ? (n8 + 255) / 256 : 4096;
    bwd_dq_convert_kernel<BF16><<<(unsigned)blocks, 256, 0, stream>>>(
        a.dq_acc, static_cast<uint16_t*>(a.dq), n8);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace bwd

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.D == 64) return a.bf16 ? bwd::launch_t<64, true>(a, stream) : bwd::launch_t<64, false>(a, stream);
  return a.bf16 ? bwd::launch_t<128, true>(a, stream) : bwd::launch_t<128, false>(a, stream);
}

cudaError_t read_bwd_status(unsigned* out, cudaStream_t stream) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, bwd::g_status, sizeof(unsigned), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(bwd::g_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace ea
