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
//    dP^T = V dO^T into TMEM; eight compute warps (two threads per key row, each
//    with 64 of the tile's 128 queries; TMEM lane = key) form P^T = 2^(S^T c - LSE_2) and dS^T = P^T (dP^T - delta), write
//    both to TMEM as 16-bit (over the columns they came from) and dS^T also to a
//    128-byte-swizzled shared-memory tile; then dV += P^T dO and dK += dS^T Q (A
//    from TMEM) and dQ_part = dS K (A: the dS^T tile read M-major) over dP^T's
//    columns; the compute warps add scale * dQ_part (TMEM lane = query row) into
//    an fp32 accumulator with 16-byte vector atomics;
//  * Q and dO are double-buffered (the next Q tile's loads run during this one's
//    MMAs) and the next S^T is issued before the compute warps have read this
//    dQ_part, so the tensor core has work queued while they add it;
//  * a last kernel rounds the dQ accumulator to the input type.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace ea {
namespace bwd {

__device__ unsigned g_status;

constexpr int BM = 128;  // queries per Q tile
constexpr int BN = 128;  // keys per K/V tile (= TMEM lanes)
constexpr int THREADS = 288;  // warps 0-7 compute, warp 8 loads and issues
constexpr int ISSUER_WARP = 8;
constexpr int NCOMP = 256;    // compute threads: warps w and w + 4 share TMEM lanes 32 (w mod 4) ...
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: S^T at 0 (P^T over its first 64), dP^T at 128 (dS^T over its first
// 64; dQ_part over its first D once dK has read dS^T), dV at 256, dK at 256 + D

struct Params {
  const float* lse;    // [B, Hq, Sq], natural log
  const float* delta;  // [B, Hq, Sq]
  float* dq_acc;       // [B, Hq, Sq, D], zero at launch
  uint16_t* dk;        // [B, Hkv, Skv, D]
  uint16_t* dv;
  int B, Hq, Hkv, Sq, Skv, group, causal;
  int kv_slowest;  // 1: grid (KV head, batch, key tile), 0: (key tile, KV head, batch)
  float c2;     // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
  int debug_fault;  // 3: CTA (0, 0, 0) withholds the Q/dO loads of its iteration 1
};

template <int D>
struct Layout {
  static constexpr int REGION = 128 * 128;  // 128 rows x 64 16-bit columns, 128-byte swizzle
  static constexpr int NREG = D / 64;
  static constexpr int TILE = NREG * REGION;  // 128 x D
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE;
  static constexpr int Q_OFF = 2 * TILE;                // two buffers
  static constexpr int DO_OFF = 4 * TILE;               // two buffers
  static constexpr int DS_OFF = 6 * TILE;               // dS^T: 128 keys x 128 queries
  static constexpr int VEC_OFF = DS_OFF + 2 * REGION;   // LSE (log2 units), delta of the Q tile
  static constexpr int BAR_OFF = VEC_OFF + 2 * BM * 4;
  enum { KV_FULL, QD_FULL, S_FULL = QD_FULL + 2, P_FULL, DQ_FULL, DQ_FREE, VEC_READY, DRAIN, NUM_BARS };
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

  // Key tiles vary fastest: CTAs that run at the same time share a few heads, whose
  // fp32 dQ rows then stay in L2 for their atomics, and within a head the causal
  // tiles that most Q tiles see start first.  When one CTA's work is a large share
  // of an SM's, key tiles vary slowest instead, so those long CTAs start first.
  const int n0 = (p.kv_slowest ? blockIdx.z : blockIdx.x) * BN;
  const int hk = p.kv_slowest ? blockIdx.x : blockIdx.y, b = p.kv_slowest ? blockIdx.y : blockIdx.z;
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
    mbar_init(bar(L::QD_FULL + 1), 1);
    mbar_init(bar(L::S_FULL), 1);
    mbar_init(bar(L::P_FULL), NCOMP);
    mbar_init(bar(L::DQ_FULL), 1);
    mbar_init(bar(L::DQ_FREE), NCOMP);
    mbar_init(bar(L::VEC_READY), NCOMP);
    mbar_init(bar(L::DRAIN), 1);
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
      const uint64_t k_mn = sdesc_sw128(sb + L::K_OFF, L::REGION, 1024);
      const uint64_t ds_mn = sdesc_sw128(sb + L::DS_OFF, L::REGION, 1024);
      constexpr uint32_t idesc_s = umma_idesc_f16(BF16, BN, BM, false, false);
      constexpr uint32_t idesc_kv = umma_idesc_f16(BF16, BN, D, false, true);
      constexpr uint32_t idesc_dq = umma_idesc_f16(BF16, BM, D, true, true);
      const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 256 + D;
      // bounded-wait test: one CTA never issues iteration 1's loads, so the waits run out
      const int withheld =
          (p.debug_fault == 3 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) ? 1 : -1;
      // Q, dO of iteration i go to buffer i & 1
      auto load_qd = [&](int i) {
        if (i == withheld) return;
        const int h = hk * p.group + i / per_head, m = m_lo + i % per_head;
        const uint32_t fb = bar(L::QD_FULL + (i & 1));
        mbar_expect_tx(fb, 2 * L::TILE);
        for (int rr = 0; rr < L::NREG; ++rr) {
          tma_load_3d(sb + L::Q_OFF + (i & 1) * L::TILE + rr * L::REGION, &tmq, fb, rr * 64, m * BM,
                      b * p.Hq + h, pol_q);
          tma_load_3d(sb + L::DO_OFF + (i & 1) * L::TILE + rr * L::REGION, &tmdo, fb, rr * 64, m * BM,
                      b * p.Hq + h, pol_q);
        }
      };
      int n_qd = 0;  // Q/dO loads issued
      load_qd(0);
      ++n_qd;
      if (n_iter > 1) {
        load_qd(1);
        ++n_qd;
      }
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        const uint32_t qo = (it & 1) * L::TILE;
        const uint64_t q_km = sdesc_sw128(sb + L::Q_OFF + qo, 16, 1024);
        const uint64_t do_km = sdesc_sw128(sb + L::DO_OFF + qo, 16, 1024);
        const uint64_t q_mn = sdesc_sw128(sb + L::Q_OFF + qo, L::REGION, 1024);
        const uint64_t do_mn = sdesc_sw128(sb + L::DO_OFF + qo, L::REGION, 1024);
        if (!(ok = mbar_wait(bar(L::QD_FULL + (it & 1)), (it >> 1) & 1, abort_flag, &g_status, lim)))
          break;
        if (it == 0 && !(ok = mbar_wait(bar(L::KV_FULL), 0, abort_flag, &g_status, lim))) break;
        tc_fence_after();
        // S^T = K Q^T: its columns' last P^T was read by the last dV, issued before
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::REGION + (kk & 3) * 32) >> 4;
          umma_ss(t_s, k_km + off, q_km + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        // dP^T's columns held the last dQ_part: the compute warps must have read it
        if (it > 0 && !(ok = mbar_wait(bar(L::DQ_FREE), (it - 1) & 1, abort_flag, &g_status, lim)))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::REGION + (kk & 3) * 32) >> 4;
          umma_ss(t_dp, v_km + off, do_km + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(L::S_FULL));
        // the other buffer's last reader, iteration it - 1, has completed (its DQ_FULL
        // preceded DQ_FREE): load iteration it + 1 into it
        if (it > 0 && it + 1 < n_iter) {
          load_qd(it + 1);
          ++n_qd;
        }
        if (!(ok = mbar_wait(bar(L::P_FULL), it & 1, abort_flag, &g_status, lim))) break;
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q over the tile's 128 queries, 16 per MMA
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_ts(t_dv, t_s + kk * 8, do_mn + kk * 128, idesc_kv, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_ts(t_dk, t_dp + kk * 8, q_mn + kk * 128, idesc_kv, (it > 0 || kk > 0) ? 1u : 0u);
        // dQ_part = dS K over the tile's 128 keys, into dP^T's columns (after dK read dS^T)
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ss(t_dp, ds_mn + kk * 128, k_mn + kk * 128, idesc_dq, kk > 0 ? 1u : 0u);
        umma_commit(bar(L::DQ_FULL));
      }
      // nothing may be in flight when the CTA exits: the last load into each buffer
      // (no later phase follows, so none is missed) and every MMA issued above (one
      // more commit, on a barrier of its own, tracks them all, also after an abort)
      drain_wait(bar(L::KV_FULL), 0, lim);
      for (int i = max(0, n_qd - 2); i < n_qd; ++i)
        if (i != withheld) drain_wait(bar(L::QD_FULL + (i & 1)), (i >> 1) & 1, lim);
      umma_commit(bar(L::DRAIN));
      drain_wait(bar(L::DRAIN), 0, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ compute warps: two threads per key row
    // TMEM lane r: key n0 + r (S^T, dP^T, dK, dV), query m0 + r (dQ_part); warps w and
    // w + 4 share the lanes of quarter w and split the columns between them
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_t = tmem + ((uint32_t)(quarter * 32) << 16);
    float* v_lse = reinterpret_cast<float*>(smem + L::VEC_OFF);
    float* v_dl = v_lse + BM;
    const int key = n0 + r;
    const int c0 = half * 64;  // this thread's 64 of the tile's 128 queries
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b_, ph_, abort_flag, &g_status, lim));
    };
    // row r's LSE (half 0, log2 units) or delta (half 1) for iteration i, loaded one
    // iteration ahead so its latency hides behind the current one
    auto row_value = [&](int i) -> float {
      const int hi = hk * p.group + i / per_head, qi = (m_lo + i % per_head) * BM + r;
      if (qi >= p.Sq) return half == 0 ? INFINITY : 0.f;
      const size_t idx = ((size_t)b * p.Hq + hi) * p.Sq + qi;
      return half == 0 ? p.lse[idx] * 1.4426950408889634f : p.delta[idx];
    };
    float next_v = n_iter > 0 ? row_value(0) : 0.f;
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      const int h = hk * p.group + it / per_head, m = m_lo + it % per_head;
      const int m0 = m * BM;
      const size_t bh = (size_t)b * p.Hq + h;
      // the row vectors of this Q tile: every thread read the last ones before P_FULL
      // completed, which the last DQ_FULL implies
      (half == 0 ? v_lse : v_dl)[r] = next_v;
      mbar_arrive(bar(L::VEC_READY));
      if (it + 1 < n_iter) next_v = row_value(it + 1);
      if (!(ok = wait_warp(bar(L::VEC_READY), it & 1))) break;
      if (!(ok = wait_warp(bar(L::S_FULL), it & 1))) break;
      tc_fence_after();
      {
        uint32_t pp[32], dd[32];  // this thread's 64 queries of P^T, dS^T as 16-bit pairs
#pragma unroll
        for (int g = 0; g < 2; ++g) {  // 32 queries at a time
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_t + c0 + 32 * g, sr);
          tmem_ld32(lane_t + 128 + c0 + 32 * g, dr);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float pv[2], dsv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int cq = c0 + 32 * g + j + u;  // query column in the tile
              const int q = m0 + cq;
              const bool vis = q < p.Sq && key < p.Skv && (!p.causal || key <= q + dlen);
              const float x = fmaf(__uint_as_float(sr[j + u]), p.c2, -v_lse[cq]);
              pv[u] = vis ? ex2(x) : 0.f;
              dsv[u] = pv[u] * (__uint_as_float(dr[j + u]) - v_dl[cq]);
            }
            pp[16 * g + (j >> 1)] = pack2<BF16>(pv[0], pv[1]);
            dd[16 * g + (j >> 1)] = pack2<BF16>(dsv[0], dsv[1]);
          }
        }
        tmem_st32(lane_t + (c0 >> 1), pp);        // P^T over S^T's columns
        tmem_st32(lane_t + 128 + (c0 >> 1), dd);  // dS^T over dP^T's columns
        // dS^T row r, queries c0 .. c0 + 63: 16-byte chunk c at chunk c ^ (r mod 8)
        const uint32_t reg = sb + L::DS_OFF + half * L::REGION + r * 128;
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
      // dQ_part row r (query m0 + r), this half's D / 2 columns, into the fp32 accumulator
      const bool live = m0 + r < p.Sq;
      float* dst = p.dq_acc + (bh * p.Sq + (live ? m0 + r : 0)) * D + half * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_t + 128 + half * (D / 2) + 32 * c, v);
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
    // this tile's dV rows (half 0) and dK rows (half 1); zero when no query sees the key
    if (ok) {
      const float f = half == 0 ? 1.f : p.scale;
      uint16_t* grad = half == 0 ? p.dv : p.dk;
      uint4* row = reinterpret_cast<uint4*>(grad + (((size_t)b * p.Hkv + hk) * p.Skv + key) * D);
      if (n_iter == 0) {
        if (key < p.Skv)
          for (int i = 0; i < D / 8; ++i) row[i] = make_uint4(0, 0, 0, 0);
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_t + 256 + half * D + 32 * c, v);
          if (key < p.Skv) {
#pragma unroll
            for (int i = 0; i < 4; ++i) row[4 * c + i] = pack8<BF16>(v + 8 * i, f);
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
    p.debug_fault = a.debug_fault;
    // the longest CTA (key tile 0) against an SM's share of all (query head, Q tile)
    // iterations: above a fifth, start the long CTAs first
    const long long n_kt = (a.Skv + BN - 1) / BN, n_mt = (a.Sq + BM - 1) / BM;
    long long total = 0;
    for (long long t = 0; t < n_kt; ++t) {
      long long m_lo = 0;
      if (a.causal) {
        const long long lo = t * BN - (a.Skv - a.Sq) - (BM - 1);
        m_lo = lo <= 0 ? 0 : ((lo + BM - 1) / BM < n_mt ? (lo + BM - 1) / BM : n_mt);
      }
      total += n_mt - m_lo;
    }
    total *= (long long)a.B * a.Hq;
    const long long longest = n_mt * (a.Hq / a.Hkv);
    p.kv_slowest = longest * 5 * (a.num_sms > 0 ? a.num_sms : 1) > total ? 1 : 0;
    const dim3 grid = p.kv_slowest ? dim3(a.Hkv, a.B, (unsigned)n_kt) : dim3((unsigned)n_kt, a.Hkv, a.B);
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
