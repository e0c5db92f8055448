// Prefill: fused exact attention O = softmax(scale * Q K^T [+ causal mask]) V
// with the per-row log-sum-exp, for sm_103a.
//
// What is computed follows the pages' algorithm (abaddon attention.rs, module
// doc "Algorithm": load a Q tile, for each K/V tile form S = Q K^T, mask,
// update the running max and sum, rescale and accumulate O += P V, divide by
// the sum at the end; rustytorch flash_attention_forward.cu,
// OnlineSoftmaxState: LSE = m + log(l)).  How it is computed is GB300-native:
//
//  * a work item is two 128-row Q tiles (256 consecutive query rows) of one
//    (batch, query head); the K/V tiles of the matching KV head are streamed
//    once for both; KV head = query head / (Hq / Hkv) (abaddon
//    flash_attention_f16, GQA mapping);
//  * the grid is persistent (one CTA per SM): the loader warp claims work
//    items from a global counter and queues them in shared memory for the
//    other warps; items are ordered so each group of heads' K and V stays in
//    L2 and, within a group, the longest causal items come first; the next
//    item's Q, K, V loads and first S MMAs overlap the current item's last
//    P V and epilogue (O is handed back through an mbarrier as soon as the
//    epilogue has read it from TMEM);
//  * warp 8 streams Q once and K, V 128-key tiles through a 4-stage ring with
//    TMA (3-D tensor maps, 128-byte swizzle, mbarrier transaction counts);
//  * one thread of warp 9 + i issues the tcgen05.mma of Q tile i: S_i = Q_i K_j^T
//    into TMEM, O_i += P_i V_j with P read from TMEM and V from shared memory.
//    The two issuers hand a token back and forth, so per KV tile their batches
//    reach the tensor core in the order P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1):
//    S_0 completes a whole tile's MMAs before S_1, and softmax 0 runs while the
//    tensor core works for Q tile 1 and the other way round.  (Issuers that do
//    not take turns let the tensor core interleave both streams; both S tiles
//    then finish together and the softmax warpgroups fall into step.)  Each
//    issuer makes its other waits (its P, the K/V ring, O free) while the other
//    one's batch executes, so only the hand-off lies between two batches: the
//    tensor core queues just two or three MMAs, and a single issuer's barrier
//    checks between batches idled it.  Both Q tiles step through every KV tile
//    of an item; the shorter one's extra steps are empty batches.  No commit
//    frees a ring slot: after S_i(c) completes (issued after every MMA of its
//    issuer that reads K(c) or V(c-1)), softmax warpgroup i, which waits for
//    it anyway, releases its use of both slots with plain arrives;
//  * warpgroup i (warps 4i..4i+3) owns the rows of Q tile i, one row per
//    thread (TMEM lane = row): load S, mask, row max, exponentiate with exp2
//    (scale * log2 e folded into one FMA), accumulate the row sum, write P
//    (16-bit) over the S columns it has consumed, and rescale the O row in
//    TMEM only when the running max grew by more than 2^8 (exact: O and l
//    share the same stale max).  Completion of S_i(j) implies completion of
//    every earlier MMA, so O_i already holds P V up to tile j-1 and P_i(j-1)
//    has been consumed: the softmax never waits on O inside the loop;
//  * causal: KV tiles wholly after a Q tile's last row are never loaded or
//    multiplied (abaddon flash_attention_f16, causal `break`); only tiles
//    that cross the diagonal or the end of the keys are masked element-wise.
//    Alignment is bottom-right: key j is visible to row i iff j <= i + (Skv - Sq);
//  * epilogue: O / l rounded to the input dtype and written through a
//    128-byte-swizzled shared-memory staging region per warpgroup with TMA
//    stores (rows past Sq fall outside the tensor map); LSE = ln 2 * (m +
//    log2 l); a row with no visible key gets O = 0, LSE = -inf.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace ea {
namespace fwd {

__device__ unsigned g_status;

constexpr int BM = 128;             // rows per Q tile (= TMEM lanes)
constexpr int NQ = 2;               // Q tiles per CTA
constexpr int BN = 128;             // keys per KV tile
constexpr int NS = 4;               // K/V ring stages
constexpr int NITEM = 4;            // claimed work items queued from the loader to the others
constexpr int NQS = 3;              // Q ring: single-tile slots
constexpr int NUM_THREADS = 512;    // warpgroups 0, 1: softmax; warpgroup 2: epilogue; warp 12
                                    // K/V loader, warps 13, 14 MMA, warp 15 work items and Q
constexpr int EPI_WARP = 8;         // first warp of the epilogue warpgroup
constexpr int KV_WARP = 12;
constexpr int MMA_WARP = 13;        // warp 13 + i issues the MMAs of Q tile i
constexpr int QLOAD_WARP = 15;
constexpr float RESCALE_LOG2 = 8.0f;  // rescale O when the max grows by more than 2^8
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: S_i at 128 i (P_i overwrites its first 64 columns), O_i at 256 + 128 i
constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_O = 256;

struct Params {
  void* o;
  float* lse;
  int* work_counter;  // zeroed before the launch; CTAs claim work items from it
  int B, Hq, Hkv, Sq, Skv, group, num_m_blocks, causal, neg, zero;
  int heads_per_group;  // flattened (batch, head) rows per scheduling group
  float c2;  // scale * log2(e); 1 when scale == 0 (then every visible score is set to 0)
  uint64_t wait_limit_ns;
  int debug_fault;
  // token-major layouts (attn_fwd_varlen, attn_fwd_qkvpacked; the VL kernels): Q, K, V
  // and O are [tokens, heads, D] (row strides in the tensor maps); sequence b's
  // queries are tokens [cu_q[b], cu_q[b+1]) and its keys [cu_k[b], cu_k[b+1]), or
  // b * Sq and b * Skv onwards when cu_q is null; Sq and Skv are then the longest
  // lengths.  LSE of head h, token t is at h * total_q + t.
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  int win_left, win_right;  // sliding-window bounds (-1: none); causal is win_right = 0
  int o_rstride;            // elements between consecutive tokens of O
  int o_align32;            // O is 32-byte aligned (so is every row): 32-byte stores
};

// Query and key rows of one sequence in the token-major layouts.
struct Seq {
  int q0, nq;  // first query token, query count
  int k0, nk;  // first key token, key count
};

// Offsets outside the arrays, decreasing offsets and lengths above the longest
// length are clamped (no access leaves the arrays) and reported in the status word.
__device__ __forceinline__ Seq seq_of(const Params& p, int b) {
  Seq s;
  if (!p.cu_q) {
    s.q0 = b * p.Sq;
    s.nq = p.Sq;
    s.k0 = b * p.Skv;
    s.nk = p.Skv;
    return s;
  }
  const int a = p.cu_q[b], e = p.cu_q[b + 1], c = p.cu_k[b], f = p.cu_k[b + 1];
  s.q0 = min(max(a, 0), p.total_q);
  s.nq = min(min(max(e, s.q0), p.total_q) - s.q0, p.Sq);
  s.k0 = min(max(c, 0), p.total_k);
  s.nk = min(min(max(f, s.k0), p.total_k) - s.k0, p.Skv);
  if (s.q0 != a || s.nq != e - a || s.k0 != c || s.nk != f - c) atomicOr(&g_status, kStatusSeqLenClamped);
  return s;
}

// A claimed work item as queued in shared memory: its index (-1: no more work),
// its KV steps n_kv (both Q tiles step through all of them), the steps [a, e) that
// Q tile i multiplies, and the tensor-map coordinates of its Q tile 0 and K/V tile 0.
struct ItemEntry {
  int w, n_kv, a[2], e[2], q_y, q_z, k_y0, kv_z;
};

template <int D>
struct Layout {
  static constexpr int REGION = 128 * 128;    // 128 rows x 128 bytes (64 columns), swizzled
  static constexpr int NREG = D / 64;
  static constexpr int TILE = NREG * REGION;  // a 128 x D 16-bit tile
  static constexpr int Q_OFF = 0;             // Q ring: NQS single-tile slots
  static constexpr int RING_OFF = Q_OFF + NQS * TILE;
  static constexpr int INVL_OFF = RING_OFF + NS * TILE;  // 1 / l of each row, per Q tile
  static constexpr int BAR_OFF = INVL_OFF + NQ * BM * 4;
  enum {
    Q_FULL, Q_EMPTY = Q_FULL + NQS, RING_FULL = Q_EMPTY + NQS, RING_EMPTY = RING_FULL + NS,
    S_FULL = RING_EMPTY + NS, P_FULL = S_FULL + NQ, O_DONE = P_FULL + NQ, O_FREE = O_DONE + NQ,
    ITEM_FULL = O_FREE + NQ, ITEM_EMPTY = ITEM_FULL + NITEM, TOK = ITEM_EMPTY + NITEM,
    DRAIN = TOK + NQ, INVL_FULL = DRAIN + NQ, INVL_EMPTY = INVL_FULL + NQ, NUM_BARS = INVL_EMPTY + NQ
  };
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int ITEM_OFF = MISC_OFF + 16;           // NITEM claimed work items (ItemEntry)
  static constexpr int BYTES = ITEM_OFF + NITEM * (int)sizeof(ItemEntry);
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 bytes
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(TILE % 1024 == 0 && RING_OFF % 1024 == 0,
                "128-byte-swizzled tiles need 1024-byte alignment");
  static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
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

__device__ __forceinline__ void zero_row(const Params& p, int bh, int row, int D) {
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)bh * p.Sq + row) * D);
  for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
  if (p.lse) p.lse[(size_t)bh * p.Sq + row] = -INFINITY;
}

// The same for a row of the token-major layouts (O row stride o_rstride, LSE [Hq, total_q]).
__device__ __forceinline__ void zero_row_tm(const Params& p, const Seq& s, int hq, int row, int D) {
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                        (size_t)(s.q0 + row) * p.o_rstride + (size_t)hq * D);
  for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
  if (p.lse) p.lse[(size_t)hq * p.total_q + s.q0 + row] = -INFINITY;
}

// KV tiles a Q tile starting at row m0 needs, and the first that may need masking.
__device__ __forceinline__ void tile_range(const Params& p, int m0, int* n_tiles, int* mask_from) {
  if (m0 >= p.Sq) {
    *n_tiles = 0;
    *mask_from = 0;
    return;
  }
  const int last_row = min(m0 + BM, p.Sq) - 1;
  const int delta = p.Skv - p.Sq;
  int n_keys = p.Skv;
  if (p.causal) n_keys = max(0, min(p.Skv, last_row + delta + 1));
  *n_tiles = (n_keys + BN - 1) / BN;
  int mf = p.Skv / BN;
  if (p.causal) mf = min(mf, max(0, m0 + delta + 1) / BN);
  *mask_from = mf;
}

// Token-major kernels: the KV tiles [*lo, *hi) that a Q tile at row m0 of sequence s
// needs (*lo == *hi: none), the first tile *mr holding a key past some row's right
// bound or past the keys, and the tile *ml below which tiles hold a key before some
// row's left bound.  Row i of the sequence keeps keys
// [i + d - win_left, i + d + win_right] of [0, nk), d = nk - nq (-1: no bound).
__device__ __forceinline__ void tile_span(const Params& p, const Seq& s, int m0, int* lo, int* hi,
                                          int* mr, int* ml) {
  *lo = *hi = *mr = *ml = 0;
  if (m0 >= s.nq || s.nk <= 0) return;
  const int last_row = min(m0 + BM, s.nq) - 1;
  const int delta = s.nk - s.nq;
  int k_hi = s.nk - 1, r0 = s.nk;  // last key of any row; first key past row m0's right bound
  if (p.win_right >= 0) {
    k_hi = min(k_hi, last_row + delta + p.win_right);
    r0 = min(r0, max(0, m0 + delta + p.win_right + 1));
  }
  int k_lo = 0, l1 = 0;  // first key of any row; first key of the last row
  if (p.win_left >= 0) {
    k_lo = max(0, m0 + delta - p.win_left);
    l1 = max(0, last_row + delta - p.win_left);
  }
  if (k_hi < k_lo) return;
  *lo = k_lo / BN;
  *hi = k_hi / BN + 1;
  *mr = r0 / BN;
  *ml = (l1 + BN - 1) / BN;
}

// The KV tiles of a token-major work item (two Q tiles from row m_base): both Q
// tiles step through tiles t0 .. t0 + n_kv - 1; Q tile qi multiplies steps
// [a, e) of them and masks tiles at or after mr and before ml per key.
struct ItemTiles {
  int t0, n_kv, a, e, mr, ml;
};

__device__ __forceinline__ ItemTiles item_tiles(const Params& p, const Seq& s, int m_base, int qi) {
  static_assert(NQ == 2, "two Q tiles per item");
  int lo0, hi0, mr0, ml0, lo1, hi1, mr1, ml1;
  tile_span(p, s, m_base, &lo0, &hi0, &mr0, &ml0);
  tile_span(p, s, m_base + BM, &lo1, &hi1, &mr1, &ml1);
  // rows grow with the tile, so tile 1's keys never start before tile 0's
  const bool ne0 = hi0 > lo0, ne1 = hi1 > lo1;
  ItemTiles it;
  it.t0 = ne0 ? lo0 : (ne1 ? lo1 : 0);
  it.n_kv = (ne1 ? hi1 : (ne0 ? hi0 : 0)) - it.t0;
  const bool ne = qi == 0 ? ne0 : ne1;
  it.a = ne ? (qi == 0 ? lo0 : lo1) - it.t0 : 0;
  it.e = ne ? (qi == 0 ? hi0 : hi1) - it.t0 : 0;
  it.mr = qi == 0 ? mr0 : mr1;
  it.ml = qi == 0 ? ml0 : ml1;
  return it;
}

// Work item w -> (256-row block, batch, query head).  Items are grouped by
// heads_per_group consecutive (batch, head) rows, chosen on the host so that a
// group's K and V stay resident in L2; inside a group the blocks go from the
// last (most causal work) to the first, heads innermost, so CTAs working at the
// same time share KV heads and the longest items start first.
__device__ __forceinline__ void decode_item(const Params& p, int w, int* mb, int* hq, int* b) {
  const int BH = p.B * p.Hq;
  const int full = p.num_m_blocks * p.heads_per_group;
  const int gi = w / full;
  const int g0 = gi * p.heads_per_group;
  const int size = min(p.heads_per_group, BH - g0);
  const int off = w - gi * full;
  const int hb = g0 + off % size;
  *mb = p.num_m_blocks - 1 - off / size;
  *b = hb / p.Hq;
  *hq = hb % p.Hq;
}


template <int D, bool BF16, bool VL>
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
  const int n_items = p.num_m_blocks * p.Hq * p.B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQS; ++s) {
      mbar_init(bar(L::Q_FULL + s), 1);
      mbar_init(bar(L::Q_EMPTY + s), 1);  // the issuer of the tile in the slot
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::RING_FULL + s), 1);
      mbar_init(bar(L::RING_EMPTY + s), NQ);  // freed by both softmax warpgroups (see there)
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(bar(L::S_FULL + i), 1);
      mbar_init(bar(L::P_FULL + i), BM);
      mbar_init(bar(L::O_DONE + i), 1);
      mbar_init(bar(L::O_FREE + i), BM);
      mbar_init(bar(L::TOK + i), 1);  // issuer i finished issuing a batch
      mbar_init(bar(L::DRAIN + i), 1);
      mbar_init(bar(L::INVL_FULL + i), BM);   // written by softmax warpgroup i
      mbar_init(bar(L::INVL_EMPTY + i), BM);  // read by the epilogue warpgroup
    }
    for (int q = 0; q < NITEM; ++q) {
      mbar_init(bar(L::ITEM_FULL + q), 1);
      // the K/V loader, the MMA issuers, the softmax warps and the epilogue warps
      mbar_init(bar(L::ITEM_EMPTY + q), 1 + NQ + NQ * 4 + 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  volatile ItemEntry* item_q = reinterpret_cast<volatile ItemEntry*>(smem + L::ITEM_OFF);
  if (warp == QLOAD_WARP && lane == 0) {
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

  // Everything the loaders and issuers need about work item w, computed once by the
  // thread that claims it.
  auto fill_entry = [&](int w, volatile ItemEntry* q) {
    int mb, hq, b;
    decode_item(p, w, &mb, &hq, &b);
    const int m_base = mb * (NQ * BM);
    q->w = w;
    if constexpr (VL) {
      const Seq sq = seq_of(p, b);
      const ItemTiles t0 = item_tiles(p, sq, m_base, 0), t1 = item_tiles(p, sq, m_base, 1);
      q->n_kv = t0.n_kv;
      q->a[0] = t0.a;
      q->e[0] = t0.e;
      q->a[1] = t1.a;
      q->e[1] = t1.e;
      q->q_y = sq.q0 + m_base;
      q->q_z = hq;
      q->k_y0 = sq.k0 + t0.t0 * BN;
      q->kv_z = hq / p.group;
    } else {
      int n_t[NQ], mf[NQ];
      for (int i = 0; i < NQ; ++i) tile_range(p, m_base + i * BM, &n_t[i], &mf[i]);
      q->n_kv = max(n_t[0], n_t[1]);
      q->a[0] = 0;
      q->e[0] = n_t[0];
      q->a[1] = 0;
      q->e[1] = n_t[1];
      q->q_y = m_base;
      q->q_z = b * p.Hq + hq;
      q->k_y0 = 0;
      q->kv_z = b * p.Hkv + hq / p.group;
    }
  };

  // register split: 128 threads x 72 (loaders, issuers) + 128 x 56 (epilogue) + 256 x 192
  // (softmax) = 512 threads x 128, the launch allotment (ptxas allocates each region
  // within its new limit)
  if (warp >= KV_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    if (warp == QLOAD_WARP) {
      // ------------------------------------------ work items and Q tiles (one thread)
      // Claims work items from the counter and queues them for every other role,
      // then loads the item's two Q tiles into a ring of three single-tile slots;
      // a slot is free once the last S MMA of its previous tile has completed, so
      // the next item's first Q tile is usually resident long before it is needed.
      if (lane == 0) {
        const uint64_t pol_q = policy_evict_first();
        int qt = 0;  // Q tiles loaded
        bool ok = true;
        for (int r = 0; ok; ++r) {
          const int qs = r % NITEM;
          if (!(ok = mbar_wait<false>(bar(L::ITEM_EMPTY + qs), ((r / NITEM) & 1) ^ 1, abort_flag,
                               &g_status, lim)))
            break;
          int w = atomicAdd(p.work_counter, 1);
          if (w >= n_items) w = -1;
          volatile ItemEntry* q = item_q + qs;
          if (w >= 0) fill_entry(w, q);
          else q->w = -1;
          const int n_kv = w >= 0 ? q->n_kv : 0, q_y = q->q_y, q_z = q->q_z;
          mbar_arrive(bar(L::ITEM_FULL + qs));
          if (w < 0) break;
          if (n_kv == 0) continue;
          for (int i = 0; i < NQ && ok; ++i, ++qt) {
            const int s = qt % NQS;
            if (!(ok = mbar_wait<false>(bar(L::Q_EMPTY + s), ((qt / NQS) & 1) ^ 1, abort_flag, &g_status, lim)))
              break;
            mbar_expect_tx(bar(L::Q_FULL + s), L::TILE);
            for (int rr = 0; rr < L::NREG; ++rr)
              tma_load_3d(sb + L::Q_OFF + s * L::TILE + rr * L::REGION, &tmq, bar(L::Q_FULL + s),
                          rr * 64, q_y + i * BM, q_z, pol_q);
          }
        }
        // every copy issued must have landed before the CTA may exit
        for (int t = max(0, qt - NQS); t < qt; ++t)
          drain_wait(bar(L::Q_FULL + t % NQS), (t / NQS) & 1, lim);
      }
      __syncwarp();
    } else if (warp == KV_WARP) {
      // ---------------------------------------------------- K/V loader (one thread)
      if (lane == 0) {
        const uint64_t pol_kv = policy_evict_last();
        int ld = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
          const int qs = r % NITEM;
          if (!(ok = mbar_wait<false>(bar(L::ITEM_FULL + qs), (r / NITEM) & 1, abort_flag, &g_status, lim)))
            break;
          const int w = item_q[qs].w;
          const int n_kv = item_q[qs].n_kv, k_y0 = item_q[qs].k_y0, kv_z = item_q[qs].kv_z;
          mbar_arrive(bar(L::ITEM_EMPTY + qs));
          if (w < 0) break;
          for (int l = 0; l < 2 * n_kv; ++l, ++ld) {  // K_0, V_0, K_1, V_1, ...
            const int s = ld % NS;
            if (!(ok = mbar_wait<false>(bar(L::RING_EMPTY + s), ((ld / NS) & 1) ^ 1, abort_flag, &g_status,
                                 lim)))
              break;
            if (p.debug_fault == 1 && ld == 1) continue;  // withhold V_0: consumers must time out
            mbar_expect_tx(bar(L::RING_FULL + s), L::TILE);
            const CUtensorMap* tm = (l & 1) ? &tmv : &tmk;
            for (int rr = 0; rr < L::NREG; ++rr)
              tma_load_3d(sb + L::RING_OFF + s * L::TILE + rr * L::REGION, tm,
                          bar(L::RING_FULL + s), rr * 64, k_y0 + (l >> 1) * BN, kv_z, pol_kv);
          }
        }
        for (int l = max(0, ld - NS); l < ld; ++l) {
          if (p.debug_fault == 1 && l == 1) continue;
          drain_wait(bar(L::RING_FULL + l % NS), (l / NS) & 1, lim);
        }
      }
      __syncwarp();
    } else if (warp == MMA_WARP || warp == MMA_WARP + 1) {
      // ------------------------------------------------ MMA issuers, one per Q tile
      const int qi = warp - MMA_WARP;
      if (lane == 0) {
        const uint32_t abort_s = smem_u32(misc + 1);
        constexpr uint32_t idesc_qk = umma_idesc_f16(BF16, BM, BN, false, false);
        constexpr uint32_t idesc_pv = umma_idesc_f16(BF16, BM, D, false, true);
        auto ring_wait = [&](int ld) -> bool {
          return mbar_wait_s(bar(L::RING_FULL + ld % NS), (ld / NS) & 1, abort_s, &g_status, lim);
        };
        // Shared-memory descriptors are built once; every MMA then only adds an
        // offset to the 14-bit start-address field (addresses stay below 256 KB,
        // so the addition never carries out of the field).
        // 128-byte-swizzle descriptors: the high half is one constant (stride 1024
        // bytes); the low half holds the start address and the leading byte offset
        // (16 bytes for the K-major Q and K, one 64-column region for the MN-major V)
        const uint32_t d_hi = (uint32_t)(sdesc_sw128(sb, 16, 1024) >> 32);
        const uint32_t q_lo = (uint32_t)sdesc_sw128(sb + L::Q_OFF, 16, 1024);
        const uint32_t k_lo = (uint32_t)sdesc_sw128(sb + L::RING_OFF, 16, 1024);
        const uint32_t v_lo = (uint32_t)sdesc_sw128(sb + L::RING_OFF, L::REGION, 1024);
        const uint32_t t_s = tmem + COL_S + 128u * qi, t_o = tmem + COL_O + 128u * qi;
        // S = Q K^T with Q in slot qs and K in the ring slot of load ld (the start
        // addresses stay below 256 KB, so the additions never leave their field)
        auto issue_s = [&](int qs, int ld) {
          const uint32_t a0 = q_lo + (uint32_t)((qs * L::TILE) >> 4);
          const uint32_t b0 = k_lo + (uint32_t)(((ld % NS) * L::TILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // K-major operands: 16 columns = 32 bytes inside a 128-byte swizzled row
            const uint32_t off = ((kk >> 2) * L::REGION + (kk & 3) * 32) >> 4;
            umma_ss_lo(t_s, a0 + off, d_hi, b0 + off, d_hi, idesc_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(L::S_FULL + qi));
        };
        auto issue_pv = [&](int ld, bool acc) {  // O += P V, V in the ring slot of ld
          // V is [key][d] (d contiguous): MN-major B, 16 keys = 2 swizzle atoms of 8 rows;
          // LBO steps to the next 64-column block of d, SBO to the next 8 keys.
          const uint32_t b0 = v_lo + (uint32_t)(((ld % NS) * L::TILE) >> 4);
          umma_ts_lo(t_o, t_s, b0, d_hi, idesc_pv, acc ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < BN / 16; ++kk) umma_ts_lo(t_o, t_s + kk * 8, b0 + kk * 128, d_hi, idesc_pv, 1u);
        };
        struct Steps {
          int n_kv, a, e;  // the item's KV steps; this tile multiplies steps [a, e)
        };
        // An item's first batch: S(0), or only the commit of an empty step when this
        // tile multiplies nothing there; the Q slot is released after the tile's last S.
        auto first_s = [&](const Steps& it, int qs, int ld) {
          if (it.a <= 0 && 0 < it.e) issue_s(qs, ld);
          else umma_commit(bar(L::S_FULL + qi));
          if (it.e == it.a) mbar_arrive(bar(L::Q_EMPTY + qs));
          else if (it.e == 1) umma_commit(bar(L::Q_EMPTY + qs));  // this tile's last S
        };
        // The two issuers hand a token back and forth, so their batches reach the
        // tensor core in the order P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1): S_0 then
        // completes a tile's worth of MMAs before S_1 and the softmax warpgroups
        // alternate.  Each issuer makes its other waits (its P, the K/V ring, O
        // free) while the other one's batch executes; only the hand-off lies
        // between two batches, and the tensor core queues just a couple of MMAs.
        // Both Q tiles step through every KV tile of an item: the shorter one's
        // extra steps are empty batches (a commit, no MMA) that keep the two in
        // step and release ring slots in order.  The batches run on across items:
        // an item's last batch, P V(n_kv - 1) (or nothing, for the causal
        // diagonal's shorter tile), carries the next item's S(0), so that S runs
        // while the other tile finishes the item.  Both issuers therefore issue
        // 1 + sum(n_kv) batches, and the token alternates to the end.
        int g = 0;  // batches issued
        auto token_wait = [&]() -> bool {
          if (qi == 0) return g == 0 || mbar_wait_s(bar(L::TOK + 1), (g - 1) & 1, abort_s, &g_status, lim);
          return mbar_wait_s(bar(L::TOK + 0), g & 1, abort_s, &g_status, lim);
        };
        auto token_pass = [&]() {
          tc_fence_before();
          mbar_arrive(bar(L::TOK + qi));
          ++g;
        };
        int r = 0;  // items taken from the queue
        // the next queued item with keys (or w < 0: none left); false if a wait gave up
        auto next_item = [&](int* w, Steps* it) -> bool {
          for (;;) {
            const int qs = r % NITEM;
            if (!mbar_wait_s(bar(L::ITEM_FULL + qs), (r / NITEM) & 1, abort_s, &g_status, lim))
              return false;
            *w = item_q[qs].w;
            it->n_kv = item_q[qs].n_kv;
            it->a = item_q[qs].a[qi];
            it->e = item_q[qs].e[qi];
            mbar_arrive(bar(L::ITEM_EMPTY + qs));
            ++r;
            if (*w < 0 || it->n_kv > 0) return true;
          }
        };
        // Q tile qi of the k-th item with keys sits in slot (2 k + qi) mod NQS
        auto q_wait = [&](int k) -> bool {
          const int t = 2 * k + qi;
          return mbar_wait_s(bar(L::Q_FULL + t % NQS), (t / NQS) & 1, abort_s, &g_status, lim);
        };
        int t_cnt = 0, n_done = 0;
        int w;
        Steps cur;
        bool ok = next_item(&w, &cur);
        // ---- the first batch of all: S(0) of the first item
        if (ok && w >= 0) {
          ok = q_wait(0) && ring_wait(0) && token_wait();
          if (ok) {
            tc_fence_after();
            first_s(cur, qi % NQS, 0);
            token_pass();
          }
        }
        for (int k = 0, base = 0; ok && w >= 0; ++k) {
          const int qs = (2 * k + qi) % NQS;
          const int ld_next = base + 2 * cur.n_kv;  // K_0 of the next item
          int w_next = -1;
          Steps nxt{};
          // ---- one batch per KV tile j < n_kv - 1: P V(j), then S(j+1)
          for (int j = 0; j + 1 < cur.n_kv; ++j) {
            const int ld_v = base + 2 * j + 1, ld_k = base + 2 * j + 2;
            const bool has_pv = cur.a <= j && j < cur.e;
            if (!(ok = ring_wait(ld_v) && ring_wait(ld_k))) break;
            if (!(ok = mbar_wait_s(bar(L::P_FULL + qi), t_cnt & 1, abort_s, &g_status, lim))) break;
            ++t_cnt;
            // the first P V of an item overwrites O: the last epilogue must have read it
            if (j == cur.a && has_pv && n_done > 0 &&
                !(ok = mbar_wait_s(bar(L::O_FREE + qi), (n_done - 1) & 1, abort_s, &g_status, lim)))
              break;
            if (!(ok = token_wait())) break;
            tc_fence_after();
            if (has_pv) issue_pv(ld_v, j > cur.a);
            if (cur.a <= j + 1 && j + 1 < cur.e) {
              issue_s(qs, ld_k);  // after P V(j), which read P from these columns
              if (j + 1 == cur.e - 1) umma_commit(bar(L::Q_EMPTY + qs));  // this tile's last S
            } else {
              umma_commit(bar(L::S_FULL + qi));  // an empty step for this tile
            }
            token_pass();
          }
          if (!ok) break;
          // ---- the item's last batch: P V(n_kv - 1) (if this tile has it), then the
          // next item's S(0)
          {
            const int j = cur.n_kv - 1, ld_v = base + 2 * j + 1;
            const bool has_pv = cur.a <= j && j < cur.e;
            if (!(ok = ring_wait(ld_v))) break;
            if (!(ok = mbar_wait_s(bar(L::P_FULL + qi), t_cnt & 1, abort_s, &g_status, lim))) break;
            ++t_cnt;
            if (j == cur.a && has_pv && n_done > 0 &&
                !(ok = mbar_wait_s(bar(L::O_FREE + qi), (n_done - 1) & 1, abort_s, &g_status, lim)))
              break;
            if (!(ok = next_item(&w_next, &nxt))) break;
            if (w_next >= 0 && !(ok = q_wait(k + 1) && ring_wait(ld_next))) break;
            if (!(ok = token_wait())) break;
            tc_fence_after();
            if (has_pv) issue_pv(ld_v, j > cur.a);
            umma_commit(bar(L::O_DONE + qi));
            ++n_done;
            // after P V(j), which read P from these columns
            if (w_next >= 0) first_s(nxt, (2 * (k + 1) + qi) % NQS, ld_next);
            token_pass();
          }
          base = ld_next;
          w = w_next;
          cur = nxt;
        }
        umma_commit(bar(L::DRAIN + qi));  // fires once every MMA issued above has completed
        drain_wait(bar(L::DRAIN + qi), 0, lim);
      }
      __syncwarp();
    }
  } else if (warp >= EPI_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    // ------------------------------------------------ epilogue (rows of both Q tiles)
    // Thread r owns TMEM lane r, i.e. row r of either Q tile.  Once O_i of an item
    // is complete it reads the row 32 columns at a time, hands O_i back to its
    // issuer (O_FREE) as soon as the last piece is in registers, multiplies by the
    // 1 / l the softmax warpgroup left in shared memory, rounds, and stores the
    // row (rows past the queries are not written).  Nothing here is on the
    // softmax warps' path.
    const int r_lane = threadIdx.x & 127;
    const uint32_t lane_t = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float* inv_l_s = reinterpret_cast<const float*>(smem + L::INVL_OFF);
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(b_, ph_, abort_flag, &g_status, lim));
    };
    int u_cnt = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int qs = r % NITEM;
      if (!(ok = wait_warp(bar(L::ITEM_FULL + qs), (r / NITEM) & 1))) break;
      const int w = item_q[qs].w, n_kv = item_q[qs].n_kv;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::ITEM_EMPTY + qs));
      if (w < 0) break;
      if (n_kv == 0) continue;  // no key for the item: the softmax wrote its rows
      int mb, hq, b;
      decode_item(p, w, &mb, &hq, &b);
      const int m_base = mb * (NQ * BM);
      int n_rows = p.Sq;  // query rows of the sequence
      uint16_t* o_base = static_cast<uint16_t*>(p.o) + ((size_t)(b * p.Hq + hq) * p.Sq) * D;
      size_t o_stride = D;
      if constexpr (VL) {
        const Seq sq = seq_of(p, b);
        n_rows = sq.nq;
        o_base = static_cast<uint16_t*>(p.o) + (size_t)sq.q0 * p.o_rstride + (size_t)hq * D;
        o_stride = (size_t)p.o_rstride;
      }
      for (int qi = 0; qi < NQ; ++qi) {
        const int row = m_base + qi * BM + r_lane;
        if (!(ok = wait_warp(bar(L::INVL_FULL + qi), u_cnt & 1))) break;
        const float inv_l = inv_l_s[qi * BM + r_lane];  // 0: no visible key, O = 0
        mbar_arrive(bar(L::INVL_EMPTY + qi));
        if (!(ok = wait_warp(bar(L::O_DONE + qi), u_cnt & 1))) break;
        tc_fence_after();
        const uint32_t t_o = lane_t + COL_O + 128u * qi;
        uint16_t* dst = o_base + (size_t)row * o_stride;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_o + 32u * c, v);
          if (c == D / 32 - 1) {  // the whole row is in registers: O_i may be overwritten
            tc_fence_before();
            mbar_arrive(bar(L::O_FREE + qi));
          }
          if (row < n_rows) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                pk[i] = inv_l > 0.f ? pack2<BF16>(__uint_as_float(v[16 * h + 2 * i]) * inv_l,
                                                  __uint_as_float(v[16 * h + 2 * i + 1]) * inv_l)
                                    : 0u;
              uint16_t* d16 = dst + 32 * c + 16 * h;
              if (p.o_align32) {
                st_global_v8(d16, pk);  // whole 32-byte sectors in one store
              } else {
                reinterpret_cast<uint4*>(d16)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                reinterpret_cast<uint4*>(d16)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              }
            }
          }
        }
      }
      ++u_cnt;
    }
  } else {

    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ------------------------------------------------ softmax (rows)
    const int qi = warp >> 2;             // Q tile of this warpgroup
    const int r_lane = threadIdx.x & 127; // TMEM lane == tile row
    const uint32_t lane_t = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t t_s = lane_t + COL_S + 128u * qi;
    const uint32_t t_o = lane_t + COL_O + 128u * qi;
    const float mval = p.neg ? INFINITY : -INFINITY;
    const float c2 = p.c2;
    // tcgen05.ld/st are warp-collective: every wait outcome and every rescale
    // decision below is made uniform across the warp before TMEM is touched.
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(b_, ph_, abort_flag, &g_status, lim));
    };
    float* inv_l_s = reinterpret_cast<float*>(smem + L::INVL_OFF);
    int t_cnt = 0, u_cnt = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int qs = r % NITEM;
      if (!(ok = wait_warp(bar(L::ITEM_FULL + qs), (r / NITEM) & 1))) break;
      const int w = item_q[qs].w;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::ITEM_EMPTY + qs));
      if (w < 0) break;
      int mb, hq, b;
      decode_item(p, w, &mb, &hq, &b);
      const int bh = b * p.Hq + hq;
      const int m0 = mb * (NQ * BM) + qi * BM;
      const int row = m0 + r_lane;
      // Both Q tiles step through every KV tile of the item; outside its own steps
      // [a_own, e_own) a step only passes the barriers (its issuer multiplies nothing
      // there).  Tile t0 + t at or after mfrom (or before mleft) is masked per key.
      int n_tiles, a_own, e_own, mfrom, mleft = 0, t0 = 0;
      int first_key = 0, last_key;  // the keys this row may see (last_key < first_key: none)
      Seq sq{};
      if constexpr (VL) {
        sq = seq_of(p, b);
        const ItemTiles it = item_tiles(p, sq, mb * (NQ * BM), qi);
        n_tiles = it.n_kv;
        a_own = it.a;
        e_own = it.e;
        mfrom = it.mr;
        mleft = it.ml;
        t0 = it.t0;
        if (n_tiles == 0) {  // no key for the whole item
          if (row < sq.nq) zero_row_tm(p, sq, hq, row, D);
          continue;
        }
        const int d = sq.nk - sq.nq;
        last_key = sq.nk - 1;
        if (p.win_right >= 0) last_key = min(last_key, row + d + p.win_right);
        if (p.win_left >= 0) first_key = row + d - p.win_left;
      } else {
        int n_own, n_oth, mf_oth;
        tile_range(p, m0, &n_own, &mfrom);
        tile_range(p, m0 + (qi == 0 ? BM : -BM), &n_oth, &mf_oth);
        n_tiles = max(n_own, n_oth);
        a_own = 0;
        e_own = n_own;
        if (n_tiles == 0) {  // no key for the whole item
          if (row < p.Sq) zero_row(p, bh, row, D);
          continue;
        }
        last_key = p.causal ? min(row + (p.Skv - p.Sq), p.Skv - 1) : p.Skv - 1;
      }
      float m_used = -INFINITY, l_sum = 0.f;
      for (int t = 0; t < n_tiles; ++t, ++t_cnt) {
        if (!(ok = wait_warp(bar(L::S_FULL + qi), t_cnt & 1))) break;
        tc_fence_after();
        if (r_lane == 0) {
          // Both Q tiles step through every KV tile, so S_i number t_cnt belongs to the
          // K of load 2 t_cnt (loads alternate K, V).  Its issuer issued it (or the
          // empty step's commit) after every MMA of its own that reads that K or the V
          // before it, so its completion frees this tile's use of both ring slots;
          // each slot takes one arrival per Q tile.  This warpgroup consumes every
          // completion of S_i in order and the next S_i needs its P, which keeps the
          // ring protocol exact.
          if (t_cnt > 0) mbar_arrive(bar(L::RING_EMPTY + (2 * t_cnt - 1) % NS));
          mbar_arrive(bar(L::RING_EMPTY + (2 * t_cnt) % NS));
        }
        if (t < a_own || t >= e_own) {  // an empty step: no S was computed for this tile
          tc_fence_before();
          mbar_arrive(bar(L::P_FULL + qi));
          continue;
        }
        float x[BN];
        {
          static_assert(BN == 128, "one S row is two 64-column TMEM loads");
          uint32_t rr[BN];
          tmem_ld64x2(t_s, rr);  // the whole S row in one TMEM round trip
#pragma unroll
          for (int i = 0; i < BN; ++i) x[i] = __uint_as_float(rr[i]);
        }
        if (p.zero) {
#pragma unroll
          for (int j = 0; j < BN; ++j) x[j] = 0.f;
        }
        if constexpr (VL) {
          // keys [first_key, last_key] of the row, relative to this tile; a tile at or
          // after mleft holds no key before any row's left bound and a tile before mfrom
          // none past any row's right bound, so it tests only the side it can cross
          const int tk = t0 + t;
          const int lo_v = first_key - tk * BN, hi_v = last_key + 1 - tk * BN;
          if (tk >= mfrom && tk >= mleft) {
#pragma unroll
            for (int j = 0; j < BN; ++j) x[j] = (j < hi_v) ? x[j] : mval;
          } else if (tk < mleft && tk < mfrom) {
#pragma unroll
            for (int j = 0; j < BN; ++j) x[j] = (j >= lo_v) ? x[j] : mval;
          } else if (tk < mleft) {
#pragma unroll
            for (int j = 0; j < BN; ++j) x[j] = (j >= lo_v && j < hi_v) ? x[j] : mval;
          }
        } else if (t >= mfrom) {
          // keys [t BN, t BN + vis) of this tile are visible: one compare and select per key
          const int vis = last_key + 1 - t * BN;
#pragma unroll
          for (int j = 0; j < BN; ++j) x[j] = (j < vis) ? x[j] : mval;
        }
        // row max (min when scale < 0): chain u covers x[u + 8k], k = 0..15, with
        // three-input max: (k = 0, 1, 2), then (3, 4), ..., (13, 14), then k = 15
        static_assert(BN == 128, "chains below cover exactly 128 columns");
        float a[8];
        if (!p.neg) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            a[u] = fmax3(x[u], x[u + 8], x[u + 16]);
#pragma unroll
            for (int k = 3; k < 15; k += 2) a[u] = fmax3(a[u], x[u + 8 * k], x[u + 8 * k + 8]);
            a[u] = fmaxf(a[u], x[u + 120]);
          }
          a[0] = fmax3(a[0], a[1], a[2]);
          a[3] = fmax3(a[3], a[4], a[5]);
          a[0] = fmax3(a[0], a[3], fmaxf(a[6], a[7]));
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            a[u] = fmin3(x[u], x[u + 8], x[u + 16]);
#pragma unroll
            for (int k = 3; k < 15; k += 2) a[u] = fmin3(a[u], x[u + 8 * k], x[u + 8 * k + 8]);
            a[u] = fminf(a[u], x[u + 120]);
          }
          a[0] = fmin3(a[0], a[1], a[2]);
          a[3] = fmin3(a[3], a[4], a[5]);
          a[0] = fmin3(a[0], a[3], fminf(a[6], a[7]));
        }
        const float red = a[0];
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
        const float mu = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t c2p = f2_pack(c2, c2), nmu = f2_pack(-mu, -mu);
        uint64_t ls = f2_pack(0.f, 0.f);
        uint32_t pk[BN / 2];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) {
          const uint64_t xy = fma2(f2_pack(x[2 * i], x[2 * i + 1]), c2p, nmu);
          float a0, a1;
          f2_unpack(xy, a0, a1);
          const uint64_t e = f2_pack(ex2(a0), ex2(a1));
          ls = add2(ls, e);
          float e0, e1;
          f2_unpack(e, e0, e1);
          pk[i] = pack2<BF16>(e0, e1);
        }
        tmem_st(t_s, pk);  // P over the S columns already consumed
        {
          float s0, s1;
          f2_unpack(ls, s0, s1);
          l_sum += s0 + s1;
        }
        if (__any_sync(0xffffffffu, o_scale)) {
          // S_i(t) completed, so every earlier MMA did: O_i holds P V up to tile t-1,
          // and P V(t) waits for this warpgroup's P (rare; 32 columns at a time)
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(t_o + 32u * c, rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha_o);
            tmem_st32(t_o + 32u * c, rr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::P_FULL + qi));
      }
      if (!ok) break;
      // 1 / l of this row for the epilogue warpgroup, once it has taken the last item's
      // (a row with no visible key, or no P V at all, gets 0: O = 0)
      if (!(ok = wait_warp(bar(L::INVL_EMPTY + qi), (u_cnt & 1) ^ 1))) break;
      inv_l_s[qi * BM + r_lane] = l_sum > 0.f ? 1.f / l_sum : 0.f;
      mbar_arrive(bar(L::INVL_FULL + qi));
      ++u_cnt;
      if constexpr (VL) {
        if (p.lse && row < sq.nq)
          p.lse[(size_t)hq * p.total_q + sq.q0 + row] =
              l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
      } else if (p.lse && row < p.Sq) {
        p.lse[(size_t)bh * p.Sq + row] =
            l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
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

// Every row sees no key (Skv == 0): O = 0, LSE = -inf.
__global__ void fill_empty_kernel(uint16_t* o, float* lse, size_t rows, int D) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < rows;
       i += (size_t)gridDim.x * blockDim.x) {
    uint4* dst = reinterpret_cast<uint4*>(o + i * D);
    for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    if (lse) lse[i] = -INFINITY;
  }
}

// 3-D tensor map over 16-bit elements: D contiguous, then n1 rows s1 elements
// apart, then n2 planes s2 elements apart; 64 x 128 x 1 boxes, 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, int D, long long n1, long long n2,
                     long long s1, long long s2, bool bf16) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n1, (cuuint64_t)n2};
  const cuuint64_t strides[2] = {(cuuint64_t)s1 * 2, (cuuint64_t)s2 * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool BF16, bool VL>
static cudaError_t launch_t(const FwdArgs& a, cudaStream_t stream) {
  using L = Layout<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, BF16, VL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tk, tv;
  if (VL) {
    // [tokens, heads, D] with the given token strides; with no keys at all the K/V
    // maps cover one (never read) row of q, since a map cannot be empty
    const long long tk_rows = a.total_k > 0 ? a.total_k : 1;
    const void* kb = a.total_k > 0 ? a.k : a.q;
    const void* vb = a.total_k > 0 ? a.v : a.q;
    const long long kst = a.total_k > 0 ? a.k_rstride : a.q_rstride;
    if (!make_map(&tq, a.q, D, a.total_q, a.Hq, a.q_rstride, D, BF16) ||
        !make_map(&tk, kb, D, tk_rows, a.total_k > 0 ? a.Hkv : 1, kst, D, BF16) ||
        !make_map(&tv, vb, D, tk_rows, a.total_k > 0 ? a.Hkv : 1, kst, D, BF16))
      return cudaErrorInvalidValue;
  } else if (!make_map(&tq, a.q, D, a.Sq, (long long)a.B * a.Hq, D, (long long)a.Sq * D, BF16) ||
             !make_map(&tk, a.k, D, a.Skv, (long long)a.B * a.Hkv, D, (long long)a.Skv * D, BF16) ||
             !make_map(&tv, a.v, D, a.Skv, (long long)a.B * a.Hkv, D, (long long)a.Skv * D, BF16)) {
    return cudaErrorInvalidValue;
  }
  Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.work_counter = a.work_counter;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.group = a.Hq / a.Hkv;
  p.num_m_blocks = (a.Sq + NQ * BM - 1) / (NQ * BM);
  p.causal = a.causal ? 1 : 0;
  const float c2 = a.scale * 1.4426950408889634f;
  p.zero = (c2 == 0.f) ? 1 : 0;
  p.neg = (c2 < 0.f) ? 1 : 0;
  p.c2 = p.zero ? 1.f : c2;
  p.wait_limit_ns = a.wait_limit_ns;
  p.debug_fault = a.debug_fault;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.win_left = a.win_left;
  p.win_right = a.causal ? 0 : a.win_right;
  p.o_rstride = (int)a.o_rstride;
  // rows are multiples of 128 bytes apart in every layout, so the base decides
  p.o_align32 = (reinterpret_cast<uintptr_t>(a.o) % 32) == 0 ? 1 : 0;
  // scheduling groups: as many (batch, head) rows as keep about 64 MB of K and V
  // in L2, rounded to whole GQA groups
  const double kv_head_bytes = 4.0 * (double)(a.Skv > 0 ? a.Skv : 1) * D;  // K and V of one KV head
  const int g = a.Hq / a.Hkv;
  long long hpg = (long long)(64.0 * (1 << 20) / kv_head_bytes) * g;
  if (hpg < g) hpg = g;
  if (hpg > (long long)a.B * a.Hq) hpg = (long long)a.B * a.Hq;
  p.heads_per_group = (int)hpg;
  // persistent: one CTA per SM (or one per work item when there are fewer)
  const long long n_items = (long long)p.num_m_blocks * a.Hq * a.B;
  const int grid = (int)(n_items < a.num_sms ? n_items : a.num_sms);
  attn_fwd_kernel<D, BF16, VL><<<grid, NUM_THREADS, L::ALLOC, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.vl) {
    if (a.D == 64)
      return a.bf16 ? fwd::launch_t<64, true, true>(a, stream) : fwd::launch_t<64, false, true>(a, stream);
    return a.bf16 ? fwd::launch_t<128, true, true>(a, stream) : fwd::launch_t<128, false, true>(a, stream);
  }
  if (a.D == 64)
    return a.bf16 ? fwd::launch_t<64, true, false>(a, stream) : fwd::launch_t<64, false, false>(a, stream);
  return a.bf16 ? fwd::launch_t<128, true, false>(a, stream) : fwd::launch_t<128, false, false>(a, stream);
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
