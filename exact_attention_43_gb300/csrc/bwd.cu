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
// GB300 design, three kernels and no atomics (every gradient is reproducible bit
// for bit):
//  * a prep kernel forms the row term delta_i = sum_d dO_id O_id;
//  * both product kernels are persistent (one CTA per SM claiming work items from a
//    counter) with four roles: a loader thread, an MMA-issuing thread, eight compute
//    warps (two threads per TMEM lane, 64 columns each) and an epilogue warpgroup
//    that reads the finished accumulators, hands them back and stores them while the
//    compute warps start the next item;
//  * the dK/dV kernel's work item is one 128-key tile of one KV head: K and V stay
//    in shared memory, and dK, dV accumulate in TMEM over every query head of the
//    GQA group and every Q tile that sees the keys (causal tiles that see none are
//    skipped).  Per Q tile the issuer puts S^T = K Q^T and dP^T = V dO^T into two
//    TMEM regions, then dV += P^T dO and dK += dS^T Q with A read from TMEM.  The
//    compute warps work in two phases, P^T = 2^(S^T c - LSE_2) and then
//    dS^T = P^T (dP^T - delta), each written back over the columns it came from as
//    16-bit; the MMAs are ordered dV(i), S^T(i+1), dK(i), dP^T(i+1), so each phase
//    runs while the tensor core works on two products of the tile before or after it;
//  * the dQ kernel's work item is one 128-row Q tile (and its dO): it streams the
//    K/V tiles it sees through a 5-slot ring, V before K, like the forward:
//    S = Q K^T (two TMEM buffers, so the next S is computed while this one is used),
//    dP = dO V^T, dS = P (dP - delta) written over S as 16-bit, dQ += dS K
//    accumulated in TMEM and stored once.  Recomputing S and dP costs two more
//    products per (Q tile, KV tile) than one kernel that adds dQ into memory from the
//    dK/dV kernel, but the compute warps then overlap the tensor core instead of
//    waiting on it, and dQ needs no fp32 atomics;
//  * the three kernels are chained by programmatic launches: the dK/dV kernel sets up
//    while the prep kernel's last CTAs run, and the dQ kernel, which reads nothing the
//    dK/dV kernel writes, takes each SM the dK/dV kernel's last items leave.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace ea {
namespace bwd {

__device__ unsigned g_status;

constexpr int BM = 128;        // queries per Q tile
constexpr int BN = 128;        // keys per K/V tile (= TMEM lanes in the dK/dV kernel)
// Warps 0-7 compute, 8-11 the epilogue (reads the accumulators, hands them back, rounds
// and stores), warp 12 loads, warp 13 issues the MMAs (14, 15 idle: setmaxnreg works on
// whole warpgroups).
constexpr int THREADS = 512;
constexpr int EPI_WARP = 8;
constexpr int LOAD_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr int NCOMP = 256;     // compute threads: warps w and w + 4 share TMEM lanes 32 (w mod 4) ...
constexpr int NEPI = 128;      // epilogue threads: one accumulator row (TMEM lane) each
constexpr int NS = 5;          // dQ kernel: K/V ring stages (two and a half K/V steps)
constexpr uint32_t TMEM_COLS = 512;

struct Params {
  const float* lse;    // [B, Hq, Sq], natural log
  const float* delta;  // [B, Hq, Sq]
  uint16_t* dq;        // [B, Hq, Sq, D]
  uint16_t* dk;        // [B, Hkv, Skv, D]
  uint16_t* dv;
  int B, Hq, Hkv, Sq, Skv, group, causal;
  int* work_counter;  // [0] dK/dV, [1] dQ work items claimed; zeroed before the launches
  int per_group;      // dK/dV items: (batch, KV head) planes per scheduling group
  int per_group_q;    // dQ items: (batch, query head) planes per scheduling group
  float c2;        // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
  int debug_fault;  // 3: the dK/dV CTA of work item 0 withholds that item's second Q/dO loads
  // visible keys: key j to query i iff j <= i + d + win_right (win_right >= 0) and
  // j >= i + d - win_left (win_left >= 0), d = (keys) - (queries); causal is win_right 0
  int win_left, win_right;
  // token-major layouts (attn_bwd_varlen, attn_bwd_qkvpacked; the VL kernels): q, o, dO
  // and dq are [tokens, Hq, D], k, v, dk, dv [tokens, Hkv, D] with the row strides
  // below (elements); sequence b's queries are tokens [cu_q[b], cu_q[b+1]) and its
  // keys [cu_k[b], cu_k[b+1]), or b * Sq and b * Skv onwards when cu_q is null; Sq and
  // Skv are then the longest lengths.  LSE and the row terms are [Hq, total_q].
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  long long dq_rstride, dk_rstride;
  int st32;  // dq, dk, dv and their row strides are 32-byte aligned: 32-byte stores
};

// Query and key tokens of one sequence (the token-major layouts), or the dense
// layout's one sequence per (batch, head) plane.
struct Seq {
  int q0, nq;  // first query token, query count
  int k0, nk;  // first key token, key count
};

// Offsets outside the arrays, decreasing offsets and lengths above the longest
// length are clamped (no access leaves the arrays) and reported in the status word.
template <bool VL>
__device__ __forceinline__ Seq seq_of(const Params& p, int b) {
  Seq s;
  if (!VL || !p.cu_q) {
    s.q0 = VL ? b * p.Sq : 0;
    s.nq = p.Sq;
    s.k0 = VL ? b * p.Skv : 0;
    s.nk = p.Skv;
    return s;
  }
  const int a = p.cu_q[b], e = p.cu_q[b + 1], c = p.cu_k[b], f = p.cu_k[b + 1];
  s.q0 = min(max(a, 0), p.total_q);
  s.nq = min(min(max(e, s.q0), p.total_q) - s.q0, p.Sq);
  s.k0 = min(max(c, 0), p.total_k);
  s.nk = min(min(max(f, s.k0), p.total_k) - s.k0, p.Skv);
  if ((s.q0 != a || s.nq != e - a || s.k0 != c || s.nk != f - c) && threadIdx.x == 0)
    atomicOr(&g_status, kStatusSeqLenClamped);
  return s;
}

// dK/dV kernel shared memory: K, V, two Q and two dO buffers, the row vectors.
template <int D>
struct KVLayout {
  static constexpr int REGION = 128 * 128;  // 128 rows x 64 16-bit columns, 128-byte swizzle
  static constexpr int NREG = D / 64;
  static constexpr int TILE = NREG * REGION;  // 128 x D
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE;
  static constexpr int Q_OFF = 2 * TILE;    // two buffers
  static constexpr int DO_OFF = 4 * TILE;   // two buffers
  static constexpr int VEC_OFF = 6 * TILE;  // [2 buffers][LSE_2, delta][BM] of the Q tile
  static constexpr int BAR_OFF = VEC_OFF + 2 * 2 * BM * 4;
  enum {
    KV_FULL, KV_EMPTY, Q_FULL, DO_FULL = Q_FULL + 2, QD_FREE = DO_FULL + 2, S_READY = QD_FREE + 2, DP_READY, P_READY, DS_READY, VEC_READY, DONE, ACC_FREE, ITEM_FULL,
    ITEM_EMPTY = ITEM_FULL + 2, DRAIN = ITEM_EMPTY + 2, NUM_BARS
  };
  // [0] TMEM base, [1] abort flag, [2], [3] the two queued work items
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 bytes
  static_assert(TILE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

// dQ kernel shared memory: the Q tile, its dO tile and a ring of K/V tiles.
template <int D>
struct QLayout {
  static constexpr int REGION = 128 * 128;
  static constexpr int NREG = D / 64;
  static constexpr int TILE = NREG * REGION;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = TILE;
  static constexpr int RING_OFF = 2 * TILE;
  static constexpr int BAR_OFF = RING_OFF + NS * TILE;
  enum {
    // DS_READY + b: dS of a step in TMEM buffer b.  One barrier per buffer: the compute
    // warps may write dS of the next step before the issuer waits for this one; a
    // barrier must never complete two phases ahead of a waiter, and the step after next
    // needs a hand-off from the waiter first.  S has no barrier of its own: a step's S is
    // issued before its dP by the same thread, so DP_READY's commit covers both.
    // RING_FREE + (q & 3): ring loads 2q - 1 and 2q (K of step q - 1, V of step q) may be
    // overwritten, one commit for both; the loader waits for q in order, and q + 4 cannot
    // complete before load 2q + 8 is issued, so no waiter sees a barrier two phases on.
    QD_FULL, QD_EMPTY, RING_FULL, RING_FREE = RING_FULL + NS, DP_READY = RING_FREE + 4,
    DP_FREE, DS_READY, DONE = DS_READY + 2, ACC_FREE, ITEM_FULL,
    ITEM_EMPTY = ITEM_FULL + 2, DRAIN = ITEM_EMPTY + 2, NUM_BARS
  };
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;  // as KVLayout
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(TILE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

// Work item w -> (tile, head, batch).  Items are grouped by `per_group` consecutive
// (batch, head) planes, chosen on the host so that the rows a group streams stay in
// L2; inside a group the tiles go in the order the caller gives (the longest items
// first), heads innermost.  Returns the tile's position in that order.
__device__ __forceinline__ int decode_item(int w, int n_tiles, int planes, int per_group, int* plane) {
  const int full = n_tiles * per_group;
  const int gi = w / full;
  const int g0 = gi * per_group;
  const int size = min(per_group, planes - g0);
  const int off = w - gi * full;
  *plane = g0 + off % size;
  return off / size;
}

// One key tile of one KV head (the dK/dV kernel's work item) and the (query head,
// Q tile) iterations that see it.
struct KVItem {
  int n0, hk, b;
  Seq sq;
  int dlen;              // the bottom-right alignment of the mask
  int m_lo, per_head;    // Q tiles m_lo ... m_lo + per_head - 1 of each query head
  int n_iter;            // group * per_head
  bool skip;             // past the sequence's keys: nothing to compute or write
};

template <bool VL>
__device__ __forceinline__ KVItem kv_item(const Params& p, int n_kt, int w) {
  KVItem it;
  int hb;
  it.n0 = decode_item(w, n_kt, p.B * p.Hkv, p.per_group, &hb) * BN;  // key tiles from the first
  it.b = hb / p.Hkv;
  it.hk = hb % p.Hkv;
  it.sq = seq_of<VL>(p, it.b);
  it.skip = it.n0 >= it.sq.nk;
  it.dlen = it.sq.nk - it.sq.nq;
  // the queries [i_min, i_max] that see a key of this tile
  int i_min = 0, i_max = it.sq.nq - 1;
  if (p.win_right >= 0) i_min = max(0, it.n0 - it.dlen - p.win_right);
  if (p.win_left >= 0) i_max = min(i_max, it.n0 + BN - 1 - it.dlen + p.win_left);
  it.m_lo = i_min / BM;
  it.per_head = i_min <= i_max ? i_max / BM + 1 - it.m_lo : 0;
  it.n_iter = it.skip ? 0 : p.group * it.per_head;
  return it;
}

// One Q tile of one query head (the dQ kernel's work item) and the K/V tiles it sees.
struct QItem {
  int m0, h, b;
  Seq sq;
  int dlen;
  int t_lo, n_kv;  // K/V tiles t_lo ... t_lo + n_kv - 1
  bool skip;       // past the sequence's queries: nothing to compute or write
};

template <bool VL>
__device__ __forceinline__ QItem q_item(const Params& p, int n_mt, int w) {
  QItem it;
  int hb;
  const int mi = decode_item(w, n_mt, p.B * p.Hq, p.per_group_q, &hb);
  // with a right bound (causal) the last Q tiles see the most keys: they go first
  it.m0 = (p.win_right >= 0 ? n_mt - 1 - mi : mi) * BM;
  it.b = hb / p.Hq;
  it.h = hb % p.Hq;
  it.sq = seq_of<VL>(p, it.b);
  it.skip = it.m0 >= it.sq.nq;
  it.dlen = it.sq.nk - it.sq.nq;
  // the keys [k_lo, k_hi] some row of this tile sees
  const int last_row = min(it.m0 + BM, it.sq.nq) - 1;
  int k_lo = 0, k_hi = it.sq.nk - 1;
  if (p.win_right >= 0) k_hi = min(k_hi, last_row + it.dlen + p.win_right);
  if (p.win_left >= 0) k_lo = max(0, it.m0 + it.dlen - p.win_left);
  it.t_lo = k_lo / BN;
  it.n_kv = (!it.skip && k_lo <= k_hi) ? k_hi / BN + 1 - it.t_lo : 0;
  return it;
}

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

// 32 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape), issued and not
// waited for: the registers are valid only after tmem_wait_ld_regs on them.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr)
               : "memory");
}

// Wait for this thread's TMEM loads; the registers pass through the statement, so no use
// of them can be scheduled above it.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]),
        "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]),
        "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]),
        "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
        "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]),
        "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]),
        "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
               :
               : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (not waited for).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}

// a * b on both lanes of two packed f32 values (sm_100 and later: one instruction).
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 32 consecutive fp32 values of a TMEM row, times f, as 16-bit values at dst (64 bytes):
// two 32-byte stores, each a whole sector, when dst is 32-byte aligned, else four
// 16-byte ones.
template <bool BF16>
__device__ __forceinline__ void store_row32(void* dst, const uint32_t (&v)[32], float f, bool st32) {
  if (st32) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pk[i] = pack2<BF16>(__uint_as_float(v[16 * h + 2 * i]) * f, __uint_as_float(v[16 * h + 2 * i + 1]) * f);
      st_global_v8(static_cast<char*>(dst) + 32 * h, pk);
    }
  } else {
    uint4* d = static_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = pack8<BF16>(v + 8 * i, f);
  }
}

// delta_i = sum_d dO_id O_id (rows of D contiguous elements).  D / 8 lanes share a row,
// one 16-byte load of O and of dO each; a warp covers 256 / D rows per load and issues
// the loads of DELTA_UNROLL such groups before reducing any, so enough bytes are in
// flight to keep HBM busy.  With hq_tm > 0 the rows are token-major ([tokens, hq_tm, D])
// and the result goes to the [Hq, total_q] layout of the LSE; otherwise to row order.
constexpr int DELTA_UNROLL = 4;
constexpr int DELTA_THREADS = 256;

template <int D>
constexpr int delta_rows_per_block() {
  return (DELTA_THREADS / 32) * (256 / D) * DELTA_UNROLL;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(DELTA_THREADS) bwd_delta_kernel(const uint16_t* o, const uint16_t* dout,
                                                                  float* delta, long long rows, int hq_tm,
                                                                  long long total_q) {
  constexpr int LPR = D / 8;          // lanes per row
  constexpr int RPW = 32 / LPR;       // rows per warp per load
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  const long long row0 = (long long)blockIdx.x * delta_rows_per_block<D>() + (long long)warp * RPW * DELTA_UNROLL;
  griddep_launch_dependents();  // the dK/dV kernel may start setting up on SMs this grid leaves
  uint4 a[DELTA_UNROLL], g[DELTA_UNROLL];
#pragma unroll
  for (int u = 0; u < DELTA_UNROLL; ++u) {
    const long long row = row0 + u * RPW + sub;
    if (row < rows) {
      a[u] = reinterpret_cast<const uint4*>(o + row * D)[part];
      g[u] = reinterpret_cast<const uint4*>(dout + row * D)[part];
    } else {
      a[u] = make_uint4(0, 0, 0, 0);
      g[u] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int u = 0; u < DELTA_UNROLL; ++u) {
    const uint32_t* x = reinterpret_cast<const uint32_t*>(&a[u]);
    const uint32_t* y = reinterpret_cast<const uint32_t*>(&g[u]);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 xv = unpack2<BF16>(x[e]);
      const float2 yv = unpack2<BF16>(y[e]);
      s = fmaf(xv.x, yv.x, s);
      s = fmaf(xv.y, yv.y, s);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const long long row = row0 + u * RPW + sub;
    if (part == 0 && row < rows) delta[hq_tm > 0 ? (row % hq_tm) * total_q + row / hq_tm : row] = s;
  }
}

// Shared-memory descriptors of 128-byte-swizzled tiles as two 32-bit halves: the high
// half (stride 1024 bytes, version, layout) is one constant, the low half holds the
// start address and the leading byte offset (16 bytes for K-major operands, one
// 64-column region for MN-major ones).  The issuing thread keeps one word per operand
// and adds offsets to the 14-bit address field (addresses stay below 256 KB, so the
// addition never carries out of it).
__device__ __forceinline__ uint32_t desc_hi() { return (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32); }
__device__ __forceinline__ uint32_t desc_km(uint32_t saddr) { return (uint32_t)sdesc_sw128(saddr, 16, 1024); }
__device__ __forceinline__ uint32_t desc_mn(uint32_t saddr) {
  return (uint32_t)sdesc_sw128(saddr, 128 * 128, 1024);
}

// The eight MMAs of a 128-deep product in one statement: one predicate for the first
// (accumulate or not), a constant true one for the rest, the operand addresses stepped
// by immediates, so the issuing thread spends as few instructions as possible between
// products (it blocks on the tensor core's queue, and what it does in between shows).
// K-major A and B in shared memory (D = 128: two 64-column regions of 4 steps each).
__device__ __forceinline__ void mma8_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 da, db;\n\t.reg .b32 ta, tb;\n\t"
      "setp.ne.b32 p0, %5, 0;\n\t"
      "setp.eq.b32 p1, 0, 0;\n\t"
      "mov.b64 da, {%1, %3};\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p0;\n\t"
      "add.u32 ta, %1, 2;\n\t"
      "add.u32 tb, %2, 2;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 ta, %1, 4;\n\t"
      "add.u32 tb, %2, 4;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 ta, %1, 6;\n\t"
      "add.u32 tb, %2, 6;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 ta, %1, 1024;\n\t"
      "add.u32 tb, %2, 1024;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 ta, %1, 1026;\n\t"
      "add.u32 tb, %2, 1026;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 ta, %1, 1028;\n\t"
      "add.u32 tb, %2, 1028;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 ta, %1, 1030;\n\t"
      "add.u32 tb, %2, 1030;\n\t"
      "mov.b64 da, {ta, %3};\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "}" ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc)
      : "memory");
}

// A (128 x 128, two 16-bit values per column) in TMEM in the split layout of the
// compute threads (K-rows 0-63 at columns 0-31, 64-127 at 64-95), B MN-major in
// shared memory (16 K-rows = 2048 bytes a step).
__device__ __forceinline__ void mma8_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 db;\n\t.reg .b32 ta, tb;\n\t"
      "setp.ne.b32 p0, %5, 0;\n\t"
      "setp.eq.b32 p1, 0, 0;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p0;\n\t"
      "add.u32 ta, %1, 8;\n\t"
      "add.u32 tb, %2, 128;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 16;\n\t"
      "add.u32 tb, %2, 256;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 24;\n\t"
      "add.u32 tb, %2, 384;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 64;\n\t"
      "add.u32 tb, %2, 512;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 72;\n\t"
      "add.u32 tb, %2, 640;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 80;\n\t"
      "add.u32 tb, %2, 768;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 88;\n\t"
      "add.u32 tb, %2, 896;\n\t"
      "mov.b64 db, {tb, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "}" ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc)
      : "memory");
}

// S-like product D[tmem] = A B^T over the head dimension, both operands K-major
// 128 x D tiles in shared memory (16 columns = 32 bytes of a 128-byte swizzled row).
template <int D, bool BF16>
__device__ __forceinline__ void mma_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi) {
  constexpr uint32_t idesc = umma_idesc_f16(BF16, 128, 128, false, false);
  constexpr int REGION = 128 * 128;
  if constexpr (D == 128) {
    mma8_ss(d_tmem, a_lo, b_lo, hi, idesc, 0u);
  } else {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = ((kk >> 2) * REGION + (kk & 3) * 32) >> 4;
      umma_ss_lo(d_tmem, a_lo + off, hi, b_lo + off, hi, idesc, kk > 0 ? 1u : 0u);
    }
  }
}

// D[tmem] (+)= A B over 128 K-rows: A is 128 x 128 16-bit in TMEM (two values per
// column), B a 128 x D tile in shared memory read MN-major (16 rows = two swizzle
// atoms of 8 rows per MMA; LBO steps to the next 64 columns, SBO to the next 8 rows).
// The two compute threads of a TMEM lane each write their 64 values inside the 64
// columns they read (K-rows 0-63 at columns 0-31, K-rows 64-127 at 64-95), so
// neither overwrites columns the other may still be loading.
template <int D, bool BF16>
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                           bool acc) {
  constexpr uint32_t idesc = umma_idesc_f16(BF16, 128, D, false, true);
  mma8_ts(d_tmem, a_tmem, b_lo, hi, idesc, acc ? 1u : 0u);
}

// ============================================================================ dK, dV
// Persistent: one CTA per SM claims work items (key tile, KV head, batch) from a
// counter, longest first within each group of heads.  K and V of the next item load
// as soon as the current item's last S^T and dP^T (their only readers) complete, its
// first S^T and dP^T run while the compute warps store the current dK and dV, and its
// first dV waits only for those warps to have read the accumulators.
template <int D, bool BF16, bool VL>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const Params p) {
  using L = KVLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* item_q = reinterpret_cast<volatile int*>(misc + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int n_kt = (p.Skv + BN - 1) / BN;
  const int n_items = n_kt * p.Hkv * p.B;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::KV_FULL), 1);
    mbar_init(bar(L::KV_EMPTY), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::Q_FULL + i), 1);
      mbar_init(bar(L::DO_FULL + i), 1);
      mbar_init(bar(L::QD_FREE + i), 1);
      mbar_init(bar(L::ITEM_FULL + i), 1);
      mbar_init(bar(L::ITEM_EMPTY + i), 1 + NCOMP + NEPI);  // issuer, compute and epilogue threads
    }
    mbar_init(bar(L::S_READY), 1);
    mbar_init(bar(L::DP_READY), 1);
    mbar_init(bar(L::P_READY), NCOMP);
    mbar_init(bar(L::DS_READY), NCOMP);
    mbar_init(bar(L::VEC_READY), NCOMP);
    mbar_init(bar(L::DONE), 1);
    mbar_init(bar(L::ACC_FREE), NEPI);
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
  // TMEM columns: S^T (P^T over columns 0-31 and 64-95) at 0, dP^T (dS^T likewise)
  // at 128, dV at 256, dK at 384
  constexpr uint32_t C_S = 0, C_DP = 128, C_DV = 256, C_DK = 384;
  // one branch per warpgroup, each opening with its register limit: 256 compute threads
  // x 176 + 128 epilogue x 80 + 128 (loads, MMAs, two idle warps) x 80 = 512 x 128
  if (warp >= LOAD_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    if (warp == LOAD_WARP) {
      // ------------------------------------------------ work items and loads (one thread)
      if (lane == 0) {
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmdo);
        const uint64_t pol_kv = policy_evict_first();
        const uint64_t pol_q = policy_evict_last();
        // bounded-wait test: the CTA that claims work item 0 never issues the loads of that
        // item's second iteration (global iteration held_g), so the waits run out
        int held_g = -1;
        bool ok = true;
        int g = 0;     // (query head, Q tile) iterations reached, over all items
        int n_kv = 0;  // K/V tile pairs loaded
        int n_do = 0, n_q = 0;  // the dO and Q loads of iterations [0, n_do), [0, n_q) are issued
        for (int r = 0; ok; ++r) {
          const int slot = r & 1;
          if (!(ok = mbar_wait<false>(bar(L::ITEM_EMPTY + slot), ((r >> 1) & 1) ^ 1, abort_flag, &g_status, lim)))
            break;
          int w = atomicAdd(p.work_counter, 1);
          if (w >= n_items) w = -1;
          item_q[slot] = w;
          mbar_arrive(bar(L::ITEM_FULL + slot));
          if (w < 0) break;
          const KVItem it = kv_item<VL>(p, n_kt, w);
          if (it.n_iter == 0) continue;
          // K and V, once the last item's final S^T and dP^T have completed
          if (n_kv > 0 && !(ok = mbar_wait<false>(bar(L::KV_EMPTY), (n_kv - 1) & 1, abort_flag, &g_status, lim)))
            break;
          const int kv_y = VL ? it.sq.k0 + it.n0 : it.n0, kv_z = VL ? it.hk : it.b * p.Hkv + it.hk;
          mbar_expect_tx(bar(L::KV_FULL), 2 * L::TILE);
          for (int rr = 0; rr < L::NREG; ++rr) {
            tma_load_3d(sb + L::K_OFF + rr * L::REGION, &tmk, bar(L::KV_FULL), rr * 64, kv_y, kv_z, pol_kv);
            tma_load_3d(sb + L::V_OFF + rr * L::REGION, &tmv, bar(L::KV_FULL), rr * 64, kv_y, kv_z, pol_kv);
          }
          ++n_kv;
          // iteration g's Q and dO go to buffer g & 1, once iteration g - 2's dK, the last
          // product to read either (after its dV), has completed; Q first, as S^T needs it first
          for (int i = 0, h = it.hk * p.group, m = it.m_lo; i < it.n_iter && ok;
               ++i, ++g, h += (m + 1 == it.m_lo + it.per_head), m = (m + 1 == it.m_lo + it.per_head) ? it.m_lo : m + 1) {
            const int bi = g & 1;  // query head h, Q tile m
            const int q_y = VL ? it.sq.q0 + m * BM : m * BM, q_z = VL ? h : it.b * p.Hq + h;
            const bool held = p.debug_fault == 3 && w == 0 && i == 1;
            if (held) held_g = g;
            if (g >= 2 &&
                !(ok = mbar_wait<false>(bar(L::QD_FREE + bi), ((g - 2) >> 1) & 1, abort_flag, &g_status, lim)))
              break;
            if (!held) {
              mbar_expect_tx(bar(L::Q_FULL + bi), L::TILE);
              for (int rr = 0; rr < L::NREG; ++rr)
                tma_load_3d(sb + L::Q_OFF + bi * L::TILE + rr * L::REGION, &tmq, bar(L::Q_FULL + bi),
                            rr * 64, q_y, q_z, pol_q);
              mbar_expect_tx(bar(L::DO_FULL + bi), L::TILE);
              for (int rr = 0; rr < L::NREG; ++rr)
                tma_load_3d(sb + L::DO_OFF + bi * L::TILE + rr * L::REGION, &tmdo, bar(L::DO_FULL + bi),
                            rr * 64, q_y, q_z, pol_q);
            }
            n_q = n_do = g + 1;
          }
        }
        // nothing may be in flight when the CTA exits: the last load into each buffer (a
        // buffer is reloaded only after its last load was consumed; a withheld pair was
        // never issued, and no later load of its buffer is reached)
        if (n_kv > 0) drain_wait(bar(L::KV_FULL), (n_kv - 1) & 1, lim);
        for (int i = max(0, n_do - 2); i < n_do; ++i)
          if (i != held_g) drain_wait(bar(L::DO_FULL + (i & 1)), (i >> 1) & 1, lim);
        for (int i = max(0, n_q - 2); i < n_q; ++i)
          if (i != held_g) drain_wait(bar(L::Q_FULL + (i & 1)), (i >> 1) & 1, lim);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------ MMAs (one thread)
      if (lane == 0) {
        const uint32_t hi = desc_hi();
        const uint32_t k_km = desc_km(sb + L::K_OFF), v_km = desc_km(sb + L::V_OFF);
        const uint32_t q_km0 = desc_km(sb + L::Q_OFF), do_km0 = desc_km(sb + L::DO_OFF);
        const uint32_t q_mn0 = desc_mn(sb + L::Q_OFF), do_mn0 = desc_mn(sb + L::DO_OFF);
        constexpr uint32_t BUF = L::TILE >> 4;  // one Q or dO buffer in the address field
        auto q_km = [&](int bi) { return q_km0 + bi * BUF; };
        auto do_km = [&](int bi) { return do_km0 + bi * BUF; };
        auto q_mn = [&](int bi) { return q_mn0 + bi * BUF; };
        auto do_mn = [&](int bi) { return do_mn0 + bi * BUF; };
        auto wait = [&](int bar_i, int parity) -> bool {
          return mbar_wait<false>(bar(bar_i), parity & 1, abort_flag, &g_status, lim);
        };
        bool ok = true;
        int g = 0;     // iterations issued, over all items
        int n_it = 0;  // items with iterations
        for (int r = 0; ok; ++r) {
          const int slot = r & 1;
          if (!(ok = wait(L::ITEM_FULL + slot, r >> 1))) break;
          const int w = item_q[slot];
          mbar_arrive(bar(L::ITEM_EMPTY + slot));
          if (w < 0) break;
          const int n = kv_item<VL>(p, n_kt, w).n_iter;
          if (n == 0) continue;
          // S^T(0), dP^T(0); then per iteration i: dV(i), S^T(i+1), dK(i), dP^T(i+1), so
          // that the compute warps' P phase of i + 1 runs during dK(i), dP^T(i+1) and
          // their dS phase of i during dV(i), S^T(i+1).  S^T(0) and dP^T(0) overwrite
          // S^T and dP^T of the last item, read by its dV and dK, issued before them.
          if (!(ok = wait(L::KV_FULL, n_it) && wait(L::Q_FULL + (g & 1), g >> 1))) break;
          tc_fence_after();
          mma_kmajor<D, BF16>(tmem + C_S, k_km, q_km(g & 1), hi);
          umma_commit(bar(L::S_READY));
          if (!(ok = wait(L::DO_FULL + (g & 1), g >> 1))) break;
          tc_fence_after();
          mma_kmajor<D, BF16>(tmem + C_DP, v_km, do_km(g & 1), hi);
          umma_commit(bar(L::DP_READY));
          if (n == 1) umma_commit(bar(L::KV_EMPTY));  // the item's last readers of K and V
          for (int i = 0; i < n && ok; ++i) {
            const int gi = g + i, bi = gi & 1, bn = bi ^ 1;
            if (!(ok = wait(L::P_READY, gi))) break;
            // the item's first dV overwrites dV: the compute warps must have read the last one
            if (i == 0 && n_it > 0 && !(ok = wait(L::ACC_FREE, n_it - 1))) break;
            tc_fence_after();
            mma_tmem_a<D, BF16>(tmem + C_DV, tmem + C_S, do_mn(bi), hi, i > 0);  // dV += P^T dO
            if (i + 1 < n) {
              if (!(ok = wait(L::Q_FULL + bn, (gi + 1) >> 1))) break;
              tc_fence_after();
              mma_kmajor<D, BF16>(tmem + C_S, k_km, q_km(bn), hi);  // after dV read P^T there
              umma_commit(bar(L::S_READY));
            }
            if (!(ok = wait(L::DS_READY, gi))) break;
            tc_fence_after();
            mma_tmem_a<D, BF16>(tmem + C_DK, tmem + C_DP, q_mn(bi), hi, i > 0);  // dK += dS^T Q
            umma_commit(bar(L::QD_FREE + bi));  // Q and dO of iteration i: dK reads last
            if (i + 1 < n) {
              if (!(ok = wait(L::DO_FULL + bn, (gi + 1) >> 1))) break;
              tc_fence_after();
              mma_kmajor<D, BF16>(tmem + C_DP, v_km, do_km(bn), hi);  // after dK read dS^T there
              umma_commit(bar(L::DP_READY));
              if (i + 2 == n) umma_commit(bar(L::KV_EMPTY));
            }
          }
          if (!ok) break;
          umma_commit(bar(L::DONE));  // this item's dK and dV are complete
          g += n;
          ++n_it;
        }
        umma_commit(bar(L::DRAIN));  // fires once every MMA issued above has completed
        drain_wait(bar(L::DRAIN), 0, lim);
      }
      __syncwarp();
    }
  } else if (warp < EPI_WARP) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    // ------------------------------------------------ compute warps: two threads per key row
    // TMEM lane r: key n0 + r; warps w and w + 4 share the lanes of quarter w and
    // take queries [0, 64) and [64, 128) of each Q tile
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_t = tmem + ((uint32_t)(quarter * 32) << 16);
    float* vec = reinterpret_cast<float*>(smem + L::VEC_OFF);  // [buffer][LSE_2, delta][BM]
    const int c0 = half * 64;
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(b_, ph_, abort_flag, &g_status, lim));
    };
    // row r's negated LSE (half 0, log2 units) or negated delta (half 1) for iteration i
    // of item t, loaded one iteration ahead so its latency hides behind the current one
    // (negated, so that both enter the packed f32x2 forms below as addends)
    auto row_value = [&](const KVItem& t, int hh, int mm) -> float {  // query head hk G + hh, Q tile mm
      const int hi = t.hk * p.group + hh, qi = mm * BM + r;
      if (qi >= t.sq.nq) return half == 0 ? -INFINITY : -0.f;
      const size_t idx = VL ? (size_t)hi * p.total_q + t.sq.q0 + qi : ((size_t)t.b * p.Hq + hi) * p.Sq + qi;
      return half == 0 ? -(p.lse[idx] * 1.4426950408889634f) : -p.delta[idx];
    };
    // The row terms come from the kernel before this one, which this one was launched to
    // overlap: wait for its completion; then the dQ kernel, which reads them too and
    // nothing this one writes, may take each SM this grid leaves.
    griddep_wait();
    griddep_launch_dependents();
    bool ok = true;
    int g = 0;
    for (int rq = 0; ok; ++rq) {
      const int slot = rq & 1;
      if (!(ok = wait_warp(bar(L::ITEM_FULL + slot), (rq >> 1) & 1))) break;
      const int w = item_q[slot];
      mbar_arrive(bar(L::ITEM_EMPTY + slot));
      if (w < 0) break;
      const KVItem it = kv_item<VL>(p, n_kt, w);
      if (it.n_iter == 0) continue;  // skipped, or zero rows written by the epilogue warps
      const int key = it.n0 + r;
      // iteration i is query head hk G + i / per_head, Q tile m_lo + i % per_head: kept
      // as counters (this one's and the next's) rather than divided out every iteration
      int m_i = it.m_lo, h_n = 0, m_n = it.m_lo;
      float next_v = row_value(it, 0, it.m_lo);
      for (int i = 0; i < it.n_iter && ok; ++i) {
        const int gi = g + i;
        const int m0 = m_i * BM;
        if (++m_n == it.m_lo + it.per_head) {  // the next iteration's (head, tile)
          m_n = it.m_lo;
          ++h_n;
        }
        // the row vectors of this Q tile (-LSE_2, -delta), in buffer gi & 1: every thread
        // finished iteration gi - 2's reads before it arrived on iteration gi - 1's VEC_READY
        float* v_nl = vec + (gi & 1) * 2 * BM;
        float* v_nd = v_nl + BM;
        (half == 0 ? v_nl : v_nd)[r] = next_v;
        mbar_arrive(bar(L::VEC_READY));
        if (i + 1 < it.n_iter) next_v = row_value(it, h_n, m_n);
        m_i = m_n;
        if (!(ok = wait_warp(bar(L::VEC_READY), gi & 1))) break;
        // ---- P phase: P^T = 2^(S^T c - LSE_2) on the visible (key, query) pairs
        if (!(ok = wait_warp(bar(L::S_READY), gi & 1))) break;
        tc_fence_after();
        float pv[64];
        {
          // the two 32-column halves of this thread's S^T: the second loads while the
          // first is turned into P^T and stored
          uint32_t sa[32], sb[32];
          tmem_ld32_issue(lane_t + C_S + c0, sa);
          tmem_wait_ld_regs(sa);
          tmem_ld32_issue(lane_t + C_S + c0 + 32, sb);
          // query columns [lo, hi) of this thread's 64 see key n0 + r; a tile whose every
          // query sees every key (all but the window's edges and the ragged ends) needs no test
          const int lo = p.win_right >= 0 ? key - it.dlen - p.win_right - m0 - c0 : 0;
          int hi = key < it.sq.nk ? it.sq.nq - m0 - c0 : 0;
          if (p.win_left >= 0) hi = min(hi, key - it.dlen + p.win_left - m0 - c0 + 1);
          const bool all_visible = __all_sync(0xffffffffu, lo <= 0 && hi >= 64);
          // two query columns per packed f32x2 FMA (the same rounding as one fmaf each)
          const uint64_t c2p = f2_pack(p.c2, p.c2);
          const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(v_nl + c0);
          auto p_half = [&](const uint32_t(&sx)[32], int h, bool masked) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = 32 * h + 2 * j;
              float a0, a1;
              f2_unpack(fma2(f2_pack(__uint_as_float(sx[2 * j]), __uint_as_float(sx[2 * j + 1])), c2p,
                             nl2[16 * h + j]),
                        a0, a1);
              pv[c] = (!masked || (c >= lo && c < hi)) ? ex2(a0) : 0.f;
              pv[c + 1] = (!masked || (c + 1 >= lo && c + 1 < hi)) ? ex2(a1) : 0.f;
              pk[j] = pack2<BF16>(pv[c], pv[c + 1]);
            }
            tmem_st16(lane_t + C_S + c0 + 16 * h, pk);  // P^T over S^T columns already read
          };
          if (all_visible) {
            p_half(sa, 0, false);
            tmem_wait_ld_regs(sb);
            p_half(sb, 1, false);
          } else {
            p_half(sa, 0, true);
            tmem_wait_ld_regs(sb);
            p_half(sb, 1, true);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::P_READY));
        // ---- dS phase: dS^T = P^T (dP^T - delta)
        if (!(ok = wait_warp(bar(L::DP_READY), gi & 1))) break;
        tc_fence_after();
        {
          uint32_t da[32], db[32];
          tmem_ld32_issue(lane_t + C_DP + c0, da);
          tmem_wait_ld_regs(da);
          tmem_ld32_issue(lane_t + C_DP + c0 + 32, db);
          const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(v_nd + c0);
          auto ds_half = [&](const uint32_t(&dx)[32], int h) {  // P (dP - delta), packed pairs
            uint32_t dk2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = 32 * h + 2 * j;
              float d0, d1;
              const uint64_t dd =
                  add2(f2_pack(__uint_as_float(dx[2 * j]), __uint_as_float(dx[2 * j + 1])), nd2[16 * h + j]);
              f2_unpack(mul2(f2_pack(pv[c], pv[c + 1]), dd), d0, d1);
              dk2[j] = pack2<BF16>(d0, d1);
            }
            tmem_st16(lane_t + C_DP + c0 + 16 * h, dk2);  // dS^T over dP^T columns already read
          };
          ds_half(da, 0);
          tmem_wait_ld_regs(db);
          ds_half(db, 1);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::DS_READY));
      }
      if (!ok) break;
      g += it.n_iter;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    // ------------------------------------------------ epilogue: one key row (TMEM lane) per thread
    // Once the item's last dK product completes, dV and dK of row r go from TMEM into
    // registers 32 columns at a time; after the last load the accumulators are handed
    // back (ACC_FREE) and the rows are rounded and stored, off the compute warps' path.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_t = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(b_, ph_, abort_flag, &g_status, lim));
    };
    bool ok = true;
    int n_it = 0;
    for (int rq = 0; ok; ++rq) {
      const int slot = rq & 1;
      if (!(ok = wait_warp(bar(L::ITEM_FULL + slot), (rq >> 1) & 1))) break;
      const int w = item_q[slot];
      mbar_arrive(bar(L::ITEM_EMPTY + slot));
      if (w < 0) break;
      const KVItem it = kv_item<VL>(p, n_kt, w);
      if (it.skip) continue;
      const int key = it.n0 + r;
      const size_t off = VL ? (size_t)(it.sq.k0 + key) * p.dk_rstride + (size_t)it.hk * D
                            : (((size_t)it.b * p.Hkv + it.hk) * p.Skv + key) * D;
      uint4* dv_row = reinterpret_cast<uint4*>(p.dv + off);
      uint4* dk_row = reinterpret_cast<uint4*>(p.dk + off);
      if (it.n_iter == 0) {  // no query sees these keys: dK = dV = 0
        if (key < it.sq.nk)
          for (int i = 0; i < D / 8; ++i) dv_row[i] = dk_row[i] = make_uint4(0, 0, 0, 0);
        continue;
      }
      if (!(ok = wait_warp(bar(L::DONE), n_it & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2 * (D / 32); ++c) {  // dV's D columns, then dK's
        const bool is_dk = c >= D / 32;
        uint32_t v[32];
        tmem_ld32(lane_t + (is_dk ? C_DK : C_DV) + 32 * (c % (D / 32)), v);
        if (c == 2 * (D / 32) - 1) {  // both rows are in registers or stored: hand TMEM back
          tc_fence_before();
          mbar_arrive(bar(L::ACC_FREE));
        }
        if (key < it.sq.nk) {
          store_row32<BF16>((is_dk ? dk_row : dv_row) + 4 * (c % (D / 32)), v, is_dk ? p.scale : 1.f, p.st32);
        }
      }
      ++n_it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ============================================================================ dQ
// Persistent like the dK/dV kernel: work items (Q tile, query head, batch), the Q
// tiles with the most keys first within each group of heads.  The K/V ring runs on
// across items; the next item's Q and dO load once the current item's last S and dP
// (their readers) complete, and its first dQ waits only for the compute warps to have
// read the current dQ.
template <int D, bool BF16, bool VL>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                  const Params p) {
  using L = QLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* item_q = reinterpret_cast<volatile int*>(misc + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int n_mt = (p.Sq + BM - 1) / BM;
  const int n_items = n_mt * p.Hq * p.B;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::QD_FULL), 1);
    mbar_init(bar(L::QD_EMPTY), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::RING_FULL + s), 1);
    }
    for (int q = 0; q < 4; ++q) mbar_init(bar(L::RING_FREE + q), 1);
    mbar_init(bar(L::DP_READY), 1);
    mbar_init(bar(L::DP_FREE), NCOMP);
    mbar_init(bar(L::DS_READY), NCOMP);
    mbar_init(bar(L::DS_READY + 1), NCOMP);
    mbar_init(bar(L::DONE), 1);
    mbar_init(bar(L::ACC_FREE), NEPI);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::ITEM_FULL + i), 1);
      mbar_init(bar(L::ITEM_EMPTY + i), 1 + NCOMP + NEPI);  // issuer, compute and epilogue threads
    }
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
  // TMEM columns: S of even K/V steps at 0, of odd ones at 128 (dS over columns 0-31
  // and 64-95), dP at 256, dQ at 384
  constexpr uint32_t C_S = 0, C_DP = 256, C_DQ = 384;
  // one branch per warpgroup, each opening with its register limit: 256 compute threads
  // x 176 + 128 epilogue x 80 + 128 (loads, MMAs, two idle warps) x 80 = 512 x 128
  if (warp >= LOAD_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    if (warp == LOAD_WARP) {
      // ------------------------------------------------ work items and loads (one thread)
      if (lane == 0) {
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmdo);
        const uint64_t pol_q = policy_evict_first();
        const uint64_t pol_kv = policy_evict_last();
        bool ok = true;
        int n_qd = 0;  // Q/dO tile pairs loaded
        int ld = 0;    // K/V ring loads issued, over all items
        for (int r = 0; ok; ++r) {
          const int slot = r & 1;
          if (!(ok = mbar_wait<false>(bar(L::ITEM_EMPTY + slot), ((r >> 1) & 1) ^ 1, abort_flag, &g_status, lim)))
            break;
          int w = atomicAdd(p.work_counter + 1, 1);
          if (w >= n_items) w = -1;
          item_q[slot] = w;
          mbar_arrive(bar(L::ITEM_FULL + slot));
          if (w < 0) break;
          const QItem it = q_item<VL>(p, n_mt, w);
          if (it.n_kv == 0) continue;
          // Q and dO, once the last item's final S and dP have completed
          if (n_qd > 0 && !(ok = mbar_wait<false>(bar(L::QD_EMPTY), (n_qd - 1) & 1, abort_flag, &g_status, lim)))
            break;
          const int q_y = VL ? it.sq.q0 + it.m0 : it.m0, q_z = VL ? it.h : it.b * p.Hq + it.h;
          mbar_expect_tx(bar(L::QD_FULL), 2 * L::TILE);
          for (int rr = 0; rr < L::NREG; ++rr) {
            tma_load_3d(sb + L::Q_OFF + rr * L::REGION, &tmq, bar(L::QD_FULL), rr * 64, q_y, q_z, pol_q);
            tma_load_3d(sb + L::DO_OFF + rr * L::REGION, &tmdo, bar(L::QD_FULL), rr * 64, q_y, q_z, pol_q);
          }
          ++n_qd;
          const int hk = it.h / p.group;
          const int kv_y0 = (VL ? it.sq.k0 : 0) + it.t_lo * BN, kv_z = VL ? hk : it.b * p.Hkv + hk;
          for (int l = 0; l < 2 * it.n_kv && ok; ++l, ++ld) {  // V_0, K_0, V_1, K_1, ...
            const int s = ld % NS;
            const int q = (ld - NS + 1) >> 1;  // the release that covers load ld - NS
            if (ld >= NS &&
                !(ok = mbar_wait<false>(bar(L::RING_FREE + (q & 3)), (q >> 2) & 1, abort_flag, &g_status, lim)))
              break;
            mbar_expect_tx(bar(L::RING_FULL + s), L::TILE);
            const CUtensorMap* tm = (l & 1) ? &tmk : &tmv;
            for (int rr = 0; rr < L::NREG; ++rr)
              tma_load_3d(sb + L::RING_OFF + s * L::TILE + rr * L::REGION, tm, bar(L::RING_FULL + s), rr * 64,
                          kv_y0 + (l >> 1) * BN, kv_z, pol_kv);
          }
        }
        // the last Q/dO pair and the last NS ring loads may still be in flight
        if (n_qd > 0) drain_wait(bar(L::QD_FULL), (n_qd - 1) & 1, lim);
        for (int l = max(0, ld - NS); l < ld; ++l) drain_wait(bar(L::RING_FULL + l % NS), (l / NS) & 1, lim);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------ MMAs (one thread)
      if (lane == 0) {
        const uint32_t hi = desc_hi();
        const uint32_t q_km = desc_km(sb + L::Q_OFF), do_km = desc_km(sb + L::DO_OFF);
        const uint32_t ring_km0 = desc_km(sb + L::RING_OFF), ring_mn0 = desc_mn(sb + L::RING_OFF);
        constexpr uint32_t SLOT = L::TILE >> 4;  // one ring slot in the address field
        auto wait = [&](int bar_i, int parity) -> bool {
          return mbar_wait<false>(bar(bar_i), parity & 1, abort_flag, &g_status, lim);
        };
        // a ring load as its slot and the parity of its use of the slot, stepped rather than
        // divided out per product (the issuing thread's instructions between products show)
        struct RingPos {
          int s, ph;
        };
        auto ring_pos = [&](int l) { return RingPos{l % NS, (l / NS) & 1}; };
        auto ring_next = [&](RingPos a, int k) {  // load index + k, 0 < k < NS
          a.s += k;
          if (a.s >= NS) {
            a.s -= NS;
            a.ph ^= 1;
          }
          return a;
        };
        auto ring_km = [&](RingPos a) { return ring_km0 + (uint32_t)a.s * SLOT; };
        auto ring_mn = [&](RingPos a) { return ring_mn0 + (uint32_t)a.s * SLOT; };
        auto ring_wait = [&](RingPos a) -> bool { return wait(L::RING_FULL + a.s, a.ph); };
        bool ok = true;
        // step g reads ring loads 2g (V) and 2g + 1 (K); K(g) and V(g + 1) are released
        // together once dQ(g) has read K(g) (dP(g + 1), which reads V(g + 1), is issued
        // before it), so with NS = 5 both tiles of step g + 2 land while step g runs
        int g = 0;     // K/V steps issued over all items
        int n_it = 0;  // items with K/V steps
        for (int r = 0; ok; ++r) {
          const int slot = r & 1;
          if (!(ok = wait(L::ITEM_FULL + slot, r >> 1))) break;
          const int w = item_q[slot];
          mbar_arrive(bar(L::ITEM_EMPTY + slot));
          if (w < 0) break;
          const int n = q_item<VL>(p, n_mt, w).n_kv;
          if (n == 0) continue;
          // S(0), dP(0); then per K/V step j: S(j+1) into the other S buffer, dP(j+1)
          // once the compute warps hold dP(j), dQ += dS(j) K(j) once they wrote dS(j).
          // S(0) goes to the buffer of step g, whose last dS was read by a dQ issued
          // before; dP(0) waits until the compute warps hold the last item's final dP.
          RingPos kp = ring_pos(2 * g + 1);        // K of the current step (load 2 gj + 1)
          const RingPos vp0 = ring_pos(2 * g);     // V(0)
          if (!(ok = wait(L::QD_FULL, n_it) && ring_wait(kp))) break;
          tc_fence_after();
          mma_kmajor<D, BF16>(tmem + C_S + 128u * (g & 1), q_km, ring_km(kp), hi);
          if (g > 0 && !(ok = wait(L::DP_FREE, g - 1))) break;
          if (!(ok = ring_wait(vp0))) break;
          tc_fence_after();
          mma_kmajor<D, BF16>(tmem + C_DP, do_km, ring_km(vp0), hi);
          umma_commit(bar(L::DP_READY));
          umma_commit(bar(L::RING_FREE + (g & 3)));  // V(0), and K of the step before (its dQ came first)
          if (n == 1) umma_commit(bar(L::QD_EMPTY));  // the item's last readers of Q and dO
          for (int j = 0; j < n && ok; ++j) {
            const int gj = g + j;
            const RingPos vn = ring_next(kp, 1), kn = ring_next(kp, 2);  // V(j+1), K(j+1)
            if (j + 1 < n) {
              if (!(ok = ring_wait(kn))) break;
              tc_fence_after();
              // the other buffer held dS(gj - 1), read by dQ(gj - 1), issued before
              mma_kmajor<D, BF16>(tmem + C_S + 128u * ((gj + 1) & 1), q_km, ring_km(kn), hi);
            }
            if (!(ok = wait(L::DP_FREE, gj))) break;
            if (j + 1 < n) {
              if (!(ok = ring_wait(vn))) break;
              tc_fence_after();
              mma_kmajor<D, BF16>(tmem + C_DP, do_km, ring_km(vn), hi);
              umma_commit(bar(L::DP_READY));
              if (j + 2 == n) umma_commit(bar(L::QD_EMPTY));
            }
            if (!(ok = wait(L::DS_READY + (gj & 1), gj >> 1))) break;
            // the item's first dQ overwrites dQ: the compute warps must have read the last one
            if (j == 0 && n_it > 0 && !(ok = wait(L::ACC_FREE, n_it - 1))) break;
            tc_fence_after();
            mma_tmem_a<D, BF16>(tmem + C_DQ, tmem + C_S + 128u * (gj & 1), ring_mn(kp), hi, j > 0);  // dQ += dS K
            // K(j), read by S(j) and dQ(j), and V(j+1), read by dP(j+1) issued before; at
            // the item's last step the next item's first dP releases them
            if (j + 1 < n) umma_commit(bar(L::RING_FREE + ((gj + 1) & 3)));
            kp = kn;
          }
          if (!ok) break;
          umma_commit(bar(L::DONE));
          g += n;
          ++n_it;
        }
        umma_commit(bar(L::DRAIN));
        drain_wait(bar(L::DRAIN), 0, lim);
      }
      __syncwarp();
    }
  } else if (warp < EPI_WARP) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    // ------------------------------------------------ compute warps: two threads per query row
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_t = tmem + ((uint32_t)(quarter * 32) << 16);
    const int c0 = half * 64;  // this thread's 64 of a K/V tile's 128 keys
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(b_, ph_, abort_flag, &g_status, lim));
    };
    bool ok = true;
    int g = 0;
    for (int rq = 0; ok; ++rq) {
      const int slot = rq & 1;
      if (!(ok = wait_warp(bar(L::ITEM_FULL + slot), (rq >> 1) & 1))) break;
      const int w = item_q[slot];
      mbar_arrive(bar(L::ITEM_EMPTY + slot));
      if (w < 0) break;
      const QItem it = q_item<VL>(p, n_mt, w);
      if (it.n_kv == 0) continue;  // skipped, or zero rows written by the epilogue warps
      const int row = it.m0 + r;
      const bool live = row < it.sq.nq;
      const size_t ridx =
          VL ? (size_t)it.h * p.total_q + it.sq.q0 + row : ((size_t)it.b * p.Hq + it.h) * p.Sq + row;
      const float lse2 = live ? p.lse[ridx] * 1.4426950408889634f : INFINITY;
      const float dlt = live ? p.delta[ridx] : 0.f;
      // keys of this row: [key_lo, key_hi] (none for rows past the sequence)
      int key_lo = 0, key_hi = live ? it.sq.nk - 1 : -1;
      if (p.win_right >= 0) key_hi = min(key_hi, row + it.dlen + p.win_right);
      if (p.win_left >= 0) key_lo = row + it.dlen - p.win_left;
      for (int j = 0; j < it.n_kv && ok; ++j) {
        const int gj = g + j;
        if (!(ok = wait_warp(bar(L::DP_READY), gj & 1))) break;  // S of this step, then its dP
        tc_fence_after();
        const uint32_t t_s = lane_t + C_S + 128u * (gj & 1);
        // the two 32-column halves of this thread's S and dP: the second pair loads while
        // the first is turned into dS and stored
        uint32_t s_a[32], d_a[32], s_b[32], d_b[32];
        tmem_ld32_issue(t_s + c0, s_a);
        tmem_ld32_issue(lane_t + C_DP + c0, d_a);
        tmem_wait_ld_regs(s_a, d_a);
        tmem_ld32_issue(t_s + c0 + 32, s_b);
        tmem_ld32_issue(lane_t + C_DP + c0 + 32, d_b);
        // keys kb + u, ulo <= u < uhi, are visible to this row; a tile whose every key
        // is visible to the whole warp's rows (all but the diagonal, the window's edges
        // and the ragged ends) needs no test
        const int kb = (it.t_lo + j) * BN + c0, ulo = key_lo - kb, uhi = key_hi + 1 - kb;
        const bool all_visible = __all_sync(0xffffffffu, ulo <= 0 && uhi >= 64);
        // both columns of a pair in one packed f32x2 operation (same roundings)
        const uint64_t c2p = f2_pack(p.c2, p.c2), nl = f2_pack(-lse2, -lse2), nd = f2_pack(-dlt, -dlt);
        auto ds_half = [&](const uint32_t(&sx)[32], const uint32_t(&dx)[32], int h, bool masked) {
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int c = 32 * h + 2 * u;
            float a0, a1, d0, d1;
            f2_unpack(fma2(f2_pack(__uint_as_float(sx[2 * u]), __uint_as_float(sx[2 * u + 1])), c2p, nl), a0, a1);
            const float p0 = (!masked || (c >= ulo && c < uhi)) ? ex2(a0) : 0.f;
            const float p1 = (!masked || (c + 1 >= ulo && c + 1 < uhi)) ? ex2(a1) : 0.f;
            const uint64_t dd = add2(f2_pack(__uint_as_float(dx[2 * u]), __uint_as_float(dx[2 * u + 1])), nd);
            f2_unpack(mul2(f2_pack(p0, p1), dd), d0, d1);
            pk[u] = pack2<BF16>(d0, d1);
          }
          tmem_st16(t_s + c0 + 16 * h, pk);  // dS over S columns already read
        };
        if (all_visible) ds_half(s_a, d_a, 0, false);
        else ds_half(s_a, d_a, 0, true);
        tmem_wait_ld_regs(s_b, d_b);
        tc_fence_before();
        mbar_arrive(bar(L::DP_FREE));  // dP(j + 1) may overwrite dP(j)
        if (all_visible) ds_half(s_b, d_b, 1, false);
        else ds_half(s_b, d_b, 1, true);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::DS_READY + (gj & 1)));
      }
      if (!ok) break;
      g += it.n_kv;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    // ------------------------------------------------ epilogue: one query row (TMEM lane) per thread
    // Once the item's last dQ product completes, the row goes from TMEM into registers
    // 32 columns at a time; after the last load dQ is handed back (ACC_FREE), and the
    // row is scaled, rounded and stored, off the compute warps' path.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_t = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    auto wait_warp = [&](uint32_t b_, uint32_t ph_) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(b_, ph_, abort_flag, &g_status, lim));
    };
    bool ok = true;
    int n_it = 0;
    for (int rq = 0; ok; ++rq) {
      const int slot = rq & 1;
      if (!(ok = wait_warp(bar(L::ITEM_FULL + slot), (rq >> 1) & 1))) break;
      const int w = item_q[slot];
      mbar_arrive(bar(L::ITEM_EMPTY + slot));
      if (w < 0) break;
      const QItem it = q_item<VL>(p, n_mt, w);
      if (it.skip) continue;
      const int row = it.m0 + r;
      const bool live = row < it.sq.nq;
      uint4* dst = reinterpret_cast<uint4*>(
          VL ? p.dq + (size_t)(it.sq.q0 + row) * p.dq_rstride + (size_t)it.h * D
             : p.dq + (((size_t)it.b * p.Hq + it.h) * p.Sq + row) * D);
      if (it.n_kv == 0) {  // the rows see no key: dQ = 0
        if (live)
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        continue;
      }
      if (!(ok = wait_warp(bar(L::DONE), n_it & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_t + C_DQ + 32 * c, v);
        if (c == D / 32 - 1) {  // the whole row is in registers or stored: hand dQ back
          tc_fence_before();
          mbar_arrive(bar(L::ACC_FREE));
        }
        if (live) store_row32<BF16>(dst + 4 * c, v, p.scale, p.st32);
      }
      ++n_it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  // launched to overlap the dK/dV kernel's last items: complete only after it has, so
  // that work ordered after this kernel also sees dK and dV
  griddep_wait();
}

// 3-D tensor map over 16-bit elements: D contiguous, then n1 rows s1 elements apart,
// then n2 planes s2 elements apart; 64 x 128 x 1 boxes, 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, int D, long long n1, long long n2, long long s1,
                     long long s2, bool bf16) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n1, (cuuint64_t)n2};
  const cuuint64_t strides[2] = {(cuuint64_t)s1 * 2, (cuuint64_t)s2 * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BF16, bool VL>
static cudaError_t launch_t(const BwdArgs& a, cudaStream_t stream) {
  // row terms: one per (query token, head) in either layout
  const long long rows = VL ? (long long)a.total_q * a.Hq : (long long)a.B * a.Hq * a.Sq;
  {
    cudaError_t e = cudaMemsetAsync(a.work_counter, 0, 2 * sizeof(int), stream);
    if (e != cudaSuccess) return e;
  }
  if (rows > 0) {
    constexpr int RB = delta_rows_per_block<D>();
    bwd_delta_kernel<D, BF16><<<(unsigned)((rows + RB - 1) / RB), DELTA_THREADS, 0, stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.delta, rows,
        VL ? a.Hq : 0, (long long)a.total_q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, tk, tv, tg;
  if (VL) {
    // [tokens, heads, D] with the given token strides; with no keys (or no queries) a
    // map covers one never-read row of an array that has one
    const bool nk = a.total_k > 0, nq = a.total_q > 0;
    const void* qb = nq ? a.q : a.k;
    const void* gb = nq ? a.dout : a.k;
    const void* kb = nk ? a.k : a.q;
    const void* vb = nk ? a.v : a.q;
    if (!make_map(&tq, qb, D, nq ? a.total_q : 1, nq ? a.Hq : 1, nq ? a.q_rstride : a.k_rstride, D, BF16) ||
        !make_map(&tg, gb, D, nq ? a.total_q : 1, nq ? a.Hq : 1, nq ? a.do_rstride : a.k_rstride, D, BF16) ||
        !make_map(&tk, kb, D, nk ? a.total_k : 1, nk ? a.Hkv : 1, nk ? a.k_rstride : a.q_rstride, D, BF16) ||
        !make_map(&tv, vb, D, nk ? a.total_k : 1, nk ? a.Hkv : 1, nk ? a.k_rstride : a.q_rstride, D, BF16))
      return cudaErrorInvalidValue;
  } else {
    // with no query rows the Q/dO maps cover one (never read) row of k
    const int sq_map = a.Sq > 0 ? a.Sq : 1;
    const void* qb = a.Sq > 0 ? a.q : a.k;
    const void* gb = a.Sq > 0 ? a.dout : a.k;
    const long long qp = a.Sq > 0 ? (long long)a.B * a.Hq : 1;
    if (!make_map(&tq, qb, D, sq_map, qp, D, (long long)sq_map * D, BF16) ||
        !make_map(&tg, gb, D, sq_map, qp, D, (long long)sq_map * D, BF16) ||
        !make_map(&tk, a.k, D, a.Skv, (long long)a.B * a.Hkv, D, (long long)a.Skv * D, BF16) ||
        !make_map(&tv, a.v, D, a.Skv, (long long)a.B * a.Hkv, D, (long long)a.Skv * D, BF16))
      return cudaErrorInvalidValue;
  }
  Params p{};
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq = static_cast<uint16_t*>(a.dq);
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
  p.win_left = a.win_left;
  p.win_right = a.causal ? 0 : a.win_right;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.dq_rstride = a.dq_rstride;
  p.dk_rstride = a.dk_rstride;
  p.st32 = (reinterpret_cast<uintptr_t>(a.dq) | reinterpret_cast<uintptr_t>(a.dk) |
            reinterpret_cast<uintptr_t>(a.dv)) % 32 == 0 &&
           (a.dq_rstride * 2) % 32 == 0 && (a.dk_rstride * 2) % 32 == 0;
  const long long n_kt = (a.Skv + BN - 1) / BN, n_mt = (a.Sq + BM - 1) / BM;
  // both persistent kernels claim work items from the two counters, zeroed before the
  // row terms kernel
  p.work_counter = a.work_counter;
  const int sms = a.num_sms > 0 ? a.num_sms : 1;
  const int g = a.Hq / a.Hkv;
  if (n_kt > 0) {
    using L = KVLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, BF16, VL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    // scheduling groups: as many (batch, KV head) planes as keep about 64 MB of their
    // query heads' Q and dO in L2
    const double qd_bytes = 4.0 * (double)(a.Sq > 0 ? a.Sq : 1) * D * g;
    long long per = (long long)(64.0 * (1 << 20) / qd_bytes);
    if (per < 1) per = 1;
    if (per > (long long)a.B * a.Hkv) per = (long long)a.B * a.Hkv;
    p.per_group = (int)per;
    const long long n_items = n_kt * a.Hkv * a.B;
    const int grid = (int)(n_items < sms ? n_items : sms);
    // after the row terms kernel, its CTAs set up on the SMs that kernel's CTAs leave
    // (programmatic stream serialization; the compute warps wait for its completion)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = rows > 0 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<D, BF16, VL>, tq, tk, tv, tg, p);
    if (e != cudaSuccess) return e;
  }
  if (n_mt > 0 && rows > 0) {
    using L = QLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D, BF16, VL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    // scheduling groups: as many (batch, query head) planes as keep about 64 MB of
    // their K and V in L2, rounded to whole GQA groups
    const double kv_bytes = 4.0 * (double)(a.Skv > 0 ? a.Skv : 1) * D;
    long long per = (long long)(64.0 * (1 << 20) / kv_bytes) * g;
    if (per < g) per = g;
    if (per > (long long)a.B * a.Hq) per = (long long)a.B * a.Hq;
    p.per_group_q = (int)per;
    const long long n_items = n_mt * a.Hq * a.B;
    const int grid = (int)(n_items < sms ? n_items : sms);
    // After the dK/dV kernel its CTAs start on the SMs that kernel's CTAs leave, while
    // its last items run (programmatic stream serialization; that kernel signals once
    // its compute warps have seen the row terms complete).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = n_kt > 0 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D, BF16, VL>, tq, tk, tv, tg, p);
  }
  return cudaSuccess;
}

}  // namespace bwd

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.vl) {
    if (a.D == 64)
      return a.bf16 ? bwd::launch_t<64, true, true>(a, stream) : bwd::launch_t<64, false, true>(a, stream);
    return a.bf16 ? bwd::launch_t<128, true, true>(a, stream) : bwd::launch_t<128, false, true>(a, stream);
  }
  if (a.D == 64)
    return a.bf16 ? bwd::launch_t<64, true, false>(a, stream) : bwd::launch_t<64, false, false>(a, stream);
  return a.bf16 ? bwd::launch_t<128, true, false>(a, stream) : bwd::launch_t<128, false, false>(a, stream);
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
