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
// 128-key sub-tiles (32 KB each; 2 CTAs per SM) and reads every byte once for
// all query heads of the GQA group.  A CTA takes up to four consecutive chunks
// of one (sequence, KV head) and keeps its ring streaming across them, writing
// one partial per chunk; the group's query vectors live in registers, scores
// are formed with 8 lanes per key (16-byte loads, packed f32x2 FMAs, 3 shuffle
// levels), the online max/sum run per 128-key sub-tile, and P V uses one lane
// per 4 output columns with packed FMAs.  No tensor cores: the contraction is
// too thin to pay for them and the bound is HBM.
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
  int B, Hq, Hkv, max_S, chunk, max_chunks, group, heads_per_cta;
  int cpb;  // consecutive chunks per split-kernel CTA
  float c2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  // paged cache (block_table != nullptr): k, v are [num_pages, Hkv, page_size, D] and
  // position j of sequence b is row j % page_size of page block_table[b, j / page_size]
  const int32_t* block_table;
  int page_size, max_pages, num_pages;
  // single-launch decode: one zeroed counter per (sequence, head group) CTA row
  unsigned* tickets;
  int debug_fault;  // 2: CTA (0, 0, 0) withholds load 1 (its first V sub-tile)
};

__device__ __forceinline__ int clamp_len(const Params& p, int b) {
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_S) {
    L = L < 0 ? 0 : p.max_S;
    if (threadIdx.x == 0) atomicOr(&g_status, kStatusSeqLenClamped);
  }
  return L;
}

template <int D, int G, bool PAGED>
struct SplitLayout {
  static constexpr int STAGE = SUB * D * 2;
  static constexpr int GH = (G + 1) / 2;                      // heads per cross-warp reduction pass
  static constexpr int RING_OFF = 0;
  static constexpr int SC_OFF = RING_OFF + NST * STAGE;      // scores / probabilities [SUB][G]
  static constexpr int RED_OFF = SC_OFF + SUB * G * 4;       // [WARPS][GH][D] P V partial sums
  static constexpr int PT_OFF = RED_OFF + WARPS * GH * D * 4;    // block-table slice (paged cache)
  static constexpr int PT_MAX = PAGED ? 520 : 0;                  // entries it holds
  static constexpr int STAT_OFF = PT_OFF + PT_MAX * 4;            // m, l, alpha per head
  static constexpr int BAR_OFF = (STAT_OFF + 3 * G * 4 + 15) / 16 * 16;  // NST ring barriers
  static constexpr int ABORT_OFF = BAR_OFF + NST * 8;
  static constexpr int BYTES = ABORT_OFF + 16;
  static_assert(BAR_OFF % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(STAGE % 16 == 0 && RING_OFF % 16 == 0, "bulk copies need 16-byte alignment");
  static_assert(SC_OFF % 16 == 0, "probabilities are read as float4");
};

// Two 16-bit values of one 32-bit word as an f32 pair (low half first), for the
// packed f32x2 arithmetic.
template <bool BF16>
__device__ __forceinline__ uint64_t pair_of(uint32_t w) {
  if constexpr (BF16) {
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    const float2 f = unpack2<false>(w);
    return f2_pack(f.x, f.y);
  }
}

// A CTA takes up to p.cpb consecutive chunks of one (sequence, KV head, head
// group) and streams their K and V rows through one ring that does not drain
// between its chunks (thread 0 issues load j + NST as soon as load j has been
// consumed, whichever chunk it belongs to), writing one partial per chunk.  A
// 512-key chunk is only 256 KB of K and V: with one CTA per chunk, each CTA's
// first load and epilogue went unhidden (85 % of HBM bandwidth at chunk 512
// against 94 % at chunk 2048).
template <int D, int G, bool BF16>
__device__ __forceinline__ void merge_group(const Params& p, int b, int h0, int n, float* red, float* tot);

// PG: 0 contiguous cache; 1 paged cache, thread 0 issues the copies; 2 paged cache
// with small pages, the lanes of warp 0 issue them (a 128-key sub-tile spans at
// least four pages).  Each is its own instantiation: sharing code with the
// others cost the larger-page and contiguous kernels several percent.
template <int D, int G, bool BF16, int PG, bool MERGE = false>
__global__ void __launch_bounds__(THREADS) decode_split_kernel(const Params p) {
  constexpr bool PAGED = PG != 0, WIDE = PG == 2;
  using L = SplitLayout<D, G, PAGED>;
  constexpr int EPL = D / 8;   // key elements per lane when 8 lanes share a key
  constexpr int DPL = D / 32;  // output columns per lane in P V
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  float* sc = reinterpret_cast<float*>(smem + L::SC_OFF);
  float* red = reinterpret_cast<float*>(smem + L::RED_OFF);
  float* m_run = reinterpret_cast<float*>(smem + L::STAT_OFF);
  float* l_run = m_run + G;
  float* alpha_s = l_run + G;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kvh = blockIdx.y / (p.group / G);
  const int h0 = kvh * p.group + (blockIdx.y % (p.group / G)) * G;  // first query head of this CTA
  const int b = blockIdx.z;
  const int len = clamp_len(p, b);
  const int nch = (len + p.chunk - 1) / p.chunk;                   // chunks of this sequence
  const int c0 = blockIdx.x * p.cpb;                                // first chunk of this CTA
  const int c1 = min(c0 + p.cpb, nch);                              // end of its chunks
  if (c0 >= c1) {
    if constexpr (MERGE) {
      // an empty sequence has nothing to merge: its first CTA writes O = 0
      if (len == 0 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < G * D / 2; i += THREADS)
          reinterpret_cast<uint32_t*>(p.o + ((size_t)b * p.Hq + h0) * D)[i] = 0u;
    }
    return;
  }
  const size_t row0 = ((size_t)b * p.Hkv + kvh) * p.max_S;
  auto chunk_rows = [&](int c) -> int { return min(p.chunk, len - c * p.chunk); };
  auto ring_bar = [&](int j) -> uint32_t { return sb + L::BAR_OFF + 8 * (j % NST); };

  // Paged cache: the block-table entries of this CTA's positions, checked once and
  // kept in shared memory, so the loader thread does not wait on a global load per
  // page.  (Ranges of more pages than the buffer holds read the table directly.)
  int* pt = reinterpret_cast<int*>(smem + L::PT_OFF);
  int pg_lo = 0, pg_n = 0;
  if constexpr (PAGED) {
    pg_lo = (c0 * p.chunk) / p.page_size;
    pg_n = (min(len, c1 * p.chunk) - 1) / p.page_size + 1 - pg_lo;
  }
  const bool pt_smem = pg_n <= L::PT_MAX;
  auto page_of = [&](int pg) -> int {  // physical page of logical page pg, within the pool
    int phys = __ldg(p.block_table + (size_t)b * p.max_pages + pg);
    if (phys < 0 || phys >= p.num_pages) {  // never read outside the page pool
      atomicOr(&g_status, kStatusBadPage);
      phys = 0;
    }
    return phys;
  };
  if constexpr (PAGED) {
    if (pt_smem) {
      for (int i = threadIdx.x; i < pg_n; i += THREADS) pt[i] = page_of(pg_lo + i);
      __syncthreads();
    }
  }

  // ---------------------- load stream (thread 0; all of warp 0 for the paged cache)
  int l_c = c0, l_off = 0, l_nload = 2 * ((chunk_rows(c0) + SUB - 1) / SUB), issued = 0;
  uint64_t pol = 0;
  // bounded-wait test: one CTA never issues its load 1, so the waits on it run out
  const int withheld = (p.debug_fault == 2 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) ? 1 : -1;
  auto issue_next = [&]() {  // the next K or V sub-tile of this CTA's chunks
    if (l_c >= c1) return;
    const int sub = l_off >> 1;
    const int rows = min(SUB, chunk_rows(l_c) - sub * SUB);
    if (issued == withheld) {
    } else if constexpr (!PAGED) {
      const size_t r = row0 + (size_t)l_c * p.chunk + (size_t)sub * SUB;
      const uint16_t* src = ((l_off & 1) ? p.v : p.k) + r * D;
      const uint32_t bar = ring_bar(issued);
      mbar_expect_tx(bar, rows * D * 2);
      bulk_load(sb + L::RING_OFF + (issued % NST) * L::STAGE, src, rows * D * 2, bar, pol);
    } else if constexpr (!WIDE) {
      const uint16_t* base = (l_off & 1) ? p.v : p.k;
      const uint32_t bar = ring_bar(issued);
      const uint32_t dst = sb + L::RING_OFF + (issued % NST) * L::STAGE;
      mbar_expect_tx(bar, rows * D * 2);
      // one copy per page the sub-tile's positions fall in, into one stage and one barrier
      const int pos0 = l_c * p.chunk + sub * SUB;
      int pg = pos0 / p.page_size, off = pos0 - pg * p.page_size;
      for (int done = 0; done < rows; ++pg, off = 0) {
        const int phys = pt_smem ? pt[pg - pg_lo] : page_of(pg);
        const int seg = min(rows - done, p.page_size - off);
        bulk_load(dst + done * D * 2, base + (((size_t)phys * p.Hkv + kvh) * p.page_size + off) * D,
                  seg * D * 2, bar, pol);
        done += seg;
      }
    } else {
      // the same copies, issued by the 32 lanes of warp 0 after lane 0 has set the
      // byte count
      const uint16_t* base = (l_off & 1) ? p.v : p.k;
      const uint32_t bar = ring_bar(issued);
      const uint32_t dst = sb + L::RING_OFF + (issued % NST) * L::STAGE;
      if (lane == 0) mbar_expect_tx(bar, rows * D * 2);
      __syncwarp();
      const int pos0 = l_c * p.chunk + sub * SUB;
      const int pg0 = pos0 / p.page_size, off0 = pos0 - pg0 * p.page_size;
      const int first = min(rows, p.page_size - off0);  // positions in the first page
      const int n_seg = 1 + (rows - first + p.page_size - 1) / p.page_size;
      for (int sg = lane; sg < n_seg; sg += 32) {
        const int done = sg == 0 ? 0 : first + (sg - 1) * p.page_size;
        const int off = sg == 0 ? off0 : 0;
        const int seg = min(rows - done, p.page_size - off);
        const int phys = pt_smem ? pt[pg0 + sg - pg_lo] : page_of(pg0 + sg);
        bulk_load(dst + done * D * 2, base + (((size_t)phys * p.Hkv + kvh) * p.page_size + off) * D,
                  seg * D * 2, bar, pol);
      }
    }
    ++issued;
    if (++l_off == l_nload && ++l_c < c1) {
      l_off = 0;
      l_nload = 2 * ((chunk_rows(l_c) + SUB - 1) / SUB);
    }
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(ring_bar(i), 1);
    *abort_flag = 0;
    fence_barrier_init();
    if constexpr (!WIDE) {
      pol = policy_evict_first();
      for (int i = 0; i < NST; ++i) issue_next();
    }
  }
  if constexpr (WIDE) {
    if (warp == 0) {
      __syncwarp();  // the barriers are initialised
      pol = policy_evict_first();
      for (int i = 0; i < NST; ++i) issue_next();
    }
  }

  // query vectors of the group, pre-multiplied by scale * log2 e, for this lane's key slice
  // (8 lanes share a key; lane slice s owns elements [8 (8 v + s), 8 (8 v + s) + 8) for v < D / 64),
  // as pairs of consecutive elements for the packed f32x2 FMA
  const int slice = lane & 7;
  const uint64_t zero2 = f2_pack(0.f, 0.f);
  const uint64_t c2p = f2_pack(p.c2, p.c2);
  uint64_t qr[G][EPL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4* qs = reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.Hq + h0 + g) * D);
#pragma unroll
    for (int v4 = 0; v4 < EPL / 8; ++v4) {
      const uint4 w = qs[v4 * 8 + slice];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) qr[g][v4 * 4 + i] = fma2(pair_of<BF16>(ws[i]), c2p, zero2);
    }
  }

  int gl = 0;  // loads consumed
  bool ok = true;
  uint64_t acc[G][DPL / 2];  // P V accumulators, pairs of adjacent output columns
  for (int c = c0; c < c1; ++c) {
    const int n = chunk_rows(c);
    const int nsub = (n + SUB - 1) / SUB;
    // one partial per chunk; the single-launch decode runs the online softmax on
    // across the CTA's chunks and writes one partial for all of them
    const bool fresh = !MERGE || c == c0;
    if (fresh && threadIdx.x < G) {
      m_run[threadIdx.x] = -INFINITY;
      l_run[threadIdx.x] = 0.f;
    }
    __syncthreads();
    if (fresh) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) acc[g][e] = zero2;
    }

    for (int sub = 0; sub < nsub && ok; ++sub) {
      const int rows = min(SUB, n - sub * SUB);
      // -------------------------------------------------------------- scores
      {
        ok = mbar_wait(ring_bar(gl), (gl / NST) & 1, abort_flag, &g_status, p.wait_limit_ns);
        if (__syncthreads_or(!ok)) {
          ok = false;
          break;
        }
        const uint8_t* tile = smem + L::RING_OFF + (gl % NST) * L::STAGE;
#pragma unroll
        for (int step = 0; step < KEYS_PER_WARP / 4; ++step) {
          const int key = warp * KEYS_PER_WARP + step * 4 + (lane >> 3);
          uint64_t d2[G];
#pragma unroll
          for (int g = 0; g < G; ++g) d2[g] = zero2;
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
                const uint64_t kp = pair_of<BF16>(ws[i2]);
#pragma unroll
                for (int g = 0; g < G; ++g) d2[g] = fma2(qr[g][v4 * 4 + i2], kp, d2[g]);
              }
            }
          }
          float dot[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float lo, hi;
            f2_unpack(d2[g], lo, hi);
            dot[g] = lo + hi;
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
        if (WIDE ? warp == 0 : threadIdx.x == 0) issue_next();
        ++gl;
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
      // ------------------------------------------------------------------ P V
      {
        ok = mbar_wait(ring_bar(gl), (gl / NST) & 1, abort_flag, &g_status, p.wait_limit_ns);
        if (__syncthreads_or(!ok)) {
          ok = false;
          break;
        }
        const uint8_t* tile = smem + L::RING_OFF + (gl % NST) * L::STAGE;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint64_t a2 = f2_pack(alpha_s[g], alpha_s[g]);
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e) acc[g][e] = fma2(acc[g][e], a2, zero2);
        }
#pragma unroll
        for (int kk = 0; kk < KEYS_PER_WARP; ++kk) {
          const int key = warp * KEYS_PER_WARP + kk;
          if (key < rows) {
            uint64_t vv[DPL / 2];
            if constexpr (DPL == 4) {
              const uint2 w = *reinterpret_cast<const uint2*>(tile + key * D * 2 + lane * 8);
              vv[0] = pair_of<BF16>(w.x);
              vv[1] = pair_of<BF16>(w.y);
            } else {
              vv[0] = pair_of<BF16>(*reinterpret_cast<const uint32_t*>(tile + key * D * 2 + lane * 4));
            }
            // the group's probabilities of this key in one shared-memory load
            float pr[G];
            if constexpr (G % 4 == 0) {
#pragma unroll
              for (int q4 = 0; q4 < G / 4; ++q4) {
                const float4 t = reinterpret_cast<const float4*>(sc + key * G)[q4];
                pr[4 * q4] = t.x;
                pr[4 * q4 + 1] = t.y;
                pr[4 * q4 + 2] = t.z;
                pr[4 * q4 + 3] = t.w;
              }
            } else if constexpr (G == 2) {
              const float2 t = reinterpret_cast<const float2*>(sc)[key];
              pr[0] = t.x;
              pr[1] = t.y;
            } else {
              pr[0] = sc[key];
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const uint64_t p2 = f2_pack(pr[g], pr[g]);
#pragma unroll
              for (int e = 0; e < DPL / 2; ++e) acc[g][e] = fma2(p2, vv[e], acc[g][e]);
            }
          }
        }
        __syncthreads();  // every read of this stage done
        if (WIDE ? warp == 0 : threadIdx.x == 0) issue_next();
        ++gl;
      }
    }
    if (!ok) break;
    if (MERGE && c + 1 < c1) continue;  // the CTA's partial is written after its last chunk

    // ---------------------------------------- partials: cross-warp sum of P V
    const size_t pbase = (((size_t)b * p.Hq + h0) * p.max_chunks + (MERGE ? c0 : c)) * (D + 2);
    const size_t hstride = (size_t)p.max_chunks * (D + 2);
#pragma unroll
    for (int pass = 0; pass < G / L::GH; ++pass) {
#pragma unroll
      for (int gg = 0; gg < L::GH; ++gg)
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) {
          float lo, hi;
          f2_unpack(acc[pass * L::GH + gg][e], lo, hi);
          red[(warp * L::GH + gg) * D + lane * DPL + 2 * e] = lo;
          red[(warp * L::GH + gg) * D + lane * DPL + 2 * e + 1] = hi;
        }
      __syncthreads();
      for (int idx = threadIdx.x; idx < L::GH * D; idx += THREADS) {
        const int gg = idx / D, d = idx % D;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s += red[(w * L::GH + gg) * D + d];
        p.part[pbase + (pass * L::GH + gg) * hstride + d] = s;
      }
      __syncthreads();
    }
    if (threadIdx.x < G) {
      const int g = threadIdx.x;
      p.part[pbase + g * hstride + D] = m_run[g] * 0.69314718055994531f;  // natural-log units
      p.part[pbase + g * hstride + D + 1] = l_run[g];
    }
  }

  if (!ok && threadIdx.x == 0) {
    // unwind: wait (bounded) for the copies still in flight, then leave
    const uint64_t t0 = global_timer_ns();
    for (int i = max(gl, issued - NST); i < issued; ++i)
      while (i != withheld && !mbar_try_wait(ring_bar(i), (i / NST) & 1))
        if (global_timer_ns() - t0 > p.wait_limit_ns) break;
  }

  if constexpr (MERGE) {
    // Single launch: a ticket counts the finished CTAs of this (sequence, head
    // group); the last one merges the group's partials and puts the ticket back
    // to zero for the next call.  A CTA that gave up a wait still takes its
    // ticket, so the count stays exact (its chunks' partials are not written and
    // the status word reports it).
    __threadfence();  // this thread's partial stores, ordered before the ticket
    __syncthreads();
    int* last = reinterpret_cast<int*>(smem + L::ABORT_OFF + 4);
    if (threadIdx.x == 0) {
      unsigned* t = p.tickets + (size_t)b * gridDim.y + blockIdx.y;
      const int is_last = atomicAdd(t, 1u) == (unsigned)((nch + p.cpb - 1) / p.cpb - 1);
      if (is_last) {
        atomicExch(t, 0u);
        __threadfence();  // the other CTAs' partials, ordered before this CTA's reads
      }
      *last = is_last;
    }
    __syncthreads();
    if (*last) merge_group<D, G, BF16>(p, b, h0, (nch + p.cpb - 1) / p.cpb, red, sc);
  }
}

// The reduce kernel's merge, run by the last CTA of a (sequence, head group) in
// the single-launch decode over the n partials of the group's CTAs (partial x at
// chunk slot x * cpb): WARPS / G warps per query head share the partials, each
// warp weights its partials by e^(m_x - M) with the head's overall max M, and
// the warps' sums are added in shared memory.  Partials are read from L2
// (written by other CTAs of this launch).
template <int D, int G, bool BF16>
__device__ __forceinline__ void merge_group(const Params& p, int b, int h0, int n, float* red, float* tot) {
  constexpr int DPL = D / 32;
  constexpr int WPH = WARPS / G;  // warps per query head
  constexpr int U = 4;            // chunks whose loads are issued together
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp / WPH, s = warp % WPH;
  const float* base = p.part + ((size_t)b * p.Hq + h0 + g) * p.max_chunks * (D + 2);
  float M = -INFINITY;
  const size_t step = (size_t)p.cpb * (D + 2);
  for (int c = lane; c < n; c += 32) M = fmaxf(M, __ldcg(base + c * step + D));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float total = 0.f;
  for (int cb = s * U; cb < n; cb += WPH * U) {
    float m_c[U], l_c[U], oc[U][DPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      m_c[u] = -INFINITY;
      l_c[u] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) oc[u][e] = 0.f;
      if (cb + u < n) {
        const float* pc = base + (cb + u) * step;
        m_c[u] = __ldcg(pc + D);
        l_c[u] = __ldcg(pc + D + 1);
#pragma unroll
        for (int e2 = 0; e2 < DPL / 2; ++e2) {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(pc + lane * DPL) + e2);
          oc[u][2 * e2] = t.x;
          oc[u][2 * e2 + 1] = t.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!(m_c[u] > -1e30f)) continue;  // past the last partial
      const float w = ex2((m_c[u] - M) * 1.4426950408889634f);
      total = fmaf(l_c[u], w, total);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(oc[u][e], w, acc[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < DPL; ++e) red[warp * D + lane * DPL + e] = acc[e];
  if (lane == 0) tot[warp] = total;
  __syncthreads();
  for (int i = threadIdx.x; i < G * D / 2; i += THREADS) {
    const int gg = (2 * i) / D, d = (2 * i) % D;
    float a0 = 0.f, a1 = 0.f, t = 0.f;
#pragma unroll
    for (int w = 0; w < WPH; ++w) {
      a0 += red[(gg * WPH + w) * D + d];
      a1 += red[(gg * WPH + w) * D + d + 1];
      t += tot[gg * WPH + w];
    }
    const float inv = t > 0.f ? 1.f / t : 0.f;
    reinterpret_cast<uint32_t*>(p.o + ((size_t)b * p.Hq + h0 + gg) * D)[d / 2] =
        pack2<BF16>(a0 * inv, a1 * inv);
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
  // eight chunks per pass, their loads issued together
  constexpr int U = 8;
  for (int cb = 0; cb < n; cb += U) {
    float m_c[U], l_c[U], oc[U][DPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      m_c[u] = -INFINITY;
      l_c[u] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) oc[u][e] = 0.f;
      if (cb + u < n) {
        const float* pc = base + (size_t)(cb + u) * (D + 2);
        m_c[u] = pc[D];
        l_c[u] = pc[D + 1];
        if constexpr (DPL == 4) {
          const float2 a = *reinterpret_cast<const float2*>(pc + lane * 4);
          const float2 bb = *reinterpret_cast<const float2*>(pc + lane * 4 + 2);
          oc[u][0] = a.x;
          oc[u][1] = a.y;
          oc[u][2] = bb.x;
          oc[u][3] = bb.y;
        } else {
          const float2 a = *reinterpret_cast<const float2*>(pc + lane * 2);
          oc[u][0] = a.x;
          oc[u][1] = a.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!(m_c[u] > -1e30f)) continue;  // empty chunk, or past the last one
      const float w = ex2((m_c[u] - M) * 1.4426950408889634f);
      total = fmaf(l_c[u], w, total);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(oc[u][e], w, acc[e]);
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

template <int D, int G, bool BF16, int PG, bool MERGE = false>
static cudaError_t launch_split(const DecodeArgs& a, const Params& p, cudaStream_t stream) {
  using L = SplitLayout<D, G, PG != 0>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G, BF16, PG, MERGE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((a.max_chunks + p.cpb - 1) / p.cpb, a.Hkv * (p.group / G), a.B);
  decode_split_kernel<D, G, BF16, PG, MERGE><<<grid, THREADS, L::BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int G, bool BF16>
static cudaError_t launch_t(const DecodeArgs& a, const Params& p, cudaStream_t stream) {
  if (a.max_chunks > 0 && p.tickets) return launch_split<D, G, BF16, 0, true>(a, p, stream);
  if (a.max_chunks > 0) {
    // the contiguous-cache kernel is a separate instantiation, free of the page logic
    const cudaError_t e = !p.block_table     ? launch_split<D, G, BF16, 0>(a, p, stream)
                          : p.page_size <= 32 ? launch_split<D, G, BF16, 2>(a, p, stream)
                                              : launch_split<D, G, BF16, 1>(a, p, stream);
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
  // chunks per CTA: the most of 4, 2, 1 that keeps a CTA at no more than 2048
  // keys (longer ranges balance worse over ragged sequence lengths) and still
  // leaves at least 8 CTAs per multiprocessor (counting empty chunks)
  const long long per_x = (long long)a.B * a.Hkv * (G / p.heads_per_cta);
  p.cpb = 1;
  for (int cpb = 4; cpb > 1; cpb >>= 1)
    if ((long long)cpb * a.chunk <= 2048 && per_x * ((a.max_chunks + cpb - 1) / cpb) >= 8LL * a.num_sms) {
      p.cpb = cpb;
      break;
    }
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
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.max_S = a.max_S;
  p.chunk = a.chunk;
  p.max_chunks = a.max_chunks;
  p.group = a.Hq / a.Hkv;
  p.c2 = a.scale * 1.4426950408889634f;
  p.wait_limit_ns = a.wait_limit_ns;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.tickets = a.tickets;
  p.debug_fault = a.debug_fault;
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

// Tickets of the single-launch decode (attn_decode_fused): one counter per
// (sequence, head group) row of split-kernel CTAs.  Every counter is zero
// between calls: the CTA that finds itself last in its row puts it back.  The
// array is zeroed once per device on first use, on the calling stream.  Calls
// whose kernels overlap on the GPU share the counters and must not run at once.
static __device__ unsigned g_decode_tickets[kDecodeTickets];

namespace {
unsigned* g_ticket_ptr[64];
}  // namespace

cudaError_t decode_tickets(int device, unsigned** out, cudaStream_t stream) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_ticket_ptr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_tickets);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ptr, 0, sizeof(unsigned) * kDecodeTickets, stream);
    if (e != cudaSuccess) return e;
    g_ticket_ptr[device] = static_cast<unsigned*>(ptr);
  }
  *out = g_ticket_ptr[device];
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
