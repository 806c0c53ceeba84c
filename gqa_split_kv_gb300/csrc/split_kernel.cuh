// Split-KV decode kernel: one persistent CTA per SM walks its ranges of the
// block line; for every piece it streams the K/V tiles of one (sequence, KV head,
// pass) through a TMA-fed shared-memory ring and runs the pass's query rows over
// them with head-packed bf16 tensor-core MMAs and an fp32 online softmax.  The
// rows of a KV head are its G query heads (x q_len query tokens for multi-query
// decode), in sub-groups of at most 8; a pass runs NGP sub-groups.
//
// Roles (warp-specialised):
//   warp W (producer): one elected lane waits for a free stage, posts the byte
//     count and issues the TMA tile copies (K, V and, for the first tile of a
//     piece, the query rows).  Paged caches: the lanes resolve one page-table
//     entry per box (16, 32 or 64 rows of one page), prefetched LA tiles ahead
//     with cp.async.
//   warps 0..W-1 (consumers): W / NGP warps per sub-group; warp ws of a group owns
//     the 16-token sub-blocks ws, ws + W / NGP, ... of every tile.
//
// Prior art on the pages: the two-stage cp.async ring of "perf(dspark): overlap
// KV staging with compute via cp.async" (section "Summary"); the per-warp-group
// KV stripes with their own (m, l, acc) folded in ascending order of
// "perf(qwen3.8): split the flash-decode KV range across warp-groups" (section
// "Mechanism"); MMA head packing, XOR swizzle and one page lookup per tile of
// AstrAI commits 988e013 and 69fecaf.  Here the ring is filled by the Blackwell
// tensor-memory accelerator (cp.async.bulk.tensor, 128-byte swizzle), the stage
// count is sized for the 227 KB of shared memory per CTA, and tiles are
// released through mbarriers instead of CTA-wide barriers.
//
// A segment cut into at most 8 pieces is merged by the CTA that finishes its last
// piece (log-sum-exp over the pieces' partials, ascending order), detected with
// one per-segment counter.  Longer segments (long contexts over few KV heads) are
// merged by the combine kernel, spread over many CTAs: one CTA alone would need
// several dependent rounds of L2 loads (~1 us each) to read their partials.
//
// Head packing: the MMA tile is 16 rows; query heads fill rows 0..7 and rows
// 8..15 carry the bf16 low part of the probabilities, so P = hi + lo reaches
// the fp32 accumulator with ~2^-17 relative error at no extra MMA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "plan.cuh"
#include "ptx.cuh"

namespace da {

// Device error word (bit 0: a bounded wait ran out; bit 1: a segment counter
// update gave up; bit 2: a page-table entry outside [0, num_pages)).  The
// library is one translation unit, so the definition lives here; the host reads
// and clears it through decode_device_error().
__device__ unsigned int g_error_word = 0;

struct SplitParams {
  CUtensorMap tm_k;   // K cache / pool (bf16, or int8 values)
  CUtensorMap tm_v;   // V cache / pool
  CUtensorMap tm_q;   // Q [B, Hq, D]
  CUtensorMap tm_ks;  // int8 caches: K scales per (token, KV head), head-major
  CUtensorMap tm_vs;  // int8 caches: V scales
  const int* seq_lens;
  const int* page_table;
  float* part_acc;
  float* part_ml;
  unsigned long long* seg_counters;  // one per segment (b, u): (epoch << 32) | pieces done
  __nv_bfloat16* out;
  unsigned int epoch;                // tags this call's counter updates (never 0)
  int B, Hq, G, U, ng, gr;  // Hq, G count rows: query heads x qlen query tokens
  int ngp, npass;    // sub-groups (of gr <= 8 rows) per pass over a KV head; passes per head
  int qlen;          // query tokens per sequence (1: decode; > 1: causal block at the end)
  int max_len;       // lengths are clamped to [0, max_len]
  int page_size, max_pages, num_pages;
  int box_shift;     // paged: a TMA box holds 16 << box_shift rows of one page (16, 32 or 64)
  int page_shift;    // log2(page_size) when it is a power of two, else -1
  int S;
  int spec_first;    // contiguous caches of small batches: request the guessed first tiles before the plan
  float scale_log2;  // scale * log2(e)
  unsigned long long timeout_ns;
};

// NGP: sub-groups per pass (the query-row slots per stage); KV8: int8 K/V with
// fp32 scales per (token, KV head), widened to f16 in registers by the MMA warps;
// PG: a paged cache.
template <int D, int NGP = 1, bool KV8 = false, bool PG = false>
struct SplitGeo {
  // bf16 tiles carry 32 KB (D = 32) or 64 KB of K+V so the per-tile costs (barrier
  // round trip, TMA issue, page lookups) stay small against the bytes moved; int8
  // tiles carry half as much (the many small page boxes of a paged int8 tile are
  // split over the producer warps, below).
  static constexpr int T = D <= 64 ? 256 : D <= 128 ? 128 : 64;  // tokens per tile
  // consumer warps: two per scheduler for int8 tiles up to D = 128 (their
  // per-token work is a chain of short-latency integer steps) and for bf16 at
  // D = 32 (256 tokens of softmax per 32 KB tile), else one
  static constexpr int W = (KV8 && D <= 128) || D == 32 ? 8 : 4;
  static constexpr int SB = T / 16;                 // 16-token sub-blocks per tile
  // A pass runs ngp <= NGP_MAX sub-groups of <= 8 rows, one per group of W / ngp
  // warps; the warps of a sub-group take the sub-blocks ws, ws + W / ngp, ... of a tile.
  static constexpr int NGP_MAX = D == 128 ? 2 : 4;
  // sub-blocks per softmax step
  static constexpr int NP = KV8 ? (D <= 64 ? 2 : 1) : (D == 32 ? 2 : D <= 64 ? 4 : D <= 128 ? 2 : 1);
  static constexpr int SUBW = D >= 64 ? 64 : 32;    // elements per swizzle row
  static constexpr int NSUB = D / SUBW;             // swizzle rows per token
  static constexpr int ROWB = SUBW * 2;             // 128 or 64 bytes
  static constexpr int CPR = SUBW / 8;              // 16-byte chunks per swizzle row
  static constexpr int STAGES = KV8 ? (D == 256 ? 3 : D == 32 ? 6 : 4)
                                    : (D == 256 ? 2 : D >= 64 ? 3 : 5);
  // producer warps: paged tiles are many small page boxes, and one issuing warp
  // pays its per-tile and per-copy costs in series, so NPROD producer warps take
  // tiles in turn (four at D = 32, whose 1 KB boxes are the smallest); a
  // contiguous tile is one or two large copies
  static constexpr int NPROD = PG ? (D == 32 ? 4 : 2) : 1;
  static constexpr int NTHREADS = (W + NPROD) * 32;
  // fold scratch columns per fold pass (two passes at D = 128 with extra query rows)
  static constexpr int FD = D == 128 && NGP > 1 ? 64 : D;
  // One TMA box fills all NSUB swizzle columns of its R rows, so a tile is
  // box-major, [T/R][NSUB][R][SUBW]: R = T for a contiguous cache (one box per
  // tile), R = 16, 32 or 64 rows of one page for a paged cache.
  static constexpr int LOG_SB = SB == 16 ? 4 : SB == 8 ? 3 : SB == 4 ? 2 : SB == 2 ? 1 : 0;
  static constexpr int KV_BYTES = T * D * (KV8 ? 1 : 2);  // one tensor, one stage
  // per-token scales of one tensor and stage (int8 caches): one slot of max(R, 32)
  // floats per box, so every box lands 128-byte aligned (16-row paged boxes leave
  // 16 floats unused per slot)
  static constexpr int SC_BYTES = KV8 ? T * 8 : 0;
  // int8 tiles use the same box-major form with byte rows: [T/R][NSUB8][R][SW8],
  // 128-byte swizzled rows at D >= 128, plain D-byte rows below
  static constexpr int SW8 = D >= 128 ? 128 : D;
  static constexpr int NSUB8 = D / SW8;
  static constexpr int al1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int Q_SUB_BYTES = 8 * ROWB;      // one swizzle column of 8 query rows
  static constexpr int Q_SG_BYTES = 8 * D * 2;      // the query rows of one sub-group
  static constexpr int Q_BYTES = NGP * Q_SG_BYTES;
  static constexpr int RING = 16;                   // page-entry ring slots
  static constexpr int LA = 4;                      // page-entry prefetch distance (tiles, 128-256 KB)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_KS = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_VS = OFF_KS + STAGES * SC_BYTES;
  static constexpr int OFF_Q = al1k(OFF_VS + STAGES * SC_BYTES);
  // int8 at D >= 128: each warp keeps its f16 query fragment here ([D/32][32
  // lanes][4 words]) instead of in D/8 registers
  static constexpr bool Q_SMEM = KV8 && D >= 128;
  static constexpr int QF_BYTES = Q_SMEM ? W * D / 32 * 32 * 16 : 0;
  static constexpr int OFF_QF = OFF_Q + STAGES * Q_BYTES;
  static constexpr int OFF_FACC = OFF_QF + QF_BYTES;
  static constexpr int OFF_FML = OFF_FACC + W * 8 * FD * 4;
  static constexpr int OFF_FSC = OFF_FML + W * 8 * 2 * 4;   // per-(warp, row) merge weights
  static constexpr int OFF_FROW = OFF_FSC + W * 8 * 4;      // per-row (M, L, 1/L, -), 32 rows
  static constexpr int OFF_BAR = OFF_FROW + 32 * 4 * 4;
  static constexpr int OFF_PG = OFF_BAR + 2 * STAGES * 8;
  static constexpr int OFF_MISC = OFF_PG + RING * 32 * 4;
  static constexpr int OFF_PLAN = OFF_MISC + 16;
  static constexpr int smem_bytes(int B) { return OFF_PLAN + (2 * B + 2) * 4 + 1024; }
  static_assert(SB % W == 0 && SB <= 32, "whole sub-blocks per warp; one producer lane per block");
  static_assert((1 << LOG_SB) == SB && T >= 64, "power-of-two tiles of whole 64-token units");
  static_assert((SB / W) % NP == 0, "softmax steps cover whole sub-blocks");
  static_assert(NGP <= NGP_MAX && NGP_MAX <= W && W % NGP_MAX == 0 && D % FD == 0,
                "warp groups and fold passes divide evenly");
  static_assert(RING >= LA + 2, "page ring must hold the prefetch window");
  // a producer's previous tile (n - NPROD) waited for tile n - NPROD - STAGES, which
  // must cover tile n - 2 STAGES for its stage wait to be unambiguous; the page
  // ring must hold every entry a producer can request ahead of the slowest one
  static_assert(NPROD <= STAGES && NPROD + STAGES + LA <= RING, "producer warps and rings");
  static_assert(smem_bytes(64) <= 227 * 1024, "shared memory budget");
};

template <int ROWB>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  const uint32_t off = (uint32_t)(row * ROWB + chunk * 16);
  return ROWB == 128 ? off ^ (((off >> 7) & 7u) << 4) : off ^ (((off >> 7) & 3u) << 4);
}

// Bounded mbarrier wait.  Gives up after timeout_ns: sets the device error word
// and the CTA's abort flag, after which every later wait returns at once, so
// all warps still reach the same named barriers and the CTA exits.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicOr(&g_error_word, 1u);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Page-table column of token tok (a shift for power-of-two page sizes).
__device__ __forceinline__ int page_of(const SplitParams& p, int tok) {
  return p.page_shift >= 0 ? tok >> p.page_shift : tok / p.page_size;
}

// Piece + tile cursor used by the producer (pieces without tokens are skipped).
struct TileCursor {
  PieceWalker walk;
  Piece pc;
  int t;
  bool valid;

  __device__ __forceinline__ void init(const Plan& pl, const int* lens, const int* P, int B) {
    walk.init(blockIdx.x, gridDim.x);
    valid = walk.next(pl, lens, P, B, true, pc);
    t = pc.t0;
  }
  __device__ __forceinline__ void advance(const Plan& pl, const int* lens, const int* P, int B, int T) {
    t += T;
    if (t >= pc.t1) {
      valid = walk.next(pl, lens, P, B, true, pc);
      t = pc.t0;
    }
  }
};

// One contiguous-cache tile (and, for a piece's first tile, the pass's query rows)
// of piece pc into ring stage `stage`, issued by a single thread.
template <int D, int NGP, bool KV8>
__device__ __forceinline__ void issue_contig_tile(const SplitParams& p, uint32_t sbase, int stage, const Piece& pc,
                                                  int t) {
  using Gm = SplitGeo<D, NGP, KV8, false>;
  const int h = pc.u / p.npass;
  const int g0 = (pc.u % p.npass) * p.ngp;
  const int nsg = min(p.ngp, p.ng - g0);
  const bool first_tile = t == pc.t0;
  const uint32_t full = sbase + Gm::OFF_BAR + stage * 8;
  const uint32_t qbytes = first_tile ? (uint32_t)(nsg * Gm::NSUB * p.gr * Gm::ROWB) : 0u;
  const uint32_t kvbytes = (uint32_t)(Gm::KV_BYTES + (KV8 ? Gm::T * 4 : 0));
  mbar_arrive_expect_tx(full, 2u * kvbytes + qbytes);
  tma_load_5d(sbase + Gm::OFF_K + stage * Gm::KV_BYTES, &p.tm_k, full, 0, t, 0, h, pc.b);
  tma_load_5d(sbase + Gm::OFF_V + stage * Gm::KV_BYTES, &p.tm_v, full, 0, t, 0, h, pc.b);
  if constexpr (KV8) {
    tma_load_3d(sbase + Gm::OFF_KS + stage * Gm::SC_BYTES, &p.tm_ks, full, t, h, pc.b);
    tma_load_3d(sbase + Gm::OFF_VS + stage * Gm::SC_BYTES, &p.tm_vs, full, t, h, pc.b);
  }
  if (first_tile) {
    const uint32_t qdst = sbase + Gm::OFF_Q + stage * Gm::Q_BYTES;
    for (int sg = 0; sg < nsg; ++sg)
      for (int sub = 0; sub < Gm::NSUB; ++sub)
        tma_load_4d(qdst + sg * Gm::Q_SG_BYTES + sub * Gm::Q_SUB_BYTES, &p.tm_q, full, 0, sub,
                    h * p.G + (g0 + sg) * p.gr, pc.b);
  }
}

// Whether the guessed first piece is the piece the plan gives this CTA first
// (producer and consumers decide it alike).
__device__ __forceinline__ bool guess_hit(const Plan& pl, const int* lens, const int* P, int B, const Piece& g) {
  PieceWalker w;
  w.init(blockIdx.x, gridDim.x);
  Piece f;
  return w.next(pl, lens, P, B, true, f) && f.b == g.b && f.u == g.u && f.t0 == g.t0 && f.t1 == g.t1;
}

template <int D, bool PAGED, int NGP, bool KV8>
__device__ __forceinline__ void split_producer(const SplitParams& p, const Plan& pl, const int* lens, const int* P,
                                               uint8_t* smem, uint32_t sbase, volatile int* abort_flag,
                                               const Piece& guess, int k_spec) {
  using Gm = SplitGeo<D, NGP, KV8, PAGED>;
  const int lane = threadIdx.x & 31;
  // With NPROD producer warps, warp pw issues the tiles n with n % NPROD == pw
  // (with their page entries and query boxes).  All walk every tile.  The
  // consumers release tiles in order, and a producer's previous tile (n - NPROD)
  // waited for tile n - NPROD - STAGES, so its stage wait on tile n - STAGES
  // cannot see a phase a whole ring cycle old (NPROD <= STAGES).
  const int pw = (threadIdx.x >> 5) - Gm::W;
  const uint32_t bar_full = sbase + Gm::OFF_BAR;
  const uint32_t bar_empty = bar_full + Gm::STAGES * 8;
  const uint32_t pg_ring = sbase + Gm::OFF_PG;
  const int* pg_ring_ptr = reinterpret_cast<const int*>(smem + Gm::OFF_PG);

  TileCursor cur;
  cur.init(pl, lens, P, p.B);
  TileCursor look = cur;
  const int box_rows = PAGED ? 16 << p.box_shift : Gm::T;

  // Page entries of tile k go to ring slot k % RING, one cp.async group per
  // tile.  Tile 0's group is requested first, and tiles 1 .. LA only after tile
  // 0's copies are out, so the first tile waits on one lookup, not LA of them.
  auto request_pages = [&](int k) {
    if (look.valid) {
      const int nb = (min(Gm::T, look.pc.t1 - look.t) + box_rows - 1) >> (4 + p.box_shift);
      if (k % Gm::NPROD == pw && lane < nb) {
        const int tok = look.t + lane * box_rows;
        cp_async_4(pg_ring + (uint32_t)((k % Gm::RING) * 32 + lane) * 4,
                   p.page_table + (size_t)look.pc.b * p.max_pages + page_of(p, tok));
      }
      look.advance(pl, lens, P, p.B, Gm::T);
    }
    cp_async_commit();
  };
  if (PAGED) request_pages(0);

  int n = 0;  // tiles issued
  int stage = 0;
  uint32_t parity = 0;
  if (k_spec > 0) {
    // stages 0 .. k_spec - 1 hold the guessed first tiles: on a hit they are this
    // CTA's first tiles; else they are drained (their copies land, then the stages
    // are released as if consumed) and the ring starts after them
    if (guess_hit(pl, lens, P, p.B, guess)) {
      for (int k = 0; k < k_spec; ++k) cur.advance(pl, lens, P, p.B, Gm::T);
    } else if (lane == 0) {
      for (int k = 0; k < k_spec; ++k) {
        wait_bounded(bar_full + k * 8, 0, abort_flag, p.timeout_ns);
        mbar_arrive_cnt(bar_empty + k * 8, Gm::W);
      }
    }
    __syncwarp();
    n = k_spec;
    stage = k_spec % Gm::STAGES;
    parity = (uint32_t)(k_spec / Gm::STAGES);
  }
  while (cur.valid) {
    const Piece& pc = cur.pc;
    const int h = pc.u / p.npass;
    const int g0 = (pc.u % p.npass) * p.ngp;  // first sub-group of this pass
    const int nsg = min(p.ngp, p.ng - g0);     // sub-groups in this pass
    const bool first_tile = cur.t == pc.t0;
    const int ntok = min(Gm::T, pc.t1 - cur.t);
    const int nbox = PAGED ? (ntok + box_rows - 1) >> (4 + p.box_shift) : 1;  // boxes of this tile
    const bool own = Gm::NPROD == 1 || n % Gm::NPROD == pw;  // this warp issues tile n

    int page = 0;
    if (PAGED) {
      if (n > 0) {  // groups 0 .. n + LA requested; tile n's must be complete
        request_pages(n + Gm::LA);
        cp_async_wait<Gm::LA>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      if (own && lane < nbox) {
        page = pg_ring_ptr[(n % Gm::RING) * 32 + lane];
        if ((unsigned)page >= (unsigned)p.num_pages) {  // a bad entry: flag it, read page 0 instead
          atomicOr(&g_error_word, 4u);
          page = 0;
        }
      }
    }

    if (own) {
      // wait until the consumers have released this stage (first pass: free)
      bool ok = true;
      if (lane == 0) ok = wait_bounded(bar_empty + stage * 8, parity ^ 1u, abort_flag, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;

      const uint32_t full = bar_full + stage * 8;
      const uint32_t kdst = sbase + Gm::OFF_K + stage * Gm::KV_BYTES;
      const uint32_t vdst = sbase + Gm::OFF_V + stage * Gm::KV_BYTES;
      const uint32_t qdst = sbase + Gm::OFF_Q + stage * Gm::Q_BYTES;
      const uint32_t qbytes = first_tile ? (uint32_t)(nsg * Gm::NSUB * p.gr * Gm::ROWB) : 0u;
      // K/V boxes (and, for int8 caches, their per-token scales) move whole
      const uint32_t kvbytes = PAGED ? (uint32_t)(nbox * box_rows * (D * (KV8 ? 1 : 2) + (KV8 ? 4 : 0)))
                                     : (uint32_t)(Gm::KV_BYTES + (KV8 ? Gm::T * 4 : 0));
      if (lane == 0) mbar_arrive_expect_tx(full, 2u * kvbytes + qbytes);
      __syncwarp();
      if (PAGED) {
        // tiles start on 64-token boundaries (the plan pads segments to whole
        // 64-token units) and box_rows divides both 64 and the page size, so a
        // box never crosses a page
        if (lane < nbox) {
          const int tok = cur.t + lane * box_rows;
          const int row0 = tok - page_of(p, tok) * p.page_size;
          const uint32_t off = (uint32_t)(lane * box_rows * D * (KV8 ? 1 : 2));
          tma_load_5d(kdst + off, &p.tm_k, full, 0, row0, 0, h, page);
          tma_load_5d(vdst + off, &p.tm_v, full, 0, row0, 0, h, page);
          if constexpr (KV8) {  // [rows] fp32 scale boxes, one 128-byte aligned slot per box
            const uint32_t soff = (uint32_t)(lane * max(box_rows, 32) * 4);
            tma_load_3d(sbase + Gm::OFF_KS + stage * Gm::SC_BYTES + soff, &p.tm_ks, full, row0, h, page);
            tma_load_3d(sbase + Gm::OFF_VS + stage * Gm::SC_BYTES + soff, &p.tm_vs, full, row0, h, page);
          }
        }
      } else if (lane == 0) {
        tma_load_5d(kdst, &p.tm_k, full, 0, cur.t, 0, h, pc.b);
        tma_load_5d(vdst, &p.tm_v, full, 0, cur.t, 0, h, pc.b);
        if constexpr (KV8) {
          tma_load_3d(sbase + Gm::OFF_KS + stage * Gm::SC_BYTES, &p.tm_ks, full, cur.t, h, pc.b);
          tma_load_3d(sbase + Gm::OFF_VS + stage * Gm::SC_BYTES, &p.tm_vs, full, cur.t, h, pc.b);
        }
      }
      if (first_tile && lane < nsg * Gm::NSUB) {  // one box per (sub-group, swizzle column)
        const int sg = lane / Gm::NSUB, sub = lane % Gm::NSUB;
        tma_load_4d(qdst + sg * Gm::Q_SG_BYTES + sub * Gm::Q_SUB_BYTES, &p.tm_q, full, 0, sub,
                    h * p.G + (g0 + sg) * p.gr, pc.b);
      }
    }
    if (PAGED && n == 0) {
#pragma unroll 1
      for (int k = 1; k <= Gm::LA; ++k) request_pages(k);
    }
    ++n;
    if (++stage == Gm::STAGES) {
      stage = 0;
      parity ^= 1u;
    }
    cur.advance(pl, lens, P, p.B, Gm::T);
  }
  if (PAGED) cp_async_wait<0>();

  // After an abort, let the copies this warp issued land before the CTA exits.
  if (*abort_flag && lane == 0) {
    for (int k = n > Gm::STAGES ? n - Gm::STAGES : 0; k < n; ++k) {
      if (k % Gm::NPROD != pw) continue;
      const uint32_t full = bar_full + (uint32_t)(k % Gm::STAGES) * 8;
      const uint32_t par = (uint32_t)((k / Gm::STAGES) & 1);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(full, par) && globaltimer_ns() - t0 < p.timeout_ns) {
      }
    }
  }
}

// Per-segment counters.  A counter holds (epoch << 32) | count, where the epoch
// tags the call; a value with another epoch counts as zero, so counters never
// need resetting between calls.  A finished piece adds one with a single
// acquire-release atomic; the first add of a call that finds another call's
// value replaces it by compare-and-swap.  The piece that completes a segment
// stores (epoch + 1) << 32: the next call, which normally carries epoch + 1, then
// finds a zero count of its own and takes the one-add path; any other call (a
// replayed CUDA graph carries its captured epoch) treats it as another call's value.
constexpr uint32_t kCounterError = 0xffffffffu;

// Adds one to this call's count of counter c; returns the count before the add.
__device__ __forceinline__ uint32_t counter_add(unsigned long long* c, unsigned int epoch) {
  const unsigned long long old = atom_add_acqrel(c, 1ull);
  if ((uint32_t)(old >> 32) == epoch) return (uint32_t)old;
  // another call's value (the add above went to it): replace that value with
  // this call's, or add to it if another piece of this call already did
  unsigned long long v = old + 1ull;
  for (int it = 0; it < (1 << 20); ++it) {
    const bool ours = (uint32_t)(v >> 32) == epoch;
    const unsigned long long nv = ours ? v + 1ull : ((unsigned long long)epoch << 32) | 1ull;
    const unsigned long long prev = atom_cas_acqrel(c, v, nv);
    if (prev == v) return ours ? (uint32_t)v : 0u;
    v = prev;
  }
  atomicOr(&g_error_word, 2u);
  return kCounterError;
}

// Counts one finished piece of a segment of n pieces; true for the piece that
// completes it.
__device__ __forceinline__ bool claim_last_piece(unsigned long long* c, unsigned int epoch, int n) {
  const uint32_t cnt = counter_add(c, epoch);
  if (cnt == kCounterError || (int)cnt + 1 != n) return false;
  st_relaxed_u64(c, (unsigned long long)(epoch + 1u) << 32);
  return true;
}

// Log-sum-exp merge of `count` (<= kFusedMergeMax) partial slots slot0, slot0 +
// sstride, ... of the nrows rows row0 .. row0 + nrows - 1 of sequence b, in
// ascending slot order, by the W consumer warps.  to_partial: the merged
// unnormalised partial (acc, m, l) of the slots' joint token range replaces slot
// slot0; else the bf16 output rows are written.  Partials written by other CTAs
// are read through L2 (ld.global.cg).  Every thread merges (row, 4-column)
// items, MI at a time with all of their slot loads in flight; the first items'
// loads go out before anything else, and each warp meanwhile turns the (m, l) of
// its rows into weights in shared memory (wsm: 10 floats per row, the 8 weights,
// M and the denominator), so the weights cost no L2 round trip of their own.
template <int D, int W, int MI>
__device__ __forceinline__ void merge_slots(const SplitParams& p, float* wsm, int b, int row0, int nrows, int slot0,
                                            int sstride, int count, bool to_partial) {
  constexpr int C4 = D / 4;  // float4 columns per row
  constexpr int NT = W * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float kNegInf = -__int_as_float(0x7f800000);
  const int nitems = nrows * C4;
  // item e: row e / C4, float4 column e % C4; slot i of it at acc_of(e) + i * sstride * C4
  auto acc_of = [&](int e) {
    const size_t row = (size_t)b * p.Hq + row0 + e / C4;
    return reinterpret_cast<float4*>(p.part_acc + (row * p.S + slot0) * D) + e % C4;
  };
  float4 a[MI][kFusedMergeMax];
  auto load_items = [&](int e0) {
#pragma unroll
    for (int k = 0; k < MI; ++k) {
      const int e = e0 + k * NT + tid;
      if (e < nitems) {
        const float4* acc = acc_of(e);
#pragma unroll
        for (int i = 0; i < kFusedMergeMax; ++i)
          if (i < count) a[k][i] = __ldcg(acc + (size_t)i * sstride * C4);
      }
    }
  };
  load_items(0);
  for (int r = warp; r < nrows; r += W) {
    const size_t row = (size_t)b * p.Hq + row0 + r;
    float2 v = make_float2(kNegInf, 0.f);
    if (lane < count) v = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + row * p.S + slot0 + (size_t)lane * sstride);
    float M = v.y > 0.f ? v.x : kNegInf;  // over the slots that saw a token
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
    const float w = v.y > 0.f ? exp2_approx((v.x - M) * 1.4426950408889634f) : 0.f;
    float den = 0.f;  // ascending slot order, the same in every lane
#pragma unroll
    for (int i = 0; i < kFusedMergeMax; ++i) den += __shfl_sync(0xffffffffu, w * v.y, i);
    if (lane < kFusedMergeMax) wsm[r * 10 + lane] = w;
    if (lane == 0) {
      wsm[r * 10 + 8] = M;
      wsm[r * 10 + 9] = den;
    }
  }
  named_bar_sync(1, NT);  // weights ready; every (m, l) of slot0 has been read
  if (to_partial && tid < nrows) {
    const size_t row = (size_t)b * p.Hq + row0 + tid;
    reinterpret_cast<float2*>(p.part_ml)[row * p.S + slot0] = make_float2(wsm[tid * 10 + 8], wsm[tid * 10 + 9]);
  }
  for (int e0 = 0; e0 < nitems; e0 += MI * NT) {
    if (e0 > 0) load_items(e0);
#pragma unroll
    for (int k = 0; k < MI; ++k) {
      const int e = e0 + k * NT + tid;
      if (e >= nitems) continue;
      const int r = e / C4;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kFusedMergeMax; ++i) {
        if (i < count) {
          const float wi = wsm[r * 10 + i];
          num.x += wi * a[k][i].x;
          num.y += wi * a[k][i].y;
          num.z += wi * a[k][i].z;
          num.w += wi * a[k][i].w;
        }
      }
      if (to_partial) {
        *acc_of(e) = num;  // this thread read every slot of item e above
      } else {
        const float den = wsm[r * 10 + 9];
        const float inv = den > 0.f ? 1.f / den : 0.f;  // a row that saw no token: zeros
        uint2 o;
        o.x = pack_bf16x2(num.x * inv, num.y * inv);
        o.y = pack_bf16x2(num.z * inv, num.w * inv);
        const size_t row = (size_t)b * p.Hq + row0 + r;
        *reinterpret_cast<uint2*>(p.out + row * D + 4 * (e % C4)) = o;
      }
    }
  }
}

// int8 sub-blocks (16 tokens) are multiplied straight from the int8 tile, each
// thread widening the bytes of its MMA operands to f16 in registers (exact).
//  QK^T: thread (g, c) of a warp, g = lane / 4, c = lane % 4, holds D / 4
//        consecutive bytes of token rows g and 8 + g; word w of them, bytes
//        4w .. 4w + 3, is k-chunk w of the product, its four bytes filling the
//        thread's k-slots 2c, 2c + 1, 2c + 8, 2c + 9.  The query fragment takes the
//        same d order (kq_dim), so the dot products are unchanged.
//  PV:   thread (g, c) needs, per 8-column block, token rows 2c, 2c + 1, 8 + 2c,
//        9 + 2c at one d: it loads a run of d's of those four rows and transposes
//        bytes with byte_perm.  Column n of block nt is d = pv_dim(nt, n).
template <int D>
__host__ __device__ constexpr int kq_dim(int kk, int c, int e) {  // d of k-chunk kk, k-slot group c, byte e
  return D >= 64 ? 64 * (kk / 4) + 16 * c + 4 * (kk % 4) + e : 8 * c + 4 * kk + e;
}
template <int D>
__host__ __device__ constexpr int pv_dim(int nt, int n) {
  constexpr int run = D / 8 < 16 ? D / 8 : 16;  // d's of one thread's row run
  return (nt / run) * (8 * run) + n * run + nt % run;
}

// Rows a and b, one word (the same four d's) each -> the f16 pairs (a_d, b_d) for
// d = 0 .. 3 (a in the low half).  int8 x becomes f16 0x6400 | (x ^ 0x80), which
// is 1152 + x exactly; subtracting 1152 in f16 is exact.
__device__ __forceinline__ void int8_pairs_to_f16(uint32_t a, uint32_t b, uint32_t (&o)[4]) {
  const uint32_t lo = __byte_perm(a, b, 0x5140) ^ 0x80808080u;  // a0 b0 a1 b1
  const uint32_t hi = __byte_perm(a, b, 0x7362) ^ 0x80808080u;  // a2 b2 a3 b3
  const uint32_t h0 = __byte_perm(lo, 0x64646464u, 0x5150);
  const uint32_t h1 = __byte_perm(lo, 0x64646464u, 0x5352);
  const uint32_t h2 = __byte_perm(hi, 0x64646464u, 0x5150);
  const uint32_t h3 = __byte_perm(hi, 0x64646464u, 0x5352);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(h0), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(h1), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2]) : "r"(h2), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[3]) : "r"(h3), "r"(0x64806480u));
}

// n consecutive 32-bit words of shared memory (n = 1, 2 or 4; 4n-byte aligned)
template <int N>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t* w) {
  if constexpr (N == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

template <int D, bool PAGED, int NGP, bool KV8>
__device__ __forceinline__ void split_consumer(const SplitParams& p, const Plan& pl, const int* lens, const int* P,
                                               uint8_t* smem, uint32_t sbase, volatile int* abort_flag,
                                               const Piece& guess, int k_spec) {
  using Gm = SplitGeo<D, NGP, KV8, PAGED>;
  constexpr int KCH = D / 16;  // k-chunks of the QK^T product
  constexpr int NB8 = D / 8;   // 8-column blocks of the PV product
  constexpr int NP = Gm::NP;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // MMA row (query head within the group)
  const int i4 = lane & 3;
  const uint32_t bar_full = sbase + Gm::OFF_BAR;
  const uint32_t bar_empty = bar_full + Gm::STAGES * 8;
  float* facc = reinterpret_cast<float*>(smem + Gm::OFF_FACC);
  float* fml = reinterpret_cast<float*>(smem + Gm::OFF_FML);
  const float kNegInf = -__int_as_float(0x7f800000);

  // box-major tile (see SplitGeo): a box of 16 << rsh rows spans NSUB swizzle columns
  const int rsh = PAGED ? p.box_shift : Gm::LOG_SB;
  const uint32_t col_stride = (uint32_t)(16 * Gm::ROWB) << rsh;
  const uint32_t box_bytes = col_stride * Gm::NSUB;
  const int in_box = (1 << rsh) - 1;
  auto blk_off = [&](int kb) -> uint32_t {
    return (uint32_t)(kb >> rsh) * box_bytes + (uint32_t)((kb & in_box) * 16 * Gm::ROWB);
  };
  // ldmatrix lane -> (row, chunk) patterns
  const int k_row0 = (lane & 7) + ((lane >> 4) << 3);
  const int k_chk = (lane >> 3) & 1;
  const int v_row0 = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int v_chk = lane >> 4;
  // warp group of this warp's sub-group (NGP sub-groups per pass, p.ngp == NGP),
  // and its stripe within the group
  constexpr int WS = Gm::W / NGP;  // warps per sub-group
  constexpr int SBW = Gm::SB / WS; // sub-blocks per warp and tile
  const int sg = warp / WS, ws = warp % WS;
  // int8 tiles: box-major [T/R][NSUB8][R][SW8] bytes
  constexpr int SW8 = Gm::SW8;
  const uint32_t col8 = (uint32_t)(16 * SW8) << rsh;  // one swizzle column of a box
  const uint32_t box8 = col8 * Gm::NSUB8;
  auto blk_off8 = [&](int kb) -> uint32_t {
    return (uint32_t)(kb >> rsh) * box8 + (uint32_t)((kb & in_box) * 16 * SW8);
  };
  // 16-byte chunk ch of row r (< 16) of a sub-block, swizzled at SW8 = 128
  auto chunk8 = [&](int r, int ch) -> uint32_t {
    return (uint32_t)(ch / (SW8 / 16)) * col8 +
           (SW8 == 128 ? swz<128>(r, ch % 8) : (uint32_t)(r * SW8 + (ch % (SW8 / 16)) * 16));
  };
  // K words of token rows g and 8 + g (k-chunk order), D / 4 bytes each
  auto load_k8 = [&](const uint8_t* sb8, uint32_t* w0, uint32_t* w1) {
    if constexpr (D >= 64) {
#pragma unroll
      for (int j = 0; j < D / 64; ++j) {
        const uint32_t o = chunk8(g, 4 * j + i4);
        lds_words<4>(sb8 + o, w0 + 4 * j);
        lds_words<4>(sb8 + o + 8 * SW8, w1 + 4 * j);
      }
    } else {
      const uint32_t o = (uint32_t)(g * SW8 + 8 * i4);
      lds_words<2>(sb8 + o, w0);
      lds_words<2>(sb8 + o + 8 * SW8, w1);
    }
  };
  // V words of token rows 2c, 2c + 1, 8 + 2c, 9 + 2c: D / 8 bytes each, the runs
  // of d's that pv_dim gives this thread's MMA column g
  auto load_v8 = [&](const uint8_t* sb8, uint32_t (*vw)[D / 32]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = (e & 1) + 2 * i4 + ((e >> 1) << 3);
      if constexpr (D >= 128) {
#pragma unroll
        for (int j = 0; j < D / 128; ++j) lds_words<4>(sb8 + chunk8(r, 8 * j + g), vw[e] + 4 * j);
      } else {
        lds_words<D / 32>(sb8 + r * SW8 + g * (D / 8), vw[e]);
      }
    }
  };

  if (p.S >= 2) {
    // empty sequences have no pieces on the block line: write their zero outputs
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
      if (lens[b] != 0) continue;
      uint4* o = reinterpret_cast<uint4*>(p.out + (size_t)b * p.Hq * D);
      for (int i = threadIdx.x; i < p.Hq * D / 8; i += Gm::W * 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  PieceWalker walk;
  walk.init(blockIdx.x, gridDim.x);
  Piece pc;
  int stage = 0;  // ring position of the next tile to consume
  uint32_t parity = 0;
  if (k_spec > 0 && !guess_hit(pl, lens, P, p.B, guess)) {  // the producer drains the guessed stages
    stage = k_spec % Gm::STAGES;
    parity = (uint32_t)(k_spec / Gm::STAGES);
  }
  while (walk.next(pl, lens, P, p.B, false, pc)) {
    uint32_t qa[KCH][2];
    float acc[NB8][4];
#pragma unroll
    for (int c = 0; c < NB8; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
    float m_run = kNegInf, l_run = 0.f;
    // int8: K enters the MMA as 1152 + k (int8x4_to_f16x4_biased), so every score
    // of row g carries 1152 * (sum of the row's f16 query), removed before scaling
    float kbias = 0.f;
    const int h = pc.u / p.npass;
    const int pass_u = pc.u % p.npass;
    const int gidx = pass_u * p.ngp + sg;  // this warp's sub-group
    const int first_head = h * p.G + gidx * p.gr;
    const int nrows = gidx < p.ng ? min(p.gr, p.G - gidx * p.gr) : 0;  // 0: nothing to do this piece
    // Rows are (query head, query token i); query token i of a block of qlen sees
    // the tokens before L - qlen + 1 + i.  lim_row bounds this thread's MMA row,
    // lim_min every row of the warp (qlen == 1: both are the piece end).
    int lim_row = pc.t1, lim_min = pc.t1;
    if (p.qlen > 1) {
      const int L = lens[pc.b];
      lim_row = min(pc.t1, L - (p.qlen - 1 - (gidx * p.gr + g) % p.qlen));
      lim_min = min(pc.t1, L - p.qlen + 1);
    }

    for (int t = pc.t0; t < pc.t1; t += Gm::T) {
      wait_bounded(bar_full + stage * 8, parity, abort_flag, p.timeout_ns);
      if (t == pc.t0 && nrows > 0 && KV8) {
        // f16 query fragment in kq_dim order: row g, d = kq_dim(kk, c, 0 .. 3)
        const uint8_t* qs = smem + Gm::OFF_Q + stage * Gm::Q_BYTES + sg * Gm::Q_SG_BYTES;
#pragma unroll
        for (int j = 0; j < (D >= 64 ? D / 64 : 1); ++j) {
          uint32_t w[8];
          if constexpr (D >= 64) {
            lds_words<4>(qs + j * Gm::Q_SUB_BYTES + swz<Gm::ROWB>(g, 2 * i4), w);
            lds_words<4>(qs + j * Gm::Q_SUB_BYTES + swz<Gm::ROWB>(g, 2 * i4 + 1), w + 4);
          } else {
            lds_words<4>(qs + swz<Gm::ROWB>(g, i4), w);
          }
#pragma unroll
          for (int m = 0; m < (D >= 64 ? 4 : 2); ++m) {
            const uint32_t a0 = g < nrows ? w[2 * m] : 0u, a2 = g < nrows ? w[2 * m + 1] : 0u;
            qa[(D >= 64 ? 4 : 2) * j + m][0] = pack_f16x2(bf16lo_to_f32(a0), bf16hi_to_f32(a0));
            qa[(D >= 64 ? 4 : 2) * j + m][1] = pack_f16x2(bf16lo_to_f32(a2), bf16hi_to_f32(a2));
          }
        }
        // the row's query sum, from the f16 values the MMA multiplies (each thread
        // of the quad holds a quarter of the row's d's)
        float qsum = 0.f;
#pragma unroll
        for (int kk = 0; kk < KCH; ++kk)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const __half2 hq = *reinterpret_cast<const __half2*>(&qa[kk][e]);
            const float2 fq = __half22float2(hq);
            qsum += fq.x + fq.y;
          }
        qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
        qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
        kbias = 1152.f * qsum;
        if constexpr (Gm::Q_SMEM) {  // k-chunks 2m, 2m + 1 per 16-byte slot, read back by this lane only
          uint4* qf = reinterpret_cast<uint4*>(smem + Gm::OFF_QF) + warp * (KCH / 2) * 32 + lane;
#pragma unroll
          for (int m = 0; m < KCH / 2; ++m)
            qf[m * 32] = make_uint4(qa[2 * m][0], qa[2 * m][1], qa[2 * m + 1][0], qa[2 * m + 1][1]);
        }
      }
      if (t == pc.t0 && nrows > 0 && !KV8) {
        const uint32_t qst = sbase + Gm::OFF_Q + stage * Gm::Q_BYTES + sg * Gm::Q_SG_BYTES;
#pragma unroll
        for (int jq = 0; jq < D / 32; ++jq) {
          const int c = 4 * jq + (lane >> 3);
          uint32_t r0, r1, r2, r3;
          ldsm_x4(qst + (c / Gm::CPR) * Gm::Q_SUB_BYTES + swz<Gm::ROWB>(lane & 7, c % Gm::CPR), r0, r1, r2, r3);
          qa[2 * jq][0] = r0;
          qa[2 * jq][1] = r1;
          qa[2 * jq + 1][0] = r2;
          qa[2 * jq + 1][1] = r3;
        }
        if (g >= nrows) {
#pragma unroll
          for (int c = 0; c < KCH; ++c) qa[c][0] = qa[c][1] = 0u;
        }
      }
      const uint32_t kst = sbase + Gm::OFF_K + stage * Gm::KV_BYTES;
      const uint32_t vst = sbase + Gm::OFF_V + stage * Gm::KV_BYTES;
      // int8 caches: the stage's tiles and per-token scales
      const uint8_t* kst8 = smem + Gm::OFF_K + stage * Gm::KV_BYTES;
      const uint8_t* vst8 = smem + Gm::OFF_V + stage * Gm::KV_BYTES;
      const float* ksc = reinterpret_cast<const float*>(smem + Gm::OFF_KS + stage * Gm::SC_BYTES);
      const float* vsc = reinterpret_cast<const float*>(smem + Gm::OFF_VS + stage * Gm::SC_BYTES);
      const int sc_blk = PAGED && rsh == 0 ? 32 : 16;  // floats from one sub-block's scales to the next
#pragma unroll 1
      for (int sb = 0; sb < (nrows > 0 ? SBW : 0); sb += NP) {  // idle warps only release the stage
        // NP sub-blocks of this warp share one online-softmax step
        if (t + 16 * (ws + WS * sb) >= pc.t1) break;  // later sub-blocks lie further out
        float x[NP][4];
        uint32_t vm_lo[NP], vm_hi[NP];
        bool tail[NP];
        // int8: every K word of the step is loaded before the first MMA (at D = 256
        // 64 d's at a time, next to their MMAs)
        constexpr bool K_EARLY = KV8 && D <= 128;  // (one sub-block per step at D = 128)
        uint32_t kw[KV8 ? NP : 1][2][KV8 ? KCH : 1];
        if constexpr (K_EARLY) {
#pragma unroll
          for (int i = 0; i < NP; ++i) load_k8(kst8 + blk_off8(ws + WS * (sb + i)), kw[i][0], kw[i][1]);
        }
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const int kb = ws + WS * (sb + i);
          const int tok0 = t + 16 * kb;
          const uint32_t kbase = kst + blk_off(kb);
          // even and odd k-chunks go to separate accumulators (two short dependency
          // chains per 8-token half instead of one long one), added at the end
          float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
          float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < KCH; ++kk) {
            float(&sa)[4] = (KCH >= 4 && (kk & 1)) ? s2 : s0;
            float(&sb_)[4] = (KCH >= 4 && (kk & 1)) ? s3 : s1;
            uint32_t b0, b1, b2, b3;
            if constexpr (KV8) {  // tokens 0-7 from row g's word, 8-15 from row 8 + g's
              if (!K_EARLY && kk % 4 == 0) {
                const uint8_t* sb8 = kst8 + blk_off8(kb);
                const uint32_t o = chunk8(g, kk + i4);  // 16-byte chunk 4 (kk / 4) + c
                lds_words<4>(sb8 + o, kw[i][0] + kk);
                lds_words<4>(sb8 + o + 8 * SW8, kw[i][1] + kk);
              }
              int8x4_to_f16x4_biased(kw[i][0][kk], b0, b1);
              int8x4_to_f16x4_biased(kw[i][1][kk], b2, b3);
              uint32_t a0 = qa[kk][0], a2 = qa[kk][1];
              if constexpr (Gm::Q_SMEM) {
                const uint4 q4 = reinterpret_cast<const uint4*>(smem + Gm::OFF_QF)[(warp * (KCH / 2) + kk / 2) * 32 + lane];
                a0 = kk % 2 ? q4.z : q4.x;
                a2 = kk % 2 ? q4.w : q4.y;
              }
              mma_f16_16816(sa, a0, 0u, a2, 0u, b0, b1);
              mma_f16_16816(sb_, a0, 0u, a2, 0u, b2, b3);
            } else {
              const int c = 2 * kk + k_chk;
              ldsm_x4(kbase + (c / Gm::CPR) * col_stride + swz<Gm::ROWB>(k_row0, c % Gm::CPR), b0, b1, b2, b3);
              mma_bf16_16816(sa, qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
              mma_bf16_16816(sb_, qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
            }
          }
          if (KCH >= 4) {
            s0[0] += s2[0];
            s0[1] += s2[1];
            s1[0] += s3[0];
            s1[1] += s3[1];
          }
          x[i][0] = (s0[0] - kbias) * p.scale_log2;
          x[i][1] = (s0[1] - kbias) * p.scale_log2;
          x[i][2] = (s1[0] - kbias) * p.scale_log2;
          x[i][3] = (s1[1] - kbias) * p.scale_log2;
          if constexpr (KV8) {  // K = k_i8 * k_scale: the scale of token t multiplies its score
            const float2 ka = *reinterpret_cast<const float2*>(ksc + kb * sc_blk + 2 * i4);
            const float2 kc = *reinterpret_cast<const float2*>(ksc + kb * sc_blk + 8 + 2 * i4);
            x[i][0] *= ka.x;
            x[i][1] *= ka.y;
            x[i][2] *= kc.x;
            x[i][3] *= kc.y;
          }
          // tokens at or past the row's limit: score -inf; at or past the piece end
          // also V row zeroed (its shared memory may hold anything, and 0 * NaN
          // would poison the accumulator)
          tail[i] = tok0 + 16 > lim_min;
          vm_lo[i] = vm_hi[i] = 0xffffffffu;
          if (tail[i]) {
            const int ta = tok0 + 2 * i4, tb = tok0 + 8 + 2 * i4;
            x[i][0] = ta < lim_row ? x[i][0] : kNegInf;
            x[i][1] = ta + 1 < lim_row ? x[i][1] : kNegInf;
            x[i][2] = tb < lim_row ? x[i][2] : kNegInf;
            x[i][3] = tb + 1 < lim_row ? x[i][3] : kNegInf;
            vm_lo[i] = (ta < pc.t1 ? 0x0000ffffu : 0u) | (ta + 1 < pc.t1 ? 0xffff0000u : 0u);
            vm_hi[i] = (tb < pc.t1 ? 0x0000ffffu : 0u) | (tb + 1 < pc.t1 ? 0xffff0000u : 0u);
          }
        }
        // int8: the step's V words are requested before the softmax, which hides their
        // latency (at D = 256 after it: 128 accumulators leave no room for them)
        constexpr bool V_EARLY = KV8 && D <= 64;
        uint32_t vw[KV8 ? NP : 1][4][KV8 ? D / 32 : 1];
        if constexpr (V_EARLY) {
#pragma unroll
          for (int i = 0; i < NP; ++i) load_v8(vst8 + blk_off8(ws + WS * (sb + i)), vw[i]);
        }
        float mx = kNegInf;
#pragma unroll
        for (int i = 0; i < NP; ++i) mx = fmaxf(mx, fmaxf(fmaxf(x[i][0], x[i][1]), fmaxf(x[i][2], x[i][3])));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = m_new == kNegInf ? 0.f : m_new;  // a row that has seen no token yet
        const float alpha = exp2_approx(m_run - m_use);
        float pr[NP][4];
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) pr[i][k4] = exp2_approx(x[i][k4] - m_use);
          psum += (pr[i][0] + pr[i][1]) + (pr[i][2] + pr[i][3]);
        }
        l_run = l_run * alpha + psum;
        if (__any_sync(0xffffffffu, m_new != m_run)) {
#pragma unroll
          for (int c = 0; c < NB8; ++c) {
            acc[c][0] *= alpha;
            acc[c][1] *= alpha;
            acc[c][2] *= alpha;
            acc[c][3] *= alpha;
          }
        }
        m_run = m_new;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const int kb = ws + WS * (sb + i);
          const uint32_t vbase = vst + blk_off(kb);
          uint32_t ph0, ph1, pl0, pl1;
          if constexpr (KV8) {
            // V = v_i8 * v_scale: the scale of token t multiplies its probability (tokens
            // past the piece end have p = 0 but scales that may be anything)
            const float2 va = *reinterpret_cast<const float2*>(vsc + kb * sc_blk + 2 * i4);
            const float2 vc = *reinterpret_cast<const float2*>(vsc + kb * sc_blk + 8 + 2 * i4);
            float pv[4] = {pr[i][0] * va.x, pr[i][1] * va.y, pr[i][2] * vc.x, pr[i][3] * vc.y};
            if (tail[i]) {
              const int ta = t + 16 * kb + 2 * i4, tb = ta + 8;
              pv[0] = ta < pc.t1 ? pv[0] : 0.f;
              pv[1] = ta + 1 < pc.t1 ? pv[1] : 0.f;
              pv[2] = tb < pc.t1 ? pv[2] : 0.f;
              pv[3] = tb + 1 < pc.t1 ? pv[3] : 0.f;
            }
            // P' = hi + lo in f16
            ph0 = pack_f16x2(pv[0], pv[1]);
            ph1 = pack_f16x2(pv[2], pv[3]);
            pl0 = pack_f16x2(pv[0] - f16lo_to_f32(ph0), pv[1] - f16hi_to_f32(ph0));
            pl1 = pack_f16x2(pv[2] - f16lo_to_f32(ph1), pv[3] - f16hi_to_f32(ph1));
          } else {
            // P = hi + lo in bf16: rows g (hi) and g + 8 (lo) of the A operand
            ph0 = pack_bf16x2(pr[i][0], pr[i][1]);
            ph1 = pack_bf16x2(pr[i][2], pr[i][3]);
            pl0 = pack_bf16x2(pr[i][0] - bf16lo_to_f32(ph0), pr[i][1] - bf16hi_to_f32(ph0));
            pl1 = pack_bf16x2(pr[i][2] - bf16lo_to_f32(ph1), pr[i][3] - bf16hi_to_f32(ph1));
          }
          if constexpr (KV8) {
            // int8 rows are finite whatever the tile holds past the piece end, and
            // those tokens carry P' = 0: no V mask
#pragma unroll
            for (int wi = 0; wi < D / 32; ++wi) {
              if (!V_EARLY && wi % 4 == 0) {  // the 16-byte run wi / 4 of the four rows
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  lds_words<4>(vst8 + blk_off8(kb) + chunk8((e & 1) + 2 * i4 + ((e >> 1) << 3), 2 * wi + g),
                               vw[i][e] + wi);
              }
              uint32_t o01[4], o23[4];
              int8_pairs_to_f16(vw[i][0][wi], vw[i][1][wi], o01);  // tokens 2c, 2c + 1
              int8_pairs_to_f16(vw[i][2][wi], vw[i][3][wi], o23);  // tokens 8 + 2c, 9 + 2c
#pragma unroll
              for (int e = 0; e < 4; ++e) mma_f16_16816(acc[4 * wi + e], ph0, pl0, ph1, pl1, o01[e], o23[e]);
            }
          } else {
#pragma unroll
            for (int c2 = 0; c2 < NB8 / 2; ++c2) {
              const int c = 2 * c2 + v_chk;
              uint32_t v0, v1, v2, v3;
              ldsm_x4_t(vbase + (c / Gm::CPR) * col_stride + swz<Gm::ROWB>(v_row0, c % Gm::CPR), v0, v1, v2, v3);
              if (tail[i]) {
                v0 &= vm_lo[i];
                v1 &= vm_hi[i];
                v2 &= vm_lo[i];
                v3 &= vm_hi[i];
              }
              mma_bf16_16816(acc[2 * c2], ph0, pl0, ph1, pl1, v0, v1);
              mma_bf16_16816(acc[2 * c2 + 1], ph0, pl0, ph1, pl1, v2, v3);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + stage * 8);
      if (++stage == Gm::STAGES) {
        stage = 0;
        parity ^= 1u;
      }
    }

    // ---- fold each sub-group's warps' (m, l, acc) in ascending warp order, then
    // write.  The scratch holds FD columns per warp and row; wider heads fold in
    // D / FD passes.  Rows of the pass: row0 + s * gr + r for sub-group s.
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (g < nrows && i4 == 0) {
      fml[(warp * 8 + g) * 2 + 0] = m_run;
      fml[(warp * 8 + g) * 2 + 1] = l_run;
    }
    const int tid = threadIdx.x;
    float* fsc = reinterpret_cast<float*>(smem + Gm::OFF_FSC);
    float* frow = reinterpret_cast<float*>(smem + Gm::OFF_FROW);
    const bool direct = pc.npieces == 1;
    const int nsg = min(p.ngp, p.ng - pass_u * p.ngp);     // sub-groups of this pass
    const int row0 = h * p.G + pass_u * p.ngp * p.gr;     // its first row
    const int nrows_pass = min(nsg * p.gr, p.G - pass_u * p.ngp * p.gr);
    constexpr int FD = Gm::FD;
#pragma unroll
    for (int pass = 0; pass < D / FD; ++pass) {
      if (g < nrows) {
        float* dst = facc + (warp * 8 + g) * FD;
        if constexpr (KV8) {  // column n of 8-column block c is d = pv_dim(c, n)
#pragma unroll
          for (int c = 0; c < NB8; ++c) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int d = pv_dim<D>(c, 2 * i4 + h2);
              if (d / FD == pass) dst[d - pass * FD] = acc[c][h2] + acc[c][2 + h2];
            }
          }
        } else {
#pragma unroll
          for (int c = pass * (FD / 8); c < (pass + 1) * (FD / 8); ++c)
            *reinterpret_cast<float2*>(dst + 8 * c - pass * FD + 2 * i4) =
                make_float2(acc[c][0] + acc[c][2], acc[c][1] + acc[c][3]);
        }
      }
      named_bar_sync(1, Gm::W * 32);
      if (pass == 0) {
        // one thread per row of the pass: its sub-group's warps' merge weights and
        // the row's (M, L); row sr is row r of sub-group s
        const int sr = tid;
        const int s = NGP == 1 ? 0 : sr / p.gr, r = NGP == 1 ? sr : sr - s * p.gr;
        if (sr < nrows_pass) {
          float M = kNegInf;
          for (int w = s * WS; w < (s + 1) * WS; ++w) M = fmaxf(M, fml[(w * 8 + r) * 2]);
          float L = 0.f;
          for (int w = s * WS; w < (s + 1) * WS; ++w) {
            const float mw = fml[(w * 8 + r) * 2];
            const float sc = mw == kNegInf ? 0.f : exp2_approx(mw - M);
            fsc[w * 8 + r] = sc;
            L += sc * fml[(w * 8 + r) * 2 + 1];
          }
          frow[sr * 4 + 0] = M;
          frow[sr * 4 + 1] = L;
          frow[sr * 4 + 2] = L > 0.f ? 1.f / L : 0.f;
        }
        named_bar_sync(1, Gm::W * 32);
      }
      for (int e = tid; e < nrows_pass * (FD / 2); e += Gm::W * 32) {
        const int sr = e / (FD / 2);  // row of the pass: row r of sub-group s
        const int s = NGP == 1 ? 0 : sr / p.gr, r = NGP == 1 ? sr : sr - s * p.gr;
        const int dl = 2 * (e % (FD / 2));
        const int d = pass * FD + dl;
        float a0 = 0.f, a1 = 0.f;
        for (int w = s * WS; w < (s + 1) * WS; ++w) {
          const float sc = fsc[w * 8 + r];
          const float2 v = *reinterpret_cast<const float2*>(facc + (w * 8 + r) * FD + dl);
          a0 += sc * v.x;
          a1 += sc * v.y;
        }
        const size_t row = (size_t)pc.b * p.Hq + row0 + sr;
        if (direct) {
          const float inv = frow[sr * 4 + 2];
          *reinterpret_cast<uint32_t*>(p.out + row * D + d) = pack_bf16x2(a0 * inv, a1 * inv);
        } else {
          const size_t slot = row * p.S + pc.j;
          *reinterpret_cast<float2*>(p.part_acc + slot * D + d) = make_float2(a0, a1);
          if (d == 0)
            *reinterpret_cast<float2*>(p.part_ml + slot * 2) =
                make_float2(frow[sr * 4] * 0.69314718055994531f, frow[sr * 4 + 1]);
        }
      }
      if (pass + 1 < D / FD) named_bar_sync(1, Gm::W * 32);  // scratch reused by the next pass
    }
    if (!direct && pc.npieces <= kFusedMergeMax) {
      // publish this piece; the CTA that completes the segment merges it.  The
      // barrier orders every consumer's partial stores before thread 0's
      // acquire-release counter update, which releases them.
      named_bar_sync(1, Gm::W * 32);
      volatile int* last = reinterpret_cast<volatile int*>(smem + Gm::OFF_MISC) + 1;
      if (tid == 0) *last = claim_last_piece(p.seg_counters + (size_t)pc.b * p.U + pc.u, p.epoch, pc.npieces);
      named_bar_sync(1, Gm::W * 32);
      // one item per thread in flight: two raise the bf16 D = 128 kernel from 216
      // to 248 registers, and a 192-thread paged CTA then leaves no room beside it
      // for a combine CTA (512 threads x 40 registers)
      if (*last) merge_slots<D, Gm::W, 1>(p, facc, pc.b, row0, nrows_pass, 0, 1, pc.npieces, false);
    }
    named_bar_sync(1, Gm::W * 32);
  }
}

template <int D, bool PAGED, int NGP, bool KV8>
__global__ void __launch_bounds__(SplitGeo<D, NGP, KV8, PAGED>::NTHREADS, 1)
    split_kernel(const __grid_constant__ SplitParams p) {
  using Gm = SplitGeo<D, NGP, KV8, PAGED>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  int* lens = reinterpret_cast<int*>(smem + Gm::OFF_PLAN);
  int* P = lens + p.B;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Gm::OFF_MISC);
  const int warp = threadIdx.x >> 5;

  // Contiguous caches of small batches: the first tile of the piece this CTA gets
  // if every sequence holds max_len tokens (the usual case there) is requested
  // before seq_lens is read; the plan then confirms or drains it.  One tile only:
  // DRAM serves the requests of all CTAs side by side, so a whole ring per CTA
  // requested at once would land no tile early; the rest follow once the plan
  // is built.
  Piece guess{};
  int k_spec = 0;
  if (!PAGED && p.spec_first && guess_first_piece(p.B, p.U, p.S, plan_gap_blocks(D), p.max_len, blockIdx.x, guess))
    k_spec = min(1, (guess.t1 - guess.t0 + Gm::T - 1) / Gm::T);
  // Barriers 2 (consumers) and 3, 4 (everyone) order the start.  The consumers
  // read seq_lens first (so the guessed copies do not queue ahead of it) and build
  // the plan on barrier 2; then they wait on barrier 3 for the mbarriers, which
  // lane 0 of the first producer warp initialises before the producer warps arrive
  // there, and arrive on barrier 4, where the producers wait for the plan (after
  // the guessed tiles are issued).
  constexpr int kAll = Gm::NTHREADS, kCons = Gm::W * 32;
  if (warp >= Gm::W) {
    if (threadIdx.x == Gm::W * 32) {
#pragma unroll
      for (int s = 0; s < Gm::STAGES; ++s) {
        mbar_init(sbase + Gm::OFF_BAR + s * 8, 1);
        mbar_init(sbase + Gm::OFF_BAR + (Gm::STAGES + s) * 8, Gm::W);
      }
      *abort_flag = 0;
      fence_mbar_init();
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      prefetch_tensormap(&p.tm_q);
      if (KV8) {
        prefetch_tensormap(&p.tm_ks);
        prefetch_tensormap(&p.tm_vs);
      }
    }
    __syncwarp();
    named_bar_arrive(3, kAll);
    if constexpr (!PAGED) {
      if (threadIdx.x == Gm::W * 32)
        for (int k = 0; k < k_spec; ++k) issue_contig_tile<D, NGP, KV8>(p, sbase, k, guess, guess.t0 + k * Gm::T);
    }
    // The combine kernel (launched only when a segment can have more than 8
    // pieces) may start now; it waits on the device for this grid to finish.
    pdl_launch_dependents();
    named_bar_sync(4, kAll);
  } else {
    build_plan_arrays(p.seq_lens, p.B, p.max_len, plan_gap_blocks(D), lens, P, 2, kCons);
    pdl_launch_dependents();
    named_bar_sync(3, kAll);
    named_bar_arrive(4, kAll);
  }
  const Plan pl = make_plan(p.B, p.U, p.S, plan_gap_blocks(D), P);
  if (warp >= Gm::W)
    split_producer<D, PAGED, NGP, KV8>(p, pl, lens, P, smem, sbase, abort_flag, guess, k_spec);
  else
    split_consumer<D, PAGED, NGP, KV8>(p, pl, lens, P, smem, sbase, abort_flag, guess, k_spec);
}

}  // namespace da
