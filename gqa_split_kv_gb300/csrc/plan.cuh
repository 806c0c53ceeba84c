// Device-side split plan: the partition of every (sequence, KV-head sub-group)
// token range into pieces, one contiguous range of 16-token blocks per CTA.
//
// The pages choose one split count for all sequences and cap it by the tile
// count (AstrAI commit 988e013 "csrc", split-KV items).  This library instead
// lays all segments end to end on one weighted line and cuts the line into equal
// ranges, so a persistent grid stays balanced for any mix of lengths.  The line
// is head-major (every sequence of slot u, then of slot u + 1), so CTAs that run
// at the same time read the KV heads of the same tokens, which share DRAM pages.  Every
// segment is preceded by a gap of c positions that stands for the fixed cost of
// a piece (epilogue, partial tile, query load), so a range full of short
// sequences holds fewer blocks than one inside a long sequence.  Segments are
// padded to whole 64-token units, so every piece starts on a 64-token boundary
// of its sequence (a paged tile then never splits a box of 16, 32 or 64 rows
// across pages).
//
//   n_b  = ceil(L_b / 16)                     blocks of sequence b
//   w_b  = 4 ceil(n_b / 4) + c if n_b > 0, else 0   line positions of one segment
//   c    = 4 ceil((2816 / head_dim) / 4)      (about 176 KB of K+V streaming)
//   P_b  = w_0 + ... + w_{b-1}                (prefix, P_B = line length / U)
//   U    = Hkv * passes                       segment slots per sequence (a pass runs
//                                             one or more sub-groups of <= 8 rows)
//   segment (b, u) = positions [s0, s0 + w_b), s0 = u P_B + P_b; its blocks
//                    sit at [s0 + c, s0 + c + n_b), the rest hold none
//   S >= 2: q = ceil(U P_B / ((S - 1) U)) rounded up to a multiple of 4
//           positions (at least 4), range r = [r q, (r + 1) q); a piece is the
//           blocks of one segment inside one range (ranges that meet none of a
//           segment's blocks give no piece of it)
//   S == 1: range r = segment (r / U, r % U), whole.
#pragma once

#include <cstdint>

namespace da {

constexpr int kBlockTokens = 16;
constexpr int kRangeQuantum = 4;  // ranges start on 64-token units of the line
// Segments cut into at most this many pieces are merged inside the split kernel
// by the CTA that finishes the last piece; longer ones by the combine kernel.
constexpr int kFusedMergeMax = 8;

// Line positions charged to every segment for the fixed cost of a piece (a
// multiple of 4, so segments keep 64-token alignment on the line).
__host__ __device__ constexpr int plan_gap_blocks(int head_dim) { return (2816 / head_dim + 3) / 4 * 4; }

// Line positions of one segment with n blocks (0 for an empty sequence).
__host__ __device__ __forceinline__ int segment_width(int nb, int gap) { return nb > 0 ? ((nb + 3) & ~3) + gap : 0; }


// Block counts are 32-bit: the host rejects problems with 2^30 blocks or more.
struct Plan {
  int NB;      // positions on the line (blocks and gaps)
  int q;       // blocks per range (S >= 2)
  int ranges;  // ranges that hold work
  int U;             // segment slots per sequence (KV head x pass)
  int S;             // partial slots per (b, h)
  int gap;           // positions before each segment's blocks
};

struct Piece {
  int b, u;      // sequence, segment slot
  int t0, t1;    // token range [t0, t1) within the sequence
  int j;         // piece index within the segment (partial slot)
  int npieces;   // pieces of this segment
};

// lens[b] = clamp(seq_lens[b] or max_len, 0, max_len); P[0..B] = prefix of the
// segment widths w_b (segment_width); P[B + 1] = the largest block count of one
// sequence.  Run by the first nthreads threads of the block, which synchronise on
// named barrier bar_id (bar_id 0 with every thread: __syncthreads).
__device__ __forceinline__ void build_plan_arrays(const int* __restrict__ seq_lens, int B, int max_len, int gap,
                                                  int* lens, int* P, int bar_id, int nthreads) {
  for (int b = threadIdx.x; b < B; b += nthreads) {
    int L = seq_lens ? __ldg(seq_lens + b) : max_len;
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    lens[b] = L;
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (B + 31) / 32;
    const int b0 = lane * per;
    const int b1 = min(B, b0 + per);
    int s = 0, mx = 0;
    for (int b = b0; b < b1; ++b) {
      const int nb = (lens[b] + kBlockTokens - 1) / kBlockTokens;
      s += segment_width(nb, gap);
      mx = max(mx, nb);
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    int run = incl - s;
    for (int b = b0; b < b1; ++b) {
      P[b] = run;
      const int nb = (lens[b] + kBlockTokens - 1) / kBlockTokens;
      run += segment_width(nb, gap);
    }
    if (lane == 31) {
      P[B] = incl;
      P[B + 1] = mx;
    }
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
}

__host__ __device__ __forceinline__ Plan make_plan(int B, int U, int S, int gap, const int* P) {
  Plan pl;
  pl.U = U;
  pl.S = S;
  pl.gap = gap;
  pl.NB = U * P[B];
  if (S == 1) {
    pl.q = 0;
    pl.ranges = B * U;
  } else {
    const int R = (S - 1) * U;
    pl.q = (pl.NB + R - 1) / R;
    pl.q = (pl.q + kRangeQuantum - 1) / kRangeQuantum * kRangeQuantum;
    if (pl.q < kRangeQuantum) pl.q = kRangeQuantum;
    pl.ranges = (pl.NB + pl.q - 1) / pl.q;
  }
  return pl;
}

// Number of pieces of segment (b, u) under plan pl (S >= 2).
__host__ __device__ __forceinline__ int segment_pieces(const Plan& pl, const int* lens, const int* P, int B, int b, int u) {
  const int nb = (lens[b] + kBlockTokens - 1) / kBlockTokens;
  if (nb == 0) return 0;
  const int bs = u * P[B] + P[b] + pl.gap;  // first block
  return (bs + nb - 1) / pl.q - bs / pl.q + 1;
}

// S >= 2: the blocks of the segment at line position x that lie in [x, xe), the
// rest of range r.  Returns the position where the next segment of the range
// starts (or xe); pc.t0 == pc.t1 when [x, xe) meets none of the segment's blocks.
__host__ __device__ __forceinline__ int piece_at(const Plan& pl, const int* lens, const int* P, int B, int x, int xe, int r,
                                        Piece& pc) {
  // slot u, then sequence b: the last with P[b] <= x - u P_B (sequences with no
  // blocks are skipped because the following non-empty one shares their prefix)
  const int u = x / P[B];
  const int y = x - u * P[B];
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P[mid] <= y)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int b = lo;
  const int nb = (lens[b] + kBlockTokens - 1) / kBlockTokens;
  const int w = segment_width(nb, pl.gap);
  const int s0 = u * P[B] + P[b];
  const int bs = s0 + pl.gap;  // first block of the segment
  const int be = bs + nb;      // end of its blocks
  const int pe = xe < be ? xe : be;
  const int x0 = x > bs ? x : bs;
  pc.b = b;
  pc.u = u;
  pc.t0 = (x0 - bs) * kBlockTokens;
  const int te = (pe - bs) * kBlockTokens;
  pc.t1 = pe > x0 ? (te < lens[b] ? te : lens[b]) : pc.t0;
  pc.j = r - bs / pl.q;
  pc.npieces = (be - 1) / pl.q - bs / pl.q + 1;
  return xe < s0 + w ? xe : s0 + w;
}

// The first piece of range r if every sequence held max_len tokens: a guess made
// before seq_lens is read, so that the first tiles can be requested early.  False
// when the guess gives the range no piece.
__host__ __device__ __forceinline__ bool guess_first_piece(int B, int U, int S, int gap, int max_len, int r,
                                                           Piece& pc) {
  const int nb = (max_len + kBlockTokens - 1) / kBlockTokens;
  if (nb == 0 || B <= 0) return false;
  pc.j = 0;
  if (S == 1) {
    if (r >= B * U) return false;
    pc.b = r / U;
    pc.u = r % U;
    pc.t0 = 0;
    pc.t1 = max_len;
    pc.npieces = 1;
    return true;
  }
  const int w = segment_width(nb, gap);
  const int NB = U * B * w;
  const int R = (S - 1) * U;
  int q = (NB + R - 1) / R;
  q = (q + kRangeQuantum - 1) / kRangeQuantum * kRangeQuantum;
  if (q < kRangeQuantum) q = kRangeQuantum;
  int x = r * q;
  const int xe = x + q < NB ? x + q : NB;
  for (int k = 0; k < 2 && x < xe; ++k) {
    const int seg = x / w;  // segment (b, u) starts at u * B * w + b * w
    const int s0 = seg * w, bs = s0 + gap, be = bs + nb;
    const int x0 = x > bs ? x : bs;
    const int pe = xe < be ? xe : be;
    if (pe > x0) {
      pc.b = seg % B;
      pc.u = seg / B;
      pc.t0 = (x0 - bs) * kBlockTokens;
      const int te = (pe - bs) * kBlockTokens;
      pc.t1 = te < max_len ? te : max_len;
      return true;
    }
    x = s0 + w;
  }
  return false;
}

// Walks the pieces of the ranges r0, r0 + stride, r0 + 2 stride, ... (a CTA of the
// persistent grid: r0 = blockIdx.x, stride = gridDim.x; the host walks every range
// with r0 = 0, stride = 1).
struct PieceWalker {
  int r;       // range being walked
  int x, xe;   // S >= 2: next block and end of range r
  int stride;
  bool started;

  __host__ __device__ __forceinline__ void init(int r0, int step) {
    r = r0;
    stride = step;
    started = false;
    x = xe = 0;
  }

  // Next piece in walk order; false when the CTA's work is done.  With
  // skip_empty, segments of empty sequences (S == 1 only) are skipped.
  __host__ __device__ __forceinline__ bool next(const Plan& pl, const int* lens, const int* P, int B,
                                                bool skip_empty, Piece& pc) {
    if (pl.S == 1) {
      while (true) {
        if (started) r += stride;
        started = true;
        if (r >= pl.ranges) return false;
        pc.b = r / pl.U;
        pc.u = r % pl.U;
        pc.t0 = 0;
        pc.t1 = lens[pc.b];
        pc.j = 0;
        pc.npieces = 1;
        if (!(skip_empty && pc.t1 == 0)) return true;
      }
    }
    while (true) {
      if (!started) {
        started = true;
        if (r >= pl.ranges) return false;
        x = r * pl.q;
        xe = x + pl.q < pl.NB ? x + pl.q : pl.NB;
      }
      if (x < xe) {
        x = piece_at(pl, lens, P, B, x, xe, r, pc);
        if (pc.t1 > pc.t0) return true;
        continue;  // only a gap: no piece
      }
      r += stride;
      if (r >= pl.ranges) return false;
      x = r * pl.q;
      xe = x + pl.q < pl.NB ? x + pl.q : pl.NB;
    }
  }
};

}  // namespace da
