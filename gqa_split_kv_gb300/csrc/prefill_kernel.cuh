// Causal GQA prefill / chunked prefill over the decode cache.
//
// "gqa_prefill_attn" on the AstrAI commit page ("csrc", commit 988e013) is a
// tiled shared-memory K/V kernel with mask support, and the same page's notes on
// its double-buffered rework compare it with torch SDPA.  The pages give no
// layout or mask rule, so the reading is the plain causal
// one: sequence b holds L_b cached tokens whose last q_len are the chunk, and query
// token i (position L_b - q_len + i) sees positions 0 .. L_b - q_len + i.
//
// GB300 design.  Unlike decode, a KV tile here serves many query rows, so the
// work is a dense contraction.  One CTA owns one (sequence, KV head, block of BQ
// query tokens); its rows are the block's tokens x the G query heads of the KV head
// (token-major, BQ = ROWS / G, ROWS = 64 or 128 rows).  64-token K/V tiles come in
// by TMA (the decode maps, 128- or 64-byte swizzle) up to the block's last causal
// limit; each MMA warp owns 16 rows: S = Q K^T into registers, a masked
// online softmax in log2 units, P packed to bf16 (the C fragment of S is the A
// fragment of P V), and P V accumulated in fp32.  Masks apply only to tiles that
// reach past the block's first row limit.  Blocks launch in groups of grp
// (sequence, KV head) units whose K/V fit in L2 together, and within a group the
// heaviest blocks (latest query tokens) first, so the CTAs in flight stream the
// same few K/V ranges from L2.
#pragma once

#include <cstdint>

namespace da {

struct PrefillParams {
  CUtensorMap tm_k;  // K cache / pool (bf16, swizzled boxes of 64 tokens or of R pool rows)
  CUtensorMap tm_v;
  const __nv_bfloat16* q;  // [B, q_len, Hq, D]
  __nv_bfloat16* out;      // [B, q_len, Hq, D]
  const int* seq_lens;     // [B] or null (every sequence max_len tokens)
  const int* page_table;   // paged: [B, max_pages]
  int B, q_len, Hq, Hkv, G, BQ, nqb;
  int grp;  // (sequence, KV head) units per launch group (their K/V fit in L2 together)
  int max_len;
  int page_size, max_pages, num_pages, box_shift, page_shift;
  float scale_log2;
  unsigned long long timeout_ns;
};

// Up to D = 128: two CTAs per SM, each 4 MMA warps plus a TMA producer warp.  At
// D = 256 the fp32 output accumulators allow one CTA per SM, so it has 8 MMA warps
// (two per scheduler) and no producer warp: warp 0 issues each tile's copies once
// every warp has left the stage (a CTA barrier per tile).
template <int D>
struct PrefillGeo {
  static constexpr int BK = 64;                    // keys per tile
  static constexpr bool PRODUCER = D != 256;       // a dedicated TMA producer warp
  static constexpr int W = PRODUCER ? 4 : 8;       // MMA warps, 16 rows each
  static constexpr int ROWS = 16 * W;              // query rows per CTA
  static constexpr int NTHREADS = (W + (PRODUCER ? 1 : 0)) * 32;
  static constexpr int CTAS = D == 256 ? 1 : 2;    // CTAs per SM
  static constexpr int SUBW = D >= 64 ? 64 : 32;   // elements per swizzle row
  static constexpr int NSUB = D / SUBW;
  static constexpr int ROWB = SUBW * 2;
  static constexpr int CPR = SUBW / 8;
  static constexpr int STAGES = D <= 64 ? 4 : 2;
  static constexpr int KV_BYTES = BK * D * 2;      // one tensor, one stage
  static constexpr int Q_BYTES = ROWS * D * 2;     // [NSUB][ROWS][SUBW], swizzled
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_Q = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_Q + Q_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 2 * STAGES * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(CTAS * SMEM <= 227 * 1024, "shared memory budget");
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(PrefillGeo<D>::NTHREADS, PrefillGeo<D>::CTAS)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
  using Gm = PrefillGeo<D>;
  constexpr int BK = Gm::BK;
  constexpr int KCH = D / 16;  // k-chunks of Q K^T
  constexpr int NB8 = D / 8;   // 8-column blocks of the output
  constexpr int NT = BK / 8;   // 8-key blocks of a tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t bar_full = sbase + Gm::OFF_BAR;
  const uint32_t bar_empty = bar_full + Gm::STAGES * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Gm::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float kNegInf = -__int_as_float(0x7f800000);

  // work unit: group of grp (b, h) units (the last group may be smaller), then
  // query blocks latest first, then the units of the group
  const int nbh = p.B * p.Hkv;
  const long long per_grp = (long long)p.nqb * p.grp;
  const int gi = (int)(blockIdx.x / per_grp);
  const int gsz = min(p.grp, nbh - gi * p.grp);
  const int in_g = (int)(blockIdx.x - gi * per_grp);
  const int qb = p.nqb - 1 - in_g / gsz;
  const int bh = gi * p.grp + in_g % gsz;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  int L = p.seq_lens ? __ldg(p.seq_lens + b) : p.max_len;
  L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);
  const int q0 = qb * p.BQ;
  const int nq = min(p.BQ, p.q_len - q0);
  const int base = L - p.q_len;  // position of query token 0 is base (+ i)
  // keys [0, kv_end) are seen by some row of the block; keys below lim_first by all
  const int kv_end = max(0, min(L, base + q0 + nq));
  const int lim_first = max(0, min(L, base + q0 + 1));
  const int ntiles = (kv_end + BK - 1) / BK;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < Gm::STAGES; ++s) {
      mbar_init(bar_full + s * 8, 1);
      if (Gm::PRODUCER) mbar_init(bar_empty + s * 8, Gm::W);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == (Gm::PRODUCER ? Gm::W : 0) && lane == 0) {
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
  }
  __syncthreads();

  // Tile n's page entries (paged: lane j < nbox reads box j's entry) and its copies
  // into stage st (one whole warp: lane 0 sets the expected bytes, one box per lane)
  const int box_rows = PAGED ? 16 << p.box_shift : BK;
  auto tile_boxes = [&](int n) { return PAGED ? (min(BK, kv_end - n * BK) + box_rows - 1) / box_rows : 1; };
  auto lookup_page = [&](int n) {
    int page = 0;
    if (PAGED && lane < tile_boxes(n)) {
      const int tok = n * BK + lane * box_rows;
      const int col = p.page_shift >= 0 ? tok >> p.page_shift : tok / p.page_size;
      page = __ldg(p.page_table + (size_t)b * p.max_pages + col);
      if ((unsigned)page >= (unsigned)p.num_pages) {  // a bad entry: flag it, read page 0 instead
        atomicOr(&g_error_word, 4u);
        page = 0;
      }
    }
    return page;
  };
  auto issue_tile = [&](int n, int st, int page) {
    const int t = n * BK;
    const int nbox = tile_boxes(n);
    const uint32_t full = bar_full + st * 8;
    const uint32_t kdst = sbase + Gm::OFF_K + st * Gm::KV_BYTES;
    const uint32_t vdst = sbase + Gm::OFF_V + st * Gm::KV_BYTES;
    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(2 * nbox * box_rows * D * 2));
    __syncwarp();
    if (PAGED) {
      // tiles start on 64-token boundaries and box_rows divides 64 and the page
      // size, so a box never crosses a page
      if (lane < nbox) {
        const int tok = t + lane * box_rows;
        const int row0 = tok - (p.page_shift >= 0 ? (tok >> p.page_shift) << p.page_shift
                                                   : tok / p.page_size * p.page_size);
        const uint32_t off = (uint32_t)(lane * box_rows * D * 2);
        tma_load_5d(kdst + off, &p.tm_k, full, 0, row0, 0, h, page);
        tma_load_5d(vdst + off, &p.tm_v, full, 0, row0, 0, h, page);
      }
    } else if (lane == 0) {
      tma_load_5d(kdst, &p.tm_k, full, 0, t, 0, h, b);
      tma_load_5d(vdst, &p.tm_v, full, 0, t, 0, h, b);
    }
  };
  // after an abort, let the copies already issued land before the CTA exits
  auto drain = [&](int issued) {
    for (int k = issued > Gm::STAGES ? issued - Gm::STAGES : 0; k < issued; ++k) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_full + (uint32_t)(k % Gm::STAGES) * 8, (uint32_t)((k / Gm::STAGES) & 1)) &&
             globaltimer_ns() - t0 < p.timeout_ns) {
      }
    }
  };

  if (Gm::PRODUCER && warp == Gm::W) {
    // ---- producer: tile n of K and V into stage n % STAGES, once it is free
    int stage = 0;
    uint32_t parity = 0;
    int issued = 0;
    for (int n = 0; n < ntiles; ++n) {
      const int page = lookup_page(n);  // before the wait: the lookup overlaps it
      bool ok = true;
      if (lane == 0) ok = wait_bounded(bar_empty + stage * 8, parity ^ 1u, abort_flag, p.timeout_ns);
      if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
      issue_tile(n, stage, page);
      ++issued;
      if (++stage == Gm::STAGES) {
        stage = 0;
        parity ^= 1u;
      }
    }
    if (*abort_flag && lane == 0) drain(issued);
    return;
  }
  // no producer warp: warp 0 issues the first STAGES tiles now, the rest as stages
  // free up (issued counts warp 0's tiles, for the drain after an abort)
  int issued = 0;
  if (!Gm::PRODUCER && warp == 0) {
    for (int n = 0; n < min(ntiles, Gm::STAGES); ++n) issue_tile(n, n, lookup_page(n));
    issued = min(ntiles, Gm::STAGES);
  }

  // ---- MMA warps.  Query tile: row r = (token r / G, head r % G) of the block,
  // zero past the block; [NSUB][ROWS][SUBW] with the bf16 tile swizzle.
  const int nrows = nq * p.G;
  for (int e = threadIdx.x; e < Gm::ROWS * (D / 8); e += Gm::W * 32) {
    const int r = e / (D / 8), ch = e % (D / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < nrows) {
      const int i = q0 + r / p.G, hq = h * p.G + r % p.G;
      v = __ldg(reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.q_len + i) * p.Hq + hq) * D) + ch);
    }
    const int col = (8 * ch) / Gm::SUBW, cc = ((8 * ch) % Gm::SUBW) / 8;
    *reinterpret_cast<uint4*>(smem + Gm::OFF_Q + col * (Gm::ROWS * Gm::ROWB) + swz<Gm::ROWB>(r, cc)) = v;
  }
  named_bar_sync(1, Gm::W * 32);

  const int g = lane >> 2, c4 = lane & 3;
  const int r0 = 16 * warp;
  // key limits of this thread's two MMA rows (0 for rows past the block)
  auto row_limit = [&](int r) { return r < nrows ? max(0, min(L, base + q0 + r / p.G + 1)) : 0; };
  const int limA = row_limit(r0 + g), limB = row_limit(r0 + g + 8);
  // ldmatrix lane patterns: Q (A operand, rows x k), K (B, keys x k), V (B, keys x d, transposed)
  const int qa_row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3), qa_chk = lane >> 4;
  const int k_row0 = (lane & 7) + ((lane >> 4) << 3), k_chk = (lane >> 3) & 1;
  const int v_row0 = (lane & 7) + (((lane >> 3) & 1) << 3), v_chk = lane >> 4;
  const int rsh = PAGED ? p.box_shift : 2;  // a box holds 16 << rsh rows
  const uint32_t col_stride = (uint32_t)(16 * Gm::ROWB) << rsh;
  const uint32_t box_bytes = col_stride * Gm::NSUB;
  const int in_box = (1 << rsh) - 1;
  auto blk_off = [&](int kb) -> uint32_t {
    return (uint32_t)(kb >> rsh) * box_bytes + (uint32_t)((kb & in_box) * 16 * Gm::ROWB);
  };
  const uint32_t qs = sbase + Gm::OFF_Q;

  float o[NB8][4];
#pragma unroll
  for (int c = 0; c < NB8; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;
  float mA = kNegInf, mB = kNegInf, lA = 0.f, lB = 0.f;
  int stage = 0;
  uint32_t parity = 0;
  const bool warp_has_rows = r0 < nrows;

  for (int n = 0; n < ntiles; ++n) {
    wait_bounded(bar_full + stage * 8, parity, abort_flag, p.timeout_ns);
    const int t = n * BK;
    if (warp_has_rows && !*abort_flag) {
      const uint32_t kst = sbase + Gm::OFF_K + stage * Gm::KV_BYTES;
      const uint32_t vst = sbase + Gm::OFF_V + stage * Gm::KV_BYTES;
      float s[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KCH; ++kk) {
        uint32_t a0, a1, a2, a3;
        const int qc = 2 * kk + qa_chk;
        ldsm_x4(qs + (qc / Gm::CPR) * (Gm::ROWS * Gm::ROWB) + swz<Gm::ROWB>(qa_row, qc % Gm::CPR), a0, a1, a2, a3);
        const int kc = 2 * kk + k_chk;
#pragma unroll
        for (int kb = 0; kb < BK / 16; ++kb) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + blk_off(kb) + (kc / Gm::CPR) * col_stride + swz<Gm::ROWB>(k_row0, kc % Gm::CPR), b0, b1, b2,
                  b3);
          mma_bf16_16816(s[2 * kb], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(s[2 * kb + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // scale to log2 units; -inf at or past each row's limit (only tiles that reach
      // past the block's first limit)
      const bool masked = t + BK > lim_first;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int key = t + 8 * j + 2 * c4;
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] *= p.scale_log2;
        if (masked) {
          s[j][0] = key < limA ? s[j][0] : kNegInf;
          s[j][1] = key + 1 < limA ? s[j][1] : kNegInf;
          s[j][2] = key < limB ? s[j][2] : kNegInf;
          s[j][3] = key + 1 < limB ? s[j][3] : kNegInf;
        }
      }
      float xA = kNegInf, xB = kNegInf;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        xA = fmaxf(xA, fmaxf(s[j][0], s[j][1]));
        xB = fmaxf(xB, fmaxf(s[j][2], s[j][3]));
      }
      xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
      xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
      xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
      xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
      const float mnA = fmaxf(mA, xA), mnB = fmaxf(mB, xB);
      // a row that has seen no key keeps a finite reference, so its weights are exactly 0
      const float muA = mnA == kNegInf ? 0.f : mnA, muB = mnB == kNegInf ? 0.f : mnB;
      const float alA = exp2_approx(mA - muA), alB = exp2_approx(mB - muB);
      mA = mnA;
      mB = mnB;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        s[j][0] = exp2_approx(s[j][0] - muA);
        s[j][1] = exp2_approx(s[j][1] - muA);
        s[j][2] = exp2_approx(s[j][2] - muB);
        s[j][3] = exp2_approx(s[j][3] - muB);
        sumA += s[j][0] + s[j][1];
        sumB += s[j][2] + s[j][3];
      }
      lA = lA * alA + sumA;
      lB = lB * alB + sumB;
#pragma unroll
      for (int c = 0; c < NB8; ++c) {
        o[c][0] *= alA;
        o[c][1] *= alA;
        o[c][2] *= alB;
        o[c][3] *= alB;
      }
      // keys at or past kv_end: the tile's V rows there may hold anything (0 * NaN)
      const bool tail = t + BK > kv_end;
#pragma unroll
      for (int kb = 0; kb < BK / 16; ++kb) {
        // P of keys 16 kb .. 16 kb + 15 as the A operand: rows g / g + 8, key pairs
        const uint32_t a0 = pack_bf16x2(s[2 * kb][0], s[2 * kb][1]);
        const uint32_t a1 = pack_bf16x2(s[2 * kb][2], s[2 * kb][3]);
        const uint32_t a2 = pack_bf16x2(s[2 * kb + 1][0], s[2 * kb + 1][1]);
        const uint32_t a3 = pack_bf16x2(s[2 * kb + 1][2], s[2 * kb + 1][3]);
        uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
        if (tail) {
          const int ka = t + 16 * kb + 2 * c4, kb8 = ka + 8;
          vm_lo = (ka < kv_end ? 0x0000ffffu : 0u) | (ka + 1 < kv_end ? 0xffff0000u : 0u);
          vm_hi = (kb8 < kv_end ? 0x0000ffffu : 0u) | (kb8 + 1 < kv_end ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int c2 = 0; c2 < NB8 / 2; ++c2) {
          const int c = 2 * c2 + v_chk;
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vst + blk_off(kb) + (c / Gm::CPR) * col_stride + swz<Gm::ROWB>(v_row0, c % Gm::CPR), v0, v1, v2,
                    v3);
          if (tail) {
            v0 &= vm_lo;
            v1 &= vm_hi;
            v2 &= vm_lo;
            v3 &= vm_hi;
          }
          mma_bf16_16816(o[2 * c2], a0, a1, a2, a3, v0, v1);
          mma_bf16_16816(o[2 * c2 + 1], a0, a1, a2, a3, v2, v3);
        }
      }
    }
    if constexpr (Gm::PRODUCER) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + stage * 8);
    } else {
      // every warp has left the stage: warp 0 refills it with tile n + STAGES
      named_bar_sync(1, Gm::W * 32);
      if (warp == 0 && n + Gm::STAGES < ntiles && !*abort_flag) {
        issue_tile(n + Gm::STAGES, stage, lookup_page(n + Gm::STAGES));
        ++issued;
      }
    }
    if (++stage == Gm::STAGES) {
      stage = 0;
      parity ^= 1u;
    }
  }

  if (!Gm::PRODUCER && *abort_flag && threadIdx.x == 0) drain(issued);

  // ---- normalise and write rows of the block (a row that saw nothing: zeros)
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const float invA = lA > 0.f ? 1.f / lA : 0.f, invB = lB > 0.f ? 1.f / lB : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = r0 + g + 8 * half;
    if (r >= nrows) continue;
    const float inv = half ? invB : invA;
    __nv_bfloat16* dst = p.out + (((size_t)b * p.q_len + q0 + r / p.G) * p.Hq + h * p.G + r % p.G) * D;
#pragma unroll
    for (int c = 0; c < NB8; ++c)
      *reinterpret_cast<uint32_t*>(dst + 8 * c + 2 * c4) =
          pack_bf16x2(o[c][2 * half] * inv, o[c][2 * half + 1] * inv);
  }
}

}  // namespace da
