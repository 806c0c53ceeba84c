// Causal GQA prefill / chunked prefill on the 5th-generation tensor cores
// (tcgen05, tensor memory), head_dim 64, 128 and 256.
//
// What is computed is the prefill of prefill_kernel.cuh (the reading of
// "gqa_prefill_attn" on the AstrAI commit page, "csrc", commit 988e013): query
// token i of a chunk of q_len (position L - q_len + i) attends to cached
// positions 0 .. L - q_len + i.  Only the engine differs.
//
// A CTA owns NQT query tiles of 128 rows (NQT = 2 up to head_dim 128, 1 at 256).
// A tile is a block of 128 / G query tokens x the G query heads of one KV head
// (token-major, as prefill_kernel), and its rows live in the 128 lanes of tensor
// memory:
//   S = Q K^T   tcgen05.mma, Q and the K tile K-major in shared memory (128-byte
//               swizzle), fp32 into an S buffer of BK columns;
//   softmax     one thread per row (TMEM lane = row) loads its row of S, masks,
//               and writes P = exp2(s - m) as bf16 pairs over the first BK / 2
//               columns of the same S buffer;
//   O += P V    tcgen05.mma with P from tensor memory and the V tile MN-major in
//               shared memory, fp32 into D columns of tensor memory.
// The running maximum m is only raised (and O, l rescaled) when a row's maximum
// grows by more than 8 in log2 units; otherwise the stale m stays in both l and
// O and cancels in O / l.
//
// Overlap.  With two query tiles (A, B) each has one S buffer and its own
// softmax warpgroup, and the tensor cores alternate between them: while the
// softmax of A works on key tile j + 1, the tensor cores run P_B V_j and
// S_B = Q_B K_{j+1}^T, and the other way round.  Tensor memory: S_A, S_B (BK
// columns each), O_A, O_B (D each), 512 columns at D = 128.  With one query tile
// (head_dim 256: two O of 256 columns would not fit) S is double-buffered
// instead and S of tile j + 1 is computed while the softmax works on tile j.
// The MMAs of one thread run in issue order, so an S buffer can be overwritten
// by the next Q K^T as soon as the P V that reads its P has been issued.
//
// Warp roles: one lane of warp 0 issues the K tile copies (TMA) and one of warp 2
// the V tile copies, into one ring of slots in the order the MMAs use them (K_0,
// V_0, K_1, V_1, ...); warp 1 allocates tensor memory and one lane issues every
// MMA and commits it to an mbarrier; the last NQT * NH warpgroups run the softmax
// and the epilogue (NH = 1 thread per row with two query tiles, 2 with one: each
// takes half of the row's keys and of its O, and the two exchange the row's
// maximum through shared memory); all warps stage the query rows first.  With two
// query tiles the first warpgroup gives registers up (setmaxnreg) to the softmax
// warpgroups; the host launches that form only when the kernel's register budget
// covers the split.  Every wait is bounded: after the limit the kernel sets the
// device error word, lets the work it issued finish, frees its tensor memory and
// exits.
#pragma once

#include <cstdint>

#include "prefill_kernel.cuh"
#include "tc05.cuh"

namespace da {

template <int D>
struct PrefillTcGeo {
  static constexpr int NQT = D <= 128 ? 2 : 1;     // query tiles per CTA
  static constexpr int M = 128;                    // rows per query tile (tensor memory lanes)
  static constexpr int ROWS = NQT * M;             // query rows per CTA
  static constexpr int BK = D == 256 ? 64 : 128;   // keys per tile (N of Q K^T)
  static constexpr int NSUB = D / 64;              // 64-element swizzle columns
  // one ring of NSLOT slots holds K and V tiles in the order the MMAs use and
  // free them: item 2 j is K_j, item 2 j + 1 is V_j, item n in slot n % NSLOT.  A
  // slot frees when the last MMA that reads it completes; each load starts as soon
  // as its slot is free, whatever tensor the slot held before
  static constexpr int KV_BYTES = BK * D * 2;      // one tile of K or V: [NSUB][BK][64]
  static constexpr int QT_BYTES = M * D * 2;       // one query tile: [NSUB][M][64]
  static constexpr int NSLOT = D == 64 ? 8 : 5;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + NQT * QT_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * KV_BYTES;
  // barriers: full[NSLOT], empty[NSLOT], then s[2], p[2], o[2] (two query tiles:
  // one each per tile, o completing once after the last P V; one query tile: by
  // key-tile parity), fin (the last MMA)
  static constexpr int BAR_FULL = 0, BAR_EMPTY = NSLOT, BAR_S = 2 * NSLOT, BAR_P = BAR_S + 2, BAR_O = BAR_S + 4,
                       BAR_FIN = BAR_S + 6, NBAR = BAR_S + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] tensor memory base, [1] abort flag
  // softmax threads per row: two with one query tile (one per half of the keys;
  // they exchange the row's maximum and sum through one float per (query tile,
  // row) and read the loop decision of the step from one word per query tile),
  // one with two query tiles, where four softmax warpgroups would leave too few
  // registers for each
  static constexpr int NH = NQT == 1 ? 2 : 1;
  static constexpr int OFF_XCH = OFF_MISC + 16;
  static constexpr int OFF_DEC = OFF_XCH + NQT * M * 4;
  static constexpr int SMEM = OFF_DEC + 16 + 1024;    // + alignment slack
  // tensor memory columns: S buffer i at i * BK (two of them either way), O of
  // query tile t at 2 * BK + t * D
  static constexpr int TCOL_O = 2 * BK;
  static constexpr int TCOLS_USED = 2 * BK + NQT * D;
  static constexpr uint32_t TMEM_COLS = TCOLS_USED <= 256 ? 256u : 512u;
  static constexpr int NTHREADS = 128 * (1 + NQT * NH);
  // registers per thread after the split (two query tiles): the first warpgroup
  // (producers, MMA issue, an idle warp) drops to REG_LOW, the softmax
  // warpgroups rise to REG_HIGH; the launch must provide
  // 128 * REG_LOW + 256 * REG_HIGH registers
  static constexpr int REG_LOW = 56, REG_HIGH = 216;
  static constexpr int REG_POOL_NEEDED = 128 * REG_LOW + 128 * NQT * NH * REG_HIGH;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(TCOLS_USED <= 512, "tensor memory budget");
};

__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned long long timeout_ns) {
  return wait_bounded(bar, parity, abort_flag, timeout_ns);
}

template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(PrefillTcGeo<D>::NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Gm = PrefillTcGeo<D>;
  constexpr int BK = Gm::BK;
  constexpr int NQT = Gm::NQT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  auto bar = [&](int i) -> uint32_t { return sbase + Gm::OFF_BAR + 8 * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Gm::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Gm::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float kNegInf = -__int_as_float(0x7f800000);

  // work unit: as prefill_kernel (groups of grp (b, h) units, latest query blocks first)
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
  const int BQT = p.BQ / NQT;  // query tokens per query tile
  const int q0 = qb * p.BQ;
  const int nq = min(p.BQ, p.q_len - q0);
  const int base = L - p.q_len;  // position of query token 0
  const int kv_end = max(0, min(L, base + q0 + nq));  // keys some row sees
  const int ntiles = (kv_end + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Gm::NSLOT; ++i) {
      mbar_init(bar(Gm::BAR_FULL + i), 1);
      mbar_init(bar(Gm::BAR_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Gm::BAR_S + i), 1);
      mbar_init(bar(Gm::BAR_P + i), 128 * Gm::NH);  // every softmax thread of the query tile
      mbar_init(bar(Gm::BAR_O + i), 1);
    }
    mbar_init(bar(Gm::BAR_FIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(sbase + Gm::OFF_MISC, Gm::TMEM_COLS);
    tmem_relinquish();
  }
  // query rows: row r of tile t = (token t * BQT + r / G, head r % G) of the block,
  // zero past it; [NSUB][M][64] per tile with the 128-byte swizzle (the K-major
  // layout the MMA reads)
  for (int e = threadIdx.x; e < Gm::ROWS * (D / 8); e += Gm::NTHREADS) {
    const int rr = e / (D / 8), ch = e % (D / 8);
    const int t = rr / Gm::M, r = rr % Gm::M;
    const int tok = t * BQT + r / p.G;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < BQT * p.G && tok < nq) {
      const int i = q0 + tok, hq = h * p.G + r % p.G;
      v = __ldg(reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.q_len + i) * p.Hq + hq) * D) + ch);
    }
    *reinterpret_cast<uint4*>(smem + Gm::OFF_Q + t * Gm::QT_BYTES + (ch / 8) * (Gm::M * 128) + swz<128>(r, ch % 8)) =
        v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ---- first warpgroup: every warp gives registers up at the same instruction
    if constexpr (NQT == 2) setmaxnreg_dec<Gm::REG_LOW>();
    if (warp == 0 || warp == 2) {
      // ---- producers: warp 0 issues the K items (even n), warp 2 the V items (odd
      // n), each in order and once its slot is free.  One thread issues copies one
      // after another, so two issuing threads double the rate for the small page
      // boxes.  A producer waits for the free of item n - NSLOT by phase parity.
      // Its previous item, n - 2, needed item n - 2 - NSLOT freed, and the MMAs
      // free items at most one place out of order, so item n - 2 NSLOT is freed by
      // then: the parity it waits on is never a whole ring cycle stale.
      const int first = warp == 0 ? 0 : 1;
      int last = -1;  // last item this producer issued
      if (lane == 0) {
        // one tensor's tile j into dst, counted on the mbarrier full
        auto load = [&](const CUtensorMap* map, uint32_t dst, uint32_t full, int j) {
          const int t = j * BK;
          if (!PAGED) {
            mbar_arrive_expect_tx(full, (uint32_t)Gm::KV_BYTES);
            tma_load_5d(dst, map, full, 0, t, 0, h, b);  // box [64][BK][NSUB]
          } else {
            // boxes of R rows of one page and one swizzle column: [NSUB][BK][64]
            const int R = 16 << p.box_shift;
            const int nbox = (min(BK, kv_end - t) + R - 1) / R;
            mbar_arrive_expect_tx(full, (uint32_t)(nbox * R * 128 * Gm::NSUB));
            for (int bx = 0; bx < nbox; ++bx) {
              const int tok = t + bx * R;
              const int col = p.page_shift >= 0 ? tok >> p.page_shift : tok / p.page_size;
              int page = __ldg(p.page_table + (size_t)b * p.max_pages + col);
              if ((unsigned)page >= (unsigned)p.num_pages) {  // a bad entry: flag it, read page 0 instead
                atomicOr(&g_error_word, 4u);
                page = 0;
              }
              const int row0 = tok - col * p.page_size;
#pragma unroll
              for (int sub = 0; sub < Gm::NSUB; ++sub)
                tma_load_5d(dst + (uint32_t)(sub * BK * 128 + bx * R * 128), map, full, 0, row0, sub, h, page);
            }
          }
        };
        for (int n = first; n < 2 * ntiles; n += 2) {
          const int slot = n % Gm::NSLOT;
          if (n >= Gm::NSLOT &&
              !tc_wait(bar(Gm::BAR_EMPTY + slot), (uint32_t)(((n / Gm::NSLOT) & 1) ^ 1), abort_flag, p.timeout_ns))
            break;
          load(n & 1 ? &p.tm_v : &p.tm_k, sbase + Gm::OFF_KV + slot * Gm::KV_BYTES, bar(Gm::BAR_FULL + slot), n >> 1);
          last = n;
        }
        // after an abort, let this producer's copies still in flight (its items
        // among the last NSLOT) land before the CTA exits
        if (*abort_flag) {
          for (int k = last; k >= 0 && k > last - Gm::NSLOT; k -= 2) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(Gm::BAR_FULL + k % Gm::NSLOT), (uint32_t)((k / Gm::NSLOT) & 1)) &&
                   globaltimer_ns() - t0 < p.timeout_ns) {
            }
          }
        }
      }
    } else if (warp == 1) {
      // ---- MMA issue (lane 0); the warp zeroes V rows past the keys of the last tile
      const uint32_t id_s = tc_idesc_bf16(Gm::M, BK, false, false);
      const uint32_t id_o = tc_idesc_bf16(Gm::M, D, false, true);
      // the whole warp waits (the tail zeroing writes what the copy wrote)
      auto wait_all = [&](uint32_t b_, uint32_t par) {
        const bool w = tc_wait(b_, par, abort_flag, p.timeout_ns);
        return __all_sync(0xffffffffu, w);
      };
      // ring slot (shared-memory address) and mbarrier parity of K_j (item 2 j) and
      // V_j (item 2 j + 1)
      auto slot_addr = [&](int n) { return sbase + Gm::OFF_KV + (uint32_t)((n % Gm::NSLOT) * Gm::KV_BYTES); };
      auto full_bar = [&](int n) { return bar(Gm::BAR_FULL + n % Gm::NSLOT); };
      auto empty_bar = [&](int n) { return bar(Gm::BAR_EMPTY + n % Gm::NSLOT); };
      auto full_par = [&](int n) { return (uint32_t)((n / Gm::NSLOT) & 1); };
      // S buffer sb = Q_t K_j^T over D in steps of 16
      auto issue_qk = [&](int t, int j, int sb) {
        const uint32_t kst = slot_addr(2 * j);
        const uint32_t qt = sbase + Gm::OFF_Q + t * Gm::QT_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk / 4) * (Gm::M * 128) + (kk % 4) * 32;
          const uint32_t ko = (kk / 4) * (BK * 128) + (kk % 4) * 32;
          tc_mma_ss(tmem + sb * BK, tc_sdesc(qt + qo, 16, 1024, kTcSwizzle128B),
                    tc_sdesc(kst + ko, 16, 1024, kTcSwizzle128B), id_s, kk > 0);
        }
      };
      // O_t += P (S buffer sb) V_j over the tile's keys in steps of 16
      auto issue_pv = [&](int t, int j, int sb) {
        const uint32_t vst = slot_addr(2 * j + 1);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_ts(tmem + Gm::TCOL_O + t * D, tmem + sb * BK + 8 * kk,
                    tc_sdesc(vst + kk * 16 * 128, BK * 128, 1024, kTcSwizzle128B), id_o, j > 0 || kk > 0);
      };
      // V rows at or past kv_end may hold anything (0 * NaN would poison O): zero them
      auto zero_tail = [&](int j) {
        const int t = j * BK;
        if (t + BK <= kv_end) return;
        const int r0 = kv_end - t;
        uint8_t* vs = smem + Gm::OFF_KV + ((2 * j + 1) % Gm::NSLOT) * Gm::KV_BYTES;
        for (int e = r0 * 8 + lane; e < BK * 8; e += 32) {
          const int r = e / 8, ch = e % 8;
#pragma unroll
          for (int sub = 0; sub < Gm::NSUB; ++sub)
            *reinterpret_cast<uint4*>(vs + sub * (BK * 128) + swz<128>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      };
      bool ok = ntiles > 0 && wait_all(full_bar(0), full_par(0));
      const bool issued_any = ok;
      if (ok && lane == 0) {
        tc_fence_after();
        for (int t = 0; t < NQT; ++t) {
          issue_qk(t, 0, t);
          tc_commit(bar(Gm::BAR_S + t));
        }
        tc_commit(empty_bar(0));
      }
      __syncwarp();
      for (int j = 0; j < ntiles && ok; ++j) {
        const bool more = j + 1 < ntiles;
        if constexpr (NQT == 2) {
          // A: P_A V_j, then S_A of tile j + 1; B: the same, then V_j and K_{j+1} free
          // their slots
          ok = wait_all(full_bar(2 * j + 1), full_par(2 * j + 1));
          if (!ok) break;
          zero_tail(j);
          for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_all(bar(Gm::BAR_P + t), (uint32_t)(j & 1));
            if (ok && more && t == 0)
              ok = wait_all(full_bar(2 * j + 2), full_par(2 * j + 2));
            if (!ok) break;
            if (lane == 0) {
              tc_fence_after();
              issue_pv(t, j, t);
              if (t == 1) tc_commit(empty_bar(2 * j + 1));
              if (more) {
                issue_qk(t, j + 1, t);
                tc_commit(bar(Gm::BAR_S + t));
                if (t == 1) tc_commit(empty_bar(2 * j + 2));
              } else {
                tc_commit(bar(Gm::BAR_O + t));
              }
            }
            __syncwarp();
          }
        } else {
          // Q K^T of the next tile goes ahead of this tile's P V, so the softmax of
          // tile j + 1 can start as soon as that of tile j ends
          if (more) {
            ok = wait_all(full_bar(2 * j + 2), full_par(2 * j + 2));
            if (!ok) break;
            if (lane == 0) {
              tc_fence_after();
              issue_qk(0, j + 1, (j + 1) & 1);
              tc_commit(bar(Gm::BAR_S + ((j + 1) & 1)));
              tc_commit(empty_bar(2 * j + 2));
            }
            __syncwarp();
          }
          ok = wait_all(full_bar(2 * j + 1), full_par(2 * j + 1));
          if (!ok) break;
          zero_tail(j);
          ok = wait_all(bar(Gm::BAR_P + (j & 1)), (uint32_t)((j >> 1) & 1));
          if (!ok) break;
          if (lane == 0) {
            tc_fence_after();
            issue_pv(0, j, j & 1);
            tc_commit(bar(Gm::BAR_O + (j & 1)));
            tc_commit(empty_bar(2 * j + 1));
          }
          __syncwarp();
        }
      }
      // before the tensor memory is freed, every MMA issued must have completed
      if (lane == 0 && issued_any) {
        tc_commit(bar(Gm::BAR_FIN));
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar(Gm::BAR_FIN), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
        }
      }
      __syncwarp();
    }  // warp 3: idle
  } else {
    // ---- softmax and epilogue of query tile qt: NH threads per row, one per part
    // of the key columns (tensor memory lane = row; warps w and w + 4 reach the
    // same lanes); two halves exchange the row's maximum every key tile and the
    // row's sum at the end, and each handles its part of O
    if constexpr (NQT == 2) setmaxnreg_inc<Gm::REG_HIGH>();
    constexpr int NH = Gm::NH;
    constexpr int HK = BK / NH, HD = D / NH;
    const int sw = warp - 4;
    const int qt = sw / (4 * NH), hh = NH == 2 ? (sw >> 2) & 1 : 0;
    const int row = lane + 32 * (warp & 3);
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    volatile float* xch = reinterpret_cast<volatile float*>(smem + Gm::OFF_XCH) + qt * Gm::M + row;
    volatile int* dec = reinterpret_cast<volatile int*>(smem + Gm::OFF_DEC) + qt;
    const int tok = qt * BQT + row / p.G;  // this row's token within the block
    const bool has_row = row < BQT * p.G && tok < nq;
    const int lim = has_row ? max(0, min(L, base + q0 + tok + 1)) : 0;  // keys this row sees
    const int lim_first = max(0, min(L, base + q0 + qt * BQT + 1));      // keys every row of the tile sees
    const uint32_t o_addr = tmem + lane_addr + Gm::TCOL_O + qt * D + hh * HD;
    // the 256 threads of the query tile meet on named barrier 1 + qt; a step's
    // decision to stop (the CTA's abort flag, read once by one thread between the
    // two meetings) is the same for all of them, so none waits for a partner that
    // left
    auto meet = [&]() { named_bar_sync(1 + qt, 128 * NH); };
    float m = kNegInf, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = NQT == 2 ? qt : (j & 1);  // S buffer
      const uint32_t spar = NQT == 2 ? (uint32_t)(j & 1) : (uint32_t)((j >> 1) & 1);
      bool ok_s = tc_wait(bar(Gm::BAR_S + sb), spar, abort_flag, p.timeout_ns);
      ok_s = __all_sync(0xffffffffu, ok_s);
      const uint32_t sAddr = tmem + lane_addr + sb * BK;
      const int t = j * BK + hh * HK;  // first key of this half
      // x = s * scale_log2, or (fold: scale_log2 > 0) x = s, with the scale applied
      // in the exponent's fma and to the maximum; -inf at or past this row's limit
      // (only tiles that reach past the first row's).  Max and sum run in eight
      // independent chains.
      const bool fold = p.scale_log2 > 0.f;  // uniform over the grid
      const float sc = fold ? p.scale_log2 : 1.f;
      float x[HK];
      if (ok_s) {
        tc_fence_after();
        uint32_t r[HK];
#pragma unroll
        for (int c0 = 0; c0 < HK; c0 += 32) tmem_ld32(sAddr + hh * HK + c0, *reinterpret_cast<uint32_t(*)[32]>(r + c0));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < HK; ++i) x[i] = fold ? __uint_as_float(r[i]) : __uint_as_float(r[i]) * p.scale_log2;
        if (j * BK + BK > lim_first) {
#pragma unroll
          for (int i = 0; i < HK; ++i) x[i] = t + i < lim ? x[i] : kNegInf;
        }
      }
      auto tile_max = [&]() {  // this thread's maximum of x, scaled
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(x[k], x[k + 8]);
#pragma unroll
        for (int i = 16; i < HK; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], fmaxf(x[i + k], x[i + 8 + k]));
        const float mxh =
            fmaxf(fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3])), fmaxf(fmaxf(mk[4], mk[5]), fmaxf(mk[6], mk[7])));
        return fold ? mxh * p.scale_log2 : mxh;
      };
      // P = exp2(x sc - mu) as bf16 pairs, stored over this part's columns of the S
      // buffer, [hh HK / 2, (hh + 1) HK / 2); returns the sum of the weights
      auto weights = [&](float mu_) {
        float sk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sk[k] = 0.f;
        constexpr int CH = HK / 2 >= 32 ? 32 : HK / 2;  // columns per store
#pragma unroll
        for (int c0 = 0; c0 < HK / 2; c0 += CH) {
          uint32_t pk[CH];
#pragma unroll
          for (int i = 0; i < CH; ++i) {
            const float e0 = exp2_approx(fmaf(x[2 * (c0 + i)], sc, -mu_));
            const float e1 = exp2_approx(fmaf(x[2 * (c0 + i) + 1], sc, -mu_));
            sk[i & 7] += e0 + e1;
            pk[i] = pack_bf16x2(e0, e1);
          }
          if constexpr (CH == 32) {
            tmem_st32(sAddr + hh * (HK / 2) + c0, pk);
          } else {
            static_assert(CH == 16, "a part of P is 16 or a multiple of 32 columns");
            tmem_st16(sAddr + hh * (HK / 2) + c0, pk);
          }
        }
        return ((sk[0] + sk[1]) + (sk[2] + sk[3])) + ((sk[4] + sk[5]) + (sk[6] + sk[7]));
      };
      // The running maximum m is raised (and O, l rescaled) only when needed.  Two
      // threads per row: when the row's maximum, exchanged every step, exceeds m
      // by more than 8.  One thread per row: the weights are first taken against
      // the current m, and only a row that has seen no key yet or whose weights
      // sum past 2^14 takes its maximum and raises m to it; every weight then
      // stays below 2^14.
      float mx = kNegInf, sum = 0.f;
      bool need_max = true, have_weights = false;
      if constexpr (NH == 2) {
        const float mxh = ok_s ? tile_max() : kNegInf;
        // the row's maximum: half 0 posts its own, half 1 combines and posts the
        // row's, half 0 reads it
        mx = mxh;
        if (hh == 0) *xch = mxh;
        meet();
        if (hh == 1) {
          mx = fmaxf(mx, *xch);
          *xch = mx;
          if (row == 0) *dec = *abort_flag;
        }
        meet();
        if (hh == 0) mx = *xch;
        if (*dec) {
          ok = false;
          break;
        }
      } else {
        if (!ok_s) {
          ok = false;
          break;
        }
        // weights() ends in a tensor-memory store that the whole warp executes:
        // every call is warp-uniform, each lane with its own m (a warp none of
        // whose rows has seen a key skips this pass: they all take the maximum)
        have_weights = __any_sync(0xffffffffu, m != kNegInf);
        if (have_weights) sum = weights(m == kNegInf ? 0.f : m);
        need_max = m == kNegInf || !(sum <= 16384.f);
        if (need_max) mx = tile_max();
      }
      const bool raise = need_max && (NH == 2 ? mx > m + 8.f : mx > m);
      const float m_new = raise ? mx : m;
      const float alpha = raise ? exp2_approx(m - m_new) : 1.f;  // 0 while m is still -inf
      if (__any_sync(0xffffffffu, raise && m != kNegInf) && j > 0) {
        // O holds the P V of tiles < j.  Two query tiles: S of tile j was issued
        // after P V of tile j - 1, and its commit covers every MMA before it, so
        // O is complete.  One query tile: wait for tile j - 1's P V (tile j - 3's,
        // the previous completion of that barrier, is done: S of tile j was
        // committed after it).  A wait that gives up leaves O as it is; the
        // next step's decision stops the loop.
        bool ok_o = true;
        if constexpr (NQT == 1) {
          ok_o = tc_wait(bar(Gm::BAR_O + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort_flag, p.timeout_ns);
          ok_o = __all_sync(0xffffffffu, ok_o);
          tc_fence_after();
        }
        if (ok_o) {
#pragma unroll 1
          for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(o_addr + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(o_addr + c0, o);
          }
          tmem_st_wait();
        }
      }
      m = m_new;
      // weights against the new m (replacing those taken against the old one; a
      // lane that did not raise writes the same values again); a row that has seen
      // no key yet takes 0, so its weights are exactly 0
      if (!have_weights || __any_sync(0xffffffffu, raise)) sum = weights(m == kNegInf ? 0.f : m);
      l = l * alpha + sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Gm::BAR_P + sb));
    }
    // ---- normalise and write the tile's rows (a row that saw nothing: zeros):
    // the row's sum from both halves, then each half writes its half of O
    if constexpr (NH == 2) {
      if (hh == 1) *xch = l;
      meet();
      if (hh == 0) {
        l += *xch;
        *xch = l;
      }
      meet();
      if (hh == 1) l = *xch;
    }
    if (ok && ntiles > 0) {
      // the last P V of this tile (it completes after every earlier one)
      const int ob = NQT == 2 ? qt : ((ntiles - 1) & 1);
      const uint32_t opar = NQT == 2 ? 0u : (uint32_t)(((ntiles - 1) >> 1) & 1);
      ok = tc_wait(bar(Gm::BAR_O + ob), opar, abort_flag, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = p.out + (((size_t)b * p.q_len + q0 + tok) * p.Hq + h * p.G + row % p.G) * D + hh * HD;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t r[32];
        if (ntiles > 0) {
          tmem_ld32(o_addr + c0, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (has_row) {
          uint4* o = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            o[k] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                              pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                              pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                              pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

}  // namespace da
