// Causal GQA prefill / chunked prefill on the 5th-generation tensor cores
// (tcgen05, tensor memory), head_dim 64, 128 and 256.
//
// What is computed is the prefill of prefill_kernel.cuh (the reading of
// "gqa_prefill_attn" on the AstrAI commit page, "csrc", commit 988e013): query
// token i of a chunk of q_len (position L - q_len + i) attends to cached
// positions 0 .. L - q_len + i.  Only the engine differs.
//
// One CTA owns 128 query rows: a block of BQ = 128 / G query tokens x the G query
// heads of one KV head (token-major, as prefill_kernel).  The rows live in the
// 128 lanes of tensor memory:
//   S = Q K^T   tcgen05.mma, Q and the K tile K-major in shared memory (128-byte
//               swizzle), fp32 into one of two S buffers of BK columns;
//   softmax     one thread per row (warps 4-7, TMEM lane = row) loads its row of S,
//               masks, and writes P = exp2(s - m) as bf16 pairs over the first
//               BK / 2 columns of the same S buffer;
//   O += P V    tcgen05.mma with P from tensor memory and the V tile MN-major in
//               shared memory, fp32 into D columns of tensor memory.
// The running maximum m is only raised (and O, l rescaled) when a row's maximum
// grows by more than 8 in log2 units; otherwise the stale m stays in both l and
// O and cancels in O / l.  While the softmax works on tile j the tensor cores
// compute S for tile j + 1 into the other buffer.
//
// Warp roles: warp 0 one lane issues the K and V tile copies (TMA) into two rings
// (K of tile j + 1 can land while tile j's P V still holds its V); warp 1 allocates tensor memory and one lane issues every MMA and
// commits it to an mbarrier; warps 4-7 run the softmax and the epilogue; all
// warps stage the query rows first.  Every wait is bounded: after the limit the
// kernel sets the device error word, lets the work it issued finish, frees its
// tensor memory and exits.
#pragma once

#include <cstdint>

#include "prefill_kernel.cuh"
#include "tc05.cuh"

namespace da {

template <int D>
struct PrefillTcGeo {
  static constexpr int M = 128;                      // query rows per CTA (tensor memory lanes)
  static constexpr int BK = D == 256 ? 64 : 128;     // keys per tile (N of Q K^T)
  static constexpr int NSUB = D / 64;                // 64-element swizzle columns
  // K and V have rings of their own: a K stage frees once its Q K^T is done, a V
  // stage once its P V is
  static constexpr int KST = D == 64 ? 4 : 3;
  static constexpr int VST = D == 64 ? 4 : D == 128 ? 3 : 2;
  static constexpr int KV_BYTES = BK * D * 2;        // one tensor, one stage: [NSUB][BK][64]
  static constexpr int Q_BYTES = M * D * 2;          // [NSUB][M][64]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + VST * KV_BYTES;
  // barriers: k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], s_full[2],
  // p_full[2], o_done[2] (P V of even / odd tiles, so every wait knows its phase),
  // fin (the last MMA)
  static constexpr int BAR_K_FULL = 0, BAR_K_EMPTY = KST, BAR_V_FULL = 2 * KST, BAR_V_EMPTY = 2 * KST + VST,
                       BAR_S = 2 * KST + 2 * VST, BAR_P = BAR_S + 2, BAR_O = BAR_S + 4, BAR_FIN = BAR_S + 6,
                       NBAR = BAR_S + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] tensor memory base, [1] abort flag
  static constexpr int SMEM = OFF_MISC + 16 + 1024;    // + alignment slack
  static constexpr int TCOL_S0 = 0, TCOL_S1 = BK, TCOL_O = 2 * BK;
  static constexpr uint32_t TMEM_COLS = 2 * BK + D <= 256 ? 256u : 512u;
  static constexpr int NTHREADS = 256;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(2 * BK + D <= 512, "tensor memory budget");
};

__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned long long timeout_ns) {
  return wait_bounded(bar, parity, abort_flag, timeout_ns);
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(256, 1) prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Gm = PrefillTcGeo<D>;
  constexpr int BK = Gm::BK;
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
  const int q0 = qb * p.BQ;
  const int nq = min(p.BQ, p.q_len - q0);
  const int base = L - p.q_len;  // position of query token 0
  const int kv_end = max(0, min(L, base + q0 + nq));   // keys some row sees
  const int lim_first = max(0, min(L, base + q0 + 1)); // keys every row sees
  const int ntiles = (kv_end + BK - 1) / BK;
  const int nrows = nq * p.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Gm::KST; ++i) {
      mbar_init(bar(Gm::BAR_K_FULL + i), 1);
      mbar_init(bar(Gm::BAR_K_EMPTY + i), 1);
    }
    for (int i = 0; i < Gm::VST; ++i) {
      mbar_init(bar(Gm::BAR_V_FULL + i), 1);
      mbar_init(bar(Gm::BAR_V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Gm::BAR_S + i), 1);
      mbar_init(bar(Gm::BAR_P + i), 128);
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
  // query rows: row r = (token r / G, head r % G) of the block, zero past it;
  // [NSUB][M][64] with the 128-byte swizzle (the K-major layout the MMA reads)
  for (int e = threadIdx.x; e < Gm::M * (D / 8); e += Gm::NTHREADS) {
    const int r = e / (D / 8), ch = e % (D / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < nrows) {
      const int i = q0 + r / p.G, hq = h * p.G + r % p.G;
      v = __ldg(reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.q_len + i) * p.Hq + hq) * D) + ch);
    }
    *reinterpret_cast<uint4*>(smem + Gm::OFF_Q + (ch / 8) * (Gm::M * 128) + swz<128>(r, ch % 8)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- producer: K of tile j, then V of tile j - 1 (the order the tensor cores
    // free their stages in), each once its stage is free
    int k_issued = 0, v_issued = 0;
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
      for (int j = 0; j <= ntiles; ++j) {
        if (j < ntiles) {
          const int st = j % Gm::KST;
          if (j >= Gm::KST &&
              !tc_wait(bar(Gm::BAR_K_EMPTY + st), (uint32_t)(((j / Gm::KST) & 1) ^ 1), abort_flag, p.timeout_ns))
            break;
          load(&p.tm_k, sbase + Gm::OFF_K + st * Gm::KV_BYTES, bar(Gm::BAR_K_FULL + st), j);
          ++k_issued;
        }
        if (j >= 1) {
          const int jv = j - 1, st = jv % Gm::VST;
          if (jv >= Gm::VST &&
              !tc_wait(bar(Gm::BAR_V_EMPTY + st), (uint32_t)(((jv / Gm::VST) & 1) ^ 1), abort_flag, p.timeout_ns))
            break;
          load(&p.tm_v, sbase + Gm::OFF_V + st * Gm::KV_BYTES, bar(Gm::BAR_V_FULL + st), jv);
          ++v_issued;
        }
      }
      // after an abort, let the copies already issued land before the CTA exits
      if (*abort_flag) {
        auto drain = [&](int base_bar, int nst, int issued) {
          for (int k = issued > nst ? issued - nst : 0; k < issued; ++k) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(base_bar + k % nst), (uint32_t)((k / nst) & 1)) &&
                   globaltimer_ns() - t0 < p.timeout_ns) {
            }
          }
        };
        drain(Gm::BAR_K_FULL, Gm::KST, k_issued);
        drain(Gm::BAR_V_FULL, Gm::VST, v_issued);
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
    // S[j & 1] = Q K_j^T over D in steps of 16; the K stage frees when it is done
    auto issue_qk = [&](int j) {
      const int st = j % Gm::KST;
      const uint32_t kst = sbase + Gm::OFF_K + st * Gm::KV_BYTES;
      const uint32_t dS = tmem + (j & 1 ? Gm::TCOL_S1 : Gm::TCOL_S0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk / 4) * (Gm::M * 128) + (kk % 4) * 32;
        const uint32_t ko = (kk / 4) * (BK * 128) + (kk % 4) * 32;
        tc_mma_ss(dS, tc_sdesc(sbase + Gm::OFF_Q + qo, 16, 1024, kTcSwizzle128B),
                  tc_sdesc(kst + ko, 16, 1024, kTcSwizzle128B), id_s, kk > 0);
      }
      tc_commit(bar(Gm::BAR_S + (j & 1)));
      tc_commit(bar(Gm::BAR_K_EMPTY + st));
    };
    int done_o = -1;  // last tile whose P V was issued
    bool ok = ntiles > 0 && wait_all(bar(Gm::BAR_K_FULL), 0);
    if (ok && lane == 0) {
      tc_fence_after();
      issue_qk(0);
    }
    for (int j = 0; j < ntiles && ok; ++j) {
      // Q K^T of the next tile goes ahead of this tile's P V, so the softmax of
      // tile j + 1 can start as soon as that of tile j ends
      if (j + 1 < ntiles) {
        const int st1 = (j + 1) % Gm::KST;
        ok = wait_all(bar(Gm::BAR_K_FULL + st1), (uint32_t)(((j + 1) / Gm::KST) & 1));
        if (!ok) break;
        if (lane == 0) {
          tc_fence_after();
          issue_qk(j + 1);
        }
      }
      const int st = j % Gm::VST;
      ok = wait_all(bar(Gm::BAR_V_FULL + st), (uint32_t)((j / Gm::VST) & 1));
      if (!ok) break;
      const int t = j * BK;
      const uint32_t vst = sbase + Gm::OFF_V + st * Gm::KV_BYTES;
      if (t + BK > kv_end) {
        // V rows at or past kv_end may hold anything (0 * NaN would poison O): zero them
        const int r0 = kv_end - t;
        for (int e = r0 * 8 + lane; e < BK * 8; e += 32) {
          const int r = e / 8, ch = e % 8;
#pragma unroll
          for (int sub = 0; sub < Gm::NSUB; ++sub)
            *reinterpret_cast<uint4*>(smem + Gm::OFF_V + st * Gm::KV_BYTES + sub * (BK * 128) + swz<128>(r, ch)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      ok = wait_all(bar(Gm::BAR_P + (j & 1)), (uint32_t)((j >> 1) & 1));
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t aP = tmem + (j & 1 ? Gm::TCOL_S1 : Gm::TCOL_S0);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_ts(tmem + Gm::TCOL_O, aP + 8 * kk, tc_sdesc(vst + kk * 16 * 128, BK * 128, 1024, kTcSwizzle128B),
                    id_o, j > 0 || kk > 0);
        tc_commit(bar(Gm::BAR_O + (j & 1)));
        tc_commit(bar(Gm::BAR_V_EMPTY + st));
      }
      done_o = j;
      __syncwarp();
    }
    // before the tensor memory is freed, every MMA issued must have completed
    if (lane == 0 && (done_o >= 0 || ntiles > 0)) {
      tc_commit(bar(Gm::BAR_FIN));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(Gm::BAR_FIN), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- softmax and epilogue: thread = row = tensor memory lane
    const int row = threadIdx.x - 128;
    const uint32_t lane_addr = (uint32_t)((warp - 4) * 32) << 16;
    const int lim = row < nrows ? max(0, min(L, base + q0 + row / p.G + 1)) : 0;  // keys this row sees
    float m = kNegInf, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      ok = tc_wait(bar(Gm::BAR_S + (j & 1)), (uint32_t)((j >> 1) & 1), abort_flag, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sAddr = tmem + lane_addr + (j & 1 ? Gm::TCOL_S1 : Gm::TCOL_S0);
      const int t = j * BK;
      float x[BK];
#pragma unroll
      for (int c0 = 0; c0 < BK; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(sAddr + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c0 + i] = __uint_as_float(r[i]) * p.scale_log2;
      }
      // -inf at or past this row's limit (only tiles that reach past the first row's)
      if (t + BK > lim_first) {
#pragma unroll
        for (int i = 0; i < BK; ++i) x[i] = t + i < lim ? x[i] : kNegInf;
      }
      float mx = kNegInf;
#pragma unroll
      for (int i = 0; i < BK; ++i) mx = fmaxf(mx, x[i]);
      // raise m (and rescale O and l) only when the row's maximum grew by more than 8
      const bool raise = mx > m + 8.f;
      const float m_new = raise ? mx : m;
      const float alpha = raise ? exp2_approx(m - m_new) : 1.f;  // 0 while m is still -inf
      if (__any_sync(0xffffffffu, raise && m != kNegInf) && j > 0) {
        // O holds the P V of tiles < j: wait for tile j - 1's (tile j - 3's, the previous
        // completion of that barrier, is done: S of tile j was committed after it),
        // then scale this warp's rows
        ok = tc_wait(bar(Gm::BAR_O + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort_flag, p.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_addr + Gm::TCOL_O + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tmem + lane_addr + Gm::TCOL_O + c0, r);
        }
        tmem_st_wait();
      }
      m = m_new;
      const float mu = m == kNegInf ? 0.f : m;  // a row that has seen no key: weights exactly 0
      float sum = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < BK; c0 += 64) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a = exp2_approx(x[c0 + 2 * i] - mu), c = exp2_approx(x[c0 + 2 * i + 1] - mu);
          sum += a + c;
          r[i] = pack_bf16x2(a, c);
        }
        tmem_st32(sAddr + c0 / 2, r);
      }
      l = l * alpha + sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Gm::BAR_P + (j & 1)));
    }
    // ---- normalise and write the block's rows (a row that saw nothing: zeros)
    if (ok && ntiles > 0) {
      // the last tile's P V (it completes after every earlier one)
      ok = tc_wait(bar(Gm::BAR_O + ((ntiles - 1) & 1)), (uint32_t)(((ntiles - 1) >> 1) & 1), abort_flag,
                   p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = p.out + (((size_t)b * p.q_len + q0 + row / p.G) * p.Hq + h * p.G + row % p.G) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        if (ntiles > 0) {
          tmem_ld32(tmem + lane_addr + Gm::TCOL_O + c0, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (row < nrows) {
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
