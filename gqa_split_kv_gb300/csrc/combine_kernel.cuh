// Log-sum-exp combine of split partials into the bf16 output.
//
// For one (b, h): M = max_j m_j over live slots (l_j > 0), w_j = exp(m_j - M),
// out = sum_j w_j acc_j / sum_j w_j l_j (the merge of "perf(qwen3.8): split the
// flash-decode KV range across warp-groups", section "Mechanism"; the
// partial/merge split of AstrAI commit 988e013 "csrc", split-KV items).
//
// Work items are (row, 128-column chunk) pairs, grid-strided over CTAs; a CTA's
// items are classified one per thread, and each item that needs merging is then
// handled by the whole CTA, one at a time.  Warp 0 loads the row's (m, l) once
// and turns them into M and the weights in shared memory while every thread's
// first acc loads are in flight; the slot x
// column products are spread over the 512 threads (JL slot lanes x D/4 column
// groups of 4), each thread keeping KB loads in flight; the JL lane sums
// are added in ascending lane order.  The summation order is fixed, so results
// are bitwise reproducible.
//
// Two modes:
//   planned:  after the split kernel (programmatic dependent launch), for the
//             segments with more than kFusedMergeMax pieces: the split kernel
//             merges smaller segments itself, and a longer run of partials is
//             spread over many CTAs here.
//             A row's slot count is its segment's piece count under the split plan.
//   plain:    decode_combine: every S slot of every row, skipping slots with l == 0.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "plan.cuh"
#include "ptx.cuh"

namespace da {

struct CombineParams {
  const float* part_acc;
  const float* part_ml;
  __nv_bfloat16* out;
  const int* seq_lens;  // planned mode
  int B, Hq, S;
  int planned;
  int G, U, ng, gr, ngp, npass, max_len;  // rows per KV head, segments per sequence, grouping
};

template <int D>
struct CombineGeo {
  static constexpr int NTHREADS = 512;
  static constexpr int CW = D < 128 ? D : 128;    // columns per work item (a row has D / CW items)
  static constexpr int NCH = D / CW;
  static constexpr int TPS = CW / 4;              // threads per slot (4 columns each)
  static constexpr int JL = NTHREADS / TPS;       // slot lanes
  static constexpr int KB = 4;                    // slot loads in flight per thread
  // shared: plan arrays (2B+2 ints) | weights (S floats) | lane sums (NTHREADS float4) | misc (32 floats)
  //         | row list (1 + 2 CLS ints)
  static constexpr int CLS = 128;                 // rows classified per round
  static int smem_bytes(int B, int S, bool planned) {
    return ((planned ? (2 * B + 2) * 4 : 0) + 15) / 16 * 16 + ((S * 4 + 15) / 16) * 16 + NTHREADS * 16 + 128 +
           (1 + 2 * CLS) * 4;
  }
};

template <int D>
__global__ void __maxnreg__(40) combine_kernel(const CombineParams p) {  // 512 threads; fits beside a split CTA
  using Cg = CombineGeo<D>;
  extern __shared__ __align__(16) uint8_t csm[];
  int* lens = reinterpret_cast<int*>(csm);
  int* P = lens + p.B;
  const int plan_bytes = p.planned ? (2 * p.B + 2) * 4 : 0;
  float* wts = reinterpret_cast<float*>(csm + ((plan_bytes + 15) / 16) * 16);
  float4* lane_sum = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(wts) + ((p.S * 4 + 15) / 16) * 16);
  float* red = reinterpret_cast<float*>(lane_sum + Cg::NTHREADS);  // [17] den

  Plan pl{};
  if (p.planned) {
    // seq_lens is not written by the split kernel: read it before waiting on it.
    build_plan_arrays(p.seq_lens, p.B, p.max_len, plan_gap_blocks(D), lens, P, 0, blockDim.x);
    pl = make_plan(p.B, p.U, p.S, plan_gap_blocks(D), P);
  }
  // A segment of n blocks meets at most (n - 1) / q + 2 ranges; when even the
  // longest sequence stays within kFusedMergeMax pieces, the split kernel merged
  // everything (batch workloads) and the CTA only waits for it.
  if (p.planned && threadIdx.x == 0) {
    const int nb_max = P[p.B + 1];
    red[31] = (nb_max == 0 || (nb_max - 1) / pl.q + 2 <= kFusedMergeMax) ? 1.f : 0.f;
  }
  const int tid = threadIdx.x, lane = tid & 31;
  const int jl = tid / Cg::TPS, c4 = tid % Cg::TPS;
  const float kNegInf = -__int_as_float(0x7f800000);
  const int items = p.B * p.Hq * Cg::NCH;        // (row, column chunk) pairs
  int* todo = reinterpret_cast<int*>(red + 32);  // [0] count, then (item, n) pairs
  // CLS threads classify one of this CTA's items each (the items base, base +
  // gridDim.x, ...); the items to merge go to the list.  The plan depends only on
  // seq_lens, so the first round is classified before the wait on the split kernel.
  auto classify = [&](int base) {
    if (tid == 0) todo[0] = 0;
    __syncthreads();
    if (tid < Cg::CLS) {
      const int item = base + tid * gridDim.x;
      const int row = item / Cg::NCH;
      if (item < items) {
        int n = p.S;
        if (p.planned) {
          const int b = row / p.Hq, h = row % p.Hq;
          const int u = (h / p.G) * p.npass + (h % p.G) / p.gr / p.ngp;
          n = segment_pieces(pl, lens, P, p.B, b, u);
        }
        if (!p.planned || n > kFusedMergeMax) {  // smaller segments were merged by the split kernel
          const int k = atomicAdd(&todo[0], 1);
          todo[1 + 2 * k] = item;
          todo[2 + 2 * k] = n;
        }
      }
    }
    __syncthreads();
  };
  __syncthreads();
  const bool nothing = p.planned && red[31] != 0.f;
  if (!nothing) classify(blockIdx.x);
  pdl_wait_primary();
  if (nothing) return;

  for (int base = blockIdx.x; base < items; base += Cg::CLS * gridDim.x) {
    if (base != blockIdx.x) classify(base);
    const int count = todo[0];
    for (int it = 0; it < count; ++it) {
      const int item = todo[1 + 2 * it];
      const int row = item / Cg::NCH;
      const int col0 = (item % Cg::NCH) * Cg::CW;  // first column of this item
      const int n = todo[2 + 2 * it];
      const float2* ml = reinterpret_cast<const float2*>(p.part_ml + (size_t)row * p.S * 2);
      const float4* acc = reinterpret_cast<const float4*>(p.part_acc + (size_t)row * p.S * D + col0) + c4;
      // this thread's first KB slot loads go out first
      float4 a[Cg::KB];
#pragma unroll
      for (int u = 0; u < Cg::KB; ++u) {
        const int j = jl + u * Cg::JL;
        a[u] = j < n ? acc[(size_t)j * (D / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // warp 0 turns the row's (m, l) into weights in shared memory, one L2 round
      // trip (the first 64 slots stay in registers) while the acc loads are in flight
      if (tid < 32) {
        float2 v[2];
        float M = kNegInf;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = lane + 32 * k;
          v[k] = j < n ? ml[j] : make_float2(kNegInf, 0.f);
          if (v[k].y > 0.f) M = fmaxf(M, v[k].x);
        }
        for (int j = lane + 64; j < n; j += 32) {
          const float2 x = ml[j];
          if (x.y > 0.f) M = fmaxf(M, x.x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float den = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = lane + 32 * k;
          if (j < n) {
            const float w = v[k].y > 0.f ? expf(v[k].x - M) : 0.f;
            wts[j] = w;
            den += w * v[k].y;
          }
        }
        for (int j = lane + 64; j < n; j += 32) {
          const float2 x = ml[j];
          const float w = x.y > 0.f ? expf(x.x - M) : 0.f;
          wts[j] = w;
          den += w * x.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane == 0) red[17] = den;
      }
      __syncthreads();
      // weighted column sums over this thread's slots (jl, jl + JL, ...)
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = jl; j0 < n; j0 += Cg::KB * Cg::JL) {
        if (j0 != jl) {
#pragma unroll
          for (int u = 0; u < Cg::KB; ++u) {
            const int j = j0 + u * Cg::JL;
            a[u] = j < n ? acc[(size_t)j * (D / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < Cg::KB; ++u) {
          const int j = j0 + u * Cg::JL;
          const float w = j < n ? wts[j] : 0.f;
          s.x += w * a[u].x;
          s.y += w * a[u].y;
          s.z += w * a[u].z;
          s.w += w * a[u].w;
        }
      }
      lane_sum[tid] = s;
      __syncthreads();
      if (jl == 0) {
        float4 t = lane_sum[c4];
        for (int k = 1; k < Cg::JL; ++k) {
          const float4 u4 = lane_sum[k * Cg::TPS + c4];
          t.x += u4.x;
          t.y += u4.y;
          t.z += u4.z;
          t.w += u4.w;
        }
        const float den = red[17];
        const float inv = den > 0.f ? 1.f / den : 0.f;
        uint2 o;
        o.x = pack_bf16x2(t.x * inv, t.y * inv);
        o.y = pack_bf16x2(t.z * inv, t.w * inv);
        *reinterpret_cast<uint2*>(p.out + (size_t)row * D + col0 + 4 * c4) = o;
      }
      __syncthreads();
    }
    __syncthreads();
  }
}

}  // namespace da
